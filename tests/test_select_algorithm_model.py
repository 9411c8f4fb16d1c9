"""The selection's pruning, modelled in numpy and checked against the oracle's
full sort (no GPU).

Two-stage candidate selection (article "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化",
section 3.3) as the CUDA path realises it: logits grouped into tiles of 8192
(or, when there are fewer than 2W tiles, into each tile's 128 interleaved
sub-chunks of 64), each group's best score key, a threshold L -- the lower
edge of the bin of 2^16 keys holding the 2W-th largest group key, counted down
from the largest key over 4096 bins, else that key itself -- and the
candidates: the logits scoring >= L in groups whose best key is >= L.  The
model repeats those steps in numpy with the kernels' fp32 score arithmetic;
the test requires every one of the oracle's 2W best (parent, token) pairs to
be a candidate, on random logits, heavy ties, a dominant token per row (the
threshold then lies beyond the 4096 bins), and vocabularies with a ragged last
tile.  A flaw in the pruning argument, the group layout or the threshold's
bin arithmetic would drop a winner here.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_packed_varlen_gb300 import workloads as wl

TILE = 8192
SUB = 128      # sub-chunks per tile
BINS = 4096    # threshold histogram bins of 2^16 keys


def f32_key(f: np.ndarray) -> np.ndarray:
    """Order-preserving uint32 key of fp32 values (-0 as +0)."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32).copy()
    u[u == 0x80000000] = 0
    neg = (u & 0x80000000) != 0
    return np.where(neg, ~u, u | np.uint32(0x80000000)).astype(np.uint32)


def sub_chunk_of(pos: np.ndarray) -> np.ndarray:
    """Sub-chunk (0..127) of tile position pos: the consumer lane l that
    reads it in chunks 2q and 2q + 1 gives sub-chunk q * 32 + l."""
    ch = pos // 1024
    lane = (pos % 256) // 8
    return (ch // 2) * 32 + lane


def model_candidates(logits: torch.Tensor, cum: np.ndarray, lse: np.ndarray, K: int):
    x = logits.float().numpy().astype(np.float32)
    W_in, V = x.shape
    nt = -(-V // TILE)
    score = (cum.astype(np.float32)[:, None] + (x - lse.astype(np.float32)[:, None]).astype(np.float32))
    keys = f32_key(score.astype(np.float32))
    n_tiles = W_in * nt
    tile_level = n_tiles >= K
    pos = np.arange(V)
    tile = (np.arange(W_in)[:, None] * nt + pos[None, :] // TILE)
    group = tile if tile_level else tile * SUB + sub_chunk_of(pos % TILE)[None, :]
    n_groups = n_tiles if tile_level else n_tiles * SUB
    gkey = np.zeros(n_groups, dtype=np.uint32)        # absent positions (ragged tail) are -inf: never the max
    np.maximum.at(gkey, group.ravel(), keys.ravel())
    exact = False
    if n_groups <= K:
        L = 0
    else:
        top = int(gkey.max()) >> 16
        d = top - (gkey.astype(np.int64) >> 16)
        hist = np.bincount(d[d < BINS], minlength=BINS)
        cumc = np.cumsum(hist)
        hit = np.nonzero(cumc >= K)[0]
        if hit.size:
            L = (top - int(hit[0])) << 16
        else:  # further down than the histogram: the K-th largest key itself
            L = int(np.sort(gkey)[::-1][K - 1])
            exact = True
    sel = (gkey[group] >= L) & (keys >= L)
    b, t = np.nonzero(sel)
    return set(zip(b.tolist(), t.tolist())), L, n_groups, tile_level, exact


def check(logits: torch.Tensor, cum: torch.Tensor, W: int):
    K = 2 * W
    cum_np = cum.numpy().astype(np.float32)
    lse = oracle.beam_select(logits, cum_np, K)[3]          # the oracle's fp32 normalisers
    tok, par, _, _ = oracle.beam_select(logits, cum_np, K, lse_in=lse)
    cand, L, n_groups, tile_level, exact = model_candidates(logits, cum_np, lse, K)
    missing = [(int(p), int(t)) for p, t in zip(par, tok) if (int(p), int(t)) not in cand]
    assert not missing, f"{len(missing)} of the 2W best are not candidates (L={L:#x}, groups {n_groups})"
    assert len(cand) >= K
    return len(cand), tile_level, n_groups, exact


@pytest.mark.parametrize("W_in,V,W,seed", [
    (1, 40000, 16, 1), (1, 40000, 64, 2), (3, 20000, 8, 3), (8, 40000, 16, 4),
    (8, 40000, 100, 5), (4, 1001, 4, 6), (2, 16385, 300, 7), (6, 9000, 3, 8),
])
def test_random_logits_keep_every_winner(W_in, V, W, seed):
    s = wl.select_inputs(W_in, V, W, seed=seed)
    n, _, n_groups, exact = check(s.logits, s.cum, W)
    # With many more groups than 2W (Gaussian logits) the 2W-th key lies
    # within the histogram and the list stays short.  When 2W nears the
    # number of groups (2 rows of 16,385: 768 sub-chunk groups, 254 of them
    # empty, for 2W = 600) the threshold falls among the empty groups' keys
    # and nearly every logit is a candidate, which the kernel's exact path
    # takes.
    if n_groups >= 8 * 2 * W:
        assert not exact
        assert n < 20 * 2 * W + 4096


@pytest.mark.parametrize("W_in,V,W,levels", [(4, 20000, 8, 1), (4, 20000, 8, 2), (8, 5000, 16, 5), (2, 40000, 50, 3)])
def test_heavy_ties_keep_every_winner(W_in, V, W, levels):
    logits = wl.quantized_logits(W_in, V, levels=levels, seed=V + levels)
    cum = torch.zeros(W_in, dtype=torch.float32)
    cum[W_in // 2:] = -0.5
    check(logits, cum, W)


@pytest.mark.parametrize("W_in,W", [(1, 16), (1, 100), (12, 16)])
def test_dominant_token_threshold_below_the_bins(W_in, W):
    # each row's one dominant logit puts its candidate's score at ~0 and the
    # 2W-th group key dozens of binades lower: the exact fallback decides L
    V = 30000
    s = wl.select_inputs(W_in, V, W, seed=50 + W_in, step=0 if W_in == 1 else 1)
    logits = s.logits.clone()
    cols = torch.arange(W_in) * 997 % V
    logits[torch.arange(W_in), cols] = 60.0
    cum = s.cum.clone()
    cum[0] = 0.0
    assert check(logits, cum, W)[3]  # the exact fallback took the threshold


def test_model_takes_both_group_levels():
    # a first step (one row, fewer tiles than 2W) groups by sub-chunks; wide
    # beams group by tiles
    s1 = wl.select_inputs(1, 40000, 64, seed=11)
    assert check(s1.logits, s1.cum, 64)[1] is False
    s2 = wl.select_inputs(8, 40000, 8, seed=12)
    assert check(s2.logits, s2.cum, 8)[1] is True
