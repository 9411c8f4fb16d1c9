"""Pins for the beam-selection oracle (CPU only).

The oracle follows section 3.3 of the article "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化":
FP32 log-softmax over the full vocabulary, candidate score = cumulative beam
score + log-probability, global candidates from the flattened beams.  It sorts
every W x V entry.  The pins check it against exhaustive enumeration, the
two-stage 2W-per-beam method (the article's pruning claim), the monotonicity
claim (IDs from logits = IDs from log-probs), a library sort, closed forms and
a hand-derived case.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from attention_packed_varlen_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _scores(x32, cum, lse):
    lp = (x32 - lse[:, None]).astype(np.float32)
    return (cum[:, None].astype(np.float32) + lp).astype(np.float32)


def exhaustive_select(logits, cum, n_keep):
    """Repeatedly take the best remaining entry (no sort): higher score, then
    lower parent, higher logit, lower token id."""
    x = logits.to(torch.float32).numpy()
    W_in, V = x.shape
    lse = np.array([np.float32(scipy.special.logsumexp(x[b].astype(np.float64))) for b in range(W_in)],
                   dtype=np.float32)
    sc = _scores(x, cum.numpy(), lse)
    taken = np.zeros_like(sc, dtype=bool)
    out = []
    for _ in range(n_keep):
        best = None
        for b in range(W_in):
            for v in range(V):
                if taken[b, v]:
                    continue
                key = (-sc[b, v], b, -x[b, v], v)
                if best is None or key < best[0]:
                    best = (key, b, v)
        _, b, v = best
        taken[b, v] = True
        out.append((v, b, sc[b, v]))
    return out


def two_stage_select(logits, cum, W, lse):
    """The article's method, restated: per-beam top-2W on the bf16 logits
    (lowest id on ties), scores read from the FP32 log-softmax, plus the
    cumulative score, flattened W x 2W, stable global sort by score."""
    x = logits.to(torch.float32).numpy()
    W_in, V = x.shape
    K = 2 * W
    ids = np.argsort(-x, axis=1, kind="stable")[:, :K]           # [W_in, 2W]
    lp = (np.take_along_axis(x, ids, axis=1) - lse[:, None]).astype(np.float32)
    cand = (cum.numpy()[:, None] + lp).astype(np.float32)         # [W_in, 2W]
    flat = cand.reshape(-1)
    order = np.argsort(-flat, kind="stable")                      # ties: lower flat index
    parent = order // K
    token = ids.reshape(-1)[order]
    return token.astype(np.int32), parent.astype(np.int32), flat[order]


@pytest.mark.parametrize("W_in,V,W,seed", [(3, 7, 3, 1), (4, 16, 4, 2), (1, 9, 2, 3), (2, 5, 2, 4)])
def test_select_matches_exhaustive_enumeration(W_in, V, W, seed):
    s = wl.select_inputs(W_in, V, W, seed=seed)
    n_keep = min(2 * W, W_in * V)
    tok, par, sc, _ = oracle.beam_select(s.logits, s.cum, n_keep)
    ex = exhaustive_select(s.logits, s.cum, n_keep)
    assert list(tok) == [e[0] for e in ex]
    assert list(par) == [e[1] for e in ex]
    np.testing.assert_array_equal(sc, np.array([e[2] for e in ex], dtype=np.float32))


def test_select_exhaustive_with_heavy_ties():
    logits = wl.quantized_logits(3, 12, levels=3, seed=7)
    # beam 1 holds beam 0's logits reversed: same lse, and with the same
    # cumulative score every value of beam 0 ties exactly with one of beam 1
    logits[1] = logits[0].flip(0)
    cum = torch.tensor([0.0, 0.0, -0.5], dtype=torch.float32)
    tok, par, sc, _ = oracle.beam_select(logits, cum, 6)
    ex = exhaustive_select(logits, cum, 6)
    assert list(zip(tok, par)) == [(e[0], e[1]) for e in ex]


@pytest.mark.parametrize("W,V,seed", [(8, 500, 1), (20, 3000, 2), (4, 64, 3)])
def test_two_stage_pruning_equals_full_sort(W, V, seed):
    # article, section 3.3: a token ranked below 2W in its own beam cannot enter
    # the global top 2W, so per-beam pruning does not change the candidates
    s = wl.select_inputs(W, V, W, seed=seed)
    tok, par, sc, lse = oracle.beam_select(s.logits, s.cum, 2 * W)
    t2, p2, s2 = two_stage_select(s.logits, s.cum, W, lse)
    np.testing.assert_array_equal(tok, t2[:2 * W])
    np.testing.assert_array_equal(par, p2[:2 * W])
    np.testing.assert_array_equal(sc, s2[:2 * W])


def test_two_stage_pruning_with_ties():
    W, V = 6, 40
    logits = wl.quantized_logits(W, V, levels=4, seed=3)
    cum = torch.tensor([0, 0, -0.25, -0.25, -1, -1], dtype=torch.float32)
    tok, par, sc, lse = oracle.beam_select(logits, cum, 2 * W)
    t2, p2, _ = two_stage_select(logits, cum, W, lse)
    np.testing.assert_array_equal(tok, t2[:2 * W])
    np.testing.assert_array_equal(par, p2[:2 * W])


def test_two_stage_orders_equal_scores_by_logit():
    # Distinct bf16 logits whose fp32 log-probabilities round to one value
    # (all below half an fp32 ulp of the row's lse = ln 4): their scores tie
    # exactly, and the article's per-beam Top-K on the logits (section 3.3)
    # puts the higher logit first even when it has the higher token id.
    V, W = 16, 2
    x = torch.full((2, V), -30.0)
    x[:, :4] = torch.tensor([0.0, 2.0 ** -27, 2.0 ** -26, 2.0 ** -25])
    logits = x.to(torch.bfloat16)
    cum = torch.tensor([0.0, -1.0])
    tok, par, sc, lse = oracle.beam_select(logits, cum, 2 * W)
    assert len(set(sc[:4].tolist())) == 1, "the case needs four exactly tied scores"
    t2, p2, _ = two_stage_select(logits, cum, W, lse)
    np.testing.assert_array_equal(tok, t2[:2 * W])
    np.testing.assert_array_equal(par, p2[:2 * W])
    assert tok.tolist() == [3, 2, 1, 0]


def test_ids_from_logits_equal_ids_from_log_probs():
    # article, section 3.3: log-softmax is strictly monotone within a row, so
    # Top-K on bf16 logits and on fp64 log-probabilities pick the same ids
    s = wl.select_inputs(5, 2000, 10, seed=4)
    x = s.logits.to(torch.float64).numpy()
    lp = x - scipy.special.logsumexp(x, axis=1, keepdims=True)
    for b in range(5):
        a = np.argsort(-x[b], kind="stable")[:20]
        c = np.argsort(-lp[b], kind="stable")[:20]
        np.testing.assert_array_equal(a, c)
    # and the oracle's global picks are consistent with it
    tok, par, _, _ = oracle.beam_select(s.logits, s.cum, 20)
    for t, p in zip(tok, par):
        assert t in np.argsort(-x[p], kind="stable")[:20]


def test_select_matches_library_sort():
    # library routine: successive stable torch sorts on the four keys
    s = wl.select_inputs(6, 300, 6, seed=5)
    tok, par, sc, lse = oracle.beam_select(s.logits, s.cum, 12)
    x = s.logits.to(torch.float32)
    score = torch.from_numpy(_scores(x.numpy(), s.cum.numpy(), lse))
    W_in, V = x.shape
    b_idx = torch.arange(W_in).repeat_interleave(V)
    v_idx = torch.arange(V).repeat(W_in)
    keys = [v_idx, -x.reshape(-1), b_idx, -score.reshape(-1)]  # least significant first
    perm = torch.arange(W_in * V)
    for key in keys:
        order = torch.sort(key[perm], stable=True).indices
        perm = perm[order]
    top = perm[:12]
    np.testing.assert_array_equal(tok, v_idx[top].numpy())
    np.testing.assert_array_equal(par, b_idx[top].numpy())


def test_row_lse_closed_forms():
    V = 151936
    # all logits equal c -> lse = c + ln V
    x = torch.full((2, V), 2.5, dtype=torch.bfloat16)
    x[1] = -7.0
    lse = oracle.row_lse(x)
    assert lse[0] == np.float32(2.5 + math.log(V))
    assert lse[1] == np.float32(-7.0 + math.log(V))
    # against the library log-sum-exp in fp64, rounded once
    s = wl.select_inputs(3, V, 3, seed=6)
    lse = oracle.row_lse(s.logits)
    ref = scipy.special.logsumexp(s.logits.to(torch.float64).numpy(), axis=1).astype(np.float32)
    np.testing.assert_array_equal(lse, ref)


def test_first_step_single_row():
    # W_in = 1 (first-step candidate init): top-2W of one row, lowest id on ties
    logits = wl.quantized_logits(1, 50, levels=5, seed=8)
    cum = torch.zeros(1)
    W = 4
    tok, par, sc, lse = oracle.beam_select(logits, cum, 2 * W)
    x = logits.to(torch.float32).numpy()[0]
    np.testing.assert_array_equal(tok, np.argsort(-x, kind="stable")[:2 * W])
    assert not par.any()
    np.testing.assert_array_equal(sc, (x[tok] - lse[0]).astype(np.float32))


def test_select_hand_derived_case():
    g = json.load(open(os.path.join(GOLDEN, "select_hand.json")))
    logits = torch.tensor(g["logits"], dtype=torch.float32).to(torch.bfloat16)
    cum = torch.tensor(g["cum"], dtype=torch.float32)
    tok, par, sc, lse = oracle.beam_select(logits, cum, len(g["token"]))
    assert list(tok) == g["token"]
    assert list(par) == g["parent"]
    want = [float(eval(e, {"ln": math.log, "exp": math.exp})) for e in g["score"]]
    np.testing.assert_allclose(sc, np.array(want, dtype=np.float32), rtol=0, atol=1e-6)
    want_lse = [float(eval(e, {"ln": math.log, "exp": math.exp})) for e in g["lse"]]
    np.testing.assert_allclose(lse, np.array(want_lse, dtype=np.float32), rtol=0, atol=1e-6)


def test_select_rejects_bad_arguments():
    s = wl.select_inputs(2, 4, 2, seed=1)
    with pytest.raises(ValueError):
        oracle.beam_select(s.logits, s.cum, 9)
