"""GPU parity of the operations around the attention path against the oracle
(article "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化"): fused SwiGLU + per-token
E4M3 (section 3.4), last-token label scores (sections 1.1, 3.1), finished-beam
handling and the token-history reorder (sections 2.3, 3.3).
"""
import numpy as np
import pytest
import torch

from attention_packed_varlen_gb300 import _binding as slm
from attention_packed_varlen_gb300 import build, workloads as wl
from oracle import heads as H

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    slm.load()


def check_e4m3(gu_cpu, q_gpu, scale_gpu):
    """Scales within 4 ulp; codes equal in value except where the oracle's
    scaled value lies within 2^-17 (relative) of a rounding boundary, and
    there the GPU code is one of the two neighbours."""
    codes, scale, x = H.swiglu_quant_e4m3(gu_cpu)
    sg = scale_gpu.cpu().numpy()
    assert np.all(np.abs(sg.astype(np.float64) - scale) <= 4 * np.spacing(scale.astype(np.float32)).astype(np.float64))
    got = H.e4m3_decode(q_gpu.cpu().numpy())
    want = H.e4m3_decode(codes)
    diff = got != want
    near = H.e4m3_boundary_distance(x) < 2.0 ** -17
    assert not (diff & ~near).any(), f"{int((diff & ~near).sum())} codes differ away from a rounding boundary"
    if diff.any():  # neighbouring magnitudes only
        cg = q_gpu.cpu().numpy()[diff].astype(np.int64)
        co = codes[diff].astype(np.int64)
        assert (np.abs((cg & 0x7F) - (co & 0x7F)) <= 1).all()
    return int(diff.sum())


@pytest.mark.parametrize("T,I,std", [(37, 5632, 2.0), (5, 64, 1.0), (3, 16384, 3.0), (130, 1024, 8.0)])
def test_swiglu_quant_matches_oracle(T, I, std):
    g = torch.Generator().manual_seed(T * 7 + I)
    gu = (torch.randn((T, 2 * I), generator=g) * std).to(torch.bfloat16)
    gu[0] = 0.0                       # an all-zero row: scale 1, zero codes
    if T > 2:
        gu[2, :I] = 60.0              # saturating SiLU, one dominant value per row
    q, scale = slm.slm_swiglu_quant_e4m3(gu.to(DEV))
    torch.cuda.synchronize()
    flips = check_e4m3(gu, q, scale)
    assert flips <= max(2, T * I // 100000)


def test_swiglu_quant_full_size_sampled_rows():
    # the concurrent Prefill-Only batch: one token row per token (T ~ 130k),
    # d_model 2048, intermediate 5632; the oracle checks 64 sampled rows
    T = sum(int(x) for x in wl.draw_lengths(240, 64, 1024, wl.workload_seed(3)))
    I = 5632
    g = torch.Generator(device=DEV).manual_seed(11)
    gu = (torch.randn((T, 2 * I), generator=g, device=DEV) * 2.0).to(torch.bfloat16)
    q, scale = slm.slm_swiglu_quant_e4m3(gu)
    torch.cuda.synchronize()
    rows = np.random.default_rng(5).choice(T, 64, replace=False)
    rows.sort()
    idx = torch.from_numpy(rows).to(DEV)
    check_e4m3(gu[idx].cpu(), q[idx], scale[idx])


def test_label_scores_matches_oracle():
    g = torch.Generator().manual_seed(21)
    lengths = [int(x) for x in wl.draw_lengths(15, 100, 500, wl.workload_seed(2))]
    lengths[3] = 0
    lengths[7] = 1
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    T, d = int(cu[-1]), 2048
    hidden = torch.randn((T, d), generator=g).to(torch.bfloat16)
    for n in (2, 8, 32):
        w = (torch.randn((n, d), generator=g) * 0.05).to(torch.bfloat16)
        logits, probs = slm.slm_label_scores(hidden.to(DEV), cu.to(DEV), w.to(DEV))
        torch.cuda.synchronize()
        lo, po = H.label_scores(hidden, cu.numpy(), w)
        lg, pg = logits.cpu().numpy().astype(np.float64), probs.cpu().numpy().astype(np.float64)
        empty = np.array(lengths) == 0
        assert np.isnan(lg[empty]).all() and np.isnan(pg[empty]).all()
        # fp32 accumulation of d products: |error| <= d * 2^-24 * sum |h_j w_j|
        hl = hidden.double().numpy()[cu.numpy()[1:][~empty] - 1]
        bound = d * 2.0 ** -24 * (np.abs(hl) @ np.abs(w.double().numpy()).T) + 1e-30
        assert (np.abs(lg[~empty] - lo[~empty]) <= bound).all()
        np.testing.assert_allclose(pg[~empty], po[~empty], rtol=0, atol=1e-5)


def test_label_scores_flags_bad_boundary():
    hidden = torch.randn((8, 64), device=DEV).to(torch.bfloat16)
    w = torch.randn((2, 64), device=DEV).to(torch.bfloat16)
    cu = torch.tensor([0, 5, 3, 8], dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    logits, _ = slm.slm_label_scores(hidden, cu, w, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 1
    assert torch.isnan(logits[1]).all()


@pytest.mark.parametrize("W,seed", [(1, 1), (5, 2), (100, 3), (400, 4), (1024, 5)])
def test_split_finished_matches_oracle(W, seed):
    rng = np.random.default_rng(seed)
    stop = 7
    tok = rng.integers(0, 20, 2 * W).astype(np.int32)
    # at most one stop per parent beam, as a real row holds the stop token once
    par = rng.integers(0, W, 2 * W).astype(np.int32)
    seen = set()
    for i in range(2 * W):
        if tok[i] == stop:
            if par[i] in seen:
                tok[i] = stop + 1
            seen.add(par[i])
    sc = np.sort(rng.normal(0, 1, 2 * W).astype(np.float32))[::-1].copy()
    res = slm.slm_beam_split_finished(torch.from_numpy(tok).to(DEV), torch.from_numpy(par).to(DEV),
                                      torch.from_numpy(sc).to(DEV), stop)
    torch.cuda.synchronize()
    active, finished = H.split_finished(tok, par, sc, W, stop)
    n_act = min(W, len(active))
    assert [tuple(x) for x in zip(res["token"].cpu().tolist()[:n_act], res["parent"].cpu().tolist()[:n_act],
                                  res["score"].cpu().tolist()[:n_act])] == [(a, b, np.float32(c).item())
                                                                           for a, b, c in active[:n_act]]
    nf = int(res["fin_count"].item())
    assert nf == len(finished)
    assert list(zip(res["fin_parent"].cpu().tolist()[:nf], res["fin_score"].cpu().tolist()[:nf])) == \
        [(b, np.float32(c).item()) for _, b, c in finished]


def test_reorder_history_matches_oracle():
    rng = np.random.default_rng(9)
    W, W_in, max_len = 400, 400, 5
    hist = torch.from_numpy(rng.integers(0, 151936, (W_in, max_len)).astype(np.int32))
    for t in range(max_len):
        parent = torch.from_numpy(rng.integers(0, W_in, W).astype(np.int32))
        token = torch.from_numpy(rng.integers(0, 151936, W).astype(np.int32))
        out = torch.zeros((W, max_len), dtype=torch.int32, device=DEV)
        slm.slm_beam_reorder_history(hist.to(DEV), parent.to(DEV), token.to(DEV), t, out)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.cpu().numpy()[:, :t + 1], H.reorder_history(hist.numpy(), parent, token, t))


def test_reorder_history_first_step_from_one_row():
    # t = 0: the first beams' tokens, no parent rows (W_in = 1, identity parents ignored)
    W = 100
    token = torch.arange(W, dtype=torch.int32, device=DEV) * 7
    out = torch.full((W, 5), -1, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    slm.slm_beam_reorder_history(None, None, token, 0, out, dev_status=status)
    slm.slm_check_status(status)
    np.testing.assert_array_equal(out[:, 0].cpu().numpy(), token.cpu().numpy())
    assert (out[:, 1:].cpu() == -1).all()
