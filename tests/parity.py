"""Comparison helpers for the GPU-vs-oracle parity tests.

Attention outputs.  The gate is max-abs 1e-2 and mean-abs 1e-3 against the
fp64 oracle.  It is applied as it stands to the fp32 output of the test
variants of the kernels (``fp32_gate=True``): that is the attention
arithmetic itself.  The product output is bf16.  The kernel's fp32 result is
off by the bf16 rounding of the softmax weights P before P V (relative 2^-8
each, the unit roundoff of an 8-bit significand: at most 2^-8 sum_j w_j |v_j|)
plus fp32 summation error, e32 <= 2^-8 sum_j w_j |v_j| + 1e-4; rounding that
result to bf16 adds at most half a bf16 ulp of it (0.0078 for |O| in [2, 4),
0.0156 in [4, 8)).  The bf16 output is therefore held per element to
max(1e-2, e32 + half an ulp of |ref| + e32) when the caller passes
sum_j w_j |v_j| (``weighted_abs_v``, the oracle run on |V|), else to the same
with e32 = 1e-3; the mean-abs bound stays 1e-3.

Beam selection: given the GPU's own fp32 log-normalisers, the oracle's full
sort must give the GPU's candidates bit for bit.  Against the oracle's own
correctly rounded normalisers (a few ulp away), any difference must be a near
tie that the normalisers' difference explains; those are counted.
"""
import numpy as np
import torch

ATOL_MAX = 1e-2
ATOL_MEAN = 1e-3


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    a = np.abs(x)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def check_attention(got: torch.Tensor, ref: np.ndarray, what: str = "", weighted_abs_v=None,
                    fp32_gate: bool = False):
    """got: the GPU output (bf16, or fp32 with fp32_gate); ref: the oracle's
    fp64 result; weighted_abs_v (optional, same shape as ref): sum_j w_j |v_j|
    per output.  Returns (max abs error, mean abs error)."""
    g = got.float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref)
    if fp32_gate:
        assert got.dtype == torch.float32, "the gate applies to the fp32 output"
        tol = np.full_like(ref, ATOL_MAX)
    else:
        e32 = 2.0 ** -8 * weighted_abs_v + 1e-4 if weighted_abs_v is not None else np.full_like(ref, 1e-3)
        tol = np.maximum(ATOL_MAX, e32 + 0.5 * bf16_ulp(np.abs(ref) + e32))
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} elements out of tolerance; worst err {err.max():.4g} "
                           f"at {np.unravel_index(err.argmax(), err.shape)} (ref {ref.flat[err.argmax()]:.4g})")
    assert err.mean() <= ATOL_MEAN, f"{what}: mean abs error {err.mean():.3g} > {ATOL_MEAN}"
    return float(err.max()), float(err.mean())


def check_lse(got: torch.Tensor, ref: np.ndarray, what: str = "", atol: float = 1e-4):
    g = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    assert err.max() <= atol + 1e-6 * np.abs(ref).max(), f"{what}: lse error {err.max():.3g}"


def f32_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    ai = np.asarray(a, dtype=np.float32).view(np.int32).astype(np.int64)
    bi = np.asarray(b, dtype=np.float32).view(np.int32).astype(np.int64)
    ai = np.where(ai < 0, -(ai & 0x7FFFFFFF), ai)
    bi = np.where(bi < 0, -(bi & 0x7FFFFFFF), bi)
    return np.abs(ai - bi)


def selection_scores(x32: np.ndarray, cum: np.ndarray, lse: np.ndarray) -> np.ndarray:
    """fp32 score of every candidate, fl32(cum_b + fl32(x_bv - lse_b)), [W_in, V]."""
    lp = (x32 - lse.astype(np.float32)[:, None]).astype(np.float32)
    return (cum.astype(np.float32)[:, None] + lp).astype(np.float32)


def _np(a, dtype):
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


def check_selection(res, oracle_cand, logits, cum_gpu, W, cum_oracle=None, max_lse_ulp=4):
    """Checks one GPU selection; returns (near ties, delta).

    res: the GPU result dict (2W sorted candidates, next beams, lse);
    oracle_cand: (token, parent, score, lse) of the oracle's full sort over
    ``cum_oracle`` (default: the GPU's own ``cum_gpu``) with its own
    correctly rounded log-normalisers.

    1. The GPU lse is within ``max_lse_ulp`` fp32 ulp of the oracle's.
    2. Conditional, bit-exact: the oracle's full sort of the scores formed
       from the GPU's own fp32 lse and cumulative scores gives exactly the
       GPU's 2W tokens, parents and scores.  This fixes the tie rule (score,
       lower parent, higher logit, lower id) and excludes duplicates.
    3. Unconditional: the largest change any candidate's score sees between
       the two normalisers, delta, is no more than the lse and cumulative
       differences plus one rounding of each fp32 step; and at every rank the
       GPU's candidate scores, by the oracle's own scores, within 2 * delta
       of the oracle's candidate at that rank (the k-th largest of values
       perturbed by at most delta moves by at most delta).  Positions where
       the two lists differ are near ties explained by that band; their
       number is returned."""
    o_tok, o_par, o_sc, o_lse = oracle_cand
    cum_g = _np(cum_gpu, np.float32)
    cum_o = cum_g if cum_oracle is None else _np(cum_oracle, np.float32)
    g_lse = _np(res["lse"], np.float32)
    g_tok = _np(res["cand_token"], np.int32)
    g_par = _np(res["cand_parent"], np.int32)
    g_sc = _np(res["cand_score"], np.float32)
    V = int(logits.shape[1])

    d_ulp = f32_ulp_diff(g_lse, o_lse)
    assert d_ulp.max() <= max_lse_ulp, f"lse differs by {d_ulp.max()} ulp"
    # the next beams are the first W candidates
    np.testing.assert_array_equal(_np(res["token"], np.int32), g_tok[:W])
    np.testing.assert_array_equal(_np(res["parent"], np.int32), g_par[:W])
    np.testing.assert_array_equal(_np(res["score"], np.float32).view(np.int32), g_sc[:W].view(np.int32))
    pairs = g_par.astype(np.int64) * V + g_tok
    assert len(np.unique(pairs)) == len(pairs), "a (parent, token) candidate appears twice"

    import oracle
    c_tok, c_par, c_sc, _ = oracle.beam_select(logits, cum_g, len(g_tok), lse_in=g_lse)
    np.testing.assert_array_equal(g_tok, c_tok, err_msg="token ids differ from the ranking on the GPU's own lse")
    np.testing.assert_array_equal(g_par, c_par, err_msg="parents differ from the ranking on the GPU's own lse")
    np.testing.assert_array_equal(g_sc.view(np.int32), c_sc.view(np.int32),
                                  err_msg="scores differ from the ranking on the GPU's own lse")

    x = logits.to(torch.float32).numpy() if isinstance(logits, torch.Tensor) else np.asarray(logits, np.float32)
    delta = 0.0
    s_o_of_g = np.zeros(len(g_tok), np.float64)
    top_lp = top_s = 0.0
    for r0 in range(0, x.shape[0], 64):  # row blocks keep the W x V temporaries small
        sl = slice(r0, r0 + 64)
        s_o = selection_scores(x[sl], cum_o[sl], o_lse[sl])
        s_g = selection_scores(x[sl], cum_g[sl], g_lse[sl])
        delta = max(delta, float(np.abs(s_o.astype(np.float64) - s_g.astype(np.float64)).max()))
        top_lp = max(top_lp, float(np.abs(x[sl] - o_lse[sl, None]).max()))
        top_s = max(top_s, float(np.abs(s_o).max()))
        hit = (g_par >= r0) & (g_par < r0 + s_o.shape[0])
        s_o_of_g[hit] = s_o[g_par[hit] - r0, g_tok[hit]]
    bound = (float(np.abs(g_lse.astype(np.float64) - o_lse.astype(np.float64)).max())
             + float(np.abs(cum_g.astype(np.float64) - cum_o.astype(np.float64)).max())
             + float(np.spacing(np.float32(top_lp))) + float(np.spacing(np.float32(top_s))))
    assert delta <= bound, f"scores move by {delta:.3g} between the normalisers, more than {bound:.3g}"
    gap = np.abs(s_o_of_g - o_sc.astype(np.float64))
    assert (gap <= 2 * delta).all(), (
        f"rank {int(gap.argmax())}: the GPU's candidate scores {s_o_of_g[gap.argmax()]!r} by the oracle's "
        f"normalisers, the oracle's candidate there {float(o_sc[gap.argmax()])!r}; band {2 * delta:.3g}")
    near = int(((g_tok != o_tok) | (g_par != o_par)).sum())
    return near, delta
