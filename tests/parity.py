"""Comparison helpers for the GPU-vs-oracle parity tests.

Attention outputs: the GPU writes bf16 O from fp32 accumulators; the oracle
is fp64.  Per element the error must stay within max(1e-2, one bf16 ulp of
the oracle value) -- above |O| = 2 a bf16 ulp exceeds 1e-2, so no bf16 output
could meet 1e-2 there -- and the mean absolute error within 1e-3.

Beam selection: token ids and parents must match exactly.  The GPU's fp32
log-normaliser may differ from the oracle's correctly rounded one by a few
ulp; that can only reorder candidates of different beams whose oracle scores
lie within that band of each other.  Such near ties are reported and checked
for validity instead of identity.
"""
import numpy as np
import torch

ATOL_MAX = 1e-2
ATOL_MEAN = 1e-3


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    a = np.abs(x)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def check_attention(got: torch.Tensor, ref: np.ndarray, what: str = "", weighted_abs_v=None):
    """weighted_abs_v (optional, same shape as ref): sum_j w_j |v_j| per
    output, for inputs whose softmax is so peaked that the bf16 rounding of
    the weights P (relative 2^-9 each) dominates: the element bound then
    becomes 2^-9 * sum_j w_j |v_j| + one bf16 ulp of the output."""
    g = got.float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref)
    tol = np.maximum(ATOL_MAX, bf16_ulp(ref))
    if weighted_abs_v is not None:
        tol = np.maximum(tol, 2.0 ** -9 * weighted_abs_v + bf16_ulp(ref))
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


def check_selection(res, o_tok, o_par, o_sc, o_lse, logits, cum, W, max_lse_ulp=4):
    """res: GPU result dict; o_*: oracle's sorted top-2W and its lse."""
    g_lse = res["lse"].cpu().numpy()
    d_ulp = f32_ulp_diff(g_lse, o_lse)
    assert d_ulp.max() <= max_lse_ulp, f"lse differs by {d_ulp.max()} ulp"
    g_tok = res["cand_token"].cpu().numpy()
    g_par = res["cand_parent"].cpu().numpy()
    g_sc = res["cand_score"].cpu().numpy()
    # the next beams are the first W candidates
    np.testing.assert_array_equal(res["token"].cpu().numpy(), g_tok[:W])
    np.testing.assert_array_equal(res["parent"].cpu().numpy(), g_par[:W])
    np.testing.assert_array_equal(res["score"].cpu().numpy(), g_sc[:W])
    # GPU scores are its own fp32 log-softmax plus the cumulative score
    x = logits.to(torch.float32).numpy()
    cum = cum.numpy().astype(np.float32)
    lp = (x[g_par, g_tok] - g_lse[g_par]).astype(np.float32)
    np.testing.assert_array_equal(g_sc, (cum[g_par] + lp).astype(np.float32))
    assert (np.diff(g_sc) <= 0).all(), "GPU candidates not in descending score order"
    if np.array_equal(g_tok, o_tok) and np.array_equal(g_par, o_par):
        # same candidates: scores may differ by the beam's lse difference plus
        # one rounding of the score
        allowed = (np.abs(g_lse[g_par].astype(np.float64) - o_lse[g_par].astype(np.float64))
                   + np.spacing(np.abs(o_sc)).astype(np.float64))
        assert (np.abs(g_sc.astype(np.float64) - o_sc.astype(np.float64)) <= allowed).all()
        return 0
    # near-tie path: explain every difference by the lse band
    lp_o = (x - o_lse[:, None]).astype(np.float32)
    score_o = (cum[:, None] + lp_o).astype(np.float32)
    band = float(np.max(np.abs(g_lse.astype(np.float64) - o_lse.astype(np.float64)))) * 2 + 1e-5
    cut = float(o_sc[-1])
    got_o = score_o[g_par, g_tok].astype(np.float64)
    assert (got_o >= cut - band).all(), "GPU kept a candidate well below the oracle's cut"
    must = set(zip(o_par[o_sc > cut + band].tolist(), o_tok[o_sc > cut + band].tolist()))
    assert must <= set(zip(g_par.tolist(), g_tok.tolist())), "GPU dropped a clear candidate"
    diff = np.nonzero((g_tok != o_tok) | (g_par != o_par))[0]
    for i in diff:
        assert abs(got_o[i] - float(o_sc[i])) <= band, f"position {i}: not a near tie"
    return len(diff)
