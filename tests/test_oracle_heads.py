"""Pins for the oracle of the operations around the attention path (CPU only):
E4M3 codes, fused SwiGLU + per-token E4M3 (article "SLM 生成式高并发推理引擎：
延迟约束下的有效吞吐优化", section 3.4), last-token label scores (sections 1.1 and
3.1), finished-beam handling and the token-history reorder (sections 2.3, 3.3).
"""
import math

import numpy as np
import pytest
import torch

from oracle import heads as H


def test_e4m3_decode_known_codes():
    # OCP E4M3: bias 7, 3 mantissa bits, S.1111.111 = NaN, max 448
    assert H.e4m3_decode(0x7E) == 448.0
    assert H.e4m3_decode(0xFE) == -448.0
    assert H.e4m3_decode(0x38) == 1.0
    assert H.e4m3_decode(0x08) == 2.0 ** -6            # smallest normal
    assert H.e4m3_decode(0x01) == 2.0 ** -9            # smallest subnormal
    assert H.e4m3_decode(0x3C) == 1.5
    assert np.isnan(H.e4m3_decode(0x7F)) and np.isnan(H.e4m3_decode(0xFF))
    vals = H.e4m3_decode(np.arange(0x7F))
    assert (np.diff(vals) > 0).all()                     # codes 0..0x7E increase


def test_e4m3_encode_matches_library_conversion():
    # torch's float8_e4m3fn rounds to nearest even inside the finite range
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(0, 40, 20000), rng.uniform(-448, 448, 20000),
                        (H.e4m3_decode(np.arange(0x7E)) + H.e4m3_decode(np.arange(1, 0x7F))) / 2,  # midpoints
                        -(H.e4m3_decode(np.arange(0x7E)) + H.e4m3_decode(np.arange(1, 0x7F))) / 2,
                        H.e4m3_decode(np.arange(0x7F)), 2.0 ** -np.arange(5, 12)])
    x = x.astype(np.float32).astype(np.float64)          # fp32 inputs, as the kernel sees them
    mine = H.e4m3_encode(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(H.e4m3_decode(mine), H.e4m3_decode(ref))


def test_e4m3_encode_saturates_and_keeps_sign():
    assert H.e4m3_encode(500.0) == 0x7E
    assert H.e4m3_encode(-1e9) == 0xFE
    assert H.e4m3_encode(464.0) == 0x7E                  # beyond the last midpoint: still 448 (saturate)
    assert H.e4m3_encode(1.0625) == 0x38                 # halfway between 1 and 1.125: even code
    assert H.e4m3_encode(1.1875) == 0x3A                 # halfway between 1.125 and 1.25: even code
    assert H.e4m3_encode(-2.0 ** -11) == 0x80            # rounds to zero, sign kept


def _gate_up(T, I, seed, std=2.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn((T, 2 * I), generator=g) * std).to(torch.bfloat16)


def test_swiglu_quant_row_maximum_maps_to_448_and_error_bound():
    gu = _gate_up(64, 256, 1)
    codes, scale, x = H.swiglu_quant_e4m3(gu)
    g = gu[:, :256].double().numpy()
    u = gu[:, 256:].double().numpy()
    h = g / (1 + np.exp(-g)) * u                              # SiLU(g) * u, plain formula
    amax = np.abs(h).max(axis=1)
    np.testing.assert_allclose(scale, amax / 448.0, rtol=1e-6)
    dec = H.e4m3_decode(codes)
    # the largest element of each row maps to +-448
    i = np.abs(h).argmax(axis=1)
    assert (np.abs(dec[np.arange(64), i]) == 448.0).all()
    # dequantised values: within half an E4M3 step (relative 2^-4) of h, or
    # of the subnormal spacing 2^-9 * scale
    err = np.abs(dec * scale[:, None].astype(np.float64) - h)
    bound = np.maximum(np.abs(h) * 2.0 ** -4, 2.0 ** -10 * scale[:, None]) * 1.0001
    assert (err <= bound).all()


def test_swiglu_quant_closed_forms():
    # gate 0 -> SiLU 0 -> all zero row: scale 1, codes +-0
    gu = torch.zeros((2, 16), dtype=torch.bfloat16)
    gu[1, 8:] = 3.0
    codes, scale, _ = H.swiglu_quant_e4m3(gu)
    assert (H.e4m3_decode(codes) == 0).all() and (scale == 1.0).all()
    # large gate: SiLU(g) ~ g, so h ~ g * u; with one dominant element the
    # others are its exact fractions
    gu = torch.zeros((1, 8), dtype=torch.bfloat16)
    gu[0, :4] = torch.tensor([40.0, 20.0, 10.0, 5.0])
    gu[0, 4:] = 1.0
    codes, scale, _ = H.swiglu_quant_e4m3(gu)
    np.testing.assert_array_equal(H.e4m3_decode(codes[0]), [448.0, 224.0, 112.0, 56.0])
    assert scale[0] == np.float32(40.0 / 448.0)


def test_label_scores_match_library_and_closed_forms():
    g = torch.Generator().manual_seed(3)
    lengths = [5, 0, 17, 1]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    T, d, n = int(cu[-1]), 64, 3
    hidden = torch.randn((T, d), generator=g).to(torch.bfloat16)
    w = torch.randn((n, d), generator=g).to(torch.bfloat16)
    logits, probs = H.label_scores(hidden, cu, w)
    for b, L in enumerate(lengths):
        if L == 0:
            assert np.isnan(logits[b]).all() and np.isnan(probs[b]).all()
            continue
        z = hidden[cu[b + 1] - 1].double() @ w.double().T
        np.testing.assert_allclose(logits[b], z.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(probs[b], torch.softmax(z, dim=0).numpy(), rtol=0, atol=1e-14)
    # one-hot hidden state: the logits are a column of w
    hidden = torch.zeros((2, d), dtype=torch.bfloat16)
    hidden[1, 7] = 1.0
    logits, probs = H.label_scores(hidden, np.array([0, 2]), w)
    np.testing.assert_array_equal(logits[0], w[:, 7].double().numpy())
    assert math.isclose(probs[0].sum(), 1.0, rel_tol=1e-15)


def test_split_finished_hand_example():
    # W = 3; 2W = 6 candidates in global order; stop id 7
    tok = [7, 4, 5, 7, 9, 7]
    par = [0, 1, 0, 2, 1, 1]
    sc = [-1.0, -1.5, -2.0, -2.5, -3.0, -3.5]
    active, finished = H.split_finished(tok, par, sc, 3, 7)
    assert active == [(4, 1, -1.5), (5, 0, -2.0), (9, 1, -3.0)]
    assert finished == [(7, 0, -1.0)]                     # the stop at rank 3 is below the first W
    # no stop token: the first W candidates, nothing finished
    active, finished = H.split_finished(tok, par, sc, 3, 8)
    assert [a[0] for a in active] == [7, 4, 5] and finished == []


def test_reorder_history_hand_example():
    hist = np.array([[1, 2], [3, 4], [5, 6]])
    out = H.reorder_history(hist, [2, 2, 0], [7, 8, 9], 2)
    np.testing.assert_array_equal(out, [[5, 6, 7], [5, 6, 8], [1, 2, 9]])
    out = H.reorder_history(None, None, [4, 5], 0)
    np.testing.assert_array_equal(out, [[4], [5]])
