"""Pins for the packed-prefill oracle (CPU only).

The oracle follows section 3.1 of the article "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化"
(packed layout, block-diagonal causal mask from the sequence boundary).  Each
test below checks it against something other than itself: a dense brute force
with an explicit mask, the library attention routine, closed forms, a
hand-derived case and the sequence-isolation invariant.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from attention_packed_varlen_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f64(x):
    return x.to(torch.float64).numpy()


def dense_masked_attention(q, k, v, cu, scale):
    """Brute force: the full T x T score matrix per head with an explicit
    block-diagonal causal mask, then a row softmax (numpy fp64)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    seq = np.zeros(T, dtype=np.int64)
    for b in range(len(cu) - 1):
        seq[cu[b]:cu[b + 1]] = b
    pos = np.arange(T)
    allowed = (seq[:, None] == seq[None, :]) & (pos[None, :] <= pos[:, None])
    o = np.zeros_like(q)
    lse = np.zeros((Hq, T))
    for h in range(Hq):
        s = scale * q[:, h, :] @ k[:, h // G, :].T
        s = np.where(allowed, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(axis=1, keepdims=True)
        o[:, h, :] = (p / l) @ v[:, h // G, :]
        lse[h] = (m + np.log(l))[:, 0]
    return o, lse


def sdpa_reference(q, k, v, cu, scale):
    """Library routine: torch scaled_dot_product_attention in fp64 on CPU,
    sequence by sequence, is_causal=True, K/V heads repeated for GQA."""
    T, Hq, D = q.shape
    G = Hq // k.shape[1]
    out = torch.zeros(T, Hq, D, dtype=torch.float64)
    for b in range(len(cu) - 1):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        if s1 == s0:
            continue
        qs = q[s0:s1].to(torch.float64).transpose(0, 1)
        ks = k[s0:s1].to(torch.float64).repeat_interleave(G, dim=1).transpose(0, 1)
        vs = v[s0:s1].to(torch.float64).repeat_interleave(G, dim=1).transpose(0, 1)
        ob = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, is_causal=True, scale=scale)
        out[s0:s1] = ob.transpose(0, 1)
    return out.numpy()


@pytest.mark.parametrize("lengths,hq,hkv,d", [
    ((37, 64, 91, 128), 4, 2, 64),   # the tiny packed-prefill workload
    ((1, 2, 3, 5, 8), 2, 2, 16),     # MHA, very short sequences
    ((7, 0, 13, 0, 1), 6, 2, 32),    # zero-length sequences in the boundary
    ((19,), 8, 1, 8),                # single sequence, MQA
])
def test_prefill_matches_dense_brute_force(lengths, hq, hkv, d):
    inp = wl.prefill_inputs(lengths, hq, hkv, d, seed=11)
    cu = inp.cu_seqlens.numpy()
    o, lse = oracle.packed_prefill(inp.q, inp.k, inp.v, cu, inp.softmax_scale, want_lse=True)
    ob, lseb = dense_masked_attention(inp.q, inp.k, inp.v, cu, inp.softmax_scale)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lseb, rtol=0, atol=1e-12)


@pytest.mark.parametrize("lengths,hq,hkv,d", [
    ((37, 64, 91, 128), 4, 2, 64),
    ((100, 3, 250), 16, 8, 128),
    ((5, 17), 14, 2, 64),
])
def test_prefill_matches_library_sdpa(lengths, hq, hkv, d):
    inp = wl.prefill_inputs(lengths, hq, hkv, d, seed=5)
    cu = inp.cu_seqlens.numpy()
    o = oracle.packed_prefill(inp.q, inp.k, inp.v, cu, inp.softmax_scale)
    ref = sdpa_reference(inp.q, inp.k, inp.v, cu, inp.softmax_scale)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_prefill_hand_derived_case():
    g = json.load(open(os.path.join(GOLDEN, "prefill_hand.json")))
    to_bf16 = lambda a: torch.tensor(a, dtype=torch.float32).to(torch.bfloat16)
    q, k, v = to_bf16(g["q"]), to_bf16(g["k"]), to_bf16(g["v"])
    o, lse = oracle.packed_prefill(q, k, v, np.array(g["cu_seqlens"]), math.log(3.0), want_lse=True)
    np.testing.assert_allclose(o, np.array(g["o"], dtype=np.float64), rtol=0, atol=1e-15)
    ln = {"ln2": math.log(2.0), "ln4": math.log(4.0)}
    want_lse = np.array([[ln.get(x, x) for x in row] for row in g["lse"]], dtype=np.float64)
    np.testing.assert_allclose(lse, want_lse, rtol=0, atol=1e-15)


def test_prefill_single_token_sequences_return_v():
    # closed form: a query alone in its sequence attends only to itself -> O = V
    inp = wl.prefill_inputs([1] * 9, 4, 2, 32, seed=3)
    o = oracle.packed_prefill(inp.q, inp.k, inp.v, inp.cu_seqlens.numpy(), inp.softmax_scale)
    v = _f64(inp.v)
    for h in range(4):
        np.testing.assert_array_equal(o[:, h, :], v[:, h // 2, :])


def test_prefill_constant_keys_give_running_mean():
    # closed form: equal scores -> uniform weights over positions 0..r of the
    # sequence -> O_r = mean(v_0..v_r); LSE = scale*q.k + ln(r+1)
    lengths = (5, 12, 1)
    inp = wl.prefill_inputs(lengths, 2, 1, 16, seed=4)
    k = torch.zeros_like(inp.k)
    o, lse = oracle.packed_prefill(inp.q, k, inp.v, inp.cu_seqlens.numpy(), 0.7, want_lse=True)
    v = _f64(inp.v)[:, 0, :]
    cu = inp.cu_seqlens.numpy()
    for b in range(len(lengths)):
        s0, s1 = cu[b], cu[b + 1]
        run = np.cumsum(v[s0:s1], axis=0) / np.arange(1, s1 - s0 + 1)[:, None]
        for h in range(2):
            np.testing.assert_allclose(o[s0:s1, h, :], run, rtol=0, atol=1e-14)
            np.testing.assert_allclose(lse[h, s0:s1], np.log(np.arange(1, s1 - s0 + 1)), atol=1e-14)


def test_prefill_dominant_key_selects_its_value():
    # closed form limit: one key far above the rest -> O = that key's value
    T, D = 6, 8
    q = torch.zeros(T, 1, D); q[:, 0, 0] = 1.0
    k = torch.zeros(T, 1, D); k[2, 0, 0] = 64.0        # token 2 dominates for rows >= 2
    v = torch.randn(T, 1, D, generator=torch.Generator().manual_seed(1))
    o = oracle.packed_prefill(q.bfloat16(), k.bfloat16(), v.bfloat16(), np.array([0, T]), 1.0)
    vb = _f64(v.bfloat16())
    for t in range(2, T):
        np.testing.assert_allclose(o[t, 0], vb[2, 0], rtol=0, atol=1e-20)


def test_prefill_sequence_isolation():
    # invariant (section 3.1): packed attention equals running each sequence alone
    lengths = (13, 1, 40, 0, 7)
    inp = wl.prefill_inputs(lengths, 4, 2, 32, seed=9)
    cu = inp.cu_seqlens.numpy()
    o = oracle.packed_prefill(inp.q, inp.k, inp.v, cu, inp.softmax_scale)
    for b in range(len(lengths)):
        s0, s1 = cu[b], cu[b + 1]
        if s1 == s0:
            continue
        ob = oracle.packed_prefill(inp.q[s0:s1], inp.k[s0:s1], inp.v[s0:s1],
                                   np.array([0, s1 - s0]), inp.softmax_scale)
        np.testing.assert_array_equal(o[s0:s1], ob)


def test_prefill_rows_match_full_pass():
    inp = wl.prefill_inputs((30, 77, 2), 4, 2, 64, seed=21)
    cu = inp.cu_seqlens.numpy()
    o, lse = oracle.packed_prefill(inp.q, inp.k, inp.v, cu, inp.softmax_scale, want_lse=True)
    rng = np.random.default_rng(0)
    rows = np.stack([rng.integers(0, inp.total_tokens, 40), rng.integers(0, 4, 40)], axis=1)
    orow, lrow = oracle.packed_prefill_rows(inp.q, inp.k, inp.v, cu, inp.softmax_scale, rows)
    for i, (t, h) in enumerate(rows):
        np.testing.assert_array_equal(orow[i], o[t, h])
        assert lrow[i] == lse[h, t]


def test_prefill_rejects_bad_boundary():
    inp = wl.prefill_inputs((4, 4), 2, 1, 8, seed=1)
    with pytest.raises(ValueError):
        oracle.packed_prefill(inp.q, inp.k, inp.v, np.array([0, 5, 3]), 1.0)
    with pytest.raises(ValueError):
        oracle.packed_prefill(inp.q, inp.k[:, :1].repeat(1, 3, 1), inp.v, inp.cu_seqlens.numpy(), 1.0)
