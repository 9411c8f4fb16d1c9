"""Pins for the shared-prefix decode oracle (CPU only).

The oracle follows section 3.2 of the article "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化":
O_b = Attention(Q_b, [prefix_K; suffix_K[b]], [prefix_V; suffix_V[b]]), with the
suffix reordered by parent index (sections 3.2, 3.3).  The oracle builds the
concatenation explicitly; the pins below check it against a two-state
online-softmax merge (the method's own formulation, written independently
here), the library attention routine, the prefill oracle's last row, and
closed forms.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_packed_varlen_gb300 import workloads as wl


def _f64(x):
    return x.to(torch.float64).numpy() if isinstance(x, torch.Tensor) else x


def _bits_to_f64(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def attention_state(q, keys, vals, scale):
    """(m, l, acc) of one query against a key list, unnormalised (numpy fp64)."""
    s = scale * keys @ q
    m = s.max()
    p = np.exp(s - m)
    return m, p.sum(), p @ vals


def merge_states(a, b):
    m = max(a[0], b[0])
    ca, cb = np.exp(a[0] - m), np.exp(b[0] - m)
    return m, a[1] * ca + b[1] * cb, a[2] * ca + b[2] * cb


@pytest.mark.parametrize("W,Lp,L_prev,Hq,Hkv,D", [
    (5, 9, 2, 14, 2, 64),
    (3, 1, 0, 4, 2, 16),
    (7, 33, 4, 6, 3, 32),
])
def test_decode_two_state_merge_equals_concatenation(W, Lp, L_prev, Hq, Hkv, D):
    inp = wl.decode_inputs(W, Lp, L_prev, L_prev + 2, Hq, Hkv, D, seed=31)
    o, lse, ks_out, vs_out = oracle.shared_prefix_decode(
        inp.q, inp.kp, inp.vp, inp.ks, inp.vs, inp.k_new, inp.v_new, inp.parent,
        inp.L_prev, inp.softmax_scale)
    q, kp, vp = _f64(inp.q), _f64(inp.kp), _f64(inp.vp)
    ks, vs = _f64(inp.ks), _f64(inp.vs)
    kn, vn = _f64(inp.k_new), _f64(inp.v_new)
    par = inp.parent.numpy()
    G = Hq // Hkv
    for b in range(W):
        for h in range(Hq):
            kv = h // G
            pre = attention_state(q[b, h], kp[:, kv], vp[:, kv], inp.softmax_scale)
            # suffix of beam b: its parent's history, then its own new row
            sk = np.concatenate([ks[par[b], :L_prev, kv], kn[b, kv][None]], axis=0)
            sv = np.concatenate([vs[par[b], :L_prev, kv], vn[b, kv][None]], axis=0)
            suf = attention_state(q[b, h], sk, sv, inp.softmax_scale)
            m, l, acc = merge_states(pre, suf)
            np.testing.assert_allclose(o[b, h], acc / l, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[b, h], m + np.log(l), rtol=0, atol=1e-12)


def test_decode_suffix_reorder_rows():
    W, L_prev, Smax = 6, 3, 5
    inp = wl.decode_inputs(W, 4, L_prev, Smax, 4, 2, 16, seed=2)
    _, _, ks_out, vs_out = oracle.shared_prefix_decode(
        inp.q, inp.kp, inp.vp, inp.ks, inp.vs, inp.k_new, inp.v_new, inp.parent,
        inp.L_prev, inp.softmax_scale)
    ks_bits = inp.ks.view(torch.int16).numpy().view(np.uint16)
    vs_bits = inp.vs.view(torch.int16).numpy().view(np.uint16)
    kn_bits = inp.k_new.view(torch.int16).numpy().view(np.uint16)
    par = inp.parent.numpy()
    for b in range(W):
        # each output beam carries its parent's rows, untouched
        np.testing.assert_array_equal(ks_out[b, :L_prev], ks_bits[par[b], :L_prev])
        np.testing.assert_array_equal(vs_out[b, :L_prev], vs_bits[par[b], :L_prev])
        np.testing.assert_array_equal(ks_out[b, L_prev], kn_bits[b])
        assert not ks_out[b, L_prev + 1:].any()
    # the prefix is never part of the reorder: beams with the same parent share history
    same = [(a, c) for a in range(W) for c in range(W) if a < c and par[a] == par[c]]
    for a, c in same:
        np.testing.assert_array_equal(ks_out[a, :L_prev], ks_out[c, :L_prev])


def test_decode_matches_library_sdpa():
    W, Lp, L_prev, Hq, Hkv, D = 4, 17, 3, 14, 2, 64
    inp = wl.decode_inputs(W, Lp, L_prev, 5, Hq, Hkv, D, seed=8)
    o, _, ks_out, vs_out = oracle.shared_prefix_decode(
        inp.q, inp.kp, inp.vp, inp.ks, inp.vs, inp.k_new, inp.v_new, inp.parent,
        inp.L_prev, inp.softmax_scale)
    G = Hq // Hkv
    kso, vso = _bits_to_f64(ks_out), _bits_to_f64(vs_out)
    for b in range(W):
        kc = np.concatenate([_f64(inp.kp), kso[b, :L_prev + 1]], axis=0)   # [n, Hkv, D]
        vc = np.concatenate([_f64(inp.vp), vso[b, :L_prev + 1]], axis=0)
        qq = torch.from_numpy(_f64(inp.q)[b][:, None, :])                    # [Hq, 1, D]
        kk = torch.from_numpy(kc).repeat_interleave(G, dim=1).transpose(0, 1)
        vv = torch.from_numpy(vc).repeat_interleave(G, dim=1).transpose(0, 1)
        ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=inp.softmax_scale)
        np.testing.assert_allclose(o[b], ref[:, 0, :].numpy(), rtol=0, atol=1e-12)


def test_decode_single_beam_is_prefill_last_row():
    # W = 1: decode over [prefix; suffix] is the last row of causal prefill over
    # that sequence (the last query sees every key).
    Lp, L_prev, Hq, Hkv, D = 10, 2, 4, 2, 32
    inp = wl.decode_inputs(1, Lp, L_prev, 4, Hq, Hkv, D, seed=6, identity_parent=True)
    o, lse, _, _ = oracle.shared_prefix_decode(
        inp.q, inp.kp, inp.vp, inp.ks, inp.vs, inp.k_new, inp.v_new, None,
        inp.L_prev, inp.softmax_scale)
    k = torch.cat([inp.kp, inp.ks[0, :L_prev], inp.k_new])
    v = torch.cat([inp.vp, inp.vs[0, :L_prev], inp.v_new])
    T = k.shape[0]
    q = torch.zeros(T, Hq, D, dtype=torch.bfloat16)
    q[-1] = inp.q[0]
    op, lsep = oracle.packed_prefill(q, k, v, np.array([0, T]), inp.softmax_scale, want_lse=True)
    np.testing.assert_allclose(o[0], op[-1], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0], lsep[:, -1], rtol=0, atol=1e-13)


def test_decode_only_new_key_returns_new_value():
    # closed form: no prefix, no history -> each beam attends to its own new row
    inp = wl.decode_inputs(5, 0, 0, 1, 4, 2, 16, seed=12)
    o, lse, _, _ = oracle.shared_prefix_decode(
        inp.q, inp.kp, inp.vp, inp.ks, inp.vs, inp.k_new, inp.v_new, inp.parent,
        0, inp.softmax_scale)
    vn = _f64(inp.v_new)
    for h in range(4):
        np.testing.assert_array_equal(o[:, h], vn[:, h // 2])


def test_decode_identity_parent_without_history_is_plain_attention():
    # parent = identity and L_prev = 0 reduce to single-query attention over
    # [prefix; new row]; checked against the dense formula directly.
    W, Lp, Hq, Hkv, D = 3, 12, 2, 1, 8
    inp = wl.decode_inputs(W, Lp, 0, 1, Hq, Hkv, D, seed=13, identity_parent=True)
    o, _, _, _ = oracle.shared_prefix_decode(
        inp.q, inp.kp, inp.vp, inp.ks, inp.vs, inp.k_new, inp.v_new, None, 0, inp.softmax_scale)
    for b in range(W):
        kc = np.concatenate([_f64(inp.kp)[:, 0], _f64(inp.k_new)[b]], axis=0)
        vc = np.concatenate([_f64(inp.vp)[:, 0], _f64(inp.v_new)[b]], axis=0)
        for h in range(Hq):
            s = inp.softmax_scale * kc @ _f64(inp.q)[b, h]
            p = np.exp(s - s.max()); p /= p.sum()
            np.testing.assert_allclose(o[b, h], p @ vc, rtol=0, atol=1e-13)


def test_decode_rejects_bad_parent():
    inp = wl.decode_inputs(4, 3, 1, 2, 2, 1, 8, seed=1)
    bad = torch.tensor([0, 1, 4, 2], dtype=torch.int32)
    with pytest.raises(ValueError):
        oracle.shared_prefix_decode(inp.q, inp.kp, inp.vp, inp.ks, inp.vs, inp.k_new,
                                    inp.v_new, bad, 1, 1.0)
