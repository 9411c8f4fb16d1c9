"""GPU parity of slm_shared_prefix_decode_attn against the fp64 oracle.

Shared-prefix beam decode (article "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化",
sections 3.2-3.3): every step of the two beam workloads, chained so that each
step's reordered suffix feeds the next, plus edge cases (no prefix, a prefix
that is not a multiple of the 128-key block, one beam, no appended row,
identity parents, head_dim 128) and an out-of-range parent index.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_packed_varlen_gb300 import _binding as slm
from attention_packed_varlen_gb300 import build, workloads as wl
from tests.parity import bf16_ulp, check_attention, check_lse

pytestmark = pytest.mark.gpu
DEV = "cuda"
THREADS = oracle.default_threads()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    slm.load()


def bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def run_step(d, ks_dev, vs_dev, Smax, with_new=True, parent=True, workspace=None, fp32=False):
    dev = torch.device(DEV)
    W, Hq, D = d.q.shape
    Hkv = d.kp.shape[1] if d.kp is not None else d.k_new.shape[1]
    ks_out = torch.zeros((W, Smax, Hkv, D), dtype=torch.bfloat16, device=dev)
    vs_out = torch.zeros_like(ks_out)
    lse = torch.empty((W, Hq), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kp = d.kp.to(dev) if d.kp.shape[0] > 0 else None
    vp = d.vp.to(dev) if d.vp.shape[0] > 0 else None
    fn = slm.slm_shared_prefix_decode_attn_f32 if fp32 else slm.slm_shared_prefix_decode_attn
    o = fn(
        d.q.to(dev), kp, vp, ks_dev, vs_dev,
        d.k_new.to(dev) if with_new else None, d.v_new.to(dev) if with_new else None,
        d.parent.to(dev) if parent else None, d.L_prev, d.softmax_scale,
        ks_out=ks_out, vs_out=vs_out, lse=lse, dev_status=status, workspace=workspace)
    slm.slm_check_status(status)
    return o, lse, ks_out, vs_out


def check_step(d, ks_host, vs_host, o, lse, ks_out, vs_out, what, with_new=True, parent=True, o32=None):
    args = (d.k_new if with_new else None, d.v_new if with_new else None, d.parent if parent else None,
            d.L_prev, d.softmax_scale)
    ref, ref_lse, ks_ref, vs_ref = oracle.shared_prefix_decode(d.q, d.kp, d.vp, ks_host, vs_host, *args,
                                                               n_threads=THREADS)
    # sum_j w_j |v_j| per output: the oracle with |V| everywhere
    absv = lambda t: None if t is None else t.abs()
    wabs, _, _, _ = oracle.shared_prefix_decode(d.q, d.kp, absv(d.vp), ks_host, absv(vs_host), args[0],
                                                absv(args[1]), *args[2:], n_threads=THREADS)
    check_attention(o, ref, what, weighted_abs_v=wabs)
    check_lse(lse, ref_lse, what)
    if o32 is not None:  # the fp32 output of the same kernels: the 1e-2 / 1e-3 gate, and o is its rounding
        check_attention(o32, ref, what + " (fp32 output)", fp32_gate=True)
        # within one bf16 ulp of the fp32 result rounded: the last split to
        # arrive merges the key splits, so their fp32 summation order varies
        # between calls (measured run to run: below 1e-7 absolute, which near
        # zero is several bf16 ulps, hence the 2^-20 absolute term)
        r32 = o32.cpu().to(torch.bfloat16).float().numpy().astype(np.float64)
        ob = o.cpu().float().numpy().astype(np.float64)
        gap = np.abs(ob - r32)
        lim = bf16_ulp(np.maximum(np.abs(ob), np.abs(r32))) + 2.0 ** -20
        k = np.unravel_index((gap / lim).argmax(), gap.shape)
        assert (gap <= lim).all(), (what, k, ob[k], float(o32.cpu()[k]), ref[k], gap[k] / lim[k])
    Ls = d.L_prev + (1 if with_new else 0)
    np.testing.assert_array_equal(bits(ks_out)[:, :Ls], ks_ref[:, :Ls], err_msg=f"{what}: K suffix reorder")
    np.testing.assert_array_equal(bits(vs_out)[:, :Ls], vs_ref[:, :Ls], err_msg=f"{what}: V suffix reorder")


@pytest.mark.parametrize("workload,index", [(wl.SHORT_PROMPT_BEAM, 4), (wl.LONG_PROMPT_WIDE_BEAM, 5)])
def test_beam_workload_all_steps_chained(workload, index):
    W, Smax = workload.beams, workload.max_suffix
    dev = torch.device(DEV)
    ks_dev = vs_dev = None
    ks_host = vs_host = None
    for step in range(workload.steps):
        d = wl.decode_inputs(W, workload.prefix_len, step, Smax, workload.n_q_heads, workload.n_kv_heads,
                             workload.head_dim, seed=wl.workload_seed(index, step))
        # the prompt K/V is the same every step: one copy per request
        base = wl.decode_inputs(W, workload.prefix_len, 0, Smax, workload.n_q_heads, workload.n_kv_heads,
                                workload.head_dim, seed=wl.workload_seed(index, 0))
        d.kp, d.vp = base.kp, base.vp
        if step == 0:
            ks_host, vs_host = d.ks, d.vs
            ks_dev, vs_dev = ks_host.to(dev), vs_host.to(dev)
        o, lse, ks_out, vs_out = run_step(d, ks_dev, vs_dev, Smax)
        o32 = run_step(d, ks_dev, vs_dev, Smax, fp32=True)[0]
        check_step(d, ks_host, vs_host, o, lse, ks_out, vs_out, f"{workload.name} step {step}", o32=o32)
        # the next step reads this step's reordered suffix
        ks_dev, vs_dev = ks_out, vs_out
        ks_host, vs_host = ks_out.cpu(), vs_out.cpu()


@pytest.mark.parametrize("W,Lp,L_prev,Smax,hq,hkv,D,with_new,parent", [
    (16, 0, 2, 4, 14, 2, 64, True, True),       # no prefix: suffix only
    (16, 129, 1, 3, 14, 2, 64, True, True),     # prefix spills into a second key block
    (1, 96, 3, 5, 14, 2, 64, True, True),       # one beam
    (40, 64, 3, 5, 14, 2, 64, False, True),     # nothing appended
    (40, 64, 0, 1, 14, 2, 64, True, False),     # identity parents, no history
    (3, 200, 2, 4, 4, 2, 128, True, True),      # head_dim 128, fewer beams than a tile
    (130, 1, 0, 2, 8, 8, 64, True, True),       # MHA, a one-token prompt, several tiles
])
def test_decode_edge_cases(W, Lp, L_prev, Smax, hq, hkv, D, with_new, parent):
    d = wl.decode_inputs(W, Lp, L_prev, Smax, hq, hkv, D, seed=W + Lp + L_prev, identity_parent=not parent)
    dev = torch.device(DEV)
    o, lse, ks_out, vs_out = run_step(d, d.ks.to(dev), d.vs.to(dev), Smax, with_new=with_new, parent=parent)
    o32 = run_step(d, d.ks.to(dev), d.vs.to(dev), Smax, with_new=with_new, parent=parent, fp32=True)[0]
    check_step(d, d.ks, d.vs, o, lse, ks_out, vs_out, f"W={W} Lp={Lp} L_prev={L_prev}", with_new, parent, o32=o32)


@pytest.mark.parametrize("W,Lp,L_prev,hq,hkv,D", [
    (400, 1024, 4, 14, 2, 64),     # the wide beam's last step: 8 key blocks over 24 tiles x heads
    (37, 1000, 2, 4, 2, 128),      # head_dim 128, a ragged last key block
    (5, 2000, 1, 8, 8, 64),        # MHA: more splits than the SMs need
])
def test_decode_key_split_matches_oracle_and_unsplit(W, Lp, L_prev, hq, hkv, D):
    # the prompt's key blocks split over CTAs (workspace of the library's size) and
    # not split (empty workspace) give the oracle's result; the two differ only by
    # fp32 summation order
    Smax = L_prev + 1
    assert slm.slm_shared_prefix_decode_workspace_size(W, Lp, hq, hkv, D) > 0
    d = wl.decode_inputs(W, Lp, L_prev, Smax, hq, hkv, D, seed=W * 7 + Lp)
    dev = torch.device(DEV)
    outs = {}
    for name, ws in (("split", None), ("unsplit", torch.empty(0, dtype=torch.uint8, device=dev))):
        o, lse, ks_out, vs_out = run_step(d, d.ks.to(dev), d.vs.to(dev), Smax, workspace=ws)
        check_step(d, d.ks, d.vs, o, lse, ks_out, vs_out, f"{name} W={W} Lp={Lp}")
        outs[name] = o.float()
    assert (outs["split"] - outs["unsplit"]).abs().max().item() < 2e-2


def test_decode_workspace_serves_calls_of_other_shapes_and_too_small_runs_unsplit():
    # one zero-filled workspace, sized for the widest call, serves calls of other
    # shapes in turn (a completed call leaves its tickets at zero again); a
    # workspace far too small is ignored and the call runs unsplit
    dev = torch.device(DEV)
    ws = torch.zeros(slm.slm_shared_prefix_decode_workspace_size(400, 1024, 14, 2, 64), dtype=torch.uint8,
                     device=dev)
    tiny = torch.zeros(256, dtype=torch.uint8, device=dev)
    for i, (W, Lp, L_prev, w) in enumerate(((400, 1024, 2, ws), (37, 300, 1, ws), (400, 1024, 0, ws),
                                             (130, 600, 3, ws), (400, 1024, 1, tiny))):
        d = wl.decode_inputs(W, Lp, L_prev, L_prev + 1, 14, 2, 64, seed=100 + i)
        o, lse, ks_out, vs_out = run_step(d, d.ks.to(dev), d.vs.to(dev), L_prev + 1, workspace=w)
        check_step(d, d.ks, d.vs, o, lse, ks_out, vs_out, f"call {i}: W={W} Lp={Lp} L_prev={L_prev}")


def test_decode_bad_parent_sets_device_status():
    d = wl.decode_inputs(8, 32, 1, 3, 14, 2, 64, seed=3)
    dev = torch.device(DEV)
    parent = d.parent.clone()
    parent[5] = 8                                  # == W: out of range
    ks_out = torch.zeros((8, 3, 2, 64), dtype=torch.bfloat16, device=dev)
    vs_out = torch.zeros_like(ks_out)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    slm.slm_shared_prefix_decode_attn(d.q.to(dev), d.kp.to(dev), d.vp.to(dev), d.ks.to(dev), d.vs.to(dev),
                                      d.k_new.to(dev), d.v_new.to(dev), parent.to(dev), 1, d.softmax_scale,
                                      ks_out=ks_out, vs_out=vs_out, dev_status=status)
    with pytest.raises(slm.SlmError):
        slm.slm_check_status(status)
    assert int(status.item()) & 2
