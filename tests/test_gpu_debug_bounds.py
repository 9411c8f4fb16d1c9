"""The debug-bounds build on the tiny workload and the edge shapes (GPU).

``libslm_attn_debug.so`` is the library built with ``-DSLM_DEBUG_BOUNDS``
(every index the attention kernels and the prefill schedule compute is
checked against its buffer; a failed check sets SLM_DEV_BOUNDS in the device
status word and skips the access, never trapping) and ``-DSLM_NVTX``.  It
stands in for a memory checker, which this pool does not offer.  On valid
inputs no check may fail, and the results must be those of the product
library bit for bit (the checks only read).
"""
import numpy as np
import pytest
import torch

from attention_packed_varlen_gb300 import _binding as slm
from attention_packed_varlen_gb300 import build, workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def libs():
    prod = slm.load(build.build())
    dbg = slm.load(build.build(debug=True))
    return prod, dbg


def with_lib(lib, fn):
    saved = slm._lib
    slm._lib = lib
    try:
        return fn()
    finally:
        slm._lib = saved


def bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy()


PREFILL_CASES = [
    ("tiny", None),
    ("edges", ((1, 0, 1, 2, 0, 63, 64, 65, 127, 128, 129, 191, 192, 255, 256, 257), 16, 8, 128)),
    ("mha", ((5, 130, 64, 1, 300), 8, 8, 64)),
    ("g4", ((100, 37, 260), 16, 4, 128)),
    ("g7", ((96, 33, 200, 1), 14, 2, 64)),
    ("long", ((2000,), 16, 8, 128)),
]


@pytest.mark.parametrize("name,case", PREFILL_CASES)
def test_prefill_debug_bounds_clean_and_identical(libs, name, case):
    prod, dbg = libs
    inp = (wl.prefill_workload_inputs(wl.TINY_PREFILL, seed=wl.workload_seed(1)) if case is None
           else wl.prefill_inputs(case[0], case[1], case[2], case[3], seed=sum(case[0]) + case[1]))
    dev = torch.device(DEV)
    q, k, v, cu = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), inp.cu_seqlens.to(dev)
    outs = []
    for lib in (prod, dbg):
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        T, Hq = q.shape[0], q.shape[1]
        lse = torch.empty((Hq, T), dtype=torch.float32, device=dev)
        o = with_lib(lib, lambda: slm.slm_packed_prefill_attn(q, k, v, cu, max(1, inp.max_seqlen), inp.softmax_scale,
                                                              lse=lse, dev_status=status))
        with_lib(lib, lambda: slm.slm_check_status(status))
        outs.append((bits(o), lse.cpu().numpy()))
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    np.testing.assert_array_equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("W,Lp,L_prev,Smax,hq,hkv,D", [
    (16, 129, 1, 3, 14, 2, 64),
    (400, 1024, 4, 5, 14, 2, 64),   # the prompt's key blocks split over CTAs
    (37, 1000, 2, 3, 4, 2, 128),
    (130, 1, 0, 2, 8, 8, 64),
])
def test_decode_debug_bounds_clean(libs, W, Lp, L_prev, Smax, hq, hkv, D):
    prod, dbg = libs
    d = wl.decode_inputs(W, Lp, L_prev, Smax, hq, hkv, D, seed=W + Lp)
    dev = torch.device(DEV)
    args = [t.to(dev) for t in (d.q, d.kp, d.vp, d.ks, d.vs, d.k_new, d.v_new, d.parent)]
    res = []
    for lib in (prod, dbg):
        ks_out = torch.zeros((W, Smax, hkv, D), dtype=torch.bfloat16, device=dev)
        vs_out = torch.zeros_like(ks_out)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        n = with_lib(lib, lambda: slm.slm_shared_prefix_decode_workspace_size(W, Lp, hq, hkv, D))
        ws = torch.zeros(max(n, 16), dtype=torch.uint8, device=dev) if n else None
        o = with_lib(lib, lambda: slm.slm_shared_prefix_decode_attn(*args, L_prev, d.softmax_scale, ks_out=ks_out,
                                                                    vs_out=vs_out, dev_status=status, workspace=ws))
        with_lib(lib, lambda: slm.slm_check_status(status))
        res.append((o.float().cpu().numpy(), bits(ks_out), bits(vs_out)))
    # the key split's merge order varies between calls, so O agrees to fp32
    # summation order (below one bf16 ulp); the reordered suffix exactly
    assert np.abs(res[0][0] - res[1][0]).max() <= 2.0 ** -6
    np.testing.assert_array_equal(res[0][1], res[1][1])
    np.testing.assert_array_equal(res[0][2], res[1][2])
