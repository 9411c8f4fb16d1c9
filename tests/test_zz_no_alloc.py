"""GPU test of slm_packed_prefill_attn_noalloc, the prefill entry point for
callers that cannot allocate device memory where they run attention (for
example code inside a frozen, ahead-of-time compiled graph with a fixed memory
plan, or a host that owns every allocation).  Instead of a caller workspace it
keeps its tile schedule in a fixed array of the library's own device memory.

The test calls it through the C ABI twice in a row, on different inputs, and
checks each output against the workspace entry point slm_packed_prefill_attn
on the same inputs, within the attention tolerance of the parity tests (the
two run the same kernels, so they are expected to agree exactly), and against
the CPU oracle, so that a fault in the schedule both share cannot pass.  It
also checks that a request too large for the built-in array is refused
cleanly.
The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from attention_packed_varlen_gb300 import _binding as slm
from attention_packed_varlen_gb300 import build, workloads as wl
from tests.parity import check_attention, check_lse

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    build.build()
    return slm.load()


def _noalloc(lib, inp, out, lse):
    dev = torch.device(DEV)
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    cu = inp.cu_seqlens.to(dev)
    T, Hq, D = q.shape
    st = lib.slm_packed_prefill_attn_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(cu.data_ptr()), None, len(inp.lengths), T, max(1, inp.max_seqlen), Hq, k.shape[1], D,
        inp.softmax_scale, ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()), None,
        ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    assert st == slm.SLM_OK, lib.slm_last_error().decode()
    return q, k, v, cu


def test_noalloc_prefill_matches_workspace_entry_point(lib):
    dev = torch.device(DEV)
    cases = [wl.prefill_workload_inputs(wl.PREFILL_ONLY_REQUEST, seed=wl.workload_seed(2)),
             wl.prefill_workload_inputs(wl.TINY_PREFILL, seed=wl.workload_seed(1))]
    for inp in cases:  # two calls in a row; the second must not see the first's schedule
        T, Hq, D = inp.q.shape
        out = torch.full((T, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full((Hq, T), float("nan"), dtype=torch.float32, device=dev)
        q, k, v, cu = _noalloc(lib, inp, out, lse)
        ref_lse = torch.empty_like(lse)
        ref = slm.slm_packed_prefill_attn(q, k, v, cu, max(1, inp.max_seqlen), inp.softmax_scale, lse=ref_lse)
        torch.cuda.synchronize()
        a, b = out.float().cpu().numpy(), ref.float().cpu().numpy()
        assert np.isfinite(a).all()
        err = np.abs(a - b)
        assert err.max() <= 1e-2 and err.mean() <= 1e-3, (err.max(), err.mean())
        assert np.abs(lse.cpu().numpy() - ref_lse.cpu().numpy()).max() <= 1e-4
        o_ref, lse_ref = oracle.packed_prefill(inp.q, inp.k, inp.v, inp.cu_seqlens.numpy(), inp.softmax_scale,
                                               want_lse=True, n_threads=oracle.default_threads())
        check_attention(out.cpu(), o_ref, "no-allocation entry point vs oracle")
        check_lse(lse.cpu(), lse_ref, "no-allocation entry point vs oracle")


def test_noalloc_prefill_refuses_requests_beyond_its_buffer(lib):
    # 16 query / 8 KV heads: 64 tokens per sub-tile, so 4 million tokens in
    # one sequence need about 32,800 work items, above the 16,383 it holds
    st = lib.slm_packed_prefill_attn_noalloc(
        ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16), None, 1,
        4_194_304, 4_194_304, 16, 8, 128, 0.088, ctypes.c_void_p(32), None, None, None)
    assert st == 2
    assert b"built-in buffer" in lib.slm_last_error()
