"""The attention kernels' bounded waits run out without hanging (GPU).

Failure detection as the article "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化"
asks of the serving path (section 2.5: bounded waiting, never an unbounded
hang), tested without faulting the GPU: the wait limit is set to zero through
the C ABI, so every pipeline wait that is not already complete gives up at
once.  The call must return, the kernel must end early with the
pipeline-timeout bit in the device status word, and the next call with the
default limit must be correct again (the kernel drained its copies and MMAs
and freed its tensor memory).  Both the prefill kernel and the decode kernel
with the prompt's key blocks split over CTAs (whose tickets a unit that gave
up never takes) are covered.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_packed_varlen_gb300 import _binding as slm
from attention_packed_varlen_gb300 import build, workloads as wl
from tests.parity import check_attention

pytestmark = pytest.mark.gpu
DEV = "cuda"
TIMEOUT_BIT = 4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    slm.load()


class zero_wait_limit:
    def __enter__(self):
        self.prev = slm.slm_set_wait_timeout_ns(0)
        return self

    def __exit__(self, *exc):
        assert slm.slm_set_wait_timeout_ns(self.prev) == 0


def test_prefill_wait_timeout_returns_status_and_next_call_is_correct():
    inp = wl.prefill_workload_inputs(wl.PREFILL_ONLY_REQUEST, seed=wl.workload_seed(2))
    dev = torch.device(DEV)
    q, k, v, cu = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), inp.cu_seqlens.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    with zero_wait_limit():
        slm.slm_packed_prefill_attn(q, k, v, cu, inp.max_seqlen, inp.softmax_scale, dev_status=status)
        torch.cuda.synchronize()  # returns: the kernel ended
    assert int(status.item()) & TIMEOUT_BIT
    with pytest.raises(slm.SlmError) as e:
        slm.slm_check_status(status)
    assert b"pipeline-timeout" in slm.load().slm_last_error()
    # the default limit again: a normal, correct result
    status.zero_()
    o = slm.slm_packed_prefill_attn(q, k, v, cu, inp.max_seqlen, inp.softmax_scale, dev_status=status)
    slm.slm_check_status(status)
    ref = oracle.packed_prefill(inp.q, inp.k, inp.v, inp.cu_seqlens.numpy(), inp.softmax_scale,
                                n_threads=oracle.default_threads())
    check_attention(o, ref, "prefill after a timed-out call")


def test_split_decode_wait_timeout_returns_status_and_next_call_is_correct():
    W, Lp, L_prev, Hq, Hkv, D = 400, 1024, 2, 14, 2, 64
    d = wl.decode_inputs(W, Lp, L_prev, L_prev + 1, Hq, Hkv, D, seed=41)
    dev = torch.device(DEV)
    args = [t.to(dev) for t in (d.q, d.kp, d.vp, d.ks, d.vs, d.k_new, d.v_new, d.parent)]
    ks_out = torch.zeros((W, L_prev + 1, Hkv, D), dtype=torch.bfloat16, device=dev)
    vs_out = torch.zeros_like(ks_out)
    n = slm.slm_shared_prefix_decode_workspace_size(W, Lp, Hq, Hkv, D)
    assert n > 0
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    with zero_wait_limit():
        ws = torch.zeros(n, dtype=torch.uint8, device=dev)
        slm.slm_shared_prefix_decode_attn(*args, L_prev, d.softmax_scale, ks_out=ks_out, vs_out=vs_out,
                                          dev_status=status, workspace=ws)
        torch.cuda.synchronize()
    assert int(status.item()) & TIMEOUT_BIT
    with pytest.raises(slm.SlmError):
        slm.slm_check_status(status)
    # a fresh zero-filled workspace (the timed-out call may have left tickets
    # taken), default limit: the oracle's result
    status.zero_()
    ws = torch.zeros(n, dtype=torch.uint8, device=dev)
    o = slm.slm_shared_prefix_decode_attn(*args, L_prev, d.softmax_scale, ks_out=ks_out, vs_out=vs_out,
                                          dev_status=status, workspace=ws)
    slm.slm_check_status(status)
    ref, _, ks_ref, _ = oracle.shared_prefix_decode(d.q, d.kp, d.vp, d.ks, d.vs, d.k_new, d.v_new, d.parent, L_prev,
                                                    d.softmax_scale, n_threads=oracle.default_threads())
    check_attention(o, ref, "decode after a timed-out call")
    np.testing.assert_array_equal(ks_out.cpu().view(torch.int16).numpy().view(np.uint16), ks_ref)
    # the workspace is fit for the next call again
    assert not ws[:4 * 16384].view(torch.int32).any()
