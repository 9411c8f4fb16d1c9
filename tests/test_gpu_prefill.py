"""GPU parity of slm_packed_prefill_attn against the fp64 oracle.

Packed causal GQA attention (article "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化",
section 3.1) on the seeded workloads and on edge cases: empty and one-token
sequences, tails of every length around the 64-token tile and the 128-key
block, one long sequence, head groups of 1, 2, 4 and 7, large score ranges
that force the running-max rescale, and a malformed boundary.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_packed_varlen_gb300 import _binding as slm
from attention_packed_varlen_gb300 import build, workloads as wl
from tests.parity import check_attention, check_lse

pytestmark = pytest.mark.gpu
DEV = "cuda"
THREADS = oracle.default_threads()


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    slm.load()


def run_gpu(inp, want_lse=True, fp32=False):
    dev = torch.device(DEV)
    T, Hq = inp.q.shape[0], inp.q.shape[1]
    lse = torch.full((Hq, T), float("nan"), device=dev) if want_lse else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    fn = slm.slm_packed_prefill_attn_f32 if fp32 else slm.slm_packed_prefill_attn
    o = fn(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), inp.cu_seqlens.to(dev), max(1, inp.max_seqlen),
           inp.softmax_scale, lse=lse, dev_status=status, cu_seqlens_host=inp.cu_seqlens)
    slm.slm_check_status(status)
    return o, lse


def oracle_with_weights(inp):
    """The oracle's O and LSE, and sum_j w_j |v_j| per output (the oracle on |V|)."""
    cu = inp.cu_seqlens.numpy()
    ref, ref_lse = oracle.packed_prefill(inp.q, inp.k, inp.v, cu, inp.softmax_scale, want_lse=True,
                                         n_threads=THREADS)
    wabs = oracle.packed_prefill(inp.q, inp.k, inp.v.abs(), cu, inp.softmax_scale, n_threads=THREADS)
    return ref, ref_lse, wabs


def full_check(inp, what):
    o, lse = run_gpu(inp)
    ref, ref_lse, wabs = oracle_with_weights(inp)
    check_attention(o, ref, what, weighted_abs_v=wabs)
    check_lse(lse, ref_lse, what)
    # the same kernels with an fp32 output: the max-abs 1e-2 / mean-abs 1e-3 gate on the arithmetic
    o32, lse32 = run_gpu(inp, fp32=True)
    err_max, err_mean = check_attention(o32, ref, what + " (fp32 output)", fp32_gate=True)
    check_lse(lse32, ref_lse, what + " (fp32 output)")
    # the bf16 output is the fp32 result rounded once to nearest
    np.testing.assert_array_equal(o.cpu().view(torch.int16).numpy(),
                                  o32.cpu().to(torch.bfloat16).view(torch.int16).numpy())
    print(f"{what}: fp32 output max-abs {err_max:.3g}, mean-abs {err_mean:.3g}")


def test_tiny_packed_prefill_workload():
    inp = wl.prefill_workload_inputs(wl.TINY_PREFILL, seed=wl.workload_seed(1))
    full_check(inp, "tiny")


def test_prefill_only_request_workload():
    inp = wl.prefill_workload_inputs(wl.PREFILL_ONLY_REQUEST, seed=wl.workload_seed(2))
    full_check(inp, "prefill-only request")


@pytest.mark.parametrize("lengths,hq,hkv,d", [
    ((1, 0, 1, 2, 0, 63, 64, 65, 127, 128, 129, 191, 192, 255, 256, 257), 16, 8, 128),
    ((5, 130, 64, 1, 300), 8, 8, 64),            # G = 1 (MHA)
    ((100, 37, 260), 16, 4, 128),                # G = 4
    ((96, 33, 200, 1), 14, 2, 64),               # G = 7: 18 tokens x 7 heads = 126 rows per tile
    ((2000,), 16, 8, 128),                       # one long sequence: 16 key blocks
    ((1,), 4, 2, 64),                            # a single token
])
def test_prefill_edge_shapes(lengths, hq, hkv, d):
    inp = wl.prefill_inputs(lengths, hq, hkv, d, seed=sum(lengths) + hq)
    full_check(inp, f"{lengths} {hq}/{hkv} D={d}")


def test_prefill_large_score_range_rescales():
    # q scaled up: scores span tens of units, so the running max jumps by more
    # than the lazy-rescale threshold across key blocks and O is rescaled in
    # TMEM.  The softmax is then so peaked that the bf16 rounding of P bounds
    # the error (tests/parity.check_attention states the bound).
    inp = wl.prefill_inputs((700, 300, 129), 16, 8, 128, seed=77)
    inp.q = (inp.q.float() * 6.0).to(torch.bfloat16)
    o, lse = run_gpu(inp)
    ref, ref_lse, wabs = oracle_with_weights(inp)
    check_attention(o, ref, "large scores", weighted_abs_v=wabs)
    check_lse(lse, ref_lse, "large scores")
    # fp32 output: within the bf16 rounding of the weights P, 2^-8 sum_j w_j |v_j|
    o32, _ = run_gpu(inp, fp32=True)
    err = np.abs(o32.cpu().numpy().astype(np.float64) - ref)
    assert (err <= 2.0 ** -8 * wabs + 1e-4).all(), err.max()


def test_concurrent_batch_sampled_rows():
    # one layer of the 240-sequence concurrent batch at full size; the oracle
    # computes sampled rows one by one: random rows plus every row of the
    # first and last tile of a few sequences
    inp = wl.prefill_workload_inputs(wl.CONCURRENT_PREFILL_BATCH, seed=wl.workload_seed(3))
    o, lse = run_gpu(inp)
    T, Hq = inp.q.shape[0], inp.q.shape[1]
    rng = np.random.default_rng(0)
    rows = [np.stack([rng.integers(0, T, 3000), rng.integers(0, Hq, 3000)], axis=1)]
    cu = inp.cu_seqlens.numpy()
    for b in (0, 1, len(cu) // 2, len(cu) - 2):
        for t in list(range(cu[b], min(cu[b] + 64, cu[b + 1]))) + list(range(max(cu[b], cu[b + 1] - 64), cu[b + 1])):
            rows.append(np.array([[t, h] for h in range(Hq)]))
    rows = np.concatenate(rows)
    ref, ref_lse = oracle.packed_prefill_rows(inp.q, inp.k, inp.v, cu, inp.softmax_scale, rows, n_threads=THREADS)
    got = o[torch.from_numpy(rows[:, 0]).to(o.device), torch.from_numpy(rows[:, 1]).to(o.device)]
    check_attention(got, ref, "concurrent batch (sampled)")
    check_lse(lse[torch.from_numpy(rows[:, 1]).to(o.device), torch.from_numpy(rows[:, 0]).to(o.device)],
              ref_lse, "concurrent batch lse")
    # property over every row: finite, and |O| bounded by the largest |V| of the head
    assert torch.isfinite(o.float()).all()
    assert o.float().abs().max() <= inp.v.float().abs().max() * 1.01


def test_prefill_bad_boundary_sets_device_status():
    inp = wl.prefill_inputs((10, 10, 10), 4, 2, 64, seed=1)
    dev = torch.device(DEV)
    cu = torch.tensor([0, 20, 10, 30], dtype=torch.int32, device=dev)   # decreasing
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    slm.slm_packed_prefill_attn(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), cu, 30, 0.125, dev_status=status)
    with pytest.raises(slm.SlmError) as e:
        slm.slm_check_status(status)
    assert e.value.status == 5 and int(status.item()) & 1


def test_prefill_repeatable():
    # the prefill has no order-dependent reduction: repeated calls agree bit
    # for bit (a race in the pipeline would show up as a call that differs)
    inp = wl.prefill_workload_inputs(wl.PREFILL_ONLY_REQUEST, seed=5)
    a, _ = run_gpu(inp, want_lse=False)
    for _ in range(10):
        b, _ = run_gpu(inp, want_lse=False)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
