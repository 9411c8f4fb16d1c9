"""GPU parity of slm_beam_select against the oracle's full W x V sort:
bit-exact given the GPU's own fp32 log-normalisers, and every difference from
the oracle's own ranking explained by the normalisers' few-ulp difference.

Two-stage candidate selection (article "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化",
section 3.3) on the two beam workloads at full size (V = 151,936), the first
step (one row), heavy ties (few distinct logits, all-equal rows), a
vocabulary that is not a multiple of 8, 2W = V, W = 1, rows long enough for
the three-kernel path, and a dominant token that pushes the threshold far
below the largest score.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_packed_varlen_gb300 import _binding as slm
from attention_packed_varlen_gb300 import build, workloads as wl
from tests.parity import check_selection

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    slm.load()


def run_and_check(logits, cum, W):
    dev = torch.device(DEV)
    res = slm.slm_beam_select(logits.to(dev), cum.to(dev), W)
    torch.cuda.synchronize()
    near, _ = check_selection(res, oracle.beam_select(logits, cum, 2 * W), logits, cum, W)
    return res, near


@pytest.mark.parametrize("workload,index", [(wl.SHORT_PROMPT_BEAM, 4), (wl.LONG_PROMPT_WIDE_BEAM, 5)])
def test_beam_workload_selection(workload, index):
    s = wl.select_inputs(workload.beams, workload.vocab, workload.beams, seed=wl.workload_seed(index, 1), step=1)
    _, near = run_and_check(s.logits, s.cum, workload.beams)
    print(f"{workload.name}: {near} near ties against the oracle's own normalisers, all explained")


@pytest.mark.parametrize("W", [100, 400])
def test_first_step_single_row(W):
    s = wl.select_inputs(1, 151936, W, seed=W, step=0)
    run_and_check(s.logits, s.cum, W)


@pytest.mark.parametrize("W_in,V,W,levels", [(8, 1000, 8, 5), (6, 40000, 6, 3), (3, 70000, 3, 1)])
def test_heavy_ties(W_in, V, W, levels):
    logits = wl.quantized_logits(W_in, V, levels=levels, seed=V)
    cum = torch.zeros(W_in, dtype=torch.float32)
    cum[W_in // 2:] = -0.5
    run_and_check(logits, cum, W)


@pytest.mark.parametrize("W_in,V,W", [(5, 1001, 5), (8, 16, 8), (4, 20000, 1), (32, 50000, 32)])
def test_odd_sizes(W_in, V, W):
    s = wl.select_inputs(W_in, V, W, seed=V + W)
    run_and_check(s.logits, s.cum, W)


def test_select_repeatable():
    s = wl.select_inputs(100, 151936, 100, seed=9)
    dev = torch.device(DEV)
    a = slm.slm_beam_select(s.logits.to(dev), s.cum.to(dev), 100)
    b = slm.slm_beam_select(s.logits.to(dev), s.cum.to(dev), 100)
    for key in a:
        assert torch.equal(a[key], b[key]), key


def test_sampled_threshold_miss():
    # A row whose few very large logits sit exactly where the threshold's
    # sample looks: the sample then overstates the row's top, fewer than 2W
    # logits pass the threshold, and the beam must be redone exactly.  The
    # sample positions are those of the 16-byte runs the selection reads
    # (512 runs of 8 logits, evenly spaced, 8-aligned).
    W_in, V, W = 8, 151936, 100
    s = wl.select_inputs(W_in, V, W, seed=77)
    logits = s.logits.clone()
    runs = [(j * (V - 8) // 511) & ~7 for j in range(30)]
    for b in range(W_in):
        logits[b, runs] = 20.0
    run_and_check(logits, s.cum, W)


@pytest.mark.parametrize("W_in,V,W", [(2, 600000, 2), (1, 600000, 50)])
def test_long_rows_three_kernel_path(W_in, V, W):
    # Rows of more than 64 tiles of 8192 take the path with the separate
    # row-statistics kernel and the global histogram: tile groups (2 rows,
    # 4 candidates) and sub-chunk groups (one row, 100 candidates).
    s = wl.select_inputs(W_in, V, W, seed=V + W_in)
    run_and_check(s.logits, s.cum, W)


@pytest.mark.parametrize("W_in,W", [(1, 100), (100, 100)])
def test_dominant_token_threshold_far_below_top(W_in, W):
    # One logit per row far above the rest, and a zero cumulative score for
    # beam 0: its candidate scores exactly 0 (the log-normaliser rounds to
    # the dominant logit), while the 2W-th group key lies near -50, dozens of
    # binades further down and outside the select kernel's shared histogram
    # window, so the threshold is taken by exact radix selection instead.
    V = 151936
    s = wl.select_inputs(W_in, V, W, seed=31 + W_in, step=0 if W_in == 1 else 1)
    logits = s.logits.clone()
    cols = torch.arange(W_in) * 997 % V
    logits[torch.arange(W_in), cols] = 60.0
    cum = s.cum.clone()
    cum[0] = 0.0
    res, _ = run_and_check(logits, cum, W)
    kept = set(zip(res["parent"].cpu().tolist(), res["token"].cpu().tolist()))
    assert all((b, int(cols[b])) in kept for b in range(W_in))
