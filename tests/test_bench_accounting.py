"""The benchmark's algorithmic FLOP and byte counts (the numerators of its
roofline fractions), checked on the CPU against counts made another way:
enumerated causal pairs, element counts of the tensors each call must read and
write, and the workloads' own sizes."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from attention_packed_varlen_gb300 import workloads as wl  # noqa: E402


def test_prefill_flops_count_the_causal_pairs():
    lengths = [1, 5, 64, 130]
    Hq, D = 4, 64
    pairs = sum(int(np.tril(np.ones((L, L))).sum()) for L in lengths)  # (query, key) with key <= query
    # QK^T and PV: 2 multiply-adds of length D per pair = 4 D flops
    assert bench.prefill_flops(lengths, Hq, D) == 4 * D * pairs * Hq


def test_concurrent_batch_sizes():
    L = wl.draw_lengths(240, 64, 1024, bench.PREFILL_SEED)
    T = int(np.sum(L))
    assert T == 130794
    assert abs(bench.prefill_flops(L, 16, 128) - 368.7e9) < 0.05e9
    # Q, K, V read once, O written once, bf16
    elems = T * 16 * 128 + T * 8 * 128 + T * 8 * 128 + T * 16 * 128
    assert bench.prefill_bytes(T, 16, 8, 128) == elems * 2
    assert abs(bench.prefill_bytes(T, 16, 8, 128) - 1.607e9) < 0.001e9


def test_selection_reads_the_logits_once():
    assert bench.select_bytes(400, 151936) == 400 * 151936 * 2
    assert bench.select_bytes(1, 151936) == 151936 * 2


def test_decode_bytes_are_the_tensors_the_call_moves():
    W, Lp, L_prev, Hq, Hkv, D = 400, 1024, 4, 14, 2, 64
    row = Hkv * D  # one token's K (or V) row over the KV heads, elements
    reads = (W * Hq * D                        # q
             + 2 * Lp * row                    # prompt K and V
             + 2 * W * L_prev * row            # each beam's parent history, K and V
             + 2 * W * row)                    # the new rows
    writes = W * Hq * D + 2 * W * (L_prev + 1) * row  # o and the reordered suffix
    assert bench.decode_attn_bytes(W, Lp, L_prev, Hq, Hkv, D) == (reads + writes) * 2
    assert abs(bench.decode_attn_bytes(W, Lp, L_prev, Hq, Hkv, D) - 4.0e6) < 0.01e6
    assert abs(bench.decode_attn_bytes(100, 96, 3, Hq, Hkv, D) - 0.82e6) < 0.01e6


def test_loop_bytes_sum_its_steps():
    bw = wl.LONG_PROMPT_WIDE_BEAM
    want = 151936 * 2 + sum(
        bench.decode_attn_bytes(bw.beams, bw.prefix_len, t, bw.n_q_heads, bw.n_kv_heads, bw.head_dim)
        + bw.beams * 151936 * 2 for t in range(bw.steps))
    assert bench.loop_bytes(bw) == want


def test_selection_launch_count_follows_the_fused_path():
    # stream + select while the group keys fit the select kernel's shared
    # memory (rows of at most 64 tiles of 8192, at most 16,384 groups); a
    # row-statistics kernel in between otherwise
    assert bench.select_launches(100, 151936, 100) == 2      # 1,900 tile groups
    assert bench.select_launches(400, 151936, 400) == 2      # 7,600 tile groups
    assert bench.select_launches(1, 151936, 400) == 2        # 19 tiles < 2W: 2,432 sub-chunk groups
    assert bench.select_launches(900, 151936, 200) == 3      # 17,100 tile groups
    assert bench.select_launches(8, 151936, 100) == 3        # 152 tiles < 2W: 19,456 sub-chunk groups
    assert bench.select_launches(2, 600000, 2) == 3          # 74 tiles per row
    # the loops' launch counts: first step (selection + history), then per
    # step attention + selection + history
    bw = wl.LONG_PROMPT_WIDE_BEAM
    per_step = 1 + bench.select_launches(bw.beams, bw.vocab, bw.beams) + 1
    assert bench.select_launches(1, bw.vocab, bw.beams) + 1 + bw.steps * per_step == 23
