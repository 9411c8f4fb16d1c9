"""Seeded synthetic inputs for the attention hot path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic. Both the CUDA path (tests, bench) and the CPU oracle are
fed from here, so the two always see identical bf16 bit patterns.

Recipe (the pages ran on business traffic and print no data, so seeded draws
stand in for it):

* values: ``torch.Generator('cpu').manual_seed(seed)`` then fp32 ``randn``
  scaled by ``std`` and rounded to bf16 (round-to-nearest-even, torch's cast);
* sequence lengths: ``numpy.random.default_rng(seed)`` uniform integers with
  inclusive bounds;
* parent indices: uniform over ``0..W-1`` from the same numpy generator;
* cumulative beam scores at step ``t``: ``-sort(|N(0,1)|) * t`` in fp32,
  distinct and descending (a beam list as a previous selection leaves it).

Workload shapes follow the article "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化":
Prefill-Only requests of 15 samples with prompts of a few hundred tokens
(section 1.2 and 4.3), beam search with W about 100 (up to 400) beams and at
most 5 generated tokens over a 151,936-entry vocabulary (section 1.2, 3.3).
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np
import torch


# ----------------------------------------------------------------------------
# Named workloads
# ----------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    name: str
    lengths: Optional[Sequence[int]]  # fixed lengths, or None to draw
    n_seqs: int
    len_lo: int
    len_hi: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    layers: int = 1  # independent Q/K/V sets called back to back

    @property
    def softmax_scale(self) -> float:
        return 1.0 / float(self.head_dim) ** 0.5


@dataclasses.dataclass(frozen=True)
class BeamWorkload:
    name: str
    prefix_len: int
    beams: int
    steps: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    vocab: int = 151936
    logit_std: float = 3.0

    @property
    def softmax_scale(self) -> float:
        return 1.0 / float(self.head_dim) ** 0.5

    @property
    def max_suffix(self) -> int:
        return self.steps


TINY_PREFILL = PrefillWorkload(
    name="tiny packed prefill: L={37,64,91,128}, T=320, 4q/2kv, D=64",
    lengths=(37, 64, 91, 128), n_seqs=4, len_lo=0, len_hi=0,
    n_q_heads=4, n_kv_heads=2, head_dim=64)

PREFILL_ONLY_REQUEST = PrefillWorkload(
    name="Prefill-Only request: 15 seqs L~U[100,500], 16q/8kv, D=128",
    lengths=None, n_seqs=15, len_lo=100, len_hi=500,
    n_q_heads=16, n_kv_heads=8, head_dim=128)

CONCURRENT_PREFILL_BATCH = PrefillWorkload(
    name="concurrent Prefill-Only batch: 240 seqs L~U[64,1024], 16q/8kv, D=128, 28 layers",
    lengths=None, n_seqs=240, len_lo=64, len_hi=1024,
    n_q_heads=16, n_kv_heads=8, head_dim=128, layers=28)

SHORT_PROMPT_BEAM = BeamWorkload(
    name="short-prompt beam: Lp=96, W=100, 4 steps, 14q/2kv, D=64, V=151936",
    prefix_len=96, beams=100, steps=4, n_q_heads=14, n_kv_heads=2, head_dim=64)

LONG_PROMPT_WIDE_BEAM = BeamWorkload(
    name="long-prompt wide beam: Lp=1024, W=400, 5 steps, 14q/2kv, D=64, V=151936",
    prefix_len=1024, beams=400, steps=5, n_q_heads=14, n_kv_heads=2, head_dim=64)


def workload_seed(workload_index: int, step_or_layer: int = 0, k: int = 0) -> int:
    """Seed convention: 1000 * workload + 10 * layer_or_step + k."""
    return 1000 * workload_index + 10 * step_or_layer + k


# ----------------------------------------------------------------------------
# Primitive draws
# ----------------------------------------------------------------------------
def bf16_randn(shape, seed: int, std: float = 1.0) -> torch.Tensor:
    g = torch.Generator("cpu").manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(torch.bfloat16)


def draw_lengths(n: int, lo: int, hi: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(int(seed))
    return rng.integers(lo, hi + 1, size=n).astype(np.int64)


def cu_seqlens_from_lengths(lengths: Sequence[int]) -> torch.Tensor:
    """Sequence boundary: prefix sums of the lengths, int32 [B+1]."""
    cs = np.zeros(len(lengths) + 1, dtype=np.int64)
    cs[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return torch.from_numpy(cs.astype(np.int32))


# ----------------------------------------------------------------------------
# Packed prefill inputs
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class PrefillInputs:
    q: torch.Tensor  # bf16 [T, Hq, D]
    k: torch.Tensor  # bf16 [T, Hkv, D]
    v: torch.Tensor  # bf16 [T, Hkv, D]
    cu_seqlens: torch.Tensor  # int32 [B+1]
    lengths: np.ndarray
    softmax_scale: float

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def max_seqlen(self) -> int:
        return int(self.lengths.max()) if len(self.lengths) else 0


def prefill_inputs(lengths: Sequence[int], n_q_heads: int, n_kv_heads: int,
                   head_dim: int, seed: int, std: float = 1.0,
                   softmax_scale: Optional[float] = None) -> PrefillInputs:
    lengths = np.asarray(lengths, dtype=np.int64)
    T = int(lengths.sum())
    q = bf16_randn((T, n_q_heads, head_dim), seed * 4 + 1, std)
    k = bf16_randn((T, n_kv_heads, head_dim), seed * 4 + 2, std)
    v = bf16_randn((T, n_kv_heads, head_dim), seed * 4 + 3, std)
    scale = softmax_scale if softmax_scale is not None else 1.0 / float(head_dim) ** 0.5
    return PrefillInputs(q, k, v, cu_seqlens_from_lengths(lengths), lengths, scale)


def prefill_workload_inputs(wl: PrefillWorkload, seed: int) -> PrefillInputs:
    if wl.lengths is not None:
        lengths = np.asarray(wl.lengths, dtype=np.int64)
    else:
        lengths = draw_lengths(wl.n_seqs, wl.len_lo, wl.len_hi, seed)
    return prefill_inputs(lengths, wl.n_q_heads, wl.n_kv_heads, wl.head_dim, seed)


# ----------------------------------------------------------------------------
# Beam decode inputs
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class DecodeInputs:
    q: torch.Tensor        # bf16 [W, Hq, D]
    kp: torch.Tensor       # bf16 [Lp, Hkv, D]
    vp: torch.Tensor       # bf16 [Lp, Hkv, D]
    ks: torch.Tensor       # bf16 [W, Smax, Hkv, D] rows < L_prev valid, previous beam order
    vs: torch.Tensor       # bf16 [W, Smax, Hkv, D]
    k_new: torch.Tensor    # bf16 [W, Hkv, D] new beam order
    v_new: torch.Tensor    # bf16 [W, Hkv, D]
    parent: torch.Tensor   # int32 [W]
    L_prev: int
    softmax_scale: float


def decode_inputs(W: int, Lp: int, L_prev: int, Smax: int, n_q_heads: int,
                  n_kv_heads: int, head_dim: int, seed: int,
                  std: float = 1.0, identity_parent: bool = False,
                  softmax_scale: Optional[float] = None) -> DecodeInputs:
    if L_prev + 1 > Smax:
        raise ValueError("suffix buffer too short for the appended row")
    q = bf16_randn((W, n_q_heads, head_dim), seed * 8 + 1, std)
    kp = bf16_randn((Lp, n_kv_heads, head_dim), seed * 8 + 2, std)
    vp = bf16_randn((Lp, n_kv_heads, head_dim), seed * 8 + 3, std)
    ks = torch.zeros((W, Smax, n_kv_heads, head_dim), dtype=torch.bfloat16)
    vs = torch.zeros((W, Smax, n_kv_heads, head_dim), dtype=torch.bfloat16)
    if L_prev > 0:
        ks[:, :L_prev] = bf16_randn((W, L_prev, n_kv_heads, head_dim), seed * 8 + 4, std)
        vs[:, :L_prev] = bf16_randn((W, L_prev, n_kv_heads, head_dim), seed * 8 + 5, std)
    k_new = bf16_randn((W, n_kv_heads, head_dim), seed * 8 + 6, std)
    v_new = bf16_randn((W, n_kv_heads, head_dim), seed * 8 + 7, std)
    if identity_parent:
        parent = torch.arange(W, dtype=torch.int32)
    else:
        rng = np.random.default_rng(int(seed))
        parent = torch.from_numpy(rng.integers(0, W, size=W).astype(np.int32))
    scale = softmax_scale if softmax_scale is not None else 1.0 / float(head_dim) ** 0.5
    return DecodeInputs(q, kp, vp, ks, vs, k_new, v_new, parent, L_prev, scale)


# ----------------------------------------------------------------------------
# Beam selection inputs
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class SelectInputs:
    logits: torch.Tensor   # bf16 [W_in, V]
    cum: torch.Tensor      # fp32 [W_in]
    W: int


def cumulative_scores(W_in: int, step: int, seed: int) -> torch.Tensor:
    g = torch.Generator("cpu").manual_seed(int(seed) * 4 + 3)
    a = torch.randn(W_in, generator=g, dtype=torch.float32).abs()
    a, _ = torch.sort(a)
    return (-a * float(step)).contiguous()


def select_inputs(W_in: int, V: int, W: int, seed: int, step: int = 1,
                  std: float = 3.0) -> SelectInputs:
    logits = bf16_randn((W_in, V), seed * 4 + 2, std)
    return SelectInputs(logits, cumulative_scores(W_in, step, seed), W)


def quantized_logits(W_in: int, V: int, levels: int, seed: int) -> torch.Tensor:
    """Logits drawn from a handful of values: a heavy-tie stress input."""
    rng = np.random.default_rng(int(seed))
    vals = rng.integers(0, levels, size=(W_in, V)).astype(np.float32) * 0.5
    return torch.from_numpy(vals).to(torch.bfloat16)


# ----------------------------------------------------------------------------
# Fixed-depth beam search loop inputs
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class DecodeLoopInputs:
    logits0: torch.Tensor        # bf16 [1, V]: the prompt's last-row logits
    kp: torch.Tensor             # bf16 [Lp, Hkv, D]: shared prompt K/V
    vp: torch.Tensor
    steps: list                  # per decode step: (q [W, Hq, D], k_new [W, Hkv, D], v_new, logits [W, V])
    stop_id: Optional[int]
    softmax_scale: float


def decode_loop_inputs(bw: BeamWorkload, seed: int, n_steps: Optional[int] = None,
                       stop_id: Optional[int] = None, stop_rows: float = 0.0) -> DecodeLoopInputs:
    """Synthetic inputs of the fixed-depth loop: prompt K/V, first-step logits,
    and per decode step the new rows' q/k/v and the step's logits (the stand-in
    for the prediction head, whose weights are not part of this path).  With a
    stop id, a fraction `stop_rows` of each step's rows gets the stop token
    among its highest logits (just above the row's maximum), so stop
    candidates reach the global list."""
    n_steps = bw.steps if n_steps is None else n_steps
    W, V, Hq, Hkv, D = bw.beams, bw.vocab, bw.n_q_heads, bw.n_kv_heads, bw.head_dim
    kp = bf16_randn((bw.prefix_len, Hkv, D), seed * 16 + 1)
    vp = bf16_randn((bw.prefix_len, Hkv, D), seed * 16 + 2)
    rng = np.random.default_rng(int(seed))

    def logits_rows(n, s):
        x = bf16_randn((n, V), s, bw.logit_std)
        if stop_id is not None and stop_rows > 0:
            rows = np.nonzero(rng.random(n) < stop_rows)[0]
            if len(rows):
                top = x[rows].float().max(dim=1).values
                x[rows, stop_id] = (top + 0.5).to(torch.bfloat16)
        return x

    logits0 = logits_rows(1, seed * 16 + 3)
    steps = []
    for t in range(n_steps):
        base = seed * 16 + 4 + 4 * t
        steps.append((bf16_randn((W, Hq, D), base * 7 + 1), bf16_randn((W, Hkv, D), base * 7 + 2),
                      bf16_randn((W, Hkv, D), base * 7 + 3), logits_rows(W, base * 7 + 4)))
    return DecodeLoopInputs(logits0, kp, vp, steps, stop_id, bw.softmax_scale)
