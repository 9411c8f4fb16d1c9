"""Fixed-depth beam search as one enqueued program (article "SLM 生成式高并发推理引擎：
延迟约束下的有效吞吐优化", section 2.3): first-step candidates from the prompt's
last-row logits, then a fixed number of steps of

    shared-prefix decode attention with parent-index suffix reorder
    -> the step's logits (given: the prediction head is outside this path)
    -> two-stage beam selection over the cumulative scores
    -> optional finished-beam split (stop token; W active beams go on)
    -> token-history reorder.

Every buffer is allocated once, when the loop is built; ``record`` only
enqueues C-ABI calls on the current CUDA stream, so the whole loop can be
captured into a single CUDA graph (``capture``) and replayed with new inputs
copied into the same tensors.  All per-step results stay in their own buffers
and can be read after the run.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _binding as slm


class BeamDecodeLoop:
    def __init__(self, W: int, V: int, n_steps: int, prefix_len: int, n_q_heads: int, n_kv_heads: int,
                 head_dim: int, stop_id: Optional[int] = None, softmax_scale: Optional[float] = None,
                 device="cuda"):
        dev = torch.device(device)
        self.W, self.V, self.n_steps, self.Lp = W, V, n_steps, prefix_len
        self.Hq, self.Hkv, self.D = n_q_heads, n_kv_heads, head_dim
        self.stop_id = stop_id
        self.scale = softmax_scale if softmax_scale is not None else 1.0 / float(head_dim) ** 0.5
        self.n_tokens = n_steps + 1
        Smax = max(1, n_steps)
        i32, f32, bf16 = torch.int32, torch.float32, torch.bfloat16
        # suffix K/V after each step (step 0: empty), attention outputs per step
        self.ks = [torch.zeros((W, Smax, n_kv_heads, head_dim), dtype=bf16, device=dev) for _ in range(n_steps + 1)]
        self.vs = [torch.zeros((W, Smax, n_kv_heads, head_dim), dtype=bf16, device=dev) for _ in range(n_steps + 1)]
        self.o = [torch.empty((W, n_q_heads, head_dim), dtype=bf16, device=dev) for _ in range(n_steps)]
        self.hist = [torch.zeros((W, self.n_tokens), dtype=i32, device=dev) for _ in range(n_steps + 1)]
        self.cum0 = torch.zeros(1, dtype=f32, device=dev)
        ws = max(slm.slm_beam_select_workspace_size(1, V, W), slm.slm_beam_select_workspace_size(W, V, W))
        if ws == 0:
            raise slm.SlmError(2, f"unsupported beam sizes W={W} V={V}")
        self.ws = torch.empty(ws, dtype=torch.uint8, device=dev)
        dws = slm.slm_shared_prefix_decode_workspace_size(W, prefix_len, n_q_heads, n_kv_heads, head_dim)
        self.dec_ws = torch.zeros(dws, dtype=torch.uint8, device=dev) if dws else None
        self.sel = []
        for t in range(n_steps + 1):
            w_in = 1 if t == 0 else W
            self.sel.append({"token": torch.empty(W, dtype=i32, device=dev),
                             "parent": torch.empty(W, dtype=i32, device=dev),
                             "score": torch.empty(W, dtype=f32, device=dev),
                             "cand_token": torch.empty(2 * W, dtype=i32, device=dev),
                             "cand_parent": torch.empty(2 * W, dtype=i32, device=dev),
                             "cand_score": torch.empty(2 * W, dtype=f32, device=dev),
                             "lse": torch.empty(w_in, dtype=f32, device=dev)})
        self.fin = None
        if stop_id is not None:
            self.fin = [{k: torch.empty(W, dtype=i32, device=dev) for k in ("token", "parent", "fin_token",
                                                                             "fin_parent")}
                        for _ in range(n_steps + 1)]
            for f in self.fin:
                f["score"] = torch.empty(W, dtype=f32, device=dev)
                f["fin_score"] = torch.empty(W, dtype=f32, device=dev)
                f["fin_count"] = torch.empty(1, dtype=i32, device=dev)
        self.status = torch.zeros(1, dtype=i32, device=dev)
        self.graph = None

    def active(self, t: int) -> dict:
        """Beams that go on after step t: (token, parent, score) [W]."""
        return self.fin[t] if self.fin is not None else self.sel[t]

    def _select(self, t: int, logits: torch.Tensor, cum: torch.Tensor):
        lib = slm.load()
        r = self.sel[t]
        P = slm._ptr
        w_in = logits.shape[0]
        slm._check(lib.slm_beam_select(
            P(logits), P(cum), w_in, self.V, self.W, P(r["token"]), P(r["parent"]), P(r["score"]),
            P(r["cand_token"]), P(r["cand_parent"]), P(r["cand_score"]), P(r["lse"]), P(self.ws), self.ws.numel(),
            slm._stream(logits.device)))
        if self.fin is not None:
            f = self.fin[t]
            slm._check(lib.slm_beam_split_finished(
                P(r["cand_token"]), P(r["cand_parent"]), P(r["cand_score"]), self.W, int(self.stop_id),
                P(f["token"]), P(f["parent"]), P(f["score"]), P(f["fin_token"]), P(f["fin_parent"]),
                P(f["fin_score"]), P(f["fin_count"]), slm._stream(logits.device)))

    def record(self, logits0: torch.Tensor, kp: torch.Tensor, vp: torch.Tensor, steps) -> None:
        """Enqueues the whole loop on the current stream.  steps[t - 1] =
        (q, k_new, v_new, logits) of decode step t = 1..n_steps, in the order
        of the beams that step t runs for (those chosen at step t - 1)."""
        if len(steps) != self.n_steps:
            raise ValueError(f"expected {self.n_steps} steps, got {len(steps)}")
        self._select(0, logits0, self.cum0)
        a = self.active(0)
        slm.slm_beam_reorder_history(None, None, a["token"], 0, self.hist[0], dev_status=self.status)
        for t in range(1, self.n_steps + 1):
            q, k_new, v_new, logits = steps[t - 1]
            prev = self.active(t - 1)
            slm.slm_shared_prefix_decode_attn(
                q, kp, vp, self.ks[t - 1], self.vs[t - 1], k_new, v_new, prev["parent"], t - 1, self.scale,
                ks_out=self.ks[t], vs_out=self.vs[t], out=self.o[t - 1], dev_status=self.status,
                workspace=self.dec_ws)
            self._select(t, logits, prev["score"])
            a = self.active(t)
            slm.slm_beam_reorder_history(self.hist[t - 1], a["parent"], a["token"], t, self.hist[t],
                                         dev_status=self.status)

    def capture(self, logits0, kp, vp, steps) -> torch.cuda.CUDAGraph:
        """Records the loop into one CUDA graph over these (static) tensors;
        ``replay()`` reruns it after new values are copied into them."""
        s = torch.cuda.Stream(device=logits0.device)
        s.wait_stream(torch.cuda.current_stream(logits0.device))
        with torch.cuda.stream(s):  # one eager run: library set-up outside the capture
            self.record(logits0, kp, vp, steps)
        torch.cuda.current_stream(logits0.device).wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.record(logits0, kp, vp, steps)
        self.graph = g
        return g

    def replay(self) -> None:
        if self.graph is None:
            raise RuntimeError("capture() first")
        self.graph.replay()
