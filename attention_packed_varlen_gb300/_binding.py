"""Thin ctypes binding of the C ABI in ``include/slm_attn.h``.

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, their device pointers and the current CUDA stream are handed to
the library, and every step of the computation runs in its CUDA kernels.
There is no fallback: if the library is missing or fails to load, calls
raise.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libslm_attn.so")

SLM_OK = 0
STATUS_NAMES = {0: "SLM_OK", 1: "SLM_ERR_INVALID_ARG", 2: "SLM_ERR_UNSUPPORTED", 3: "SLM_ERR_CUDA",
                4: "SLM_ERR_WORKSPACE", 5: "SLM_ERR_DEVICE_CHECK"}

EXPORTS = ("slm_last_error", "slm_abi_version", "slm_packed_prefill_attn", "slm_prefill_workspace_size",
           "slm_shared_prefix_decode_attn", "slm_beam_select", "slm_beam_select_workspace_size",
           "slm_check_status", "slm_packed_prefill_attn_noalloc", "slm_swiglu_quant_e4m3", "slm_label_scores",
           "slm_beam_split_finished", "slm_beam_reorder_history", "slm_shared_prefix_decode_workspace_size",
           "slm_packed_prefill_attn_f32", "slm_shared_prefix_decode_attn_f32", "slm_set_wait_timeout_ns")


class SlmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load(path: Optional[str] = None):
    """Loads the CUDA library (built by ``attention_packed_varlen_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"CUDA library not built: {p} is missing "
                               "(run `python -m attention_packed_varlen_gb300.build`)")
        lib = ctypes.CDLL(p)
        P, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
        lib.slm_last_error.restype = ctypes.c_char_p
        lib.slm_last_error.argtypes = []
        lib.slm_abi_version.restype = i32
        lib.slm_abi_version.argtypes = []
        lib.slm_packed_prefill_attn.restype = ctypes.c_int
        lib.slm_packed_prefill_attn.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32, P, P, P, sz, P, P]
        lib.slm_packed_prefill_attn_f32.restype = ctypes.c_int
        lib.slm_packed_prefill_attn_f32.argtypes = lib.slm_packed_prefill_attn.argtypes
        lib.slm_set_wait_timeout_ns.restype = ctypes.c_uint64
        lib.slm_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
        lib.slm_prefill_workspace_size.restype = sz
        lib.slm_prefill_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        lib.slm_shared_prefix_decode_attn.restype = ctypes.c_int
        lib.slm_shared_prefix_decode_attn.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                                      f32, P, P, P, P, P, P, sz, P]
        lib.slm_shared_prefix_decode_attn_f32.restype = ctypes.c_int
        lib.slm_shared_prefix_decode_attn_f32.argtypes = lib.slm_shared_prefix_decode_attn.argtypes
        lib.slm_shared_prefix_decode_workspace_size.restype = sz
        lib.slm_shared_prefix_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        lib.slm_beam_select.restype = ctypes.c_int
        lib.slm_beam_select.argtypes = [P, P, i32, i32, i32, P, P, P, P, P, P, P, P, sz, P]
        lib.slm_beam_select_workspace_size.restype = sz
        lib.slm_beam_select_workspace_size.argtypes = [i32, i32, i32]
        lib.slm_check_status.restype = ctypes.c_int
        lib.slm_check_status.argtypes = [P, P]
        lib.slm_packed_prefill_attn_noalloc.restype = ctypes.c_int
        lib.slm_packed_prefill_attn_noalloc.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32, P, P, P, P]
        lib.slm_swiglu_quant_e4m3.restype = ctypes.c_int
        lib.slm_swiglu_quant_e4m3.argtypes = [P, i32, i32, P, P, P]
        lib.slm_label_scores.restype = ctypes.c_int
        lib.slm_label_scores.argtypes = [P, P, i32, i32, i32, P, i32, P, P, P, P]
        lib.slm_beam_split_finished.restype = ctypes.c_int
        lib.slm_beam_split_finished.argtypes = [P, P, P, i32, i32, P, P, P, P, P, P, P, P]
        lib.slm_beam_reorder_history.restype = ctypes.c_int
        lib.slm_beam_reorder_history.argtypes = [P, P, P, i32, i32, i32, i32, P, P, P]
        if path is None:
            _lib = lib
        return lib


def _check(status: int):
    if status != SLM_OK:
        raise SlmError(status, load().slm_last_error().decode(errors="replace"))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, dim: Optional[int] = None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dimensions, got {t.dim()}")


# ----------------------------------------------------------------------------
# Size queries
# ----------------------------------------------------------------------------
def slm_prefill_workspace_size(num_seqs: int, total_tokens: int, max_seqlen: int, n_q_heads: int,
                               n_kv_heads: int) -> int:
    return int(load().slm_prefill_workspace_size(num_seqs, total_tokens, max_seqlen, n_q_heads, n_kv_heads))


def slm_beam_select_workspace_size(W_in: int, V: int, W: int) -> int:
    return int(load().slm_beam_select_workspace_size(W_in, V, W))


def slm_shared_prefix_decode_workspace_size(W: int, Lp: int, n_q_heads: int, n_kv_heads: int, head_dim: int) -> int:
    """Bytes of workspace that let the decode attention split the prompt's key blocks (0: never split)."""
    return int(load().slm_shared_prefix_decode_workspace_size(W, Lp, n_q_heads, n_kv_heads, head_dim))


def slm_abi_version() -> int:
    return int(load().slm_abi_version())


def slm_set_wait_timeout_ns(ns: int) -> int:
    """Sets the limit of the attention kernels' bounded waits (test and
    diagnostic use; default 1 s) and returns the previous one."""
    return int(load().slm_set_wait_timeout_ns(int(ns)))


# ----------------------------------------------------------------------------
# Packed prefill
# ----------------------------------------------------------------------------
def slm_packed_prefill_attn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor,
                            max_seqlen: int, softmax_scale: Optional[float] = None, *,
                            cu_seqlens_host: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                            lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                            dev_status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """O [T, Hq, D] of packed causal GQA attention over sequences delimited by
    ``cu_seqlens`` (int32 [B+1], on the device).  ``lse`` (fp32 [Hq, T]) is
    filled when given."""
    return _prefill(q, k, v, cu_seqlens, max_seqlen, softmax_scale, cu_seqlens_host, out, lse, workspace,
                    dev_status, torch.bfloat16)


def slm_packed_prefill_attn_f32(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor,
                                max_seqlen: int, softmax_scale: Optional[float] = None, *,
                                cu_seqlens_host: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                                lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                                dev_status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The same attention with O returned as fp32 [T, Hq, D], before any bf16
    rounding (test and diagnostic variant)."""
    return _prefill(q, k, v, cu_seqlens, max_seqlen, softmax_scale, cu_seqlens_host, out, lse, workspace,
                    dev_status, torch.float32)


def _prefill(q, k, v, cu_seqlens, max_seqlen, softmax_scale, cu_seqlens_host, out, lse, workspace, dev_status,
             out_dtype):
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    if k.shape != (T, Hkv, D) or v.shape != (T, Hkv, D):
        raise ValueError("k and v must be [T, Hkv, D] matching q")
    B = cu_seqlens.shape[0] - 1
    scale = float(softmax_scale) if softmax_scale is not None else 1.0 / float(D) ** 0.5
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    _need(out, "out", out_dtype, 3)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    need = slm_prefill_workspace_size(B, T, int(max_seqlen), Hq, Hkv)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    host_cs = None
    if cu_seqlens_host is not None:
        host_cs = cu_seqlens_host.to(torch.int32).contiguous()
        if host_cs.is_cuda:
            raise ValueError("cu_seqlens_host must be on the CPU")
    fn = load().slm_packed_prefill_attn if out_dtype == torch.bfloat16 else load().slm_packed_prefill_attn_f32
    st = fn(
        _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(host_cs), B, T, int(max_seqlen), Hq, Hkv, D, scale,
        _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), _ptr(dev_status), _stream(q.device))
    _check(st)
    return out


# ----------------------------------------------------------------------------
# Shared-prefix decode
# ----------------------------------------------------------------------------
_decode_ws = {}  # (device, stream) -> zero-filled decode workspace, grown on demand


def _decode_workspace(device: torch.device, n: int) -> torch.Tensor:
    if torch.cuda.is_current_stream_capturing():  # never keep memory of a graph's private pool
        return torch.zeros(n, dtype=torch.uint8, device=device)
    key = (torch.device(device).index, torch.cuda.current_stream(device).cuda_stream)
    ws = _decode_ws.get(key)
    if ws is None or ws.numel() < n:
        ws = torch.zeros(n, dtype=torch.uint8, device=device)
        _decode_ws[key] = ws
    return ws


def slm_shared_prefix_decode_attn(q: torch.Tensor, kp: Optional[torch.Tensor], vp: Optional[torch.Tensor],
                                  ks: Optional[torch.Tensor], vs: Optional[torch.Tensor],
                                  k_new: Optional[torch.Tensor], v_new: Optional[torch.Tensor],
                                  parent_idx: Optional[torch.Tensor], L_prev: int,
                                  softmax_scale: Optional[float] = None, *, ks_out: torch.Tensor,
                                  vs_out: torch.Tensor, out: Optional[torch.Tensor] = None,
                                  lse: Optional[torch.Tensor] = None,
                                  dev_status: Optional[torch.Tensor] = None,
                                  workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """O [W, Hq, D] of beam decode attention over the shared prompt K/V plus
    each beam's reordered suffix; writes the reordered suffix to ks_out/vs_out.
    ``workspace`` (uint8, device, zero-filled before its first use) lets the
    prompt's key blocks be split over CTAs; when None, a zeroed one kept per
    device and stream is used (a completed call leaves it fit for the next;
    inside a CUDA graph capture a fresh one is allocated instead)."""
    return _decode(q, kp, vp, ks, vs, k_new, v_new, parent_idx, L_prev, softmax_scale, ks_out, vs_out, out, lse,
                   dev_status, workspace, torch.bfloat16)


def slm_shared_prefix_decode_attn_f32(q: torch.Tensor, kp: Optional[torch.Tensor], vp: Optional[torch.Tensor],
                                      ks: Optional[torch.Tensor], vs: Optional[torch.Tensor],
                                      k_new: Optional[torch.Tensor], v_new: Optional[torch.Tensor],
                                      parent_idx: Optional[torch.Tensor], L_prev: int,
                                      softmax_scale: Optional[float] = None, *, ks_out: torch.Tensor,
                                      vs_out: torch.Tensor, out: Optional[torch.Tensor] = None,
                                      lse: Optional[torch.Tensor] = None,
                                      dev_status: Optional[torch.Tensor] = None,
                                      workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The same decode attention with O returned as fp32 [W, Hq, D], before
    any bf16 rounding (test and diagnostic variant)."""
    return _decode(q, kp, vp, ks, vs, k_new, v_new, parent_idx, L_prev, softmax_scale, ks_out, vs_out, out, lse,
                   dev_status, workspace, torch.float32)


def _decode(q, kp, vp, ks, vs, k_new, v_new, parent_idx, L_prev, softmax_scale, ks_out, vs_out, out, lse,
            dev_status, workspace, out_dtype):
    _need(q, "q", torch.bfloat16, 3)
    W, Hq, D = q.shape
    _need(ks_out, "ks_out", torch.bfloat16, 4)
    _need(vs_out, "vs_out", torch.bfloat16, 4)
    Smax, Hkv = ks_out.shape[1], ks_out.shape[2]
    Lp = 0
    if kp is not None:
        _need(kp, "kp", torch.bfloat16, 3)
        _need(vp, "vp", torch.bfloat16, 3)
        Lp = kp.shape[0]
        if kp.shape != (Lp, Hkv, D) or vp.shape != kp.shape:
            raise ValueError("kp/vp must be [Lp, Hkv, D]")
    for name, t in (("ks", ks), ("vs", vs)):
        if t is not None:
            _need(t, name, torch.bfloat16, 4)
            if t.shape != (W, Smax, Hkv, D):
                raise ValueError(f"{name} must be [W, Smax, Hkv, D]")
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        if t is not None:
            _need(t, name, torch.bfloat16, 3)
            if t.shape != (W, Hkv, D):
                raise ValueError(f"{name} must be [W, Hkv, D]")
    if parent_idx is not None:
        _need(parent_idx, "parent_idx", torch.int32, 1)
    scale = float(softmax_scale) if softmax_scale is not None else 1.0 / float(D) ** 0.5
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    _need(out, "out", out_dtype, 3)
    if lse is not None:
        _need(lse, "lse", torch.float32, 2)
    if workspace is None:
        n = slm_shared_prefix_decode_workspace_size(W, Lp, Hq, Hkv, D)
        workspace = _decode_workspace(q.device, n) if n else None
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    fn = load().slm_shared_prefix_decode_attn if out_dtype == torch.bfloat16 else load().slm_shared_prefix_decode_attn_f32
    st = fn(
        _ptr(q), _ptr(kp), _ptr(vp), _ptr(ks), _ptr(vs), _ptr(k_new), _ptr(v_new), _ptr(parent_idx), W, Lp,
        int(L_prev), Smax, Hq, Hkv, D, scale, _ptr(ks_out), _ptr(vs_out), _ptr(out), _ptr(lse), _ptr(dev_status),
        _ptr(workspace), ws_bytes, _stream(q.device))
    _check(st)
    return out


# ----------------------------------------------------------------------------
# Beam selection
# ----------------------------------------------------------------------------
def slm_beam_select(logits: torch.Tensor, cum_scores: torch.Tensor, W: int, *, workspace=None,
                    want_candidates: bool = True, want_lse: bool = True):
    """Returns dict(token, parent, score [W]; cand_token, cand_parent,
    cand_score [2W]; lse [W_in])."""
    _need(logits, "logits", torch.bfloat16, 2)
    _need(cum_scores, "cum_scores", torch.float32, 1)
    W_in, V = logits.shape
    dev = logits.device
    need = slm_beam_select_workspace_size(W_in, V, W)
    if need == 0:
        raise SlmError(2, f"unsupported beam sizes W_in={W_in} V={V} W={W}")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    res = {
        "token": torch.empty(W, dtype=torch.int32, device=dev),
        "parent": torch.empty(W, dtype=torch.int32, device=dev),
        "score": torch.empty(W, dtype=torch.float32, device=dev),
    }
    if want_candidates:
        res["cand_token"] = torch.empty(2 * W, dtype=torch.int32, device=dev)
        res["cand_parent"] = torch.empty(2 * W, dtype=torch.int32, device=dev)
        res["cand_score"] = torch.empty(2 * W, dtype=torch.float32, device=dev)
    if want_lse:
        res["lse"] = torch.empty(W_in, dtype=torch.float32, device=dev)
    st = load().slm_beam_select(
        _ptr(logits), _ptr(cum_scores), W_in, V, W, _ptr(res["token"]), _ptr(res["parent"]), _ptr(res["score"]),
        _ptr(res.get("cand_token")), _ptr(res.get("cand_parent")), _ptr(res.get("cand_score")), _ptr(res.get("lse")),
        _ptr(workspace), workspace.numel(), _stream(dev))
    _check(st)
    return res


def slm_check_status(dev_status: torch.Tensor) -> None:
    """Raises SlmError when a kernel set a bit in ``dev_status``.  After a
    pipeline timeout the decode workspaces kept for this device are dropped:
    a unit that gave up never took its ticket, so they are not zero any more."""
    _need(dev_status, "dev_status", torch.int32)
    st = load().slm_check_status(_ptr(dev_status), _stream(dev_status.device))
    if st != SLM_OK and int(dev_status.item()) & 4:
        for key in [k for k in _decode_ws if k[0] == dev_status.device.index]:
            del _decode_ws[key]
    _check(st)


# ----------------------------------------------------------------------------
# MLP: fused SwiGLU + per-token E4M3
# ----------------------------------------------------------------------------
def slm_swiglu_quant_e4m3(gate_up: torch.Tensor):
    """Returns (q uint8 [T, I] E4M3 codes, scale fp32 [T]) for gate_up bf16 [T, 2I]."""
    _need(gate_up, "gate_up", torch.bfloat16, 2)
    T, two_i = gate_up.shape
    if two_i % 2:
        raise ValueError("gate_up must have an even number of columns")
    I = two_i // 2
    q = torch.empty((T, I), dtype=torch.uint8, device=gate_up.device)
    scale = torch.empty(T, dtype=torch.float32, device=gate_up.device)
    _check(load().slm_swiglu_quant_e4m3(_ptr(gate_up), T, I, _ptr(q), _ptr(scale), _stream(gate_up.device)))
    return q, scale


# ----------------------------------------------------------------------------
# Prefill-Only: last-token label scores
# ----------------------------------------------------------------------------
def slm_label_scores(hidden: torch.Tensor, cu_seqlens: torch.Tensor, w_label: torch.Tensor, *,
                     dev_status: Optional[torch.Tensor] = None, want_probs: bool = True):
    """Returns (logits, probs) fp32 [num_seqs, n_labels] (probs None when not wanted)."""
    _need(hidden, "hidden", torch.bfloat16, 2)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    _need(w_label, "w_label", torch.bfloat16, 2)
    T, d = hidden.shape
    n_labels = w_label.shape[0]
    if w_label.shape[1] != d:
        raise ValueError("w_label must be [n_labels, d_model]")
    B = cu_seqlens.numel() - 1
    dev = hidden.device
    logits = torch.empty((B, n_labels), dtype=torch.float32, device=dev)
    probs = torch.empty((B, n_labels), dtype=torch.float32, device=dev) if want_probs else None
    _check(load().slm_label_scores(_ptr(hidden), _ptr(cu_seqlens), B, T, d, _ptr(w_label), n_labels, _ptr(logits),
                                   _ptr(probs), _ptr(dev_status), _stream(dev)))
    return logits, probs


# ----------------------------------------------------------------------------
# Beam search state: finished hypotheses, token history
# ----------------------------------------------------------------------------
def slm_beam_split_finished(cand_token: torch.Tensor, cand_parent: torch.Tensor, cand_score: torch.Tensor,
                            stop_id: int):
    """Returns dict(token, parent, score [W]: active beams; fin_token, fin_parent, fin_score [W] and
    fin_count [1]: hypotheses finished at this step)."""
    _need(cand_token, "cand_token", torch.int32, 1)
    _need(cand_parent, "cand_parent", torch.int32, 1)
    _need(cand_score, "cand_score", torch.float32, 1)
    W = cand_token.numel() // 2
    dev = cand_token.device
    res = {k: torch.empty(W, dtype=torch.int32, device=dev) for k in ("token", "parent", "fin_token", "fin_parent")}
    res["score"] = torch.empty(W, dtype=torch.float32, device=dev)
    res["fin_score"] = torch.empty(W, dtype=torch.float32, device=dev)
    res["fin_count"] = torch.empty(1, dtype=torch.int32, device=dev)
    _check(load().slm_beam_split_finished(
        _ptr(cand_token), _ptr(cand_parent), _ptr(cand_score), W, stop_id, _ptr(res["token"]), _ptr(res["parent"]),
        _ptr(res["score"]), _ptr(res["fin_token"]), _ptr(res["fin_parent"]), _ptr(res["fin_score"]),
        _ptr(res["fin_count"]), _stream(dev)))
    return res


def slm_beam_reorder_history(hist_in: Optional[torch.Tensor], parent: Optional[torch.Tensor], token: torch.Tensor,
                             t: int, hist_out: torch.Tensor, *, dev_status: Optional[torch.Tensor] = None):
    """hist_out[b, :t] = hist_in[parent[b], :t]; hist_out[b, t] = token[b]."""
    _need(token, "token", torch.int32, 1)
    _need(hist_out, "hist_out", torch.int32, 2)
    W, max_len = hist_out.shape
    W_in = hist_in.shape[0] if hist_in is not None else 1
    _check(load().slm_beam_reorder_history(_ptr(hist_in), _ptr(parent), _ptr(token), W, W_in, t, max_len,
                                           _ptr(hist_out), _ptr(dev_status), _stream(token.device)))
    return hist_out
