"""CPU oracle for the attention hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg (and its ``--impl reference`` arm) may import this package. The product
library never calls it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C loops, fp64 attention, fp32
selection scores as the article fixes them); this module compiles it with gcc
and marshals numpy / torch arrays into it.  Sources followed, from the article
"SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化":

* ``packed_prefill`` -- section 3.1, packed Q/K/V layout and the
  block-diagonal causal mask implied by the sequence boundary;
* ``shared_prefix_decode`` -- section 3.2, the attention equation over the
  prefix/suffix concatenation, and the parent-index suffix reorder of
  sections 3.2 and 3.3;
* ``beam_select`` / ``row_lse`` -- section 3.3, FP32 log-softmax scores plus
  cumulative beam scores, global candidates from the flattened beams (here by
  a full sort of every W x V entry).

The operations around the attention path (SwiGLU + E4M3, label scores,
finished beams, the fixed-depth decode loop) are in ``oracle/heads.py``.

Pins that tie this oracle to something other than itself are in
``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.environ.get("SLM_ORACLE_LIB") or os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (IEEE semantics: no
    fast-math, no floating-point contraction).  SLM_ORACLE_LIB names a
    prebuilt library to load instead (used to check the pins themselves)."""
    if os.environ.get("SLM_ORACLE_LIB"):
        return _LIB
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.oracle_packed_prefill.argtypes = [P, P, P, P, i32, i32, i32, i32, f64, P, P, i32]
            lib.oracle_packed_prefill_rows.argtypes = [P, P, P, P, i32, i32, i32, i32, f64, P, i64, P, P, i32]
            lib.oracle_shared_prefix_decode.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32,
                                                        i32, i32, i32, f64, P, P, P, P, i32]
            lib.oracle_row_lse.argtypes = [P, i32, i64, P]
            lib.oracle_beam_select.argtypes = [P, P, i32, i64, i32, P, P, P, P, P]
            for fn in (lib.oracle_packed_prefill, lib.oracle_packed_prefill_rows,
                       lib.oracle_shared_prefix_decode, lib.oracle_row_lse,
                       lib.oracle_beam_select):
                fn.restype = ctypes.c_int
            _lib = lib
    return _lib


def _bits(x) -> np.ndarray:
    """bf16 tensor (torch) or uint16 array -> contiguous uint16 bit array."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("expected bf16 bit patterns as uint16")
        return np.ascontiguousarray(x)
    import torch
    if x.dtype != torch.bfloat16:
        raise TypeError(f"expected a bf16 tensor, got {x.dtype}")
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# ----------------------------------------------------------------------------
def packed_prefill(q, k, v, cu_seqlens, softmax_scale: float, want_lse: bool = False,
                   n_threads: int = 1):
    """fp64 O [T, Hq, D] (and LSE [Hq, T]) of packed causal GQA attention."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    T, Hq, D = qb.shape
    Hkv = kb.shape[1]
    o = np.zeros((T, Hq, D), dtype=np.float64)
    lse = np.zeros((Hq, T), dtype=np.float64) if want_lse else None
    rc = lib.oracle_packed_prefill(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(cu), len(cu) - 1,
                                   Hq, Hkv, D, float(softmax_scale), _ptr(o), _ptr(lse),
                                   int(n_threads))
    if rc != 0:
        raise ValueError("oracle_packed_prefill rejected its arguments")
    return (o, lse) if want_lse else o


def packed_prefill_rows(q, k, v, cu_seqlens, softmax_scale: float, rows, n_threads: int = 1):
    """fp64 outputs for selected (token, q head) rows only: ([n, D], lse [n])."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
    T, Hq, D = qb.shape
    Hkv = kb.shape[1]
    o = np.zeros((rows.shape[0], D), dtype=np.float64)
    lse = np.zeros((rows.shape[0],), dtype=np.float64)
    rc = lib.oracle_packed_prefill_rows(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(cu), len(cu) - 1,
                                        Hq, Hkv, D, float(softmax_scale), _ptr(rows),
                                        rows.shape[0], _ptr(o), _ptr(lse), int(n_threads))
    if rc != 0:
        raise ValueError("oracle_packed_prefill_rows rejected its arguments")
    return o, lse


def shared_prefix_decode(q, kp, vp, ks, vs, k_new, v_new, parent, L_prev: int,
                         softmax_scale: float, n_threads: int = 1):
    """Returns (o fp64 [W,Hq,D], lse fp64 [W,Hq], ks_out, vs_out as uint16 bits)."""
    lib = _load()
    qb, kpb, vpb, ksb, vsb = _bits(q), _bits(kp), _bits(vp), _bits(ks), _bits(vs)
    knb = None if k_new is None else _bits(k_new)
    vnb = None if v_new is None else _bits(v_new)
    par = None if parent is None else np.ascontiguousarray(np.asarray(parent, dtype=np.int32))
    W, Hq, D = qb.shape
    Lp, Hkv = kpb.shape[0], kpb.shape[1]
    Smax = ksb.shape[1]
    ks_out = np.zeros_like(ksb)
    vs_out = np.zeros_like(vsb)
    o = np.zeros((W, Hq, D), dtype=np.float64)
    lse = np.zeros((W, Hq), dtype=np.float64)
    rc = lib.oracle_shared_prefix_decode(_ptr(qb), _ptr(kpb), _ptr(vpb), _ptr(ksb), _ptr(vsb),
                                         _ptr(knb), _ptr(vnb), _ptr(par), W, Lp, int(L_prev), Smax,
                                         Hq, Hkv, D, float(softmax_scale), _ptr(ks_out),
                                         _ptr(vs_out), _ptr(o), _ptr(lse), int(n_threads))
    if rc != 0:
        raise ValueError("oracle_shared_prefix_decode rejected its arguments")
    return o, lse, ks_out, vs_out


def row_lse(logits) -> np.ndarray:
    lib = _load()
    lb = _bits(logits)
    W_in, V = lb.shape
    out = np.zeros((W_in,), dtype=np.float32)
    if lib.oracle_row_lse(_ptr(lb), W_in, V, _ptr(out)) != 0:
        raise ValueError("oracle_row_lse rejected its arguments")
    return out


def beam_select(logits, cum_scores, n_keep: int, lse_in=None):
    """Full sort of all W_in x V candidates; returns the first ``n_keep`` as
    (token int32, parent int32, score fp32, lse fp32 [W_in]).

    ``lse_in`` (fp32 [W_in], optional) replaces the oracle's own row
    log-normalisers: the ranking is then that of the same scores formed from
    the given normalisers (used to check a selection given its own fp32
    log-softmax)."""
    lib = _load()
    lb = _bits(logits)
    W_in, V = lb.shape
    cum = np.ascontiguousarray(np.asarray(cum_scores, dtype=np.float32))
    lse_given = None
    if lse_in is not None:
        lse_given = np.ascontiguousarray(np.asarray(lse_in, dtype=np.float32))
        if lse_given.shape != (W_in,):
            raise ValueError("lse_in must have one value per row")
    tok = np.zeros((n_keep,), dtype=np.int32)
    par = np.zeros((n_keep,), dtype=np.int32)
    sc = np.zeros((n_keep,), dtype=np.float32)
    lse = np.zeros((W_in,), dtype=np.float32)
    rc = lib.oracle_beam_select(_ptr(lb), _ptr(cum), W_in, V, int(n_keep), _ptr(lse_given),
                                _ptr(tok), _ptr(par), _ptr(sc), _ptr(lse))
    if rc == -2:
        raise MemoryError("oracle_beam_select could not allocate its sort buffer")
    if rc != 0:
        raise ValueError("oracle_beam_select rejected its arguments")
    return tok, par, sc, lse
