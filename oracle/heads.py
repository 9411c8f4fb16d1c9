"""CPU oracle for the operations around the attention path -- TEST
INFRASTRUCTURE ONLY (like the rest of ``oracle/``: only tests, the smoke
check and the benchmark's CPU legs may use it; the product library never does).

Plain numpy, fp64 unless the article fixes a precision, written from the
article "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化":

* ``e4m3_encode`` / ``e4m3_decode`` and ``swiglu_quant_e4m3`` -- section 3.4:
  FP32 SiLU(gate) x up, per-token dynamic scale, E4M3 codes;
* ``label_scores`` -- sections 1.1 and 3.1: each sequence's last valid row,
  the label tokens' logits, a softmax over the labels;
* ``split_finished`` -- section 3.3: 2W global candidates, stop-token
  candidates set aside, W active beams go on;
* ``reorder_history`` and ``beam_decode_loop`` -- section 2.3: the fixed-depth
  beam search loop and the states the parent index reorders.

Pins are in ``tests/test_oracle_heads.py``.
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------
# E4M3 (OCP 8-bit floating point, E4M3 variant): 1 sign bit, 4 exponent bits
# (bias 7), 3 mantissa bits; no infinities; S.1111.111 is NaN, so the largest
# finite magnitude is 1.75 * 2^8 = 448.
# ----------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_decode(code) -> np.ndarray:
    """Value of each E4M3 code (NaN for the two NaN codes)."""
    c = np.asarray(code, dtype=np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e.astype(np.float64) - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


# the non-negative finite codes in value order (code k has value e4m3_decode(k))
_POS_CODES = np.arange(0x7F, dtype=np.int64)      # 0x00 .. 0x7E
_POS_VALUES = e4m3_decode(_POS_CODES)             # increasing


def e4m3_encode(x) -> np.ndarray:
    """Round each value to the nearest E4M3 value, ties to the even code (last
    mantissa bit 0), magnitudes above 448 saturated to 448.  NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.searchsorted(_POS_VALUES, a, side="left")   # first value >= a
    hi = np.minimum(hi, len(_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    vlo, vhi = _POS_VALUES[lo], _POS_VALUES[hi]
    exact = vhi == a
    dlo, dhi = a - vlo, vhi - a
    pick_hi = exact | (dhi < dlo) | ((dhi == dlo) & (_POS_CODES[hi] % 2 == 0))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo])
    code = np.where(np.signbit(x), code | 0x80, code)  # the sign is kept, also on zero
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def _f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def swiglu_quant_e4m3(gate_up):
    """gate_up [T, 2I] (bf16 values; torch or numpy) -> (codes uint8 [T, I],
    scale fp32 [T], x fp64 [T, I]).

    h = fl32(SiLU(g) * u) with SiLU(g) = g / (1 + exp(-g)) evaluated in fp64
    and the product rounded once to fp32; amax = max |h|; scale =
    fl32(amax / 448); inv = fl32(448 / amax); x = fl32(h * inv); codes =
    e4m3_encode(x).  A row with amax = 0 has scale 1 and codes 0.  x is
    returned so a test can tell which codes sit on a rounding boundary."""
    gu = _as_f64(gate_up)
    T, two_i = gu.shape
    I = two_i // 2
    g, u = gu[:, :I], gu[:, I:]
    h = _f32(g / (1.0 + np.exp(-g)) * u).astype(np.float64)
    amax = np.abs(h).max(axis=1) if I else np.zeros(T)
    scale = np.where(amax > 0, _f32(amax / E4M3_MAX), np.float32(1.0)).astype(np.float32)
    inv = np.where(amax > 0, _f32(E4M3_MAX / np.where(amax > 0, amax, 1.0)), np.float32(0.0)).astype(np.float64)
    x = _f32(h * inv[:, None]).astype(np.float64)
    return e4m3_encode(x), scale, x


def e4m3_boundary_distance(x) -> np.ndarray:
    """Relative distance of each value from the nearest E4M3 rounding
    boundary (midpoint between neighbouring codes); large = safely inside."""
    a = np.minimum(np.abs(np.asarray(x, dtype=np.float64)), E4M3_MAX)
    mids = (_POS_VALUES[1:] + _POS_VALUES[:-1]) / 2.0
    i = np.clip(np.searchsorted(mids, a), 1, len(mids) - 1)
    d = np.minimum(np.abs(a - mids[i - 1]), np.abs(a - mids[i]))
    return d / np.maximum(a, 2.0 ** -9)


# ----------------------------------------------------------------------------
# Last-token label scores
# ----------------------------------------------------------------------------
def _as_f64(t):
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().to(torch.float64).cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)


def label_scores(hidden, cu_seqlens, w_label):
    """(logits, probs) fp64 [B, n_labels]: for sequence b with boundary
    [s0, s1), h = hidden[s1 - 1], logits[b, k] = h . w_label[k], probs[b] =
    softmax(logits[b]).  A sequence of length 0 gets NaN."""
    h = _as_f64(hidden)
    w = _as_f64(w_label)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    B = len(cu) - 1
    n = w.shape[0]
    logits = np.full((B, n), np.nan)
    probs = np.full((B, n), np.nan)
    for b in range(B):
        s0, s1 = cu[b], cu[b + 1]
        if s1 <= s0:
            continue
        z = np.array([np.dot(h[s1 - 1], w[k]) for k in range(n)])
        logits[b] = z
        e = np.exp(z - z.max())
        probs[b] = e / e.sum()
    return logits, probs


# ----------------------------------------------------------------------------
# Beam search state
# ----------------------------------------------------------------------------
def split_finished(cand_token, cand_parent, cand_score, W: int, stop_id: int):
    """Walks the 2W global candidates in order: a stop-token candidate ranked
    among the first W is a finished hypothesis; the first W others are the
    next active beams.  Returns (active list of (token, parent, score),
    finished list of (token, parent, score))."""
    active, finished = [], []
    for rank in range(len(cand_token)):
        tok, par, sc = int(cand_token[rank]), int(cand_parent[rank]), float(cand_score[rank])
        if tok == stop_id:
            if rank < W:
                finished.append((tok, par, sc))
        elif len(active) < W:
            active.append((tok, par, sc))
    return active, finished


def reorder_history(hist_in, parent, token, t: int):
    """New beam b: its parent's first t tokens, then token[b]."""
    W = len(token)
    out = np.zeros((W, t + 1), dtype=np.int64)
    for b in range(W):
        p = int(parent[b]) if parent is not None else b
        if t:
            out[b, :t] = np.asarray(hist_in)[p, :t]
        out[b, t] = int(token[b])
    return out


def candidate_scores(logits, cum, lse, parent, token) -> np.ndarray:
    """fp32 scores of the given (parent, token) candidates, formed as the
    article's section 3.3 fixes them: fl32(cum[p] + fl32(x[p, v] - lse[p]))
    with x the bf16 logit widened exactly and lse the fp32 log-normaliser."""
    import oracle as _o
    bits = _o._bits(logits)
    par = np.asarray(parent, dtype=np.int64)
    tok = np.asarray(token, dtype=np.int64)
    x = (bits[par, tok].astype(np.uint32) << 16).view(np.float32)
    lp = (x - np.asarray(lse, dtype=np.float32)[par]).astype(np.float32)
    return (np.asarray(cum, dtype=np.float32)[par] + lp).astype(np.float32)


def beam_decode_loop(logits0, kp, vp, steps, W: int, softmax_scale: float, stop_id=None, follow=None,
                     n_threads: int = 1):
    """Fixed-depth beam search (section 2.3), one record per step.

    Step 0 turns the prompt's last-row logits [1, V] into the first W beams
    (cumulative score 0).  Decode step t = 1..len(steps) takes steps[t-1] =
    (q [W,Hq,D], k_new, v_new [W,Hkv,D], logits [W,V]) of the beams chosen at
    step t-1 and
      1. attends over the shared prompt K/V plus each beam's suffix, the
         suffix of step t-1 reordered by that step's parent index with the
         new row appended (sections 3.2, 3.3);
      2. ranks all W x V extensions by cumulative score and keeps the top 2W
         candidates (section 3.3);
      3. with a stop id, sets finished hypotheses aside (``split_finished``);
      4. reorders the token history by the new parents (``reorder_history``).

    Each record holds ``cum`` (the cumulative scores the step's selection
    started from), ``cand`` = (token, parent, score, lse) of the top 2W,
    ``active`` = (token, parent, score) of the W beams that go on,
    ``finished`` (list of (token, parent, score)), ``hist`` [W, t+1] and, for
    t >= 1, the attention ``o``, ``lse`` and reordered suffix ``ks``/``vs``
    (bf16 bits) of that step.

    ``follow(t, rec)``, when given, returns the (token, parent) arrays of the
    beams to go on with after step t instead of the record's own -- e.g.
    those of another run whose near-equal scores were ordered differently --
    so that every later step is compared on the same beams.  Only the beams'
    identity is taken: their cumulative scores are this oracle's own,
    ``candidate_scores`` from its own log-normalisers and its own earlier
    scores.  The hypotheses ``hist`` and ``ks``/``vs`` follow the same beams."""
    import oracle as _o  # the package's C-backed attention and selection

    def split(tok, par, sc):
        if stop_id is None:
            return (tok[:W].astype(np.int32), par[:W].astype(np.int32), sc[:W].astype(np.float32)), []
        act, fin = split_finished(tok, par, sc, W, stop_id)
        return (np.array([a[0] for a in act], np.int32), np.array([a[1] for a in act], np.int32),
                np.array([a[2] for a in act], np.float32)), fin

    def go_on(t, rec, logits, cum):
        if follow is None:
            return rec["active"]
        tok, par = follow(t, rec)
        tok = np.asarray(tok, np.int32)
        par = np.asarray(par, np.int32)
        return tok, par, candidate_scores(logits, cum, rec["cand"][3], par, tok)

    recs = []
    cum = np.zeros(1, np.float32)
    cand = _o.beam_select(logits0, cum, 2 * W)
    active, fin = split(*cand[:3])
    rec = {"cum": cum, "cand": cand, "active": active, "finished": fin}
    state = go_on(0, rec, logits0, cum)
    rec["hist"] = reorder_history(None, None, state[0], 0)
    recs.append(rec)
    hist = rec["hist"]
    Hkv, D = np.asarray(_o._bits(kp)).shape[1:]
    Smax = max(1, len(steps))
    ks = np.zeros((W, Smax, Hkv, D), np.uint16)
    vs = np.zeros_like(ks)
    for t in range(1, len(steps) + 1):
        q, k_new, v_new, logits = steps[t - 1]
        parent = state[1]
        o, lse, ks, vs = _o.shared_prefix_decode(q, kp, vp, ks, vs, k_new, v_new, parent, t - 1, softmax_scale,
                                                 n_threads=n_threads)
        cum = state[2]
        cand = _o.beam_select(logits, cum, 2 * W)
        active, fin = split(*cand[:3])
        rec = {"cum": cum, "cand": cand, "active": active, "finished": fin, "o": o, "lse": lse, "ks": ks,
               "vs": vs}
        state = go_on(t, rec, logits, cum)
        hist = reorder_history(hist, state[1], state[0], t)
        rec["hist"] = hist
        recs.append(rec)
    return recs
