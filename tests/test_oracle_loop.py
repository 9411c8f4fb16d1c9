"""Pins for the oracle's fixed-depth beam search loop (article "SLM 生成式高并发推理引擎：
延迟约束下的有效吞吐优化", section 2.3), CPU only.

Each check recomputes a property of the whole loop by a route of its own:
W = 1 is greedy decoding; every kept set is the top W of all W x V
extensions found by plain enumeration; a final beam's score is the sum of
its tokens' log-probabilities along its ancestry; its suffix K/V rows and its
token history are the rows of its ancestors; its attention output is a
plain softmax over the prompt rows and those ancestor rows.
"""
import numpy as np
import torch

from attention_packed_varlen_gb300 import workloads as wl
from oracle import heads as H

W, V, LP, HQ, HKV, D, STEPS = 3, 40, 5, 4, 2, 8, 4
SCALE = 1.0 / np.sqrt(D)


def tiny(seed, W=W, stop_id=None, stop_rows=0.0):
    bw = wl.BeamWorkload("tiny loop", LP, W, STEPS, HQ, HKV, D, vocab=V, logit_std=2.0)
    return wl.decode_loop_inputs(bw, seed, stop_id=stop_id, stop_rows=stop_rows)


def f64(t):
    return t.to(torch.float64).numpy()


def logsoftmax(x):
    m = x.max(axis=-1, keepdims=True)
    return x - (m + np.log(np.exp(x - m).sum(axis=-1, keepdims=True)))


def ancestry(recs, b):
    """Row of beam b's ancestor in each kept set 0..N-1 (b is a row of the last kept set N-1 that ran step N)."""
    N = len(recs) - 1
    rows = [0] * N
    r = b
    for s in range(N - 1, -1, -1):
        rows[s] = r
        r = int(recs[s]["active"][1][r])
    return rows


def test_width_one_is_greedy():
    d = tiny(1, W=1)
    recs = H.beam_decode_loop(d.logits0, d.kp, d.vp, d.steps, 1, SCALE)
    tok = [int(np.argmax(f64(d.logits0)[0]))] + [int(np.argmax(f64(s[3])[0])) for s in d.steps]
    assert recs[-1]["hist"][0].tolist() == tok
    assert all(int(r["active"][1][0]) == 0 for r in recs)
    lp = logsoftmax(f64(d.logits0))[0, tok[0]] + sum(logsoftmax(f64(s[3]))[0, t] for s, t in zip(d.steps, tok[1:]))
    assert abs(float(recs[-1]["active"][2][0]) - lp) < 1e-4


def test_each_kept_set_is_top_w_of_all_extensions():
    d = tiny(2)
    recs = H.beam_decode_loop(d.logits0, d.kp, d.vp, d.steps, W, SCALE)
    cum = np.zeros(1)
    rows = [f64(d.logits0)] + [f64(s[3]) for s in d.steps]
    for t, rec in enumerate(recs):
        x = rows[t]
        sc = cum[:, None] + logsoftmax(x)
        order = sorted(((sc[p, v], p, v) for p in range(x.shape[0]) for v in range(V)), reverse=True)
        want = [(p, v) for _, p, v in order[:W]]
        got = list(zip(rec["active"][1].tolist(), rec["active"][0].tolist()))
        assert got == want, f"step {t}"
        cum = np.array([sc[p, v] for p, v in want])
        np.testing.assert_allclose(rec["active"][2], cum, rtol=0, atol=1e-4)


def test_final_scores_hist_and_suffix_follow_the_ancestry():
    d = tiny(3)
    recs = H.beam_decode_loop(d.logits0, d.kp, d.vp, d.steps, W, SCALE)
    N = len(d.steps)
    last = recs[N]
    ls = [logsoftmax(f64(d.logits0))] + [logsoftmax(f64(s[3])) for s in d.steps]
    kbits = [s[1].view(torch.int16).numpy().view(np.uint16) for s in d.steps]
    vbits = [s[2].view(torch.int16).numpy().view(np.uint16) for s in d.steps]
    for b in range(W):
        # beam b of the set that ran step N, extended by step N's selection
        rows = ancestry(recs, b)
        toks = [int(recs[s]["active"][0][rows[s]]) for s in range(N)]
        assert recs[N - 1]["hist"][b].tolist() == toks
        score = ls[0][0, toks[0]] + sum(ls[s][rows[s - 1], toks[s]] for s in range(1, N))
        assert abs(float(recs[N - 1]["active"][2][b]) - score) < 1e-4
        for s in range(N):  # suffix position s holds step s+1's new row of ancestor rows[s]
            np.testing.assert_array_equal(last["ks"][b, s], kbits[s][rows[s]])
            np.testing.assert_array_equal(last["vs"][b, s], vbits[s][rows[s]])
        # attention of step N: softmax over the prompt rows and the ancestor rows, per query head
        q = f64(d.steps[N - 1][0])[b]
        K = np.concatenate([f64(d.kp), np.stack([f64(d.steps[s][1])[rows[s]] for s in range(N)])])
        Vv = np.concatenate([f64(d.vp), np.stack([f64(d.steps[s][2])[rows[s]] for s in range(N)])])
        for h in range(HQ):
            g = h // (HQ // HKV)
            z = K[:, g] @ q[h] * SCALE
            p = np.exp(z - z.max())
            np.testing.assert_allclose(last["o"][b, h], (p / p.sum()) @ Vv[:, g], rtol=0, atol=1e-12)
    # the final history: the last kept set's tokens after its parents' histories
    for b in range(W):
        p = int(last["active"][1][b])
        assert last["hist"][b].tolist() == recs[N - 1]["hist"][p].tolist() + [int(last["active"][0][b])]


def test_stop_token_beams_leave_the_loop():
    stop = 7
    d = tiny(4, stop_id=stop, stop_rows=0.6)
    recs = H.beam_decode_loop(d.logits0, d.kp, d.vp, d.steps, W, SCALE, stop_id=stop)
    n_fin = 0
    for rec in recs:
        tok, par, sc, _ = rec["cand"]
        assert stop not in rec["active"][0].tolist()
        assert len(rec["active"][0]) == W
        # finished: stop candidates ranked among the first W
        want = [(int(par[i]), float(sc[i])) for i in range(W) if tok[i] == stop]
        assert [(f[1], f[2]) for f in rec["finished"]] == want
        n_fin += len(want)
        # active: the first W non-stop candidates, in rank order
        keep = [i for i in range(2 * W) if tok[i] != stop][:W]
        assert rec["active"][0].tolist() == tok[keep].tolist()
    assert n_fin > 0, "the stop token never reached the first W candidates"


def test_follow_replaces_the_kept_set():
    d = tiny(5)
    own = H.beam_decode_loop(d.logits0, d.kp, d.vp, d.steps, W, SCALE)

    def swap_first_two(t, rec):
        tok, par = (a.copy() for a in rec["active"][:2])
        tok[[0, 1]], par[[0, 1]] = tok[[1, 0]], par[[1, 0]]
        return tok, par

    fol = H.beam_decode_loop(d.logits0, d.kp, d.vp, d.steps, W, SCALE, follow=swap_first_two)
    assert fol[0]["hist"][0].tolist() == own[0]["hist"][1].tolist()
    assert fol[0]["hist"][1].tolist() == own[0]["hist"][0].tolist()
    # step 2 reorders step 1's suffix by the followed (swapped) parents
    par = swap_first_two(1, fol[1])[1]
    k1 = d.steps[0][1].view(torch.int16).numpy().view(np.uint16)
    for b in range(W):
        np.testing.assert_array_equal(fol[2]["ks"][b, 0], k1[par[b]])


def test_following_its_own_beams_changes_nothing():
    # follow() hands over only the beams' identity; the loop then scores them
    # itself.  Following its own kept beams must give every record bit for
    # bit, so the followed scores are the same fp32 arithmetic as the sort's.
    for seed, stop in ((6, None), (7, 7)):
        d = tiny(seed, stop_id=stop, stop_rows=0.5 if stop is not None else 0.0)
        own = H.beam_decode_loop(d.logits0, d.kp, d.vp, d.steps, W, SCALE, stop_id=stop)
        fol = H.beam_decode_loop(d.logits0, d.kp, d.vp, d.steps, W, SCALE, stop_id=stop,
                                 follow=lambda t, rec: rec["active"][:2])
        for a, b in zip(own, fol):
            for k in ("cum", "hist"):
                np.testing.assert_array_equal(a[k], b[k])
            for x, y in zip(a["cand"], b["cand"]):
                np.testing.assert_array_equal(np.asarray(x).view(np.int32), np.asarray(y).view(np.int32))


def test_followed_beams_are_scored_by_the_oracle():
    # a followed beam that the oracle itself did not keep gets the oracle's
    # own score for it: its cumulative score plus its fp32 log-probability
    d = tiny(8)
    last = {}

    def take_third_candidate(t, rec):
        tok, par = (a.copy() for a in rec["active"][:2])
        tok[0], par[0] = rec["cand"][0][W], rec["cand"][1][W]   # rank W: not kept by the oracle
        last[t] = (tok, par)
        return tok, par

    fol = H.beam_decode_loop(d.logits0, d.kp, d.vp, d.steps, W, SCALE, follow=take_third_candidate)
    for t in range(1, len(fol)):
        tok, par = last[t - 1]
        x = f64(d.logits0 if t == 1 else d.steps[t - 2][3])
        prev_cum = fol[t - 1]["cum"]
        lse = logsoftmax(x)
        want = np.asarray(prev_cum, np.float64)[par] + lse[par, tok]
        np.testing.assert_allclose(fol[t]["cum"], want, rtol=0, atol=1e-5)
