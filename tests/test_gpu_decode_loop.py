"""GPU parity of the fixed-depth beam search loop (article "SLM 生成式高并发推理引擎：
延迟约束下的有效吞吐优化", section 2.3) against the oracle's loop.

Every step is compared: the selection (bit-exact given the GPU's own fp32
normalisers and cumulative scores; against the oracle's own, differences
only at near ties that the normalisers explain), the finished-beam split
(exact, on the GPU's own candidates and against the oracle's own split), the
token history (exact), the attention output (within the attention tolerance),
the reordered suffix K/V (bit exact) and the cumulative scores (the oracle's
own against the GPU's, within the accumulated normaliser band).  The oracle
runs its own loop and takes only the kept beams' identity from the GPU, so
that a near tie resolved the other way cannot make later steps incomparable.
The loop captured as one CUDA graph must give the eager results bit for bit,
also after new inputs are copied into its tensors.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import heads as H
from attention_packed_varlen_gb300 import _binding as slm
from attention_packed_varlen_gb300 import build, workloads as wl
from attention_packed_varlen_gb300.decode_loop import BeamDecodeLoop
from tests.parity import check_attention, check_selection

pytestmark = pytest.mark.gpu
DEV = "cuda"
THREADS = oracle.default_threads()
STOP = 151643


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    slm.load()


def to_dev(d):
    dev = torch.device(DEV)
    return (d.logits0.to(dev), d.kp.to(dev), d.vp.to(dev),
            [tuple(x.to(dev) for x in s) for s in d.steps])


def make_loop(bw, stop_id):
    return BeamDecodeLoop(bw.beams, bw.vocab, bw.steps, bw.prefix_len, bw.n_q_heads, bw.n_kv_heads, bw.head_dim,
                          stop_id=stop_id, softmax_scale=bw.softmax_scale)


def snapshot(loop):
    """Every per-step result the loop keeps, copied to the host."""
    out = {"hist": [h.cpu().clone() for h in loop.hist], "o": [o.cpu().clone() for o in loop.o],
           "ks": [k.cpu().clone() for k in loop.ks], "vs": [v.cpu().clone() for v in loop.vs],
           "sel": [{k: v.cpu().clone() for k, v in s.items()} for s in loop.sel]}
    if loop.fin is not None:  # finished entries past the count are not written
        out["fin"] = []
        for f in loop.fin:
            n = int(f["fin_count"][0])
            out["fin"].append({k: (v[:n] if k.startswith("fin_") and k != "fin_count" else v).cpu().clone()
                               for k, v in f.items()})
    return out


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def check_against_oracle(bw, d, snap, stop_id):
    """Runs the oracle's own loop beside the GPU's.  At each step, before the
    oracle goes on, the GPU's selection is checked against the oracle's record
    of that step (bit-exact given the GPU's own normalisers and cumulative
    scores; near ties explained otherwise); then the oracle takes the GPU's
    kept beams' identity (token, parent) -- its own when nothing differed --
    and scores them itself.  So the oracle's cumulative scores never come from
    the GPU, and they are compared with the GPU's at every step."""
    W = bw.beams
    act = (lambda t: snap["fin"][t]) if stop_id is not None else (lambda t: snap["sel"][t])
    stats = {"near": 0, "fin": 0, "max_cum_diff": 0.0}
    band = [0.0]  # accumulated bound on |GPU cum - oracle cum|

    def follow(t, rec):
        what = f"{bw.name} step {t}"
        logits = d.logits0 if t == 0 else d.steps[t - 1][3]
        cum_g = np.zeros(1, np.float32) if t == 0 else act(t - 1)["score"].numpy()
        cum_o = rec["cum"]
        diff = float(np.abs(cum_g.astype(np.float64) - np.asarray(cum_o, np.float64)).max())
        assert diff <= band[0], f"{what}: cumulative scores differ by {diff:.3g} > {band[0]:.3g}"
        stats["max_cum_diff"] = max(stats["max_cum_diff"], diff)
        near, delta = check_selection(snap["sel"][t], rec["cand"], logits, cum_g, W, cum_oracle=cum_o)
        band[0] = delta  # a kept candidate's score moves by at most delta
        stats["near"] += near
        g_act = act(t)
        if near == 0:  # same candidates: the finished split must agree too
            np.testing.assert_array_equal(g_act["token"].numpy(), rec["active"][0], err_msg=what)
            np.testing.assert_array_equal(g_act["parent"].numpy(), rec["active"][1], err_msg=what)
            if stop_id is not None:
                f = snap["fin"][t]
                nf = int(f["fin_count"][0])
                assert [x[1] for x in rec["finished"]] == f["fin_parent"][:nf].tolist(), what
                got = f["fin_score"][:nf].numpy().astype(np.float64)
                want = np.array([x[2] for x in rec["finished"]], np.float64)
                assert (np.abs(got - want) <= delta).all(), what
        return g_act["token"].numpy(), g_act["parent"].numpy()

    recs = H.beam_decode_loop(d.logits0, d.kp, d.vp, d.steps, W, bw.softmax_scale, stop_id=stop_id,
                              follow=follow, n_threads=THREADS)
    for t, rec in enumerate(recs):
        what = f"{bw.name} step {t}"
        if stop_id is not None:
            g = snap["sel"][t]
            a_ref, f_ref = H.split_finished(g["cand_token"].numpy(), g["cand_parent"].numpy(),
                                            g["cand_score"].numpy(), W, stop_id)
            f = snap["fin"][t]
            nf = int(f["fin_count"][0])
            assert nf == len(f_ref), what
            stats["fin"] += nf
            assert f["fin_parent"][:nf].tolist() == [x[1] for x in f_ref], what
            np.testing.assert_array_equal(f["fin_score"][:nf].numpy(), np.array([x[2] for x in f_ref], np.float32))
            assert f["token"].tolist() == [x[0] for x in a_ref], what
            assert f["parent"].tolist() == [x[1] for x in a_ref], what
            np.testing.assert_array_equal(f["score"].numpy(), np.array([x[2] for x in a_ref], np.float32))
        np.testing.assert_array_equal(snap["hist"][t][:, :t + 1].numpy(), rec["hist"], err_msg=what)
        if t >= 1:
            check_attention(snap["o"][t - 1], rec["o"], what)
            np.testing.assert_array_equal(bits(snap["ks"][t])[:, :t], rec["ks"][:, :t], err_msg=what)
            np.testing.assert_array_equal(bits(snap["vs"][t])[:, :t], rec["vs"][:, :t], err_msg=what)
    # the GPU's final cumulative scores against the oracle's own for the same beams
    last_o = H.candidate_scores(d.steps[-1][3], recs[-1]["cum"], recs[-1]["cand"][3],
                                act(len(recs) - 1)["parent"].numpy(), act(len(recs) - 1)["token"].numpy())
    diff = float(np.abs(act(len(recs) - 1)["score"].numpy().astype(np.float64) - last_o).max())
    assert diff <= band[0], f"final cumulative scores differ by {diff:.3g} > {band[0]:.3g}"
    return stats["near"], stats["fin"]


@pytest.mark.parametrize("workload,index,stop_id", [
    (wl.SHORT_PROMPT_BEAM, 4, None), (wl.SHORT_PROMPT_BEAM, 4, STOP),
    (wl.LONG_PROMPT_WIDE_BEAM, 5, None), (wl.LONG_PROMPT_WIDE_BEAM, 5, STOP)])
def test_loop_every_step_matches_oracle(workload, index, stop_id):
    d = wl.decode_loop_inputs(workload, wl.workload_seed(index, 7), stop_id=stop_id,
                              stop_rows=0.3 if stop_id is not None else 0.0)
    loop = make_loop(workload, stop_id)
    loop.record(*to_dev(d))
    torch.cuda.synchronize()
    slm.slm_check_status(loop.status)
    n_near, n_fin = check_against_oracle(workload, d, snapshot(loop), stop_id)
    print(f"{workload.name}: {n_near} near ties over {workload.steps + 1} selections, all explained")
    if stop_id is not None:
        assert n_fin > 0, "no hypothesis finished: the stop rows did not reach the kept candidates"


@pytest.mark.parametrize("stop_id", [None, STOP])
def test_graph_replay_equals_eager_and_takes_new_inputs(stop_id):
    bw = wl.SHORT_PROMPT_BEAM
    d1 = wl.decode_loop_inputs(bw, 11, stop_id=stop_id, stop_rows=0.3 if stop_id is not None else 0.0)
    d2 = wl.decode_loop_inputs(bw, 12, stop_id=stop_id, stop_rows=0.3 if stop_id is not None else 0.0)
    static = to_dev(d1)
    loop = make_loop(bw, stop_id)
    loop.record(*static)
    torch.cuda.synchronize()
    loop.capture(*static)
    # new inputs into the captured tensors
    new = to_dev(d2)
    static[0].copy_(new[0]); static[1].copy_(new[1]); static[2].copy_(new[2])
    for s_old, s_new in zip(static[3], new[3]):
        for a, b in zip(s_old, s_new):
            a.copy_(b)
    loop.replay()
    torch.cuda.synchronize()
    slm.slm_check_status(loop.status)
    graph2 = snapshot(loop)
    check_against_oracle(bw, d2, graph2, stop_id)
    # an eager run on the second inputs must give the replay's results exactly
    loop2 = make_loop(bw, stop_id)
    loop2.record(*to_dev(d2))
    torch.cuda.synchronize()
    eager2 = snapshot(loop2)
    for key in eager2:
        for a, b in zip(eager2[key], graph2[key]):
            if isinstance(a, dict):
                for k in a:
                    assert torch.equal(a[k], b[k]), (key, k)
            else:
                assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                                   b.view(torch.int16) if b.dtype == torch.bfloat16 else b), key


@pytest.mark.parametrize("stop_id", [None, STOP])
def test_graph_replays_repeat_the_same_beams(stop_id):
    # Many replays of the wide-beam loop: every selection, history and
    # reordered suffix must repeat bit for bit (the logits are inputs, so
    # nothing upstream of a selection varies), and the attention output may
    # differ only by the key-split merge's fp32 summation order.  A race in
    # any kernel's pipeline, or between kernels that start their setup while
    # the one before still runs, would show up here as a replay that differs.
    bw = wl.LONG_PROMPT_WIDE_BEAM
    d = wl.decode_loop_inputs(bw, 21, stop_id=stop_id, stop_rows=0.3 if stop_id is not None else 0.0)
    static = to_dev(d)
    loop = make_loop(bw, stop_id)
    loop.record(*static)
    torch.cuda.synchronize()
    loop.capture(*static)
    loop.replay()
    torch.cuda.synchronize()
    first = snapshot(loop)
    ref = [{k: v.clone() for k, v in sel.items()} for sel in loop.sel]
    ref_hist = [h.clone() for h in loop.hist]
    for r in range(200):
        loop.replay()
        if r % 10 == 9:  # compared on the device every tenth replay
            torch.cuda.synchronize()
            for a, b in zip(loop.sel, ref):
                for k in a:
                    assert torch.equal(a[k], b[k]), ("replay", r, k)
            for a, b in zip(loop.hist, ref_hist):
                assert torch.equal(a, b), ("replay", r, "hist")
    torch.cuda.synchronize()
    slm.slm_check_status(loop.status)
    last = snapshot(loop)
    for key in ("hist", "ks", "vs"):
        for a, b in zip(first[key], last[key]):
            assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                               b.view(torch.int16) if b.dtype == torch.bfloat16 else b), key
    for a, b in zip(first["sel"], last["sel"]):
        for k in a:
            assert torch.equal(a[k], b[k]), ("sel", k)
    if stop_id is not None:
        for a, b in zip(first["fin"], last["fin"]):
            for k in a:
                assert torch.equal(a[k], b[k]), ("fin", k)
    for a, b in zip(first["o"], last["o"]):
        gap = (a.float() - b.float()).abs()
        lim = torch.maximum(a.float().abs(), b.float().abs()) * 2.0 ** -7 + 2.0 ** -20
        assert bool((gap <= lim).all()), float(gap.max())
