"""Replay extensions on the GPU, through the C ABI ("Tail-Replay" notes page):
* gdn_tail_replay_k (caller-chosen tail per request) and gdn_adaptive_replay_plan (section 5, the
  proposed extension) against the oracle;
* gdn_tail_replay_overlap (section 2.5, transfer / replay overlap): identical states, the copy
  delivered, and the overlapped time close to the longer of the two instead of their sum.
"""
import numpy as np
import pytest
import torch

import hybrid_model_recurrent_gb300 as gdn
import oracle
import synth
from parity_util import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gdn.build()
    gdn.lib()
    gdn.clear_status(DEV)
    yield
    assert gdn.read_status(DEV) == gdn.GDN_OK, "a kernel reported a device-side timeout"


def _inputs(seed, lens, H, d, dtype, a_lo, a_hi):
    w = synth.Workload("ext", list(lens), H, d, d, dtype, dtype, a_lo, a_hi, "uniform", seed=seed)
    return w, synth.make_inputs(w)


def _dev(inp):
    return synth.Inputs(inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV), inp.alpha.to(DEV), inp.beta.to(DEV))


@pytest.mark.parametrize("algo", ["per_token", "chunked", "two_pass"])
def test_replay_k_matches_r_based_replay_and_oracle(algo):
    lens = [300, 129, 64]
    H = 2
    w, inp = _inputs(81, lens, H, 128, torch.bfloat16, 0.9, 1.0)
    d = _dev(inp)
    cu = w.cu_seqlens
    m = [300, 100, 64]
    S_a = synth.state(3, w.B * H, 128, 128, 1.0).view(w.B, H, 128, 128)
    a = gdn.gdn_tail_replay(d.q, d.k, d.v, d.alpha, d.beta, cu, m, 1, 10, S_a=S_a.to(DEV), algo=algo)
    b = gdn.gdn_tail_replay_k(d.q, d.k, d.v, d.alpha, d.beta, cu, m, a["k"], S_a=S_a.to(DEV), algo=algo)
    torch.cuda.synchronize()
    assert torch.equal(a["S_hat"], b["S_hat"]) and torch.equal(a["S_exact"], b["S_exact"])
    ks = [7, 100, 0]
    c = gdn.gdn_tail_replay_k(d.q, d.k, d.v, d.alpha, d.beta, cu, m, ks, algo=algo)
    torch.cuda.synchronize()
    for s in range(w.B):
        sl = slice(cu[s], cu[s + 1])
        for h in range(H):
            ref = oracle.tail_replay(inp.k[sl, h], inp.v[sl, h], inp.alpha[sl, h], inp.beta[sl, h], m[s], ks[s],
                                     max(m[s], 1))
            assert_close(c["S_hat"][s, h], ref["S_hat"], f"replay_k s={s} h={h}")


def test_adaptive_plan_matches_oracle_and_meets_the_bound():
    lens = [1200, 700, 2000]
    H = 4
    w, inp = _inputs(83, lens, H, 128, torch.bfloat16, 0.9, 1.0)
    # heads that forget at different rates: head 0 fast, head 3 almost not at all
    alpha = inp.alpha.clone()
    alpha[:, 0] = alpha[:, 0] * 0.9
    alpha[:, 3] = torch.clamp(0.999 + 0.001 * alpha[:, 3], max=1.0)
    inp = synth.Inputs(inp.q, inp.k, inp.v, alpha, inp.beta)
    d = _dev(inp)
    cu = w.cu_seqlens
    m = [1200, 650, 2000]
    for eps, rmax in ((1e-2, (1, 5)), (1e-4, (1, 2)), (0.3, (1, 20))):
        ks, ex = gdn.gdn_adaptive_replay_plan(d.alpha, cu, m, eps, *rmax, H=H)
        ks_o, ex_o = oracle.adaptive_replay_plan(alpha, cu, m, eps, *rmax)
        assert (ks, ex) == (ks_o, ex_o), (eps, rmax)
    # replay the planned tails (exact twin from a seeded S_a) and check ||E|| <= eps ||S_a|| where met
    eps, rmax = 1e-2, (1, 1)
    ks, ex = gdn.gdn_adaptive_replay_plan(d.alpha, cu, m, eps, *rmax, H=H)
    S_a = synth.state(5, w.B * H, 128, 128, 1.0).view(w.B, H, 128, 128)
    r = gdn.gdn_tail_replay_k(d.q, d.k, d.v, d.alpha, d.beta, cu, m, ks, S_a=S_a.to(DEV))
    torch.cuda.synchronize()
    E = (r["S_exact"] - r["S_hat"]).double().cpu()
    for s in range(w.B):
        if ex[s]:
            continue
        for h in range(H):
            bound = eps * float(torch.linalg.norm(S_a[s, h].double()))
            assert float(torch.linalg.norm(E[s, h])) <= bound * (1 + 1e-3) + 1e-5, (s, h)


def test_adaptive_plan_reads_the_gates_after_earlier_work_on_its_stream():
    """The plan copies the gates on the caller's stream: gates that earlier work on that stream is still writing (here
    a copy queued behind a device-side delay, on a non-blocking stream) are the ones it reads."""
    lens = [800, 600]
    H = 2
    w, inp = _inputs(87, lens, H, 128, torch.bfloat16, 0.9, 1.0)
    cu = w.cu_seqlens
    m = [800, 600]
    eps, rmax = 1e-2, (1, 2)
    fast = inp.alpha * 0.5                 # forgets within a few tokens
    slow = torch.ones_like(inp.alpha)      # never forgets: the budget is too short for every head
    want_fast = oracle.adaptive_replay_plan(fast, cu, m, eps, *rmax)
    want_slow = oracle.adaptive_replay_plan(slow, cu, m, eps, *rmax)
    assert want_fast != want_slow
    side = torch.cuda.Stream()
    alpha_d = slow.to(DEV)
    fast_h = fast.pin_memory()
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        torch.cuda._sleep(20_000_000)          # ~10 ms on the side stream before the gates change
        alpha_d.copy_(fast_h, non_blocking=True)
    got = gdn.gdn_adaptive_replay_plan(alpha_d, cu, m, eps, *rmax, H=H, stream=side)
    assert got == want_fast, "the plan must see the gates written before it on its stream"
    torch.cuda.synchronize()


def _timed(stream, fn, reps=5):
    """Median device time of fn on stream.  The GPU is kept busy while the host enqueues fn, so that the
    host's own time for the call (argument checks, the launch plan) is not counted."""
    fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(2_000_000)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return float(np.median(ts))


def test_overlap_gives_identical_states_and_runs_the_legs_concurrently():
    """The copy and the replay run at the same time.  Per overlapped call, events on the two streams give the
    copy's end (B, recorded on the copy stream after the call) and the call's end (C, on the compute stream,
    which joins the copy), both from the call's start (A).  The replay is sized to take about twice as long as
    the copy, so:
      - the copy ends well before the call does (it did not wait for the replay): B - A < 0.75 (C - A);
      - the replay did not wait for the copy: C - B is shorter than the replay alone by at least half the
        copy's time in the same call, C - B < T_replay - 0.5 (B - A).
    Each bound compares times of one call, or a kernel's time on an otherwise idle GPU, so a busy host link
    moves both sides alike.  The overlap's speed-up itself is reported by the benchmark."""
    H, T = 256, 1024                       # 256 (layer, head) scans, a 1024-token tail each
    w, inp = _inputs(85, [T], H, 128, torch.bfloat16, 0.97, 1.0)
    d = _dev(inp)
    cu, m = w.cu_seqlens, [T]
    comp = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    ref = gdn.gdn_tail_replay(d.q, d.k, d.v, d.alpha, d.beta, cu, m, 1, 1)
    torch.cuda.synchronize()
    t_rep = _timed(comp, lambda: gdn.gdn_tail_replay(d.q, d.k, d.v, d.alpha, d.beta, cu, m, 1, 1))
    # size the transfer to take about half as long as the replay
    probe_h = torch.empty(64 << 20, dtype=torch.uint8).pin_memory()
    probe_d = torch.empty_like(probe_h, device=DEV)
    t_probe = _timed(comp, lambda: probe_d.copy_(probe_h, non_blocking=True))
    nbytes = int(min(max(probe_h.numel() * 0.5 * t_rep / t_probe, 1 << 20), 2 << 30)) // 4096 * 4096
    kv_h = torch.randint(0, 255, (nbytes,), dtype=torch.uint8).pin_memory()
    kv_d = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)

    def overlapped():
        return gdn.gdn_tail_replay_overlap(d.q, d.k, d.v, d.alpha, d.beta, cu, m, 1, 1, kv_h, kv_d,
                                           copy_stream=copy)

    r = overlapped()
    torch.cuda.synchronize()
    assert torch.equal(r["S_hat"], ref["S_hat"]), "the overlapped replay must not change the states"
    assert torch.equal(kv_d.cpu(), kv_h), "the copy was not delivered"
    copy_end, call_end = [], []
    for _ in range(5):
        ea, eb, ec = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        torch.cuda.synchronize()
        # keep the GPU busy while the host enqueues the call, so that its launch overhead is not timed
        torch.cuda._sleep(2_000_000)
        ea.record(comp)
        overlapped()
        eb.record(copy)
        ec.record(comp)
        torch.cuda.synchronize()
        copy_end.append(ea.elapsed_time(eb))
        call_end.append(ea.elapsed_time(ec))
    b, c = float(np.median(copy_end)), float(np.median(call_end))
    print(f"T_replay {t_rep:.3f} ms; overlapped call: copy done at {b:.3f} ms, call done at {c:.3f} ms")
    assert b < 0.75 * c, "the copy ended with the call: it waited for the replay"
    assert c - b < t_rep - 0.5 * b, "the replay started only when the copy was done"


@pytest.mark.parametrize("L,H,Dm,d,m,rn,rd", [(3, 4, 256, 64, 700, 1, 10), (2, 2, 128, 128, 300, 1, 20),
                                              (2, 3, 96, 32, 129, 1, 1)])
def test_group_replay_matches_oracle(L, H, Dm, d, m, rn, rd):
    from oracle import group as G
    w = synth.group_weights(7, L, H, Dm, d)
    h = synth.group_inputs(7, m, Dm)
    r = gdn.gdn_group_replay(h.to(DEV), w.to(DEV), L, H, Dm, d, m, rn, rd)
    torch.cuda.synchronize()
    ref = G.group_replay(h, w, L, H, Dm, d, m, rn, rd)
    assert (r["a"], r["k"]) == (ref["a"], ref["k"])
    errs = []
    for l in range(L):
        for hh in range(H):
            assert_close(r["S_hat"][l, hh], ref["S_hat"][l][hh], f"group S_hat layer {l} head {hh}")
            assert_close(r["S_exact"][l, hh], ref["S_exact"][l][hh], f"group S_exact layer {l} head {hh}")
            e = np.linalg.norm(ref["S_exact"][l][hh] - ref["S_hat"][l][hh]) / np.linalg.norm(ref["S_exact"][l][hh])
            errs.append(round(float(e), 4))
    print(f"relative replay error per (layer, head): {errs}")
    if rn == rd:
        assert torch.equal(r["S_hat"], r["S_exact"])
