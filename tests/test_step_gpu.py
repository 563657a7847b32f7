"""gdn_step (a serving step's prefills, resumes and tail replays in one launch) against the
three entry points called one by one, and against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import hybrid_model_recurrent_gb300 as gdn
import oracle
import synth
from parity_util import assert_close, check_output

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gdn.build()
    gdn.lib()
    gdn.clear_status(DEV)
    yield
    assert gdn.read_status(DEV) == gdn.GDN_OK, "a kernel reported a device-side timeout"


def _case(seed, lens, H, d, dtype):
    w = synth.Workload("step", list(lens), H, d, d, dtype, dtype, 0.9, 1.0, "sigmoid", seed=seed)
    inp = synth.make_inputs(w, device="cpu")
    dev = synth.Inputs(*(t.to(DEV) for t in (inp.q, inp.k, inp.v, inp.alpha, inp.beta)))
    return w, inp, dev


CASES = [(128, torch.bfloat16, "chunked"), (128, torch.bfloat16, "two_pass"), (128, torch.bfloat16, "chunked_mma"),
         (128, torch.bfloat16, "per_token"), (64, torch.float32, "auto"), (32, torch.bfloat16, "auto")]


@pytest.mark.parametrize("d,dtype,algo", CASES)
def test_step_equals_the_three_calls_bitwise(d, dtype, algo):
    lens = [300, 130, 77]
    H = 2
    w, inp, x = _case(41, lens, H, d, dtype)
    cu = w.cu_seqlens
    S0 = synth.state(43, w.B * H, d, d, 0.3).view(w.B, H, d, d).to(DEV)
    ck_new = [[50, 100, 290], [64], []]
    # the resumes read checkpoints an earlier prefill stored (seeded states here, another buffer)
    ck_old = [[64, 128, 192, 256], [1, 64], [77]]
    store = synth.state(47, 7 * H, d, d, 0.7).view(7, H, d, d).to(DEV)
    probes = [(0, 0), (0, 63), (0, 64), (0, 200), (0, 300), (1, 0), (1, 1), (1, 130), (2, 76), (2, 77), (0, 129)]
    m = [280, 130, 50]
    S_a = synth.state(53, w.B * H, d, d, 0.5).view(w.B, H, d, d).to(DEV)
    out = torch.bfloat16 if dtype == torch.bfloat16 else torch.float32

    pf = gdn.gdn_prefill_ckpt(x.q, x.k, x.v, x.alpha, x.beta, cu, S0=S0, ckpt_pos=ck_new, out_dtype=out, algo=algo)
    rs = gdn.gdn_resume_from_ckpt(x.q, x.k, x.v, x.alpha, x.beta, cu, store, ck_old, probes, S0=S0, out_dtype=out,
                                  algo=algo)
    rp = gdn.gdn_tail_replay(x.q, x.k, x.v, x.alpha, x.beta, cu, m, 1, 10, S_a=S_a, readout=True, out_dtype=out,
                             algo=algo)
    st = gdn.gdn_step(x.q, x.k, x.v, x.alpha, x.beta, cu, out_dtype=out, algo=algo,
                      prefill=dict(S0=S0, ckpt_pos=ck_new),
                      resume=dict(ckpt_states=store, ckpt_pos=ck_old, probes=probes, S0=S0),
                      replay=dict(m=m, r_num=1, r_den=10, S_a=S_a, readout=True))
    torch.cuda.synchronize()
    a, b = st["prefill"], pf
    assert torch.equal(a["o"], b["o"]) and torch.equal(a["S_final"], b["S_final"])
    assert torch.equal(a["ckpt_states"], b["ckpt_states"])
    a, b = st["resume"], rs
    assert a["chosen"] == b["chosen"] and a["offsets"] == b["offsets"]
    assert torch.equal(a["S_out"], b["S_out"]) and torch.equal(a["o"], b["o"])
    a, b = st["replay"], rp
    assert a["a"] == b["a"] and a["k"] == b["k"]
    assert torch.equal(a["S_hat"], b["S_hat"])
    # the replay's rows of o: only [a_b, m_b) of each sequence is written
    for s in range(w.B):
        rows = slice(cu[s] + b["a"][s], cu[s] + m[s])
        assert torch.equal(a["o"][rows], b["o"][rows])
    if algo == "per_token" or d != 128 or dtype != torch.bfloat16:
        # the per-token kernel's own twin mode splits a CTA's rows between the two scans; the step runs the
        # twin as a job of its own, so the two agree to rounding
        for s in range(w.B):
            for h in range(H):
                assert_close(a["S_exact"][s, h].cpu(), b["S_exact"][s, h].cpu().double(), f"twin s={s} h={h}")
    else:
        assert torch.equal(a["S_exact"], b["S_exact"])

    # one sequence of each part against the oracle as well
    sl = slice(cu[0], cu[1])
    for h in range(H):
        ref = oracle.prefill(inp.q[sl, h], inp.k[sl, h], inp.v[sl, h], inp.alpha[sl, h], inp.beta[sl, h],
                             S0=S0[0, h].cpu(), ckpt_pos=ck_new[0], want_o=True)
        assert_close(st["prefill"]["S_final"][0, h], ref["S"], f"prefill S h={h}")
        check_output(st["prefill"]["o"][sl, h], ref["o"], f"prefill o h={h}")
        stc = store.cpu()
        ref = oracle.resume(inp.q[sl, h], inp.k[sl, h], inp.v[sl, h], inp.alpha[sl, h], inp.beta[sl, h],
                            [stc[j, h] for j in range(4)], ck_old[0], 200, S0=S0[0, h].cpu())
        assert st["resume"]["chosen"][3] == ref["c"]
        assert_close(st["resume"]["S_out"][3, h], ref["S"], f"resume S h={h}")
        ref = oracle.tail_replay(inp.k[sl, h], inp.v[sl, h], inp.alpha[sl, h], inp.beta[sl, h], m[0], 1, 10,
                                 S_a=S_a[0, h].cpu())
        assert_close(st["replay"]["S_hat"][0, h], ref["S_hat"], f"replay S_hat h={h}")
        assert_close(st["replay"]["S_exact"][0, h], ref["S_exact"], f"replay S_exact h={h}")


def test_step_parts_are_optional_and_empty_jobs_work():
    lens = [200, 64]
    H = 2
    w, inp, x = _case(59, lens, H, 128, torch.bfloat16)
    cu = w.cu_seqlens
    ck = [[64, 128], [64]]
    store = synth.state(61, 3 * H, 128, 128, 0.7).view(3, H, 128, 128).to(DEV)
    # every probe sits on a checkpoint or at depth 0: no token to recompute
    probes = [(0, 64), (0, 128), (1, 64), (0, 0)]
    st = gdn.gdn_step(x.q, x.k, x.v, x.alpha, x.beta, cu, resume=dict(ckpt_states=store, ckpt_pos=ck,
                                                                     probes=probes, readout=False))
    rp = gdn.gdn_step(x.q, x.k, x.v, x.alpha, x.beta, cu, replay=dict(m=[0, 64], r_num=0, r_den=1))
    torch.cuda.synchronize()
    S = st["resume"]["S_out"]
    assert torch.equal(S[0], store[0]) and torch.equal(S[1], store[1]) and torch.equal(S[2], store[2])
    assert torch.count_nonzero(S[3]) == 0                # depth 0 without S0: the zero state
    assert st["resume"]["offsets"] == [0, 0, 0, 0, 0]
    assert rp["replay"]["k"] == [0, 0] and torch.count_nonzero(rp["replay"]["S_hat"]) == 0
    none = gdn.gdn_step(x.q, x.k, x.v, x.alpha, x.beta, cu)
    assert none == {}


def test_step_refuses_resumes_from_checkpoints_it_writes():
    w, inp, x = _case(67, [128], 1, 128, torch.bfloat16)
    ck = torch.zeros((2, 1, 128, 128), dtype=torch.float32, device=DEV)
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_step(x.q, x.k, x.v, x.alpha, x.beta, w.cu_seqlens,
                     prefill=dict(ckpt_pos=[[64, 128]], ckpt_states=ck),
                     resume=dict(ckpt_states=ck, ckpt_pos=[[64, 128]], probes=[(0, 100)]))
    assert e.value.status == gdn.GDN_ERR_INVALID_ARG


def test_step_at_full_size_in_the_benchmark_configuration():
    """The benchmark's step: 8 x 16 heads x 8192 tokens, 16 checkpoints, 16 resume probes from a store an
    earlier prefill wrote, 5 % tail replays, as one launch.  Bit for bit the three entry points' results, and
    sampled (sequence, head) streams against the oracle."""
    import dataclasses
    w = synth.workload("prefill")
    x = synth.make_inputs(w, device=DEV)
    cu, ck = w.cu_seqlens, w.ckpt_positions()
    probes = dataclasses.replace(w, n_probes=16).probes()
    m = list(w.seq_lens)
    ws = gdn.workspace(DEV)
    store = gdn.gdn_prefill_ckpt(x.q, x.k, x.v, x.alpha, x.beta, cu, ckpt_pos=ck, ws=ws)["ckpt_states"]
    st = gdn.gdn_step(x.q, x.k, x.v, x.alpha, x.beta, cu, ws=ws, prefill=dict(ckpt_pos=ck),
                      resume=dict(ckpt_states=store, ckpt_pos=ck, probes=probes),
                      replay=dict(m=m, r_num=1, r_den=20))
    pf = gdn.gdn_prefill_ckpt(x.q, x.k, x.v, x.alpha, x.beta, cu, ckpt_pos=ck, ws=ws)
    rs = gdn.gdn_resume_from_ckpt(x.q, x.k, x.v, x.alpha, x.beta, cu, store, ck, probes, ws=ws)
    rp = gdn.gdn_tail_replay(None, x.k, x.v, x.alpha, x.beta, cu, m, 1, 20, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(st["prefill"]["o"], pf["o"]) and torch.equal(st["prefill"]["S_final"], pf["S_final"])
    assert torch.equal(st["prefill"]["ckpt_states"], pf["ckpt_states"])
    assert torch.equal(st["prefill"]["ckpt_states"], store), "the store and the step's own dumps agree"
    assert st["resume"]["chosen"] == rs["chosen"] and st["resume"]["offsets"] == rs["offsets"]
    assert torch.equal(st["resume"]["S_out"], rs["S_out"]) and torch.equal(st["resume"]["o"], rs["o"])
    assert st["replay"]["k"] == rp["k"] == [410] * w.B and torch.equal(st["replay"]["S_hat"], rp["S_hat"])
    # sampled streams against the oracle (its checkpoints its own)
    for i, h in ((0, 5), (7, 11)):
        s, d = probes[i]
        sl = slice(cu[s], cu[s + 1])
        args = (x.q[sl, h].cpu(), x.k[sl, h].cpu(), x.v[sl, h].cpu(), x.alpha[sl, h].cpu(), x.beta[sl, h].cpu())
        ref = oracle.prefill(*args, ckpt_pos=ck[s], want_o=False)
        res = oracle.resume(*args, list(ref["ckpt"]), ck[s], d)
        assert st["resume"]["chosen"][i] == res["c"]
        assert_close(st["resume"]["S_out"][i, h], res["S"], f"step resume probe {i} h={h}")
        lo, hi = st["resume"]["offsets"][i], st["resume"]["offsets"][i + 1]
        if hi > lo:
            check_output(st["resume"]["o"][lo:hi, h], res["o"], f"step resume o probe {i} h={h}")
        rep = oracle.tail_replay(args[1], args[2], args[3], args[4], m[s], 1, 20)
        assert_close(st["replay"]["S_hat"][s, h], rep["S_hat"], f"step replay s={s} h={h}")


def test_step_lanes_never_share_a_two_pass_workspace():
    """A workspace large enough for the long lane's two-pass path but not for the whole job list: the step
    runs its two lanes side by side, so neither may take the two-pass path (they would share its schedule and
    T areas).  Bit for bit the fused kernel's results from the three entry points."""
    lens = [1024, 1024]
    H, d = 4, 128
    w, inp, x = _case(71, lens, H, d, torch.bfloat16)
    cu = w.cu_seqlens
    ck = [[256, 512, 768, 1024], [256, 512, 1024]]
    store = synth.state(73, 7 * H, d, d, 0.7).view(7, H, d, d).to(DEV)
    probes = [(0, 300), (0, 700), (1, 600), (1, 1000), (0, 256)]
    m = [1024, 900]
    L = gdn.lib()
    head = int(L.gdn_workspace_size_two_pass(sum(lens), H, len(lens)))
    tail_tokens = sum(d_ - max(c for c in [0] + ck[s] if c <= d_) for s, d_ in probes) + sum(
        -(-mm // 10) for mm in m)
    whole = int(L.gdn_workspace_size_two_pass(sum(lens) + tail_tokens, H, len(lens) + len(probes) + len(m)))
    assert head < whole
    ws = torch.zeros(head, dtype=torch.uint8, device=DEV)
    ws_fused = torch.zeros(int(L.gdn_workspace_size()), dtype=torch.uint8, device=DEV)
    for _ in range(2):
        st = gdn.gdn_step(x.q, x.k, x.v, x.alpha, x.beta, cu, ws=ws, prefill=dict(ckpt_pos=ck),
                          resume=dict(ckpt_states=store, ckpt_pos=ck, probes=probes),
                          replay=dict(m=m, r_num=1, r_den=10))
        pf = gdn.gdn_prefill_ckpt(x.q, x.k, x.v, x.alpha, x.beta, cu, ckpt_pos=ck, ws=ws_fused, algo="chunked")
        rs = gdn.gdn_resume_from_ckpt(x.q, x.k, x.v, x.alpha, x.beta, cu, store, ck, probes, ws=ws_fused,
                                      algo="chunked")
        rp = gdn.gdn_tail_replay(None, x.k, x.v, x.alpha, x.beta, cu, m, 1, 10, ws=ws_fused, algo="chunked")
        torch.cuda.synchronize()
        assert gdn.read_status(DEV, ws=ws) == gdn.GDN_OK
        assert torch.equal(st["prefill"]["o"], pf["o"]) and torch.equal(st["prefill"]["S_final"], pf["S_final"])
        assert torch.equal(st["prefill"]["ckpt_states"], pf["ckpt_states"])
        assert torch.equal(st["resume"]["S_out"], rs["S_out"]) and torch.equal(st["resume"]["o"], rs["o"])
        assert torch.equal(st["replay"]["S_hat"], rp["S_hat"])
