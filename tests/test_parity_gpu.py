"""CUDA path against the fp64 oracle, element by element, through the C ABI.

Small cases compare every output; the full-size workloads (in the launch
configuration the benchmark uses) compare sampled (sequence, head) streams that
the oracle recomputes one by one.  Inputs come from the seeded generator only;
no oracle input or expected value comes from the CUDA path.
"""
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


def _seq(t, cu, b):
    return t[cu[b]:cu[b + 1]]


def _inputs(seed, lens, H, dk, dv, dtype, a_lo=0.9, a_hi=1.0, beta="uniform", device="cpu"):
    w = synth.Workload("case", list(lens), H, dk, dv, dtype, dtype, a_lo, a_hi, beta, seed=seed)
    return w, synth.make_inputs(w, device=device)


def _oracle_prefill_head(inp, cu, b, h, S0=None, ckpt=(), want_o=True):
    sl = slice(cu[b], cu[b + 1])
    return oracle.prefill(inp.q[sl, h], inp.k[sl, h], inp.v[sl, h], inp.alpha[sl, h], inp.beta[sl, h],
                          S0=S0, ckpt_pos=ckpt, want_o=want_o)


def _dev(inp):
    return synth.Inputs(inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV), inp.alpha.to(DEV), inp.beta.to(DEV))


# ---------------------------------------------------------------------------------------------
# Tiny workload: every output of all three operations
# ---------------------------------------------------------------------------------------------
def test_tiny_prefill_resume_replay():
    w = synth.workload("tiny")
    inp = synth.make_inputs(w)
    d = _dev(inp)
    cu = w.cu_seqlens
    ck = w.ckpt_positions()
    r = gdn.gdn_prefill_ckpt(d.q, d.k, d.v, d.alpha, d.beta, cu, ckpt_pos=ck, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = [_oracle_prefill_head(inp, cu, 0, h, ckpt=ck[0]) for h in range(w.H)]
    for h in range(w.H):
        assert_close(r["o"][:, h], ref[h]["o"], f"tiny o head {h}")
        assert_close(r["S_final"][0, h], ref[h]["S"], f"tiny S_N head {h}")
        for i in range(len(ck[0])):
            assert_close(r["ckpt_states"][i, h], ref[h]["ckpt"][i], f"tiny ckpt {ck[0][i]} head {h}")

    # resume from the GPU's own checkpoints vs the oracle resuming from its own
    depths = [0, 1, 63, 64, 65, 100, 128, 129, 200, 255, 256]
    probes = [(0, dd) for dd in depths]
    rs = gdn.gdn_resume_from_ckpt(d.q, d.k, d.v, d.alpha, d.beta, cu, r["ckpt_states"], ck, probes,
                                  out_dtype=torch.float32)
    torch.cuda.synchronize()
    for i, dd in enumerate(depths):
        for h in range(w.H):
            o_ = oracle.resume(inp.q[:, h], inp.k[:, h], inp.v[:, h], inp.alpha[:, h], inp.beta[:, h],
                               ref[h]["ckpt"], ck[0], dd)
            assert rs["chosen"][i] == o_["c"], "chosen checkpoint is an index: bit-exact"
            assert_close(rs["S_out"][i, h], o_["S"], f"tiny resume d={dd} head {h}")
            lo, hi = rs["offsets"][i], rs["offsets"][i + 1]
            assert hi - lo == dd - o_["c"]
            if hi > lo:
                assert_close(rs["o"][lo:hi, h], o_["o"], f"tiny resume o d={dd} head {h}")

    # Tail-Replay r = 0.05 from m = 256 (k = 13, a = 243) with the exact twin from S_a
    a_, k_ = oracle.replay_plan(256, 1, 20)
    assert (a_, k_) == (243, 13)
    S_a = np.stack([_oracle_prefill_head(inp, cu, 0, h, ckpt=[a_], want_o=False)["ckpt"][0] for h in range(w.H)])
    S_a_t = torch.from_numpy(S_a).to(torch.float32)[None].to(DEV)
    rp = gdn.gdn_tail_replay(d.q, d.k, d.v, d.alpha, d.beta, cu, [256], 1, 20, S_a=S_a_t, readout=True,
                             out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert rp["a"] == [243] and rp["k"] == [13]
    for h in range(w.H):
        o_ = oracle.tail_replay(inp.k[:, h], inp.v[:, h], inp.alpha[:, h], inp.beta[:, h], 256, 1, 20,
                                S_a=S_a_t[0, h].cpu(), q=inp.q[:, h], want_o=True)
        assert_close(rp["S_hat"][0, h], o_["S_hat"], f"tiny S_hat head {h}")
        assert_close(rp["S_exact"][0, h], o_["S_exact"], f"tiny S_exact head {h}")
        assert_close(rp["o"][243:256, h], o_["o"], f"tiny replay o head {h}")
        E = (rp["S_exact"][0, h] - rp["S_hat"][0, h]).double().cpu().numpy()
        assert_close(E, o_["S_exact"] - o_["S_hat"], f"tiny E_m head {h}", tol=1e-3)


# ---------------------------------------------------------------------------------------------
# Ragged batches spanning several 32-token tiles with ragged tails, every d_k
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("dk,dv,dtype,out,algo", [
    (64, 64, torch.bfloat16, torch.bfloat16, "auto"), (64, 64, torch.bfloat16, torch.float32, "auto"),
    (128, 128, torch.bfloat16, torch.bfloat16, "per_token"), (128, 128, torch.bfloat16, torch.bfloat16, "chunked"),
    (128, 128, torch.bfloat16, torch.float32, "chunked"), (128, 128, torch.bfloat16, torch.bfloat16, "chunked_mma"),
    (128, 128, torch.bfloat16, torch.bfloat16, "two_pass"), (128, 128, torch.bfloat16, torch.float32, "two_pass"),
    (128, 128, torch.float32, torch.float32, "auto"),
    (32, 32, torch.bfloat16, torch.float32, "auto"), (128, 64, torch.bfloat16, torch.float32, "auto"),
    (64, 128, torch.float32, torch.bfloat16, "auto"), (32, 128, torch.bfloat16, torch.bfloat16, "auto"),
    # d_k = 128 on the per-token path with 2 and 4 warps (the warps stage their own inputs)
    (128, 32, torch.bfloat16, torch.bfloat16, "per_token"), (128, 64, torch.float32, torch.float32, "per_token"),
])
def test_ragged_prefill_with_initial_state(dk, dv, dtype, out, algo):
    lens = [100, 37, 0, 300, 1]
    H = 3
    w, inp = _inputs(11 + dk + dv, lens, H, dk, dv, dtype, 0.85, 1.0)
    cu = w.cu_seqlens
    ck = [[1, 32, 33, 100], [37], [], [64, 65, 299, 300], [1]]
    S0 = synth.state(5, w.B * H, dv, dk, 0.5).view(w.B, H, dv, dk)
    d = _dev(inp)
    r = gdn.gdn_prefill_ckpt(d.q, d.k, d.v, d.alpha, d.beta, cu, S0=S0.to(DEV), ckpt_pos=ck, out_dtype=out,
                             algo=algo)
    torch.cuda.synchronize()
    slot = 0
    slots = []
    for b in range(w.B):
        slots.append(list(range(slot, slot + len(ck[b]))))
        slot += len(ck[b])
    for b in range(w.B):
        for h in range(H):
            ref = _oracle_prefill_head(inp, cu, b, h, S0=S0[b, h], ckpt=ck[b])
            assert_close(r["S_final"][b, h], ref["S"], f"S_N b={b} h={h}")
            if lens[b]:
                check_output(r["o"][cu[b]:cu[b + 1], h], ref["o"], f"o b={b} h={h}")
            for i, s in enumerate(slots[b]):
                assert_close(r["ckpt_states"][s, h], ref["ckpt"][i], f"ckpt b={b} c={ck[b][i]} h={h}")
    # a zero-length sequence returns its initial state unchanged
    assert torch.equal(r["S_final"][2].cpu(), S0[2])


@pytest.mark.parametrize("dk,dv,algo", [(128, 128, "per_token"), (128, 128, "chunked"), (128, 128, "chunked_mma"),
                                        (128, 128, "two_pass"), (64, 32, "auto"), (128, 64, "per_token"),
                                        (128, 32, "per_token")])
def test_ragged_replay_twin_and_readout(dk, dv, algo):
    lens = [200, 71, 5, 64]
    H = 4
    w, inp = _inputs(21 + dk, lens, H, dk, dv, torch.bfloat16, 0.9, 1.0)
    cu = w.cu_seqlens
    m = [200, 50, 0, 64]
    d = _dev(inp)
    S_a = synth.state(9, w.B * H, dv, dk, 1.0).view(w.B, H, dv, dk)
    for rn, rd in ((1, 10), (1, 1), (0, 1), (3, 7)):
        rp = gdn.gdn_tail_replay(d.q, d.k, d.v, d.alpha, d.beta, cu, m, rn, rd, S_a=S_a.to(DEV), readout=True,
                                 out_dtype=torch.float32, algo=algo)
        torch.cuda.synchronize()
        for b in range(w.B):
            a_, k_ = oracle.replay_plan(m[b], rn, rd)
            assert (rp["a"][b], rp["k"][b]) == (a_, k_)
            sl = slice(cu[b], cu[b + 1])
            for h in range(H):
                o_ = oracle.tail_replay(inp.k[sl, h], inp.v[sl, h], inp.alpha[sl, h], inp.beta[sl, h], m[b], rn, rd,
                                        S_a=S_a[b, h], q=inp.q[sl, h], want_o=True)
                assert_close(rp["S_hat"][b, h], o_["S_hat"], f"S_hat b={b} h={h} r={rn}/{rd}")
                assert_close(rp["S_exact"][b, h], o_["S_exact"], f"S_exact b={b} h={h} r={rn}/{rd}")
                if k_:
                    assert_close(rp["o"][cu[b] + a_:cu[b] + m[b], h], o_["o"], f"replay o b={b} h={h}")
                else:
                    assert not torch.any(rp["S_hat"][b, h]), "k = 0 leaves the zero state"
    # state-only replay without the twin
    rp = gdn.gdn_tail_replay(d.q, d.k, d.v, d.alpha, d.beta, cu, m, 1, 10, algo=algo)
    torch.cuda.synchronize()
    for b in range(w.B):
        sl = slice(cu[b], cu[b + 1])
        for h in range(H):
            o_ = oracle.tail_replay(inp.k[sl, h], inp.v[sl, h], inp.alpha[sl, h], inp.beta[sl, h], m[b], 1, 10)
            assert_close(rp["S_hat"][b, h], o_["S_hat"], f"S_hat(no twin) b={b} h={h}")


@pytest.mark.parametrize("algo", ["per_token", "chunked", "chunked_mma", "two_pass"])
def test_resume_from_seeded_checkpoints(algo):
    """Resume with checkpoint states drawn by the generator (fed to both sides)."""
    lens = [300, 130]
    H, dk, dv = 2, 128, 128
    w, inp = _inputs(31, lens, H, dk, dv, torch.bfloat16, 0.9, 1.0, beta="sigmoid")
    cu = w.cu_seqlens
    ck = [[50, 100, 290], [1, 64]]
    ck_states = synth.state(13, 5 * H, dv, dk, 0.7).view(5, H, dv, dk)
    S0 = synth.state(17, w.B * H, dv, dk, 0.3).view(w.B, H, dv, dk)
    probes = [(0, 0), (0, 49), (0, 50), (0, 51), (0, 300), (1, 0), (1, 1), (1, 63), (1, 130), (0, 289)]
    d = _dev(inp)
    rs = gdn.gdn_resume_from_ckpt(d.q, d.k, d.v, d.alpha, d.beta, cu, ck_states.to(DEV), ck, probes,
                                  S0=S0.to(DEV), out_dtype=torch.bfloat16, algo=algo)
    torch.cuda.synchronize()
    base = [0, 3]
    for i, (s, dd) in enumerate(probes):
        sl = slice(cu[s], cu[s + 1])
        for h in range(H):
            st = [ck_states[base[s] + j, h] for j in range(len(ck[s]))]
            o_ = oracle.resume(inp.q[sl, h], inp.k[sl, h], inp.v[sl, h], inp.alpha[sl, h], inp.beta[sl, h],
                               st, ck[s], dd, S0=S0[s, h])
            assert rs["chosen"][i] == o_["c"]
            assert_close(rs["S_out"][i, h], o_["S"], f"resume probe {i} h={h}")
            lo, hi = rs["offsets"][i], rs["offsets"][i + 1]
            if hi > lo:
                check_output(rs["o"][lo:hi, h], o_["o"], f"resume o probe {i} h={h}")


def _small_alpha_inputs(seed, lens, H):
    """bf16 d = 128 streams whose gates reach down to the bottom of the supported range:
    about 6% of the tokens take alpha = 10^(-30 u) (1 down to 1e-30), and a run of tokens
    takes alpha ~ U[0.2, 0.5], so that decay products cross 2^-32 inside a 64-token window."""
    w, inp = _inputs(seed, lens, H, 128, 128, torch.bfloat16, 0.85, 1.0)
    u, _ = synth.gates(seed + 1000, 0, w.T, H, 0.0, 1.0, "uniform")
    sel, _ = synth.gates(seed + 2000, 0, w.T, H, 0.0, 1.0, "uniform")
    mid, _ = synth.gates(seed + 3000, 0, w.T, H, 0.2, 0.5, "uniform")
    alpha = inp.alpha.clone()
    alpha[100:180] = mid[100:180]
    tiny = sel < 0.06
    alpha[tiny] = torch.pow(10.0, -30.0 * u[tiny].double()).float()
    alpha = torch.clamp(alpha, min=1e-30)
    return w, synth.Inputs(inp.q, inp.k, inp.v, alpha, inp.beta)


@pytest.mark.parametrize("algo", ["per_token", "chunked", "two_pass"])
def test_small_alpha_gates(algo):
    """alpha down to 1e-30 (the bottom of the documented range), with checkpoints and a resume."""
    lens = [300, 129]
    H = 2
    w, inp = _small_alpha_inputs(61, lens, H)
    assert float(inp.alpha.min()) < 1e-25 and float(inp.alpha.max()) <= 1.0
    cu = w.cu_seqlens
    ck = [[64, 101, 150, 299], [1, 128]]
    S0 = synth.state(19, w.B * H, 128, 128, 0.5).view(w.B, H, 128, 128)
    d = _dev(inp)
    r = gdn.gdn_prefill_ckpt(d.q, d.k, d.v, d.alpha, d.beta, cu, S0=S0.to(DEV), ckpt_pos=ck,
                             out_dtype=torch.float32, algo=algo)
    torch.cuda.synchronize()
    slots = [[0, 1, 2, 3], [4, 5]]
    refs = {}
    for b in range(w.B):
        for h in range(H):
            ref = _oracle_prefill_head(inp, cu, b, h, S0=S0[b, h], ckpt=ck[b])
            refs[b, h] = ref
            assert_close(r["S_final"][b, h], ref["S"], f"S_N b={b} h={h}")
            check_output(r["o"][cu[b]:cu[b + 1], h], ref["o"], f"o b={b} h={h}")
            for i, s in enumerate(slots[b]):
                assert_close(r["ckpt_states"][s, h], ref["ckpt"][i], f"ckpt b={b} c={ck[b][i]} h={h}")
    # resume from the oracle's checkpoint states (fp32), fed to both sides
    ck_states = torch.zeros(6, H, 128, 128, dtype=torch.float32)
    for b in range(w.B):
        for h in range(H):
            for i, s in enumerate(slots[b]):
                ck_states[s, h] = torch.as_tensor(np.asarray(refs[b, h]["ckpt"][i]), dtype=torch.float32)
    probes = [(0, 120), (0, 300), (1, 77)]
    rs = gdn.gdn_resume_from_ckpt(d.q, d.k, d.v, d.alpha, d.beta, cu, ck_states.to(DEV), ck, probes,
                                  S0=S0.to(DEV), out_dtype=torch.float32, algo=algo)
    torch.cuda.synchronize()
    for i, (s, dd) in enumerate(probes):
        sl = slice(cu[s], cu[s + 1])
        for h in range(H):
            st = [ck_states[slots[s][j], h] for j in range(len(ck[s]))]
            o_ = oracle.resume(inp.q[sl, h], inp.k[sl, h], inp.v[sl, h], inp.alpha[sl, h], inp.beta[sl, h],
                               st, ck[s], dd, S0=S0[s, h])
            assert rs["chosen"][i] == o_["c"]
            assert_close(rs["S_out"][i, h], o_["S"], f"small-alpha resume probe {i} h={h}")
            lo, hi = rs["offsets"][i], rs["offsets"][i + 1]
            if hi > lo:
                check_output(rs["o"][lo:hi, h], o_["o"], f"small-alpha resume o probe {i} h={h}")


@pytest.mark.parametrize("algo", ["per_token", "chunked", "two_pass"])
def test_placement_feeds_prefill_and_resume(algo):
    """Checkpoints chosen by the placement programme ("Sparse prefix caching ...", Theorem 2) for a
    seeded depth distribution drive gdn_prefill_ckpt; resume probes at depths drawn from the same
    distribution recompute exactly f(d) tokens and match the oracle."""
    from oracle import placement as PL
    lens = [400, 257]
    H = 2
    w, inp = _inputs(71, lens, H, 128, 128, torch.bfloat16, 0.9, 1.0, beta="sigmoid")
    cu = w.cu_seqlens
    ck = []
    for b, n in enumerate(lens):
        wd = synth.depth_weights("prompts", n, 3000, seed=b)
        pos, cost = gdn.gdn_ckpt_placement(wd, 5, "dp")
        assert cost == PL.place_dp(wd, 5)[1]
        ck.append(pos)
    d = _dev(inp)
    r = gdn.gdn_prefill_ckpt(d.q, d.k, d.v, d.alpha, d.beta, cu, ckpt_pos=ck, out_dtype=torch.float32, algo=algo)
    torch.cuda.synchronize()
    probes = []
    for b, n in enumerate(lens):
        wd = synth.depth_weights("prompts", n, 3000, seed=b)
        support = [x for x in range(n + 1) if wd[x] > 0]
        picks = synth.integers(500 + b, 0, 0, 6, 0, len(support) - 1)
        probes += [(b, support[i]) for i in picks]
    rs = gdn.gdn_resume_from_ckpt(d.q, d.k, d.v, d.alpha, d.beta, cu, r["ckpt_states"], ck, probes,
                                  out_dtype=torch.float32, algo=algo)
    torch.cuda.synchronize()
    base = [0, len(ck[0])]
    for i, (s, dd) in enumerate(probes):
        assert rs["offsets"][i + 1] - rs["offsets"][i] == PL.recompute(ck[s], dd)
        sl = slice(cu[s], cu[s + 1])
        # the oracle resumes from its own checkpoint states (no oracle input comes from the GPU)
        for h in range(H):
            refh = _oracle_prefill_head(inp, cu, s, h, ckpt=ck[s])
            o_ = oracle.resume(inp.q[sl, h], inp.k[sl, h], inp.v[sl, h], inp.alpha[sl, h], inp.beta[sl, h],
                               [refh["ckpt"][j] for j in range(len(ck[s]))], ck[s], dd)
            assert rs["chosen"][i] == o_["c"]
            assert_close(rs["S_out"][i, h], o_["S"], f"placement resume probe {i} h={h}")
            lo, hi = rs["offsets"][i], rs["offsets"][i + 1]
            if hi > lo:
                check_output(rs["o"][lo:hi, h], o_["o"], f"placement resume o probe {i} h={h}")


# ---------------------------------------------------------------------------------------------
# invariants on the GPU
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("algo", ["per_token", "chunked", "chunked_mma", "two_pass"])
def test_identity_gates_leave_state_unchanged(algo):
    lens = [77]
    H, dk, dv = 2, 128, 128
    w, inp = _inputs(41, lens, H, dk, dv, torch.bfloat16)
    S0 = synth.state(3, H, dv, dk, 1.0).view(1, H, dv, dk)
    d = _dev(inp)
    ones = torch.ones_like(d.alpha)
    zeros = torch.zeros_like(d.beta)
    r = gdn.gdn_prefill_ckpt(d.q, d.k, d.v, ones, zeros, w.cu_seqlens, S0=S0.to(DEV), out_dtype=torch.float32,
                             algo=algo)
    torch.cuda.synchronize()
    assert torch.equal(r["S_final"].cpu(), S0), "alpha = 1, beta = 0 must leave S unchanged (bitwise)"


@pytest.mark.parametrize("algo", ["per_token", "chunked", "chunked_mma", "two_pass"])
def test_row_permutation_equivariance(algo):
    """Row i of the state evolves from component i of v alone (the key operator acts from the right), so
    permuting the components of v (and the rows of S0) permutes the rows of every state and the components of
    every output, whatever the chunking, rounding order or kernel: the GPU results must agree bit for bit."""
    lens = [200, 75]
    H, dk, dv = 2, 128, 128
    w, inp = _inputs(43, lens, H, dk, dv, torch.bfloat16, 0.9, 1.0, beta="sigmoid")
    cu = w.cu_seqlens
    ck = [[64, 150], [75]]
    perm = torch.from_numpy(np.random.default_rng(5).permutation(dv))
    S0 = synth.state(19, w.B * H, dv, dk, 0.5).view(w.B, H, dv, dk)
    d = _dev(inp)
    vp = d.v[:, :, perm.to(DEV)].contiguous()
    S0p = S0[:, :, perm, :].contiguous()
    a = gdn.gdn_prefill_ckpt(d.q, d.k, d.v, d.alpha, d.beta, cu, S0=S0.to(DEV), ckpt_pos=ck,
                             out_dtype=torch.float32, algo=algo)
    b = gdn.gdn_prefill_ckpt(d.q, d.k, vp, d.alpha, d.beta, cu, S0=S0p.to(DEV), ckpt_pos=ck,
                             out_dtype=torch.float32, algo=algo)
    torch.cuda.synchronize()
    pd = perm.to(DEV)
    assert torch.equal(b["S_final"], a["S_final"][:, :, pd, :]), "final states: rows permuted"
    assert torch.equal(b["ckpt_states"], a["ckpt_states"][:, :, pd, :]), "checkpoints: rows permuted"
    assert torch.equal(b["o"], a["o"][:, :, pd]), "outputs: components permuted"


@pytest.mark.parametrize("algo,dk", [("per_token", 128), ("per_token", 64), ("per_token", 32), ("chunked", 128),
                                     ("chunked_mma", 128), ("two_pass", 128)])
def test_resume_is_bitwise_equal_to_full_run_and_runs_are_deterministic(algo, dk):
    """Resume from the deepest stored checkpoint c_j <= d reproduces, bit for bit,
    the state at d of a full run that stores the same checkpoints plus d.  (Each
    stored checkpoint renormalises the running scale, so the comparison run must
    not store anything else between c_j and d.)  The per-token cases at d_k = 64 and 32
    run that kernel's 2-row lane tile with its producer warp."""
    lens = [1000]
    H, dv = 3, dk
    w, inp = _inputs(51, lens, H, dk, dv, torch.bfloat16, 0.95, 1.0, beta="sigmoid")
    d = _dev(inp)
    cu = w.cu_seqlens
    C = [321, 500, 777]
    depths = [321, 322, 400, 499, 500, 501, 776, 777, 1000]
    base = gdn.gdn_prefill_ckpt(d.q, d.k, d.v, d.alpha, d.beta, cu, ckpt_pos=[C], readout=False, algo=algo)
    again = gdn.gdn_prefill_ckpt(d.q, d.k, d.v, d.alpha, d.beta, cu, ckpt_pos=[C], readout=False, algo=algo)
    rs = gdn.gdn_resume_from_ckpt(d.q, d.k, d.v, d.alpha, d.beta, cu, base["ckpt_states"], [C],
                                  [(0, dd) for dd in depths], readout=False, algo=algo)
    torch.cuda.synchronize()
    assert torch.equal(base["ckpt_states"], again["ckpt_states"]) and torch.equal(base["S_final"], again["S_final"])
    for i, dd in enumerate(depths):
        Cd = sorted(set(C) | {dd})
        full = gdn.gdn_prefill_ckpt(d.q, d.k, d.v, d.alpha, d.beta, cu, ckpt_pos=[Cd], readout=False, algo=algo)
        torch.cuda.synchronize()
        assert rs["chosen"][i] == max(c for c in C if c <= dd)
        assert torch.equal(rs["S_out"][i], full["ckpt_states"][Cd.index(dd)]), \
            f"resume to d={dd} is not bitwise the full run"


# ---------------------------------------------------------------------------------------------
# full-size workloads, sampled
# ---------------------------------------------------------------------------------------------
def _gpu_inputs(w, t_range=None, with_q=True, alloc_full=False):
    """Streams generated on the GPU.  With alloc_full, buffers span all T rows
    but only t_range is filled (the rest is never read)."""
    t0, t1 = t_range if t_range is not None else (0, w.T)
    if not alloc_full:
        return synth.make_inputs(w, device=DEV, t_range=(t0, t1), with_q=with_q)
    T = w.T
    bufs = {}
    for name, stream, d, norm in (("q", synth.STREAM_Q, w.dk, True), ("k", synth.STREAM_K, w.dk, True),
                                  ("v", synth.STREAM_V, w.dv, False)):
        if name == "q" and not with_q:
            bufs[name] = None
            continue
        t = torch.empty((T, w.H, d), dtype=w.qkv_dtype, device=DEV)
        bufs[name] = t
    al = torch.empty((T, w.H), dtype=torch.float32, device=DEV)
    be = torch.empty((T, w.H), dtype=torch.float32, device=DEV)
    return synth.Inputs(bufs["q"], bufs["k"], bufs["v"], al, be)


def _fill_rows(buf, w, t0, t1, stream, d, norm):
    synth.rows_into(buf[t0:t1], w.seed, stream, t0, t1, w.H, d, norm)


def _fill_tail(inp, w, t0, t1, with_q):
    if with_q:
        _fill_rows(inp.q, w, t0, t1, synth.STREAM_Q, w.dk, True)
    _fill_rows(inp.k, w, t0, t1, synth.STREAM_K, w.dk, True)
    _fill_rows(inp.v, w, t0, t1, synth.STREAM_V, w.dv, False)
    a, b = synth.gates(w.seed, t0, t1, w.H, w.alpha_lo, w.alpha_hi, w.beta_kind)
    inp.alpha[t0:t1].copy_(a)
    inp.beta[t0:t1].copy_(b)


def _host_head(inp, t0, t1, h, with_q=True):
    q = inp.q[t0:t1, h].cpu() if with_q else None
    return q, inp.k[t0:t1, h].cpu(), inp.v[t0:t1, h].cpu(), inp.alpha[t0:t1, h].cpu(), inp.beta[t0:t1, h].cpu()


@pytest.mark.parametrize("algo", ["auto", "chunked", "per_token"])
def test_full_prefill_workload_sampled(algo):
    """8 x 16 heads, N = 8192, bf16, 16 equally spaced checkpoints: full run, sampled oracle."""
    w = synth.workload("prefill")
    inp = _gpu_inputs(w)
    cu = w.cu_seqlens
    ck = w.ckpt_positions()
    r = gdn.gdn_prefill_ckpt(inp.q, inp.k, inp.v, inp.alpha, inp.beta, cu, ckpt_pos=ck, algo=algo)
    r32 = gdn.gdn_prefill_ckpt(inp.q, inp.k, inp.v, inp.alpha, inp.beta, cu, ckpt_pos=ck, out_dtype=torch.float32,
                               algo=algo)
    torch.cuda.synchronize()
    assert torch.equal(r["S_final"], r32["S_final"]), "readout dtype must not change the state"
    assert torch.equal(r["ckpt_states"], r32["ckpt_states"])
    samples = [(b, (5 * b + 3) % w.H) for b in range(w.B)]   # one (sequence, head) stream per sequence
    jobs = []
    for b, h in samples:
        q, k, v, a, be = _host_head(inp, cu[b], cu[b + 1], h)
        jobs.append(lambda q=q, k=k, v=v, a=a, be=be, b=b: oracle.prefill(q, k, v, a, be, ckpt_pos=ck[b]))
    refs = oracle.run_many(jobs)
    for (b, h), ref in zip(samples, refs):
        check_output(r["o"][cu[b]:cu[b + 1], h], ref["o"], f"prefill o bf16 b={b} h={h}")
        assert_close(r32["o"][cu[b]:cu[b + 1], h], ref["o"], f"prefill o fp32 b={b} h={h}")
        assert_close(r["S_final"][b, h], ref["S"], f"prefill S_N b={b} h={h}")
        for i in range(len(ck[b])):
            assert_close(r["ckpt_states"][b * len(ck[b]) + i, h], ref["ckpt"][i], f"prefill ckpt {i} b={b} h={h}")


def test_full_long_prefill_and_resume_sampled():
    """4 x 32 heads, N = 131072, 32 checkpoints, 64 resume probes: full run; one (sequence, head) stream per
    sequence against the oracle, with every resume probe that lands on it."""
    w = synth.workload("long")
    inp = _gpu_inputs(w)
    cu = w.cu_seqlens
    ck = w.ckpt_positions()
    r = gdn.gdn_prefill_ckpt(inp.q, inp.k, inp.v, inp.alpha, inp.beta, cu, ckpt_pos=ck)
    probes = w.probes()
    rs = gdn.gdn_resume_from_ckpt(inp.q, inp.k, inp.v, inp.alpha, inp.beta, cu, r["ckpt_states"], ck, probes)
    torch.cuda.synchronize()
    for i, (s, dd) in enumerate(probes):
        j = oracle.select_ckpt(ck[s], dd)
        assert rs["chosen"][i] == (0 if j < 0 else ck[s][j])
    samples = [(b, (9 * b + 17) % w.H) for b in range(w.B)]
    hosts = [_host_head(inp, cu[b], cu[b + 1], h) for b, h in samples]
    refs = oracle.run_many([lambda x=x, b=b: oracle.prefill(*x, ckpt_pos=ck[b]) for (b, _), x in zip(samples, hosts)])
    n_probes = 0
    for (b, h), x, ref in zip(samples, hosts, refs):
        check_output(r["o"][cu[b]:cu[b + 1], h], ref["o"], f"long o b={b} h={h}")
        assert_close(r["S_final"][b, h], ref["S"], f"long S_N b={b} h={h}")
        for i in range(len(ck[b])):
            assert_close(r["ckpt_states"][b * 32 + i, h], ref["ckpt"][i], f"long ckpt {i} b={b} h={h}")
        # every resume probe on sequence b, head h, from the oracle's own checkpoints
        sel = [i for i, (s, _) in enumerate(probes) if s == b]
        outs = oracle.run_many([lambda dd=probes[i][1]: oracle.resume(*x, ref["ckpt"], ck[b], dd) for i in sel])
        for i, o_ in zip(sel, outs):
            dd = probes[i][1]
            assert_close(rs["S_out"][i, h], o_["S"], f"long resume probe {i} d={dd} h={h}")
            lo, hi = rs["offsets"][i], rs["offsets"][i + 1]
            if hi > lo:
                check_output(rs["o"][lo:hi, h], o_["o"], f"long resume o probe {i} h={h}")
            n_probes += 1
    assert n_probes == len(probes), "every probe lands on one of the sampled sequences"


def _prefix_state(w, b, h, a):
    """The oracle's exact state after the first a tokens of (sequence b, head h) of the seeded workload, rounded
    once to fp32 (the exact twin's input on both sides)."""
    cu = w.cu_seqlens
    hs = range(h, h + 1)
    k = synth.rows(w.seed, synth.STREAM_K, cu[b], cu[b] + a, w.H, w.dk, w.qkv_dtype, True, heads=hs)[:, 0]
    v = synth.rows(w.seed, synth.STREAM_V, cu[b], cu[b] + a, w.H, w.dv, w.qkv_dtype, False, heads=hs)[:, 0]
    al, be = synth.gates(w.seed, cu[b], cu[b] + a, w.H, w.alpha_lo, w.alpha_hi, w.beta_kind, heads=hs)
    return torch.from_numpy(np.asarray(oracle.scan(k, v, al[:, 0], be[:, 0], want_o=False)["S"], dtype=np.float32))


def _replay_full(name, samples, real_sa=False):
    """The workload's tail replays with the exact twin.  S_a is a seeded random state, or with real_sa the
    oracle's own state at a for the sampled streams (the exact S_a -> S_m error check of the error
    decomposition); the returned stats are ||E_m||_F / ||S_a||_F and the per-instance bound prod(alpha)."""
    w = synth.workload(name)
    cu = w.cu_seqlens
    m = list(w.seq_lens)
    rn, rd = w.replay_r
    inp = _gpu_inputs(w, with_q=False, alloc_full=True)
    plans = [oracle.replay_plan(m[b], rn, rd) for b in range(w.B)]
    for b in range(w.B):
        a_, _ = plans[b]
        _fill_tail(inp, w, cu[b] + a_, cu[b] + m[b], with_q=False)
    S_a = synth.state(w.seed + 101, w.B * w.H, w.dv, w.dk, 1.0, device=DEV).view(w.B, w.H, w.dv, w.dk)
    if real_sa:
        sas = oracle.run_many([lambda b=b, h=h: _prefix_state(w, b, h, plans[b][0]) for b, h in samples])
        for (b, h), sa in zip(samples, sas):
            S_a[b, h].copy_(sa)
    rp = gdn.gdn_tail_replay(None, inp.k, inp.v, inp.alpha, inp.beta, cu, m, rn, rd, S_a=S_a)
    torch.cuda.synchronize()
    assert [(rp["a"][b], rp["k"][b]) for b in range(w.B)] == plans, "replay indices are bit-exact"
    jobs = []
    hosts = []
    for b, h in samples:
        a_, k_ = plans[b]
        _, k, v, al, be = _host_head(inp, cu[b] + a_, cu[b] + m[b], h, with_q=False)
        Sa = S_a[b, h].cpu()
        hosts.append((al, Sa))
        jobs.append(lambda k=k, v=v, al=al, be=be, Sa=Sa, k_=k_: oracle.tail_replay(k, v, al, be, k_, 1, 1, S_a=Sa))
    refs = oracle.run_many(jobs)
    stats = []
    for (b, h), ref, (al, Sa) in zip(samples, refs, hosts):
        assert_close(rp["S_hat"][b, h], ref["S_hat"], f"{name} S_hat b={b} h={h}")
        assert_close(rp["S_exact"][b, h], ref["S_exact"], f"{name} S_exact b={b} h={h}")
        e = np.linalg.norm(ref["S_exact"] - ref["S_hat"]) / np.linalg.norm(Sa.double().numpy())
        stats.append((e, float(np.prod(al.double().numpy())), float(al.max())))
    return w, rp, stats


def test_full_tail_replay_5pct_sampled():
    """768 (layer, head) scans as 24 layers x 32 heads, m = 32768, k = 1639 from zero; the exact twin starts from
    the workload's own state at a = 31129 (computed by the oracle over rows [0, a)) for one head of every layer.
    The oracle's replay error obeys the per-instance bound ||E_m||_F <= prod(alpha) ||S_a||_F (unit keys up to
    bf16 rounding, beta <= 1), hence also the page's rho^k."""
    samples = [(0, 32 * l + (7 * l) % 32) for l in range(24)]
    w, rp, stats = _replay_full("replay5", samples, real_sa=True)
    assert rp["k"] == [1639] and rp["a"] == [31129]
    for (_, h), (e, prod_alpha, rho) in zip(samples, stats):
        assert e <= prod_alpha * (1 + 1e-9), (h, e, prod_alpha)
        assert prod_alpha <= rho ** 1639
    worst = max(stats)
    print(f"replay5, real S_a: ||E_m|| / ||S_a|| max {worst[0]:.3e} (bound prod(alpha) {worst[1]:.3e}) over "
          f"{len(samples)} streams")


def test_full_ragged_tail_replay_10pct_sampled():
    """32 requests, m_b ~ U[4096, 32768], 16 heads, k_b = ceil(m_b / 10)."""
    w = synth.workload("ragged10")
    samples = [(b, (3 * b) % w.H) for b in range(w.B)]   # one (request, head) stream per request
    _replay_full("ragged10", samples)


def test_auto_takes_two_pass_only_with_its_workspace():
    """GDN_ALGO_AUTO runs the two-pass chunked scan when the workspace holds T of every chunk, the fused
    chunked scan otherwise (the noalloc entry point's case); each is bit-identical to naming it."""
    lens = [300, 129]
    H = 2
    w, inp = _inputs(91, lens, H, 128, 128, torch.bfloat16, 0.9, 1.0)
    d = _dev(inp)
    cu = w.cu_seqlens
    ck = [[64, 150], [100]]
    small = torch.zeros(int(gdn.lib().gdn_workspace_size()), dtype=torch.uint8, device=DEV)
    big = torch.zeros(int(gdn.lib().gdn_workspace_size_two_pass(w.T, H, w.B)), dtype=torch.uint8, device=DEV)
    runs = {}
    for name, algo, ws in (("auto_small", "auto", small), ("chunked", "chunked", small), ("auto_big", "auto", big),
                           ("two_pass", "two_pass", big)):
        runs[name] = gdn.gdn_prefill_ckpt(d.q, d.k, d.v, d.alpha, d.beta, cu, ckpt_pos=ck, algo=algo, ws=ws)
    torch.cuda.synchronize()
    assert gdn.read_status(ws=small) == gdn.GDN_OK and gdn.read_status(ws=big) == gdn.GDN_OK
    for a, b in (("auto_small", "chunked"), ("auto_big", "two_pass")):
        for key in ("o", "S_final", "ckpt_states"):
            assert torch.equal(runs[a][key], runs[b][key]), (a, b, key)
    with pytest.raises(gdn.GdnError):   # naming the two-pass scan with too small a workspace
        gdn.gdn_prefill_ckpt(d.q, d.k, d.v, d.alpha, d.beta, cu, ckpt_pos=ck, algo="two_pass", ws=small)
