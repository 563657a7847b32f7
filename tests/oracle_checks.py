"""Pins for the fp64 oracle: checks against what the pages and the mathematics fix.

Each check raises AssertionError on failure.  They are collected as tests in
test_oracle_pins.py and re-run against deliberately broken copies of the
oracle in test_oracle_mutants.py, so that every plausible slip (a dropped
term, a wrong sign, a transposed operand, an off-by-one index) is shown to
fail at least one of them.

Sources: "Tail-Replay: Escaping the Curse of Linear Attention in Prefix
Caching for Hybrid LLMs" (notes page) sections 2.1-2.3, equation (1) and the
error decomposition / contraction bound of section 2.3; "Sparse prefix caching
in hybrid and recurrent LLM serving", section 3 (checkpoint resume rule).
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "index_pins.txt")


def _unit_rows(rng, n, d):
    x = rng.standard_normal((n, d))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


def brute_scan(S0, q, k, v, alpha, beta):
    """Equation (1) with the transition formed as an explicit d_k x d_k matrix
    T_t = alpha_t (I - beta_t k_t k_t^T) multiplying the state from the right
    (S in R^{d_v x d_k}), plus the write beta_t v_t k_t^T; readout S_t q_t."""
    S = np.array(S0, dtype=np.float64, copy=True)
    dk = k.shape[1]
    outs, states = [], []
    for t in range(k.shape[0]):
        T = alpha[t] * (np.eye(dk) - beta[t] * np.outer(k[t], k[t]))
        S = S @ T + beta[t] * np.outer(v[t], k[t])
        outs.append(S @ q[t])
        states.append(S.copy())
    return np.array(outs), np.array(states)


def transition_product(k, alpha, beta):
    """Phi = T_{a+1} T_{a+2} ... T_m (right-multiplied form, earliest first)."""
    dk = k.shape[1]
    Phi = np.eye(dk)
    for t in range(k.shape[0]):
        Phi = Phi @ (alpha[t] * (np.eye(dk) - beta[t] * np.outer(k[t], k[t])))
    return Phi


def _rel(x, y):
    return np.max(np.abs(x - y)) / max(np.max(np.abs(y)), 1e-300)


def check_brute_force(seed=1):
    rng = np.random.default_rng(seed)
    for dk, dv, n in ((2, 3, 5), (5, 3, 7), (8, 4, 9), (32, 32, 20), (16, 48, 12)):
        k = rng.standard_normal((n, dk))  # the recurrence is defined for any k; do not rely on unit norm
        q = rng.standard_normal((n, dk))
        v = rng.standard_normal((n, dv))
        alpha = rng.uniform(0.5, 1.0, n)
        beta = rng.uniform(0.0, 1.5, n)
        S0 = rng.standard_normal((dv, dk))
        ck = [2, n - 1, n]
        r = oracle.scan(k, v, alpha, beta, S0=S0, q=q, ckpt_pos=ck)
        o_ref, st_ref = brute_scan(S0, q, k, v, alpha, beta)
        assert _rel(r["o"], o_ref) < 1e-12, "readout differs from brute force"
        assert _rel(r["S"], st_ref[-1]) < 1e-12, "final state differs from brute force"
        for i, c in enumerate(ck):
            assert _rel(r["ckpt"][i], st_ref[c - 1]) < 1e-12, "checkpoint is not the state after token c"


def check_identity(seed=2):
    rng = np.random.default_rng(seed)
    n, dk, dv = 17, 8, 6
    S0 = rng.standard_normal((dv, dk))
    k, q, v = _unit_rows(rng, n, dk), rng.standard_normal((n, dk)), rng.standard_normal((n, dv))
    r = oracle.scan(k, v, np.ones(n), np.zeros(n), S0=S0, q=q)
    assert np.array_equal(r["S"], S0), "alpha = 1, beta = 0 must leave S unchanged"
    assert _rel(r["o"], q @ S0.T) < 1e-14, "readout of an unchanged state"


def check_beta0(seed=3):
    rng = np.random.default_rng(seed)
    n, dk, dv = 40, 6, 5
    S0 = rng.standard_normal((dv, dk))
    alpha = rng.uniform(0.8, 1.0, n)
    r = oracle.scan(_unit_rows(rng, n, dk), rng.standard_normal((n, dv)), alpha, np.zeros(n), S0=S0)
    assert _rel(r["S"], np.prod(alpha) * S0) < 1e-13, "beta = 0 must give S_N = (prod alpha) S0"


def check_delta_rule(seed=4):
    """beta = 1, unit key: S_t k_t = v_t for any alpha; with q_t = k_t, o_t = v_t."""
    rng = np.random.default_rng(seed)
    n, dk, dv = 25, 16, 12
    k = _unit_rows(rng, n, dk)
    v = rng.standard_normal((n, dv))
    alpha = rng.uniform(0.3, 1.0, n)
    S0 = rng.standard_normal((dv, dk))
    r = oracle.scan(k, v, alpha, np.ones(n), S0=S0, q=k, ckpt_pos=list(range(1, n + 1)))
    for t in range(n):
        assert _rel(r["ckpt"][t] @ k[t], v[t]) < 1e-12, "delta rule: S_t k_t must equal v_t"
    assert _rel(r["o"], v) < 1e-12, "post-update readout with q = k must return v"
    # general beta: S_t k_t = alpha (1 - beta) S_{t-1} k_t + beta v_t
    beta = rng.uniform(0.0, 1.0, n)
    r2 = oracle.scan(k, v, alpha, beta, S0=S0, ckpt_pos=list(range(1, n + 1)))
    prev = S0
    for t in range(n):
        want = alpha[t] * (1 - beta[t]) * (prev @ k[t]) + beta[t] * v[t]
        assert _rel(r2["ckpt"][t] @ k[t], want) < 1e-12, "S_t k_t identity"
        prev = r2["ckpt"][t]


def check_basis_write(seed=5):
    """k = e_j, alpha = beta = 1: column j of S is overwritten by v (associative-memory write)."""
    rng = np.random.default_rng(seed)
    dk, dv = 7, 5
    S = rng.standard_normal((dv, dk))
    js = [3, 0, 6, 3]
    for j in js:
        k = np.zeros((1, dk))
        k[0, j] = 1.0
        v = rng.standard_normal((1, dv))
        r = oracle.scan(k, v, np.ones(1), np.ones(1), S0=S)
        want = S.copy()
        want[:, j] = v[0]
        assert np.array_equal(r["S"], want), "basis-key write must overwrite exactly one column"
        S = r["S"]


def check_decomposition(seed=6):
    """E_m = S_m - S_hat_m = S_a Phi, Phi = T_{a+1} ... T_m (section 2.3, right-multiplied)."""
    rng = np.random.default_rng(seed)
    m, dk, dv = 60, 8, 6
    k, v = _unit_rows(rng, m, dk), rng.standard_normal((m, dv))
    alpha, beta = rng.uniform(0.85, 1.0, m), rng.uniform(0.0, 1.0, m)
    S0 = rng.standard_normal((dv, dk))
    a = 41
    S_a = oracle.scan(k[:a], v[:a], alpha[:a], beta[:a], S0=S0)["S"]
    rep = oracle.tail_replay(k, v, alpha, beta, m, m - a, m, S_a=S_a)  # r = (m-a)/m -> k = m - a exactly
    assert rep["a"] == a and rep["k"] == m - a
    S_m = oracle.scan(k, v, alpha, beta, S0=S0)["S"]
    assert _rel(rep["S_exact"], S_m) < 1e-12, "exact twin from S_a must reproduce the full run"
    E = S_m - rep["S_hat"]
    Phi = transition_product(k[a:m], alpha[a:m], beta[a:m])
    assert np.max(np.abs(E - S_a @ Phi)) <= 1e-12 * np.max(np.abs(S_a)), "E_m = S_a Phi"


def check_bound(seed=7):
    """||E_m||_F <= rho^k ||S_a||_F for unit keys, beta in [0, 2], alpha <= rho < 1 (section 2.3)."""
    rng = np.random.default_rng(seed)
    for trial in range(20):
        m, dk, dv = 50, 6, 5
        k, v = _unit_rows(rng, m, dk), rng.standard_normal((m, dv))
        alpha = rng.uniform(0.6, 0.95, m)
        beta = rng.uniform(0.0, 2.0, m)
        S_a = rng.standard_normal((dv, dk)) * 3
        rep = oracle.tail_replay(k, v, alpha, beta, m, 1, 5, S_a=S_a)
        kk = rep["k"]
        sl = slice(rep["a"], m)
        E = rep["S_exact"] - rep["S_hat"]
        nE, nA = np.linalg.norm(E), np.linalg.norm(S_a)
        rho = alpha[sl].max()
        assert nE <= rho ** kk * nA * (1 + 1e-12), "contraction bound rho^k"
        assert nE <= np.prod(alpha[sl]) * nA * (1 + 1e-12), "per-instance bound prod(alpha)"


def check_affinity(seed=8):
    """scan(S0) = scan(0) + S0 Phi."""
    rng = np.random.default_rng(seed)
    n, dk, dv = 30, 5, 7
    k, v = _unit_rows(rng, n, dk), rng.standard_normal((n, dv))
    alpha, beta = rng.uniform(0.7, 1.0, n), rng.uniform(0.0, 1.0, n)
    S0 = rng.standard_normal((dv, dk))
    s1 = oracle.scan(k, v, alpha, beta, S0=S0)["S"]
    s0 = oracle.scan(k, v, alpha, beta)["S"]
    Phi = transition_product(k, alpha, beta)
    assert _rel(s1, s0 + S0 @ Phi) < 1e-12, "affinity in the initial state"


def check_row_permutation(seed=9):
    rng = np.random.default_rng(seed)
    n, dk, dv = 20, 6, 9
    k, q, v = _unit_rows(rng, n, dk), rng.standard_normal((n, dk)), rng.standard_normal((n, dv))
    alpha, beta = rng.uniform(0.7, 1.0, n), rng.uniform(0.0, 1.0, n)
    S0 = rng.standard_normal((dv, dk))
    perm = rng.permutation(dv)
    r1 = oracle.scan(k, v, alpha, beta, S0=S0, q=q)
    r2 = oracle.scan(k, v[:, perm], alpha, beta, S0=S0[perm], q=q)
    assert np.array_equal(r2["S"], r1["S"][perm]), "rows of S follow the value components"
    assert np.array_equal(r2["o"], r1["o"][:, perm]), "readout rows follow the value components"


def check_resume_equals_full(seed=10):
    """Resuming from any stored checkpoint reproduces the full-run state at every d >= c, bitwise."""
    rng = np.random.default_rng(seed)
    n, dk, dv = 48, 6, 4
    k, q, v = _unit_rows(rng, n, dk), rng.standard_normal((n, dk)), rng.standard_normal((n, dv))
    alpha, beta = rng.uniform(0.8, 1.0, n), rng.uniform(0.0, 1.0, n)
    S0 = rng.standard_normal((dv, dk))
    full = oracle.scan(k, v, alpha, beta, S0=S0, q=q, ckpt_pos=list(range(1, n + 1)))
    ck = [5, 12, 13, 30, 48]
    pre = oracle.scan(k, v, alpha, beta, S0=S0, q=q, ckpt_pos=ck)
    for d in range(0, n + 1):
        r = oracle.resume(q, k, v, alpha, beta, pre["ckpt"], ck, d, S0=S0)
        want_c = max([c for c in ck if c <= d], default=0)
        assert r["c"] == want_c, "resume must start at the deepest checkpoint <= d"
        want_S = S0 if d == 0 else full["ckpt"][d - 1]
        assert np.array_equal(r["S"], want_S), "resumed state must equal the full run bitwise"
        assert r["o"].shape[0] == d - want_c, "resume recomputes exactly c_j+1 .. d"
        if d > want_c:
            assert np.array_equal(r["o"], full["o"][want_c:d]), "resumed readout equals the full run"


def check_replay_endpoints(seed=11):
    rng = np.random.default_rng(seed)
    m, dk, dv = 33, 6, 5
    k, v = _unit_rows(rng, m, dk), rng.standard_normal((m, dv))
    alpha, beta = rng.uniform(0.8, 1.0, m), rng.uniform(0.0, 1.0, m)
    full = oracle.scan(k, v, alpha, beta)["S"]
    r1 = oracle.tail_replay(k, v, alpha, beta, m, 1, 1)
    assert r1["a"] == 0 and r1["k"] == m
    assert np.array_equal(r1["S_hat"], full), "r = 1 from a zero state equals the full run"
    r0 = oracle.tail_replay(k, v, alpha, beta, m, 0, 1)
    assert r0["k"] == 0 and r0["a"] == m
    assert not np.any(r0["S_hat"]), "r = 0 (Zero-only) leaves the zero state"
    # replay window: positions a+1..m, i.e. rows [a, m)
    r5 = oracle.tail_replay(k, v, alpha, beta, m, 1, 5)
    a = r5["a"]
    direct = oracle.scan(k[a:m], v[a:m], alpha[a:m], beta[a:m])["S"]
    assert np.array_equal(r5["S_hat"], direct), "replay reads rows [a, m)"


def load_golden():
    replay, resume = [], []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == "replay":
                m, rn, rd, k, a, first, last = map(int, parts[1:8])
                replay.append((m, rn, rd, k, a, first, last, " ".join(parts[8:])))
            elif parts[0] == "resume":
                d = int(parts[1])
                cs = [int(x) for x in parts[2].split(",")]
                c, n = int(parts[3]), int(parts[4])
                resume.append((d, cs, c, n, " ".join(parts[5:])))
    return replay, resume


def check_golden_pins():
    replay, resume = load_golden()
    assert replay and resume
    for m, rn, rd, k, a, first, last, src in replay:
        aa, kk = oracle.replay_plan(m, rn, rd)
        assert (aa, kk) == (a, k), f"replay plan for {src}"
        assert (aa + 1, m) == (first, last), f"replay positions for {src}"
    for d, cs, c, n, src in resume:
        j = oracle.select_ckpt(cs, d)
        cc = 0 if j < 0 else cs[j]
        assert (cc, d - cc) == (c, n), f"resume selection for {src}"


def check_replay_plan_exhaustive(m_max=200000):
    """ceil(r m) as the least integer k with k >= r m (checked with exact rationals)."""
    for rn, rd in ((0, 1), (1, 20), (1, 10), (1, 1), (7, 100), (3, 7)):
        r = Fraction(rn, rd)
        step = 1 if m_max <= 200000 else 7
        for m in range(0, m_max + 1, step):
            a, k = oracle.replay_plan(m, rn, rd)
            assert k >= r * m and (k == 0 or k - 1 < r * m), f"ceil(r m) at m={m}, r={r}"
            assert a == m - k and 0 <= a <= m
    for bad in ((-1, 1, 20), (10, -1, 20), (10, 21, 20), (10, 1, 0)):
        try:
            oracle.replay_plan(*bad)
        except ValueError:
            continue
        raise AssertionError(f"replay plan accepted invalid {bad}")


def check_select_ckpt_random(seed=12):
    rng = np.random.default_rng(seed)
    for trial in range(300):
        N = int(rng.integers(1, 400))
        M = int(rng.integers(0, min(N, 20) + 1))
        cs = sorted(rng.choice(np.arange(1, N + 1), size=M, replace=False).tolist())
        for d in list(range(0, min(N, 40) + 1)) + cs + [N]:
            j = oracle.select_ckpt(cs, d)
            below = [i for i, c in enumerate(cs) if c <= d]
            assert j == (below[-1] if below else -1), "deepest checkpoint at or below d"


ALL_CHECKS = [
    check_brute_force, check_identity, check_beta0, check_delta_rule, check_basis_write,
    check_decomposition, check_bound, check_affinity, check_row_permutation,
    check_resume_equals_full, check_replay_endpoints, check_golden_pins,
    check_select_ckpt_random,
]
