"""Checkpoint placement ("Sparse prefix caching in hybrid and recurrent LLM serving", sections 3-5).

Oracle pins (the oracle against what the pages and the mathematics fix), then the C-ABI
implementation against the oracle: the optimal cost bit-exact (several placements can be optimal,
so the returned one is checked for validity and for reaching that cost), the deterministic
baselines position for position, and the argument checks.  Host only: no GPU needed.
"""
import itertools
import random
from fractions import Fraction

import pytest

import hybrid_model_recurrent_gb300 as gdn
import synth
from oracle import placement as P


def _weights(rng, N, zero_frac=0.3, hi=9):
    return [0 if rng.random() < zero_frac else rng.randint(0, hi) for _ in range(N + 1)]


# ---------------------------------------------------------------------------------------------
# oracle pins
# ---------------------------------------------------------------------------------------------
def test_recompute_definition_examples():
    c = [3, 7]
    # depth 0 -> nothing; below the first checkpoint -> from the start; exact hit -> 0
    assert [P.recompute(c, d) for d in range(10)] == [0, 1, 2, 0, 1, 2, 3, 0, 1, 2]
    assert P.gaps(c, 9) == [3, 4, 3] and sum(P.gaps(c, 9)) == 10
    assert P.no_cache([1, 1, 1]) == 3 == P.expected_recompute([1, 1, 1], [])


def test_segment_cost_identity_against_direct_sums():
    """C(s, t) = sum_{d=s}^{t-1} w(d)(d - s) equals the prefix-sum form used by both DPs."""
    rng = random.Random(1)
    w = _weights(rng, 40)
    W0 = [0] + list(itertools.accumulate(w))
    W1 = [0] + list(itertools.accumulate(d * x for d, x in enumerate(w)))
    for s in range(0, 41):
        for t in range(s, 42):
            direct = sum(w[d] * (d - s) for d in range(s, min(t, 41)))
            assert (W1[t] - W1[s]) - s * (W0[t] - W0[s]) == direct


def test_dp_oracle_equals_brute_force():
    rng = random.Random(2)
    for N in range(1, 11):
        for M in range(0, 5):
            for _ in range(3):
                w = _weights(rng, N)
                best, args = P.brute_force(w, M)
                pos, cost = P.place_dp(w, M)
                assert cost == best, (N, M, w)
                assert tuple(pos) in args
                assert P.expected_recompute(w, pos) == cost


def test_theorem1_uniform_depths_every_optimum_is_balanced():
    for N in range(2, 11):
        w = [0] + [1] * N            # d uniform on 1..N, p(0) = 0
        for M in range(1, N):
            best, args = P.brute_force(w, M)
            for c in args:
                g = P.gaps(c, N)
                assert max(g) - min(g) <= 1, (N, M, c)
            bal = P.balanced(N, M)
            assert P.expected_recompute(w, bal) == best
            # closed form of the proof: a gap of length g contributes g (g - 1) / 2
            assert best == sum(g * (g - 1) // 2 for g in P.gaps(bal, N))


def test_more_checkpoints_never_hurt_and_extremes():
    rng = random.Random(3)
    for _ in range(5):
        w = _weights(rng, 30)
        costs = [P.place_dp(w, M)[1] for M in range(0, 32)]
        assert costs[0] == P.no_cache(w)
        assert all(a >= b for a, b in zip(costs, costs[1:]))
        assert costs[30] == 0 and costs[31] == 0


def test_lemma1_value_is_lipschitz_in_total_variation():
    rng = random.Random(4)
    N = 12
    for _ in range(6):
        a, b = _weights(rng, N, 0.2), _weights(rng, N, 0.2)
        if sum(a) == 0 or sum(b) == 0:
            continue
        p, q = P.normalise(a), P.normalise(b)
        for M in (1, 3):
            Vp = Fraction(P.place_dp(a, M)[1], sum(a))
            Vq = Fraction(P.place_dp(b, M)[1], sum(b))
            assert abs(Vp - Vq) <= N * P.tv(p, q)


def test_theorem3_plug_in_placement_from_empirical_depths():
    """R(p, g_hat) <= V(p, M) + 2 N TV(p_hat, p) for g_hat optimal on T sampled depths."""
    rng = random.Random(5)
    N = 60
    w = synth.depth_weights("documents", N, 5000, seed=3)
    p = P.normalise(w)
    for T in (20, 200, 2000):
        for M in (2, 6):
            sample = rng.choices(range(N + 1), weights=w, k=T)
            w_hat = [0] * (N + 1)
            for d in sample:
                w_hat[d] += 1
            g_hat, _ = P.place_dp(w_hat, M)
            R_true = Fraction(P.expected_recompute(w, g_hat), sum(w))
            V = Fraction(P.place_dp(w, M)[1], sum(w))
            assert V <= R_true <= V + 2 * N * P.tv(P.normalise(w_hat), p)


def test_baselines_never_beat_the_optimum():
    N, M = 120, 5
    for kind in synth.DEPTH_KINDS:
        w = synth.depth_weights(kind, N, 3000, seed=1)
        _, opt = P.place_dp(w, M)
        for c in (P.balanced(N, M), P.block(N, M), P.greedy(w, M), P.random_place(N, M, 9)):
            assert P.expected_recompute(w, c) >= opt


def test_random_and_splitmix_reference_values():
    """splitmix64 from seed 0 starts 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4 (its published
    reference outputs); the shuffle takes distinct positions in range."""
    st, x1 = P.splitmix64(0)
    st, x2 = P.splitmix64(st)
    assert (x1, x2) == (0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4)
    c = P.random_place(50, 10, 123)
    assert c == sorted(set(c)) and len(c) == 10 and 1 <= c[0] and c[-1] <= 50


# ---------------------------------------------------------------------------------------------
# the C-ABI implementation against the oracle
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("N,Ms", [(1, [0, 1, 2]), (2, [0, 1, 2, 5]), (7, [0, 1, 3, 6, 7, 9]),
                                  (64, [1, 2, 5, 16, 63, 64]), (500, [1, 7, 16, 31]), (2048, [16, 32])])
def test_dp_matches_oracle_exactly(N, Ms):
    rng = random.Random(N)
    cases = [_weights(rng, N), _weights(rng, N, 0.9, 1000), [0] * (N + 1), [0] + [1] * N]
    cases += [synth.depth_weights(k, N, 4000, seed=N) for k in synth.DEPTH_KINDS]
    for w in cases:
        for M in Ms:
            pos, cost = gdn.gdn_ckpt_placement(w, M, "dp")
            _, ref = P.place_dp(w, M)
            assert cost == ref, (N, M)
            assert len(pos) == min(M, N) and pos == sorted(set(pos)) and (not pos or (pos[0] >= 1 and pos[-1] <= N))
            assert P.expected_recompute(w, pos) == cost
            assert gdn.gdn_expected_recompute(w, pos) == cost


def test_dp_at_the_long_prefix_size():
    """N = 131072, M = 32 (the long-prefill checkpoint budget): the product's O(N M) programme
    against the balanced placement and a local check (moving any checkpoint by one never helps)."""
    N, M = 131072, 32
    w = synth.depth_weights("prompts", N, 20000, seed=5)
    pos, cost = gdn.gdn_ckpt_placement(w, M, "dp")
    assert cost == P.expected_recompute(w, pos)
    assert cost <= gdn.gdn_ckpt_placement(w, M, "balanced")[1]
    assert cost <= gdn.gdn_ckpt_placement(w, M, "greedy")[1]
    for i in range(M):
        for delta in (-1, 1):
            c = list(pos)
            c[i] += delta
            if c == sorted(set(c)) and 1 <= c[0] and c[-1] <= N:
                assert gdn.gdn_expected_recompute(w, c) >= cost


@pytest.mark.parametrize("N,M", [(1, 1), (5, 2), (20, 3), (101, 7), (300, 12)])
def test_baselines_match_oracle_position_for_position(N, M):
    for kind in synth.DEPTH_KINDS:
        w = synth.depth_weights(kind, N, 1500, seed=M)
        for strategy, ref in (("balanced", P.balanced(N, M)), ("block", P.block(N, M)),
                              ("greedy", P.greedy(w, M)), ("random", P.random_place(N, M, 42))):
            pos, cost = gdn.gdn_ckpt_placement(w, M, strategy, seed=42)
            assert pos == ref, (strategy, N, M)
            assert cost == P.expected_recompute(w, ref)
    w = [1] * (N + 1)
    pos, _ = gdn.gdn_ckpt_placement(w, M, "block", block=3)
    assert pos == P.block(N, M, 3)


def test_expected_recompute_matches_definition():
    rng = random.Random(7)
    for N in (1, 9, 300):
        w = _weights(rng, N)
        for M in range(0, min(N, 6) + 1):
            c = sorted(rng.sample(range(1, N + 1), M))
            assert gdn.gdn_expected_recompute(w, c) == P.expected_recompute(w, c)


def test_placement_rejects_bad_arguments():
    w = [1] * 11
    with pytest.raises(gdn.GdnError):
        gdn.gdn_ckpt_placement([1, -1, 2], 1)                       # negative weight
    with pytest.raises(gdn.GdnError):
        gdn.gdn_ckpt_placement(w, -1)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_ckpt_placement(w, 2, "block", block=-3)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_ckpt_placement([5], 1)                              # N = 0
    with pytest.raises(gdn.GdnError):
        gdn.gdn_ckpt_placement([1 << 59] * 4, 1)                    # totals past 2^60
    for bad in ([3, 3], [0, 4], [4, 11], [5, 2]):
        with pytest.raises(gdn.GdnError):
            gdn.gdn_expected_recompute(w, bad)
    L = gdn.lib()
    import ctypes
    import numpy as np
    arr = np.ones(11, dtype=np.int64)
    out = np.zeros(4, dtype=np.int64)
    n, c = ctypes.c_int32(), ctypes.c_int64()
    P64 = ctypes.POINTER(ctypes.c_int64)
    rc = L.gdn_ckpt_placement(arr.ctypes.data_as(P64), 10, 2, 9, 0, 0, out.ctypes.data_as(P64), ctypes.byref(n),
                              ctypes.byref(c))
    assert rc == gdn.GDN_ERR_INVALID_ARG                             # unknown strategy
    rc = L.gdn_ckpt_placement(None, 10, 2, 0, 0, 0, out.ctypes.data_as(P64), ctypes.byref(n), ctypes.byref(c))
    assert rc == gdn.GDN_ERR_INVALID_ARG
