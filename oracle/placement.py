"""Checkpoint placement oracle -- TEST INFRASTRUCTURE (same rules as the rest of ``oracle``).

"Sparse prefix caching in hybrid and recurrent LLM serving":
* section 3: a prefix of N tokens keeps states at 1 <= c_1 < ... < c_M <= N; a request that
  overlaps it to depth d resumes from the deepest c_j <= d (the start, c_0 = 0, if none) and
  recomputes f(d) = d - c_j tokens, f(0) = 0.  The depth distribution is given as integer weights
  w[0..N], so the expected recompute is the exact integer R = sum_d w[d] f(d);
* section 4: Theorem 1 (uniform depths -> the gaps of an optimal placement differ by at most one),
  Theorem 2 (the optimum by dynamic programming), Lemma 1 and Theorem 3 (plug-in bounds);
* section 5: the baselines (no cache, uniform spacing, blocks, random, greedy).

Everything here follows those definitions directly: brute force over all placements for tiny N,
the plain O(M N^2) dynamic programme (in ``gdn_oracle.c``), and the baselines step by step.
"""
from __future__ import annotations

import bisect
import ctypes
import itertools
from fractions import Fraction
from typing import List, Sequence, Tuple

import numpy as np

from . import _load

MASK64 = (1 << 64) - 1


def recompute(c: Sequence[int], d: int) -> int:
    """f(d) of section 3: tokens recomputed for overlap depth d with checkpoints c."""
    if d == 0:
        return 0
    j = bisect.bisect_right(list(c), d)   # number of checkpoints <= d
    return d - (c[j - 1] if j > 0 else 0)


def expected_recompute(w: Sequence[int], c: Sequence[int]) -> int:
    """R = sum_d w[d] f(d) (exact integer numerator)."""
    return sum(int(w[d]) * recompute(c, d) for d in range(len(w)))


def gaps(c: Sequence[int], N: int) -> List[int]:
    """The gap vector g_1..g_K of section 3 (K = M + 1, sum g = N + 1)."""
    pts = [0] + list(c) + [N + 1]
    return [pts[i + 1] - pts[i] for i in range(len(pts) - 1)]


def brute_force(w: Sequence[int], M: int) -> Tuple[int, List[Tuple[int, ...]]]:
    """Least R over every placement of min(M, N) checkpoints, and every placement reaching it."""
    N = len(w) - 1
    m = min(M, N)
    best, arg = None, []
    for c in itertools.combinations(range(1, N + 1), m):
        r = expected_recompute(w, c)
        if best is None or r < best:
            best, arg = r, [c]
        elif r == best:
            arg.append(c)
    return best, arg


def place_dp(w: Sequence[int], M: int) -> Tuple[List[int], int]:
    """Theorem 2's dynamic programme, plain O(M N^2) (one optimal placement, its R)."""
    arr = np.ascontiguousarray(np.asarray(w, dtype=np.int64))
    N = len(arr) - 1
    m = min(M, N)
    pos = np.zeros(max(m, 1), dtype=np.int64)
    cost = ctypes.c_int64()
    rc = _load().gdn_oracle_place_dp(arr.ctypes.data, N, M, pos.ctypes.data, ctypes.byref(cost))
    if rc != 0:
        raise MemoryError("gdn_oracle_place_dp")
    return [int(x) for x in pos[:m]], cost.value


def no_cache(w: Sequence[int]) -> int:
    """R with no checkpoint: every request recomputes its whole overlap."""
    return sum(int(w[d]) * d for d in range(len(w)))


def balanced(N: int, M: int) -> List[int]:
    """Theorem 1's balanced placement: K = M + 1 gaps summing to N + 1 that differ by at most one,
    the larger ones first."""
    m = min(M, N)
    K = m + 1
    q, rho = divmod(N + 1, K)
    g = [q + 1 if i < rho else q for i in range(m)]
    return list(itertools.accumulate(g))


def block(N: int, M: int, b: int = 0) -> List[int]:
    """Block boundaries b, 2b, ... <= N, at most min(M, N) of them (b = floor(N / M) when 0)."""
    m = min(M, N)
    if m == 0:
        return []
    if b == 0:
        b = max(1, N // m)
    return [i * b for i in range(1, m + 1) if i * b <= N]


def greedy(w: Sequence[int], M: int) -> List[int]:
    """Section 5's greedy baseline: M times, add the free position whose checkpoint gives the
    lowest R (the shallowest on ties), evaluating R from its definition."""
    N = len(w) - 1
    chosen: List[int] = []
    for _ in range(min(M, N)):
        best, best_c = None, None
        for c in range(1, N + 1):
            if c in chosen:
                continue
            r = expected_recompute(w, sorted(chosen + [c]))
            if best is None or r < best:
                best, best_c = r, c
        chosen.append(best_c)
    return sorted(chosen)


def splitmix64(state: int) -> Tuple[int, int]:
    """One step of splitmix64 (Steele, Lea and Flood): (new state, output)."""
    state = (state + 0x9E3779B97F4A7C15) & MASK64
    z = state
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return state, z ^ (z >> 31)


def random_place(N: int, M: int, seed: int) -> List[int]:
    """The first min(M, N) picks of a Fisher-Yates shuffle of 1..N; the pick at step i is
    i + floor(x (N - i) / 2^64) for the i-th splitmix64 output x; sorted."""
    a = list(range(1, N + 1))
    st = seed & MASK64
    for i in range(min(M, N)):
        st, x = splitmix64(st)
        j = i + ((x * (N - i)) >> 64)
        a[i], a[j] = a[j], a[i]
    return sorted(a[:min(M, N)])


def tv(p: Sequence[Fraction], q: Sequence[Fraction]) -> Fraction:
    """Total-variation distance of two distributions on 0..N."""
    return sum(abs(Fraction(a) - Fraction(b)) for a, b in zip(p, q)) / 2


def normalise(w: Sequence[int]) -> List[Fraction]:
    tot = sum(int(x) for x in w)
    return [Fraction(int(x), tot) for x in w]
