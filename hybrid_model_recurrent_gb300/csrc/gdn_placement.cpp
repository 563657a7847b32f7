// gdn_placement.cpp - checkpoint placement for sparse prefix caching (host code).
//
// "Sparse prefix caching in hybrid and recurrent LLM serving", section 3 (problem statement) and
// section 4 (Theorems 1 and 2), section 5 (baselines): a cached prefix of N tokens keeps exact
// recurrent states at positions 1 <= c_1 < ... < c_M <= N.  A request that overlaps the prefix to
// depth d resumes from the deepest c_j <= d (c_0 = 0: the start) and recomputes f(d) = d - c_j
// tokens; f(0) = 0.  Depths follow a distribution given here as integer weights w(0..N) (counts of
// observed depths), so every expected cost is an exact integer numerator R = sum_d w(d) f(d).
//
// Strategies: the optimal placement by dynamic programming in O(N M) (Theorem 2: segment costs from
// prefix sums, minimised with the monotone convex-hull trick), the balanced placement of Theorem 1,
// fixed-size blocks, random positions and the greedy baseline.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <vector>

#include "../../include/gdn_scan.h"

#define GDN_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

typedef __int128 i128;

constexpr int64_t kMaxN = (int64_t)1 << 31;
constexpr int64_t kMaxTable = (int64_t)1 << 26;   // (M + 1) (N + 1) parent entries of the DP
constexpr int64_t kMaxScan = (int64_t)1 << 24;    // positions scanned by the greedy and random baselines

// Prefix sums W0[x] = sum_{d<x} w(d), W1[x] = sum_{d<x} d w(d), x = 0..N+1.
struct Prefix {
    std::vector<int64_t> W0, W1;
    // expected-recompute numerator of the segment [s, t): sum_{d=s}^{t-1} w(d) (d - s)
    int64_t seg(int64_t s, int64_t t) const { return (W1[t] - W1[s]) - s * (W0[t] - W0[s]); }
};

// Validates the weights and builds the prefix sums; sum_d d w(d) and N sum_d w(d) must stay below
// 2^60 so that every cost, line intercept and line value below fits in 64 bits.
gdn_status make_prefix(const int64_t* w, int64_t N, Prefix& P) {
    if (!w || N < 1 || N >= kMaxN) return N >= kMaxN ? GDN_ERR_UNSUPPORTED : GDN_ERR_INVALID_ARG;
    P.W0.assign((size_t)N + 2, 0);
    P.W1.assign((size_t)N + 2, 0);
    const i128 lim = (i128)1 << 60;
    i128 a = 0, b = 0;
    for (int64_t d = 0; d <= N; ++d) {
        if (w[d] < 0) return GDN_ERR_INVALID_ARG;
        a += w[d];
        b += (i128)w[d] * d;
        if (a >= lim || b >= lim || (i128)N * a >= lim) return GDN_ERR_UNSUPPORTED;
        P.W0[(size_t)d + 1] = (int64_t)a;
        P.W1[(size_t)d + 1] = (int64_t)b;
    }
    return GDN_OK;
}

int64_t cost_of(const Prefix& P, int64_t N, const int64_t* pos, int32_t M) {
    int64_t c = 0, prev = 0;
    for (int32_t i = 0; i < M; ++i) {
        c += P.seg(prev, pos[i]);
        prev = pos[i];
    }
    return c + P.seg(prev, N + 1);
}

bool strictly_increasing_in_range(const int64_t* pos, int32_t M, int64_t N) {
    for (int32_t i = 0; i < M; ++i) {
        if (pos[i] < 1 || pos[i] > N) return false;
        if (i > 0 && pos[i] <= pos[i - 1]) return false;
    }
    return true;
}

// Optimal placement of exactly M (<= N) checkpoints.  E_k[t] = least cost of the depths [0, t) with
// the k-th checkpoint at t; E_0 is 0 at t = 0.  E_k[t] = min_{k-1 <= s < t} E_{k-1}[s] + seg(s, t)
//   = W1[t] + min_s ( -s W0[t] + B[s] ),  B[s] = E_{k-1}[s] - W1[s] + s W0[s]:
// lines of slope -s (falling with s) read at x = W0[t] (rising with t), so a monotone lower envelope
// gives each layer in O(N).
void place_dp(const Prefix& P, int64_t N, int32_t M, int64_t* pos) {
    const size_t n1 = (size_t)N + 1;
    std::vector<int64_t> prev(n1, 0), cur(n1, 0);
    std::vector<int32_t> parent((size_t)M * n1, 0);
    // lines are kept as indices s into (slope -s, intercept B[s])
    std::vector<int64_t> hull_s(n1), hull_b(n1);
    // k = 1: the only earlier checkpoint is the start, s = 0
    for (int64_t t = 1; t <= N; ++t) {
        prev[(size_t)t] = P.seg(0, t);
        parent[(size_t)t] = 0;
    }
    for (int32_t k = 2; k <= M; ++k) {
        size_t head = 0, size = 0;
        int32_t* par = parent.data() + (size_t)(k - 1) * n1;
        for (int64_t t = k; t <= N; ++t) {
            // add the line of s = t - 1 (only s >= k - 1 is reachable with k - 1 earlier checkpoints)
            {
                const int64_t s = t - 1;
                const int64_t b = prev[(size_t)s] - P.W1[(size_t)s] + s * P.W0[(size_t)s];
                while (size - head >= 2) {
                    const int64_t s1 = hull_s[size - 2], b1 = hull_b[size - 2];
                    const int64_t s2 = hull_s[size - 1], b2 = hull_b[size - 1];
                    // slopes m1 = -s1 > m2 = -s2 > m3 = -s; line 2 never strictly lowest when
                    // (b2 - b1)(m2 - m3) >= (b - b2)(m1 - m2)
                    const i128 lhs = (i128)(b2 - b1) * (i128)(s - s2);
                    const i128 rhs = (i128)(b - b2) * (i128)(s2 - s1);
                    if (lhs >= rhs) --size;
                    else break;
                }
                hull_s[size] = s;
                hull_b[size] = b;
                ++size;
                if (head >= size) head = size - 1;
            }
            const int64_t x = P.W0[(size_t)t];
            while (head + 1 < size) {
                const i128 v0 = -(i128)hull_s[head] * x + hull_b[head];
                const i128 v1 = -(i128)hull_s[head + 1] * x + hull_b[head + 1];
                if (v1 <= v0) ++head;
                else break;
            }
            cur[(size_t)t] = P.W1[(size_t)t] - hull_s[head] * x + hull_b[head];
            par[t] = (int32_t)hull_s[head];
        }
        std::swap(prev, cur);
        for (int64_t t = 0; t < k; ++t) prev[(size_t)t] = 0;   // unreachable, never read as a line
    }
    // last checkpoint: least E_M[t] + seg(t, N + 1); ties go to the deepest t
    int64_t best_t = M, best = 0;
    for (int64_t t = M; t <= N; ++t) {
        const int64_t v = prev[(size_t)t] + P.seg(t, N + 1);
        if (t == M || v <= best) {
            best = v;
            best_t = t;
        }
    }
    int64_t t = best_t;
    for (int32_t k = M; k >= 1; --k) {
        pos[k - 1] = t;
        t = parent[(size_t)(k - 1) * n1 + (size_t)t];
    }
}

// Theorem 1: K = M + 1 gaps summing to N + 1 that differ by at most one (the larger ones first).
void place_balanced(int64_t N, int32_t M, int64_t* pos) {
    const int64_t K = (int64_t)M + 1, q = (N + 1) / K, rho = (N + 1) % K;
    int64_t c = 0;
    for (int32_t i = 0; i < M; ++i) {
        c += q + (i < rho ? 1 : 0);
        pos[i] = c;
    }
}

// Greedy baseline: add, M times, the free position whose checkpoint lowers the cost most
// (the shallowest one on ties).
void place_greedy(const Prefix& P, int64_t N, int32_t M, int64_t* pos) {
    std::vector<char> used((size_t)N + 2, 0);
    used[0] = used[(size_t)N + 1] = 1;
    std::vector<int64_t> left((size_t)N + 2), right((size_t)N + 2);
    for (int32_t it = 0; it < M; ++it) {
        // nearest checkpoint at or below / above every position
        int64_t l = 0;
        for (int64_t x = 0; x <= N + 1; ++x) {
            if (used[(size_t)x]) l = x;
            left[(size_t)x] = l;
        }
        int64_t r = N + 1;
        for (int64_t x = N + 1; x >= 0; --x) {
            if (used[(size_t)x]) r = x;
            right[(size_t)x] = r;
        }
        int64_t best_c = -1, best_gain = -1;
        for (int64_t c = 1; c <= N; ++c) {
            if (used[(size_t)c]) continue;
            const int64_t a = left[(size_t)c], b = right[(size_t)c];
            const int64_t gain = P.seg(a, b) - P.seg(a, c) - P.seg(c, b);
            if (gain > best_gain) {
                best_gain = gain;
                best_c = c;
            }
        }
        used[(size_t)best_c] = 1;
    }
    int32_t k = 0;
    for (int64_t c = 1; c <= N; ++c)
        if (used[(size_t)c]) pos[k++] = c;
}

// splitmix64 (Steele, Lea and Flood; the constants of its published definition)
uint64_t splitmix64(uint64_t& state) {
    uint64_t z = (state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Random baseline: the first M draws of a Fisher-Yates shuffle of 1..N (index = high word of
// draw * remaining), sorted.
void place_random(int64_t N, int32_t M, uint64_t seed, int64_t* pos) {
    std::vector<int64_t> a((size_t)N);
    for (int64_t i = 0; i < N; ++i) a[(size_t)i] = i + 1;
    uint64_t st = seed;
    for (int32_t i = 0; i < M; ++i) {
        const uint64_t range = (uint64_t)(N - i);
        const uint64_t j = (uint64_t)i + (uint64_t)(((unsigned __int128)splitmix64(st) * range) >> 64);
        std::swap(a[(size_t)i], a[(size_t)j]);
    }
    std::sort(a.begin(), a.begin() + M);
    std::memcpy(pos, a.data(), sizeof(int64_t) * (size_t)M);
}

}  // namespace

GDN_EXPORT gdn_status gdn_expected_recompute(const int64_t* weights, int64_t N, const int64_t* positions,
                                             int32_t M, int64_t* cost) {
    if (!cost || M < 0 || (M > 0 && !positions)) return GDN_ERR_INVALID_ARG;
    Prefix P;
    const gdn_status st = make_prefix(weights, N, P);
    if (st != GDN_OK) return st;
    if (!strictly_increasing_in_range(positions, M, N)) return GDN_ERR_INVALID_ARG;
    *cost = cost_of(P, N, positions, M);
    return GDN_OK;
}

GDN_EXPORT gdn_status gdn_ckpt_placement(const int64_t* weights, int64_t N, int32_t M, gdn_placement strategy,
                                         uint64_t seed, int64_t block, int64_t* positions, int32_t* count,
                                         int64_t* cost) {
    if (!count || !cost || M < 0 || (M > 0 && !positions)) return GDN_ERR_INVALID_ARG;
    if (strategy != GDN_PLACE_DP && strategy != GDN_PLACE_BALANCED && strategy != GDN_PLACE_BLOCK &&
        strategy != GDN_PLACE_RANDOM && strategy != GDN_PLACE_GREEDY)
        return GDN_ERR_INVALID_ARG;
    if (block < 0) return GDN_ERR_INVALID_ARG;
    Prefix P;
    const gdn_status st = make_prefix(weights, N, P);
    if (st != GDN_OK) return st;
    const int32_t m = (int64_t)M > N ? (int32_t)N : M;   // more checkpoints than positions: all of them
    if (strategy == GDN_PLACE_DP && (int64_t)(m + 1) * (N + 1) > kMaxTable) return GDN_ERR_UNSUPPORTED;
    if ((strategy == GDN_PLACE_RANDOM || strategy == GDN_PLACE_GREEDY) && N > kMaxScan) return GDN_ERR_UNSUPPORTED;
    int32_t n = m;
    if (m > 0) {
        switch (strategy) {
            case GDN_PLACE_DP: place_dp(P, N, m, positions); break;
            case GDN_PLACE_BALANCED: place_balanced(N, m, positions); break;
            case GDN_PLACE_GREEDY: place_greedy(P, N, m, positions); break;
            case GDN_PLACE_RANDOM: place_random(N, m, seed, positions); break;
            case GDN_PLACE_BLOCK: {
                const int64_t b = block > 0 ? block : std::max<int64_t>(1, N / m);
                n = 0;
                for (int32_t i = 1; i <= m && (int64_t)i * b <= N; ++i) positions[n++] = (int64_t)i * b;
                break;
            }
        }
    }
    *count = n;
    *cost = cost_of(P, N, positions, n);
    return GDN_OK;
}
