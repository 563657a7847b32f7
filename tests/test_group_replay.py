"""In-group chained replay ("Tail-Replay" notes page, section 2.2 step 3, section 2.4): oracle pins
and the C-ABI argument checks (host only; the GPU parity test is in test_replay_extensions_gpu.py)."""
import ctypes

import numpy as np
import pytest

import hybrid_model_recurrent_gb300 as gdn
import oracle
import synth
from oracle import group as G


def _case(L, H, Dm, d, m, seed=0):
    return synth.group_weights(seed, L, H, Dm, d), synth.group_inputs(seed, m, Dm)


def test_full_tail_replay_is_the_full_chain():
    w, h = _case(3, 2, 32, 16, 60)
    r = G.group_replay(h, w, 3, 2, 32, 16, 60, 1, 1)
    assert (r["a"], r["k"]) == (0, 60)
    for l in range(3):
        for hh in range(2):
            assert np.array_equal(r["S_hat"][l][hh], r["S_exact"][l][hh])


def test_first_layer_is_a_plain_tail_replay_of_its_inputs():
    L, H, Dm, d, m = 2, 2, 32, 16, 80
    w, h = _case(L, H, Dm, d, m, seed=1)
    r = G.group_replay(h, w, L, H, Dm, d, m, 1, 4)
    Ws = G.unpack(w, L, H, Dm, d)
    q, k, v, a, b = G.project(np.asarray(h, dtype=np.float64), Ws[0], H, d)
    for hh in range(H):
        ref = np.asarray(oracle.tail_replay(k[:, hh], v[:, hh], a[:, hh], b[:, hh], m, 1, 4)["S_hat"])
        # the projections of the tail rows alone and of all rows may round differently in BLAS
        assert np.abs(ref - r["S_hat"][0][hh]).max() <= 1e-12 * np.abs(ref).max()


def test_error_recursion_of_the_later_layers():
    """E_i = E_{i-1} T_i + S^_{i-1}(T_i - T^_i) + (b_i - b^_i) along the tail of every layer (the layers
    after the first see different transitions), with explicit d x d matrices."""
    L, H, Dm, d, m = 3, 1, 24, 8, 40
    w, h = _case(L, H, Dm, d, m, seed=2)
    Ws = G.unpack(w, L, H, Dm, d)
    a, k = oracle.replay_plan(m, 1, 5)
    hx = np.asarray(h, dtype=np.float64)
    _, ex_in = G.chain(hx[:m], Ws, H, d, keep_inputs=True)       # inputs of the full run, rows 1..m
    _, rp_in = G.chain(hx[a:m], Ws, H, d, keep_inputs=True)      # inputs of the replay, rows a+1..m
    I = np.eye(d)
    worst = 0.0
    for l in range(L):
        q, kk, v, al, be = (x[:, 0] if x.ndim == 3 else x[:, 0] for x in ex_in[l])
        qh, kh, vh, alh, beh = (x[:, 0] for x in rp_in[l])
        # per-token states of both runs along the tail (checkpoints at every position)
        full = oracle.scan(kk, v, al, be, ckpt_pos=list(range(1, m + 1)), want_o=False)
        S = [np.zeros((d, d))] + [np.asarray(s) for s in full["ckpt"]]
        rep = oracle.scan(kh, vh, alh, beh, ckpt_pos=list(range(1, k + 1)), want_o=False)
        Sh = [np.zeros((d, d))] + [np.asarray(s) for s in rep["ckpt"]]
        E = S[a] - Sh[0]
        for j in range(1, k + 1):
            i = a + j
            T = al[i - 1] * (I - be[i - 1] * np.outer(kk[i - 1], kk[i - 1]))
            Th = alh[j - 1] * (I - beh[j - 1] * np.outer(kh[j - 1], kh[j - 1]))
            b = be[i - 1] * np.outer(v[i - 1], kk[i - 1])
            bh = beh[j - 1] * np.outer(vh[j - 1], kh[j - 1])
            E = E @ T + Sh[j - 1] @ (T - Th) + (b - bh)
            worst = max(worst, float(np.abs(E - (S[i] - Sh[j])).max()))
        if l == 0:
            assert np.allclose(T, Th) and np.allclose(b, bh)   # the first layer's inputs are exact
    assert worst < 1e-12


def test_group_abi_rejects_bad_arguments():
    L = gdn.lib()
    P = ctypes.POINTER(gdn._Group)
    vp = lambda x: ctypes.c_void_p(x)

    def call(g, m=100, rn=1, rd=10, h=0x1000, wt=0x2000, sh=0x3000, se=None, scratch=0x4000, sb=1 << 30, ws=0x5000,
             wsb=256):
        return L.gdn_group_replay(ctypes.byref(g), vp(h) if h else None, m, rn, rd, vp(wt) if wt else None,
                                  vp(sh) if sh else None, vp(se) if se else None, None, None,
                                  vp(scratch) if scratch else None, sb, vp(ws) if ws else None, wsb, None)

    good = gdn._Group(2, 2, 64, 32)
    E = gdn.GDN_ERR_INVALID_ARG
    for bad in (gdn._Group(0, 2, 64, 32), gdn._Group(2, 0, 64, 32), gdn._Group(2, 2, 0, 32), gdn._Group(2, 2, 64, 48),
                gdn._Group(65, 2, 64, 32), gdn._Group(2, 2, 9000, 32)):
        assert call(bad) == E
        assert L.gdn_group_scratch_bytes(ctypes.byref(bad), 10) == 0
    assert call(good, m=-1) == E
    assert call(good, rn=2, rd=1) == E
    assert call(good, h=0) == E and call(good, wt=0) == E and call(good, sh=0) == E
    assert call(good, sh=0x3004) == E                      # S_hat not 16-byte aligned
    assert call(good, scratch=0) == E
    need = L.gdn_group_scratch_bytes(ctypes.byref(good), 10)   # k = ceil(100 / 10) = 10 rows
    assert need == 10 * (2 * 64 + 4 * 2 * 32 + 2 * 2) * 4
    assert call(good, sb=need - 4) == E
    assert call(good, se=0x6000, sb=need) == E             # the full chain needs m = 100 rows
    assert call(good, wsb=8) == E
