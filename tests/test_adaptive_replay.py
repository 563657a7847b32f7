"""Adaptive replay length ("Tail-Replay" notes page, section 5: the proposed extension) and the
bound it relies on (section 2.3).  Host only: oracle pins and argument checks; the C-ABI plan
itself reads device gates and is compared with the oracle in the GPU tests."""
import ctypes

import numpy as np
import pytest
import torch

import hybrid_model_recurrent_gb300 as gdn
import oracle
import synth


def _gates(seed, T, H, lo, hi):
    a, b = synth.gates(seed, 0, T, H, lo, hi, "uniform")
    return a, b


def test_plan_is_the_least_k_meeting_eps_for_every_head():
    T, H = 300, 3
    alpha, _ = _gates(3, T, H, 0.6, 1.0)
    alpha[:, 2] = torch.clamp(alpha[:, 2] * 0 + 0.995, max=1.0)   # one slow-forgetting head
    cu, m = [0, 300], [300]
    for eps, rmax in ((1e-2, (1, 10)), (1e-2, (1, 1)), (0.5, (1, 20)), (1e-6, (1, 2))):
        ks, ex = oracle.adaptive_replay_plan(alpha, cu, m, eps, *rmax)
        _, K = oracle.replay_plan(300, *rmax)
        a = alpha.numpy()
        prods = [np.cumprod(a[::-1, h].astype(np.float64)) for h in range(H)]
        if ex[0] == 0:
            k = ks[0]
            assert all(prods[h][k - 1] <= eps * (1 + 1e-5) for h in range(H))
            assert k == 1 or any(prods[h][k - 2] > eps * (1 - 1e-5) for h in range(H))
        else:
            assert ks[0] == K and any(prods[h][K - 1] > eps * (1 - 1e-5) for h in range(H))


def test_plan_edge_cases():
    alpha = torch.full((10, 2), 0.5)
    assert oracle.adaptive_replay_plan(alpha, [0, 10], [0], 0.1, 1, 10) == ([0], [0])      # empty prefix
    assert oracle.adaptive_replay_plan(alpha, [0, 10], [10], 0.1, 0, 1) == ([0], [1])      # no budget
    # 0.5^4 = 0.0625 <= 0.1 < 0.125 = 0.5^3
    assert oracle.adaptive_replay_plan(alpha, [0, 10], [10], 0.1, 1, 1) == ([4], [0])
    assert oracle.adaptive_replay_plan(alpha, [0, 10], [10], 0.1, 1, 5) == ([2], [1])     # budget 2 < 4


def test_chosen_tail_meets_the_error_bound():
    """With unit keys and beta in [0, 2]: ||S_m - S_hat_m||_F <= (prod alpha) ||S_a||_F <= eps ||S_a||_F."""
    T, H, d = 400, 3, 16
    w = synth.Workload("adaptive", [T], H, d, d, torch.float32, torch.float32, 0.7, 1.0, "uniform", seed=5)
    inp = synth.make_inputs(w)
    S_a = synth.state(7, H, d, d, 1.0)
    eps = 1e-3
    ks, ex = oracle.adaptive_replay_plan(inp.alpha, w.cu_seqlens, [T], eps, 1, 2)
    assert ex == [0]
    k = ks[0]
    for h in range(H):
        r = oracle.tail_replay(inp.k[:, h], inp.v[:, h], inp.alpha[:, h], inp.beta[:, h], T, k, T,
                               S_a=S_a[h])
        E = np.asarray(r["S_exact"]) - np.asarray(r["S_hat"])
        prod = float(np.prod(inp.alpha[T - k:T, h].double().numpy()))
        nS = float(np.linalg.norm(np.asarray(S_a[h], dtype=np.float64)))
        assert np.linalg.norm(E) <= prod * nS * (1 + 1e-9) + 1e-12
        assert prod <= eps * (1 + 1e-6)


def test_abi_rejects_bad_adaptive_arguments():
    L = gdn.lib()
    cu = np.array([0, 10], dtype=np.int64)
    pr = gdn._Problem()
    pr.num_seqs, pr.num_heads, pr.d_k, pr.d_v = 1, 2, 32, 32
    pr.cu_seqlens = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    pr.qkv_dtype = pr.out_dtype = gdn.GDN_BF16
    m = np.array([10], dtype=np.int64)
    k = np.zeros(1, dtype=np.int64)
    ex = np.zeros(1, dtype=np.int32)
    P64, P32 = ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)
    fake = ctypes.c_void_p(0x10000)
    for eps, rn, rd in ((1.0, 1, 10), (-0.1, 1, 10), (float("nan"), 1, 10), (0.1, 2, 1), (0.1, 1, 0)):
        rc = L.gdn_adaptive_replay_plan(ctypes.byref(pr), fake, m.ctypes.data_as(P64), ctypes.c_float(eps), rn, rd,
                                        k.ctypes.data_as(P64), ex.ctypes.data_as(P32), None)
        assert rc == gdn.GDN_ERR_INVALID_ARG, (eps, rn, rd)
    m2 = np.array([11], dtype=np.int64)   # m beyond the sequence
    rc = L.gdn_adaptive_replay_plan(ctypes.byref(pr), fake, m2.ctypes.data_as(P64), ctypes.c_float(0.1), 1, 10,
                                    k.ctypes.data_as(P64), ex.ctypes.data_as(P32), None)
    assert rc == gdn.GDN_ERR_INVALID_ARG
    rc = L.gdn_adaptive_replay_plan(ctypes.byref(pr), None, m.ctypes.data_as(P64), ctypes.c_float(0.1), 1, 10,
                                    k.ctypes.data_as(P64), ex.ctypes.data_as(P32), None)
    assert rc == gdn.GDN_ERR_INVALID_ARG


def test_abi_replay_k_and_overlap_reject_bad_arguments():
    L = gdn.lib()
    cu = np.array([0, 10], dtype=np.int64)
    pr = gdn._Problem()
    pr.num_seqs, pr.num_heads, pr.d_k, pr.d_v = 1, 2, 32, 32
    pr.cu_seqlens = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    pr.qkv_dtype = pr.out_dtype = gdn.GDN_BF16
    P64 = ctypes.POINTER(ctypes.c_int64)
    vp = lambda x: ctypes.c_void_p(x)
    m = np.array([10], dtype=np.int64)
    for kk in (11, -1):
        kr = np.array([kk], dtype=np.int64)
        rc = L.gdn_tail_replay_k(ctypes.byref(pr), None, vp(0x1000), vp(0x2000), vp(0x3000), vp(0x4000),
                                 m.ctypes.data_as(P64), kr.ctypes.data_as(P64), None, vp(0x5000), None, None,
                                 vp(0x8000), 256, None)
        assert rc == gdn.GDN_ERR_INVALID_ARG
    # overlap: a copy of kv_bytes > 0 needs both buffers; a bad replay argument enqueues nothing
    a_o = np.zeros(1, dtype=np.int64)
    k_o = np.zeros(1, dtype=np.int64)
    rc = L.gdn_tail_replay_overlap(ctypes.byref(pr), None, vp(0x1000), vp(0x2000), vp(0x3000), vp(0x4000),
                                   m.ctypes.data_as(P64), 1, 10, None, vp(0x5000), None, None, a_o.ctypes.data_as(P64),
                                   k_o.ctypes.data_as(P64), None, vp(0x9000), 4096, vp(0x8000), 256, None, None)
    assert rc == gdn.GDN_ERR_INVALID_ARG
    rc = L.gdn_tail_replay_overlap(ctypes.byref(pr), None, vp(0x1000), vp(0x2000), vp(0x3000), vp(0x4000),
                                   m.ctypes.data_as(P64), 1, 10, None, vp(0x5004), None, None, a_o.ctypes.data_as(P64),
                                   k_o.ctypes.data_as(P64), vp(0x7000), vp(0x9000), 4096, vp(0x8000), 256, None, None)
    assert rc == gdn.GDN_ERR_INVALID_ARG       # S_hat misaligned: rejected before the copy is enqueued
