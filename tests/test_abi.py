"""The C ABI on the host (no GPU): exports, exact index helpers against the
oracle, and argument validation that rejects bad calls before any CUDA work."""
import ctypes
import os
import re

import numpy as np
import pytest

import hybrid_model_recurrent_gb300 as gdn
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    gdn.build()
    return gdn.lib()


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if fn.endswith(".h"):
            text = open(os.path.join(inc, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"\b(gdn_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert "gdn_prefill_ckpt" in names and "gdn_tail_replay" in names and "gdn_resume_from_ckpt" in names
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"


def test_replay_plan_matches_oracle_exhaustively(L):
    for rn, rd in ((0, 1), (1, 20), (1, 10), (1, 1), (7, 100), (3, 7), (13, 64)):
        for m in range(0, 200001):
            assert gdn.gdn_replay_plan(m, rn, rd) == oracle.replay_plan(m, rn, rd), (m, rn, rd)
    for m in (2 ** 31, 2 ** 40):
        assert gdn.gdn_replay_plan(m, 1, 20) == oracle.replay_plan(m, 1, 20)
    for bad in ((-1, 1, 20), (5, 2, 1), (5, -1, 3), (5, 1, 0), (2 ** 41, 1, 2)):
        with pytest.raises(gdn.GdnError):
            gdn.gdn_replay_plan(*bad)


def test_select_ckpt_matches_oracle(L):
    rng = np.random.default_rng(0)
    for trial in range(400):
        N = int(rng.integers(1, 5000))
        M = int(rng.integers(0, min(N, 64) + 1))
        cs = sorted(rng.choice(np.arange(1, N + 1), size=M, replace=False).tolist())
        for d in [0, 1, N] + cs + [c - 1 for c in cs] + rng.integers(0, N + 1, 20).tolist():
            assert gdn.gdn_select_ckpt(cs, int(d)) == oracle.select_ckpt(cs, int(d))
    with pytest.raises(gdn.GdnError):
        gdn.gdn_select_ckpt([5, 5], 7)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_select_ckpt([9, 3], 7)


# ---- argument validation: every bad call returns its status before touching CUDA -------

FAKE = 0x7f0000000000  # never dereferenced: validation must fail first


def _vp(off=0):
    return ctypes.c_void_p(FAKE + off)


def _prob(B=2, H=2, dk=32, dv=32, cu=(0, 10, 30), qkv=gdn.GDN_BF16, out=gdn.GDN_BF16, algo=0):
    arr = np.ascontiguousarray(np.asarray(cu, dtype=np.int64))
    pr = gdn._Problem()
    pr.num_seqs, pr.num_heads, pr.d_k, pr.d_v = B, H, dk, dv
    pr.cu_seqlens = arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    pr.qkv_dtype, pr.out_dtype = qkv, out
    pr.algo = algo
    return pr, arr


def _p64(a):
    return None if a is None else np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def prefill(L, pr, *, q=_vp(0), k=_vp(0x1000), v=_vp(0x2000), al=_vp(0x3000), be=_vp(0x4000), S0=None,
            o=_vp(0x5000), Sf=_vp(0x6000), pos=None, cu=None, ck=_vp(0x7000), ws=_vp(0x8000), wsb=256):
    pa, ca = _p64(pos), _p64(cu)
    P = ctypes.POINTER(ctypes.c_int64)
    return L.gdn_prefill_ckpt(ctypes.byref(pr), q, k, v, al, be, S0, o, Sf,
                              None if pa is None else pa.ctypes.data_as(P),
                              None if ca is None else ca.ctypes.data_as(P), ck, ws, wsb, None)


def test_prefill_rejects_bad_arguments(L):
    pr, _keep = _prob()
    E, U = gdn.GDN_ERR_INVALID_ARG, gdn.GDN_ERR_UNSUPPORTED
    assert prefill(L, _prob(B=0, cu=(0,))[0]) == E
    assert prefill(L, _prob(H=0)[0]) == E
    assert prefill(L, _prob(dk=96)[0]) == U
    assert prefill(L, _prob(dv=48)[0]) == U
    assert prefill(L, _prob(cu=(0, 10, 5))[0]) == E           # decreasing cu_seqlens
    assert prefill(L, _prob(cu=(1, 10, 30))[0]) == E           # cu_seqlens[0] != 0
    assert prefill(L, _prob(qkv=7)[0]) == E
    assert prefill(L, _prob(algo=5)[0]) == E                    # unknown algorithm
    assert prefill(L, _prob(algo=-1)[0]) == E
    for a in (gdn.ALGO["chunked"], gdn.ALGO["chunked_mma"], gdn.ALGO["two_pass"]):
        assert prefill(L, _prob(algo=a)[0]) == U                # chunked needs d_k = d_v = 128 and bf16
        assert prefill(L, _prob(dk=128, dv=128, qkv=gdn.GDN_F32, algo=a)[0]) == U
    # the two-pass path needs its larger workspace (30 tokens x 2 heads, 2 sequences here)
    pr2, _k2 = _prob(dk=128, dv=128, algo=gdn.ALGO["two_pass"])
    need = L.gdn_workspace_size_two_pass(30, 2, 2)
    assert prefill(L, pr2) == E and prefill(L, pr2, wsb=need - 1) == E
    assert prefill(L, pr, k=None) == E
    assert prefill(L, pr, q=None) == E                          # readout requested without q
    assert prefill(L, pr, k=_vp(0x1008)) == E                   # k not 16-byte aligned
    assert prefill(L, pr, Sf=None) == E
    assert prefill(L, pr, Sf=_vp(0x6004)) == E
    assert prefill(L, pr, ws=None) == E
    assert prefill(L, pr, wsb=8) == E
    assert prefill(L, pr, pos=[5, 11, 3], cu=[0, 2, 3]) == E     # 11 > N_0 = 10
    assert prefill(L, pr, pos=[5, 5, 3], cu=[0, 2, 3]) == E      # not strictly increasing
    assert prefill(L, pr, pos=[0, 5, 3], cu=[0, 2, 3]) == E      # position 0
    assert prefill(L, pr, pos=[5, 10, 3], cu=[0, 2, 1]) == E     # decreasing cu_ckpt
    assert prefill(L, pr, pos=[5, 10, 3], cu=[0, 2, 3], ck=None) == E


def test_prefill_valid_call_without_gpu_reports_cuda_error(L):
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present; the compute path is covered by the gpu tests")
    except ImportError:
        pass
    pr, _keep = _prob()
    # arguments are valid: the library gets as far as CUDA, which is absent here
    assert prefill(L, pr, pos=[5, 10, 7], cu=[0, 2, 3]) == gdn.GDN_ERR_CUDA
    big = L.gdn_workspace_size_two_pass(30, 2, 2)
    for a in gdn.ALGO.values():
        pr2, _k2 = _prob(dk=128, dv=128, algo=a)
        assert prefill(L, pr2, pos=[5, 10, 7], cu=[0, 2, 3], wsb=big) == gdn.GDN_ERR_CUDA


def test_two_pass_workspace_size(L):
    base = L.gdn_workspace_size()
    f = L.gdn_workspace_size_two_pass
    assert f(0, 1, 0) == base
    # status word, chunk counts (4 B per range and head), chunk starts (4 B per token and head), T operand
    # rows (4 planes x 64 bf16 per token and head), each part 256-byte aligned
    up = lambda x: (x + 255) // 256 * 256
    for T, H, R in ((30, 2, 2), (8192 * 8, 16, 8), (1, 1, 1), (1000, 3, 7)):
        cnt = base
        beg = up(cnt + 4 * R * H)
        t = up(beg + 4 * T * H)
        assert f(T, H, R) == t + 512 * T * H
    assert f(-1, 1, 1) == 0 and f(1, 0, 1) == 0 and f(1, 1, -1) == 0
    assert f(1 << 29, 1, 1) == 0 and f(1 << 25, 16, 1) == 0     # 2^29 - 64 token-heads or more
    assert f((1 << 29) - 65, 1, 1) > 0


def test_resume_and_replay_reject_bad_arguments(L):
    pr, _keep = _prob()
    P64, P32 = ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)
    E = gdn.GDN_ERR_INVALID_ARG

    def resume(seqs, deps, S_out=_vp(0x9000), pos=(4, 8, 20), cu=(0, 2, 3)):
        s = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
        d = _p64(deps)
        pa, ca = _p64(pos), _p64(cu)
        return L.gdn_resume_from_ckpt(ctypes.byref(pr), _vp(0), _vp(0x1000), _vp(0x2000), _vp(0x3000),
                                      _vp(0x4000), None, _vp(0x7000), pa.ctypes.data_as(P64),
                                      ca.ctypes.data_as(P64), len(seqs), s.ctypes.data_as(P32),
                                      d.ctypes.data_as(P64), S_out, None, None, None, _vp(0x8000), 256, None)

    assert resume([0, 2], [3, 5]) == E        # seq 2 out of range
    assert resume([0, 1], [11, 5]) == E       # depth 11 > N_0 = 10
    assert resume([0, 1], [-1, 5]) == E
    assert resume([0, 1], [3, 5], S_out=None) == E
    assert resume([0, 1], [3, 5], pos=(4, 12, 20)) == E   # checkpoint beyond N_0

    def replay(m, rn=1, rd=20, S_a=None, S_exact=None, S_hat=_vp(0xa000)):
        mm = _p64(m)
        return L.gdn_tail_replay(ctypes.byref(pr), None, _vp(0x1000), _vp(0x2000), _vp(0x3000), _vp(0x4000),
                                 mm.ctypes.data_as(P64), rn, rd, S_a, S_hat, S_exact, None, None, None,
                                 _vp(0x8000), 256, None)

    assert replay([11, 5]) == E               # m > N
    assert replay([-1, 5]) == E
    assert replay([10, 5], rn=21) == E        # r > 1
    assert replay([10, 5], rd=0) == E
    assert replay([10, 5], S_a=_vp(0xb000)) == E               # S_a without S_exact
    assert replay([10, 5], S_hat=None) == E


def test_step_rejects_bad_arguments_and_writes_no_host_output(L):
    pr, _keep = _prob()
    P64, P32 = ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)
    E = gdn.GDN_ERR_INVALID_ARG
    pos, cu = _p64([4, 8, 20]), _p64([0, 2, 3])
    seqs = np.ascontiguousarray(np.asarray([0, 1], dtype=np.int32))
    deps = _p64([9, 15])
    mm = _p64([10, 20])

    def call(pf=True, rs=True, rp=True, q=_vp(0), resume_ck=_vp(0x20000), prefill_ck=_vp(0x7000), rs_readout=True,
             m=None):
        chosen = np.full(2, -7, dtype=np.int64)
        a_out = np.full(2, -7, dtype=np.int64)
        pa = gdn._PrefillArgs(None, _vp(0x5000), _vp(0x6000), pos.ctypes.data_as(P64), cu.ctypes.data_as(P64),
                              prefill_ck)
        ra = gdn._ResumeArgs(None, resume_ck, pos.ctypes.data_as(P64), cu.ctypes.data_as(P64), 2,
                             seqs.ctypes.data_as(P32), deps.ctypes.data_as(P64), _vp(0x9000),
                             _vp(0x30000) if rs_readout else None, chosen.ctypes.data_as(P64), None)
        m_arr = mm if m is None else _p64(m)
        ya = gdn._ReplayArgs(m_arr.ctypes.data_as(P64), 1, 20, None, _vp(0xa000), None, None,
                             a_out.ctypes.data_as(P64), None)
        rc = L.gdn_step(ctypes.byref(pr), q, _vp(0x1000), _vp(0x2000), _vp(0x3000), _vp(0x4000),
                        ctypes.byref(pa) if pf else None, ctypes.byref(ra) if rs else None,
                        ctypes.byref(ya) if rp else None, _vp(0x8000), 256, None)
        return rc, chosen, a_out

    # the resumes may not read checkpoints that the same call's prefill writes (3 slots x 2 heads x 32 x 32 fp32)
    for ck in (_vp(0x7000), _vp(0x7000 + 3 * 2 * 32 * 32 * 4 - 16), _vp(0x7000 - 3 * 2 * 32 * 32 * 4 + 16)):
        rc, chosen, a_out = call(resume_ck=ck)
        assert rc == E and (chosen == -7).all() and (a_out == -7).all()
    assert call(resume_ck=_vp(0x7000 + 3 * 2 * 32 * 32 * 4), q=None)[0] == E   # readouts without q
    assert call(rs=False, rp=False, q=None)[0] == E                               # the prefill's readout needs q
    rc, chosen, a_out = call(m=[11, 5])                                            # m > N: every part checked first
    assert rc == E and (chosen == -7).all() and (a_out == -7).all()
    import torch
    if not torch.cuda.is_available():
        # valid calls (fake pointers): the library gets as far as CUDA, which is absent here
        assert call(resume_ck=_vp(0x7000 + 3 * 2 * 32 * 32 * 4))[0] == gdn.GDN_ERR_CUDA
        assert call(pf=False, rp=False, rs_readout=False, q=None, resume_ck=_vp(0x7000))[0] == gdn.GDN_ERR_CUDA
