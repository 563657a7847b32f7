"""The allocation-free prefill entry point, called through the C ABI.

gdn_prefill_ckpt_noalloc serves callers that cannot allocate device memory:
they are handed their buffers but have no device allocator of their own, so
they cannot provide the small workspace the regular entry points take.  The
variant keeps that scratch in a static device array inside the library.  This
test checks, on two calls in a row (the array keeps the previous call's
contents), that it returns the same states, checkpoints and readout as the
regular entry point, within the parity tolerance of the other GPU tests.

It lives in its own file that pytest collects last, and must pass both alone
in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import hybrid_model_recurrent_gb300 as gdn
import synth
from parity_util import assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _entry():
    L = gdn.lib()
    f = L.gdn_prefill_ckpt_noalloc
    vp = ctypes.c_void_p
    pi64 = ctypes.POINTER(ctypes.c_int64)
    f.argtypes = [ctypes.POINTER(gdn._Problem), vp, vp, vp, vp, vp, vp, vp, vp, pi64, pi64, vp, vp]
    f.restype = ctypes.c_int
    return f


@pytest.mark.parametrize("dk,dtype", [(128, torch.bfloat16), (64, torch.float32)])
def test_noalloc_prefill_matches_regular_entry_point(dk, dtype):
    gdn.build()
    f = _entry()
    lens = [200, 0, 77, 160]
    H, dv = 3, dk
    w = synth.Workload("noalloc", lens, H, dk, dv, dtype, dtype, 0.9, 1.0, "uniform", seed=77)
    inp = synth.make_inputs(w, device=DEV)
    ck = [[1, 64, 200], [], [77], [33, 96]]
    S0 = synth.state(78, w.B * H, dv, dk, 0.5, device=DEV).view(w.B, H, dv, dk)
    ref = gdn.gdn_prefill_ckpt(inp.q, inp.k, inp.v, inp.alpha, inp.beta, w.cu_seqlens, S0=S0, ckpt_pos=ck,
                               out_dtype=torch.float32)

    cu = np.ascontiguousarray(np.asarray(w.cu_seqlens, dtype=np.int64))
    flat = np.ascontiguousarray(np.asarray([c for lst in ck for c in lst], dtype=np.int64))
    cu_ck = np.ascontiguousarray(np.asarray([0, 3, 3, 4, 6], dtype=np.int64))
    pr = gdn._Problem()
    pr.num_seqs, pr.num_heads, pr.d_k, pr.d_v = w.B, H, dk, dv
    pr.cu_seqlens = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    pr.qkv_dtype = gdn.GDN_BF16 if dtype == torch.bfloat16 else gdn.GDN_F32
    pr.out_dtype = gdn.GDN_F32
    P = ctypes.POINTER(ctypes.c_int64)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        o = torch.full((w.T, H, dv), float("nan"), dtype=torch.float32, device=DEV)
        S_final = torch.full((w.B, H, dv, dk), float("nan"), dtype=torch.float32, device=DEV)
        ckpt = torch.full((6, H, dv, dk), float("nan"), dtype=torch.float32, device=DEV)
        ptr = lambda t: ctypes.c_void_p(t.data_ptr())
        rc = f(ctypes.byref(pr), ptr(inp.q), ptr(inp.k), ptr(inp.v), ptr(inp.alpha), ptr(inp.beta), ptr(S0), ptr(o),
               ptr(S_final), flat.ctypes.data_as(P), cu_ck.ctypes.data_as(P), ptr(ckpt), stream)
        assert rc == gdn.GDN_OK, f"call {call}: {gdn.status_string(rc)}"
        torch.cuda.synchronize()
        for b in range(w.B):
            for h in range(H):
                assert_close(S_final[b, h], ref["S_final"][b, h], f"call {call} S_N b={b} h={h}")
                if lens[b]:
                    assert_close(o[w.cu_seqlens[b]:w.cu_seqlens[b + 1], h],
                                 ref["o"][w.cu_seqlens[b]:w.cu_seqlens[b + 1], h], f"call {call} o b={b} h={h}")
        for s in range(6):
            for h in range(H):
                assert_close(ckpt[s, h], ref["ckpt_states"][s, h], f"call {call} ckpt slot {s} h={h}")

    # invalid arguments are still rejected (sequence 0 has 200 tokens; 201 is out of range)
    bad = np.ascontiguousarray(np.asarray([1, 64, 201, 77, 33, 96], dtype=np.int64))
    rc = f(ctypes.byref(pr), ptr(inp.q), ptr(inp.k), ptr(inp.v), ptr(inp.alpha), ptr(inp.beta), ptr(S0), ptr(o),
           ptr(S_final), bad.ctypes.data_as(P), cu_ck.ctypes.data_as(P), ptr(ckpt), stream)
    assert rc == gdn.GDN_ERR_INVALID_ARG
