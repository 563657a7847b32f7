"""The allocation-free prefill entry point, called through the C ABI.

gdn_prefill_ckpt_noalloc serves callers that cannot allocate device memory:
they are handed their buffers but have no device allocator of their own, so
they cannot provide the small workspace the regular entry points take.  The
variant keeps that scratch in a static device array inside the library.  This
test checks, on two calls in a row (the array keeps the previous call's
contents), that it returns the same states, checkpoints and readout as the
regular entry point bit for bit: the regular call is given the same 256-byte
workspace, so both run the same kernel.  One (sequence, head) stream is also
checked against the fp64 oracle directly.

It lives in its own file that pytest collects last, and must pass both alone
in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import hybrid_model_recurrent_gb300 as gdn
import oracle
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


@pytest.mark.parametrize("dk,dtype,algo", [(128, torch.bfloat16, "chunked"), (64, torch.float32, "per_token")])
def test_noalloc_prefill_matches_regular_entry_point(dk, dtype, algo):
    gdn.build()
    f = _entry()
    lens = [200, 0, 77, 160]
    H, dv = 3, dk
    w = synth.Workload("noalloc", lens, H, dk, dv, dtype, dtype, 0.9, 1.0, "uniform", seed=77)
    inp = synth.make_inputs(w, device=DEV)
    ck = [[1, 64, 200], [], [77], [33, 96]]
    S0 = synth.state(78, w.B * H, dv, dk, 0.5, device=DEV).view(w.B, H, dv, dk)
    # the regular entry point with the smallest workspace takes the kernel the allocation-free call takes
    ws = torch.zeros(int(gdn.lib().gdn_workspace_size()), dtype=torch.uint8, device=DEV)
    ref = gdn.gdn_prefill_ckpt(inp.q, inp.k, inp.v, inp.alpha, inp.beta, w.cu_seqlens, S0=S0, ckpt_pos=ck,
                               out_dtype=torch.float32, ws=ws, algo=algo)
    torch.cuda.synchronize()
    # sequence 0, head 1 against the oracle
    cpu = [t.cpu() for t in (inp.q, inp.k, inp.v, inp.alpha, inp.beta)]
    sl = slice(w.cu_seqlens[0], w.cu_seqlens[1])
    orc = oracle.prefill(*(t[sl, 1] for t in cpu), S0=S0[0, 1].cpu(), ckpt_pos=ck[0])
    assert_close(ref["S_final"][0, 1], orc["S"], "regular S_N against the oracle")

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
        assert torch.equal(S_final, ref["S_final"]), f"call {call}: final states differ"
        assert torch.equal(o, ref["o"]), f"call {call}: readout differs"
        assert torch.equal(ckpt, ref["ckpt_states"]), f"call {call}: checkpoints differ"
        assert_close(S_final[0, 1], orc["S"], f"call {call} S_N against the oracle")
        assert_close(o[sl, 1], orc["o"], f"call {call} o against the oracle")
        for i in range(len(ck[0])):
            assert_close(ckpt[i, 1], orc["ckpt"][i], f"call {call} checkpoint {i} against the oracle")

    # invalid arguments are still rejected (sequence 0 has 200 tokens; 201 is out of range)
    bad = np.ascontiguousarray(np.asarray([1, 64, 201, 77, 33, 96], dtype=np.int64))
    rc = f(ctypes.byref(pr), ptr(inp.q), ptr(inp.k), ptr(inp.v), ptr(inp.alpha), ptr(inp.beta), ptr(S0), ptr(o),
           ptr(S_final), bad.ctypes.data_as(P), cu_ck.ctypes.data_as(P), ptr(ckpt), stream)
    assert rc == gdn.GDN_ERR_INVALID_ARG
