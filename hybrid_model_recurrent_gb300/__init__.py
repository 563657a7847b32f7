"""Python binding of the GB300 Gated DeltaNet state-scan library (libgdn_scan.so).

Argument marshalling only: every step of the scan runs in the library's CUDA
kernels.  Torch tensors are used for device memory and streams; outputs that
the caller does not pass are allocated here.  The names follow the C ABI in
``include/gdn_scan.h``:

* ``gdn_prefill_ckpt``      prefill with exact state dumps at sparse positions
* ``gdn_resume_from_ckpt``  resume at overlap depth d from the deepest stored state
* ``gdn_tail_replay``       Tail-Replay from a zero state at a = m - ceil(r m)
* ``gdn_step``              the three above for one serving step, in one launch
* host helpers ``gdn_replay_plan``, ``gdn_select_ckpt``, status utilities.

There is no fallback: if the compiled library is missing the import of a
compute entry point raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn_scan.so")

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA, GDN_ERR_DEVICE_TIMEOUT = range(5)
GDN_F32, GDN_BF16 = 0, 1
ALGO = {"auto": 0, "per_token": 1, "chunked": 2, "chunked_mma": 3, "two_pass": 4}
PLACE = {"dp": 0, "balanced": 1, "block": 2, "random": 3, "greedy": 4}

_lock = threading.Lock()
_lib = None
_workspaces: Dict[int, torch.Tensor] = {}


class _Group(ctypes.Structure):
    _fields_ = [("layers", ctypes.c_int32), ("heads", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("d_head", ctypes.c_int32)]


_vp, _pi64 = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64)


class _PrefillArgs(ctypes.Structure):
    _fields_ = [("S0", _vp), ("o", _vp), ("S_final", _vp), ("ckpt_pos", _pi64), ("cu_ckpt", _pi64),
                ("ckpt_states", _vp)]


class _ResumeArgs(ctypes.Structure):
    _fields_ = [("S0", _vp), ("ckpt_states", _vp), ("ckpt_pos", _pi64), ("cu_ckpt", _pi64),
                ("num_probes", ctypes.c_int32), ("probe_seq", ctypes.POINTER(ctypes.c_int32)),
                ("probe_depth", _pi64), ("S_out", _vp), ("o_out", _vp), ("chosen_pos", _pi64),
                ("o_offsets", _pi64)]


class _ReplayArgs(ctypes.Structure):
    _fields_ = [("m", _pi64), ("r_num", ctypes.c_int32), ("r_den", ctypes.c_int32), ("S_a", _vp), ("S_hat", _vp),
                ("S_exact", _vp), ("o", _vp), ("a_out", _pi64), ("k_out", _pi64)]


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} ({status})")
        self.status = status


class _Problem(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_heads", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("cu_seqlens", ctypes.POINTER(ctypes.c_int64)),
                ("qkv_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int), ("algo", ctypes.c_int)]


def build(force: bool = False) -> str:
    from . import _build
    return _build.build(force=force)


def lib():
    """The loaded C library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: build it with hybrid_model_recurrent_gb300.build()")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
            P = ctypes.POINTER(_Problem)
            pi64 = ctypes.POINTER(ctypes.c_int64)
            pi32 = ctypes.POINTER(ctypes.c_int32)
            L.gdn_prefill_ckpt.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, pi64, pi64, vp, vp, sz, vp]
            L.gdn_resume_from_ckpt.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, pi64, pi64, i32, pi32, pi64, vp, vp,
                                               pi64, pi64, vp, sz, vp]
            L.gdn_tail_replay.argtypes = [P, vp, vp, vp, vp, vp, pi64, i32, i32, vp, vp, vp, vp, pi64, pi64, vp, sz,
                                          vp]
            L.gdn_step.argtypes = [P, vp, vp, vp, vp, vp, ctypes.POINTER(_PrefillArgs), ctypes.POINTER(_ResumeArgs),
                                   ctypes.POINTER(_ReplayArgs), vp, sz, vp]
            L.gdn_replay_plan.argtypes = [i64, i32, i32, pi64, pi64]
            L.gdn_select_ckpt.argtypes = [pi64, i32, i64, pi32]
            L.gdn_tail_replay_k.argtypes = [P, vp, vp, vp, vp, vp, pi64, pi64, vp, vp, vp, vp, vp, sz, vp]
            L.gdn_tail_replay_overlap.argtypes = [P, vp, vp, vp, vp, vp, pi64, i32, i32, vp, vp, vp, vp, pi64, pi64,
                                                  vp, vp, sz, vp, sz, vp, vp]
            L.gdn_adaptive_replay_plan.argtypes = [P, vp, pi64, ctypes.c_float, i32, i32, pi64, pi32, vp]
            G = ctypes.POINTER(_Group)
            L.gdn_group_scratch_bytes.argtypes = [G, i64]
            L.gdn_group_scratch_bytes.restype = sz
            L.gdn_group_replay.argtypes = [G, vp, i64, i32, i32, vp, vp, vp, pi64, pi64, vp, sz, vp, sz, vp]
            L.gdn_ckpt_placement.argtypes = [pi64, i64, i32, ctypes.c_int, ctypes.c_uint64, i64, pi64, pi32, pi64]
            L.gdn_expected_recompute.argtypes = [pi64, i64, pi64, i32, pi64]
            L.gdn_workspace_size.argtypes = []
            L.gdn_workspace_size.restype = sz
            L.gdn_workspace_size_two_pass.argtypes = [i64, i32, i32]
            L.gdn_workspace_size_two_pass.restype = sz
            L.gdn_clear_status.argtypes = [vp, sz, vp]
            L.gdn_read_status.argtypes = [vp, sz, vp]
            L.gdn_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            L.gdn_set_wait_limit_ns.restype = None
            L.gdn_debug_stall_after.argtypes = [ctypes.c_int32]
            L.gdn_debug_stall_after.restype = None
            L.gdn_status_string.argtypes = [ctypes.c_int]
            L.gdn_status_string.restype = ctypes.c_char_p
            for f in ("gdn_prefill_ckpt", "gdn_resume_from_ckpt", "gdn_tail_replay", "gdn_step", "gdn_replay_plan",
                      "gdn_select_ckpt", "gdn_clear_status", "gdn_read_status"):
                getattr(L, f).restype = ctypes.c_int
            _lib = L
    return _lib


def status_string(s: int) -> str:
    return lib().gdn_status_string(int(s)).decode()


def _check(rc: int, where: str) -> None:
    if rc != GDN_OK:
        raise GdnError(rc, where)


def _i64(values) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(list(values), dtype=np.int64))


def _p64(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream, device) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return GDN_F32
    if dt == torch.bfloat16:
        return GDN_BF16
    raise ValueError(f"unsupported dtype {dt}")


def workspace(device, nbytes: int = 0) -> torch.Tensor:
    """The cached per-device workspace (holds the sticky device status word), grown to at least
    `nbytes`; growing keeps the status word."""
    device = torch.device(device)
    idx = device.index if device.index is not None else torch.cuda.current_device()
    ws = _workspaces.get(idx)
    need = max(int(lib().gdn_workspace_size()), int(nbytes))
    if ws is None or ws.numel() < need:
        new = torch.zeros(need, dtype=torch.uint8, device=torch.device("cuda", idx))
        if ws is not None:
            new[:int(lib().gdn_workspace_size())].copy_(ws[:int(lib().gdn_workspace_size())])
        ws = new
        _workspaces[idx] = ws
    return ws


def _auto_ws(dev, algo: str, k, v, tokens: int, ranges: int) -> torch.Tensor:
    """The cached workspace, large enough for the two-pass chunked path when the call may take it."""
    H, dk, dv = k.shape[1], k.shape[2], v.shape[-1]
    nbytes = 0
    if algo in ("auto", "two_pass") and dk == 128 and dv == 128 and k.dtype == torch.bfloat16 and tokens > 0:
        nbytes = int(lib().gdn_workspace_size_two_pass(int(tokens), int(H), int(ranges)))
    return workspace(dev, nbytes)


def read_status(device=None, stream=None, ws: Optional[torch.Tensor] = None) -> int:
    device = torch.device(device or "cuda")
    ws = ws if ws is not None else workspace(device)
    return lib().gdn_read_status(_ptr(ws), ws.numel(), _stream(stream, ws.device))


def clear_status(device=None, stream=None, ws: Optional[torch.Tensor] = None) -> None:
    device = torch.device(device or "cuda")
    ws = ws if ws is not None else workspace(device)
    _check(lib().gdn_clear_status(_ptr(ws), ws.numel(), _stream(stream, ws.device)), "gdn_clear_status")


def set_wait_limit_ns(ns: int) -> None:
    lib().gdn_set_wait_limit_ns(int(ns))


def debug_stall_after(chunks: int) -> None:
    """Testing hook: later launches stop issuing input copies after `chunks` chunks (-1: off)."""
    lib().gdn_debug_stall_after(int(chunks))


def gdn_replay_plan(m: int, r_num: int, r_den: int):
    """(a, k) with k = ceil(r_num * m / r_den) computed exactly, a = m - k."""
    a, k = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().gdn_replay_plan(m, r_num, r_den, ctypes.byref(a), ctypes.byref(k)), "gdn_replay_plan")
    return a.value, k.value


def gdn_select_ckpt(c: Sequence[int], d: int) -> int:
    """0-based index of the deepest c_i <= d, or -1."""
    arr = _i64(c)
    j = ctypes.c_int32()
    _check(lib().gdn_select_ckpt(_p64(arr) if len(arr) else None, len(arr), d, ctypes.byref(j)),
           "gdn_select_ckpt")
    return j.value


def gdn_ckpt_placement(weights: Sequence[int], M: int, strategy: str = "dp", seed: int = 0, block: int = 0):
    """Checkpoint positions for a prefix of N = len(weights) - 1 tokens and depth weights w[0..N].

    Returns (positions, R) with positions strictly increasing in [1, N] and R = sum_d w[d] f(d)
    the exact expected-recompute numerator of that placement."""
    w = _i64(weights)
    N = len(w) - 1
    out = np.zeros(max(int(M), 1), dtype=np.int64)
    n = ctypes.c_int32()
    cost = ctypes.c_int64()
    _check(lib().gdn_ckpt_placement(_p64(w), N, int(M), PLACE[strategy], ctypes.c_uint64(int(seed)), int(block),
                                    _p64(out), ctypes.byref(n), ctypes.byref(cost)), "gdn_ckpt_placement")
    return [int(x) for x in out[:n.value]], cost.value


def gdn_expected_recompute(weights: Sequence[int], positions: Sequence[int]) -> int:
    """R = sum_d w[d] f(d) of a placement (exact integer)."""
    w = _i64(weights)
    pos = _i64(positions)
    cost = ctypes.c_int64()
    _check(lib().gdn_expected_recompute(_p64(w), len(w) - 1, _p64(pos) if len(pos) else None, len(pos),
                                        ctypes.byref(cost)), "gdn_expected_recompute")
    return cost.value


def _problem(cu: np.ndarray, H: int, dk: int, dv: int, qkv_dtype: torch.dtype, out_dtype: torch.dtype,
             algo: str = "auto"):
    pr = _Problem()
    pr.algo = ALGO[algo]
    pr.num_seqs = len(cu) - 1
    pr.num_heads = H
    pr.d_k = dk
    pr.d_v = dv
    pr.cu_seqlens = _p64(cu)
    pr.qkv_dtype = _dtype_code(qkv_dtype)
    pr.out_dtype = _dtype_code(out_dtype)
    return pr


def _flatten_ckpts(ckpt_pos, B: int):
    """Per-sequence position lists -> (concatenated int64, cu_ckpt int64)."""
    if ckpt_pos is None:
        return None, None
    cu = [0]
    flat: List[int] = []
    for lst in ckpt_pos:
        flat.extend(int(x) for x in lst)
        cu.append(len(flat))
    if len(cu) != B + 1:
        raise ValueError("ckpt_pos must give one list per sequence")
    return _i64(flat), _i64(cu)


def gdn_prefill_ckpt(q, k, v, alpha, beta, cu_seqlens, *, S0=None, ckpt_pos=None, readout: bool = True,
                     out_dtype: Optional[torch.dtype] = None, o=None, S_final=None, ckpt_states=None,
                     stream=None, ws: Optional[torch.Tensor] = None, algo: str = "auto"):
    """Prefill with sparse checkpoints.  ckpt_pos: one list of 1-based positions per sequence.

    Returns dict(o=[T,H,dv] or None, S_final=[B,H,dv,dk], ckpt_states=[M_total,H,dv,dk])."""
    cu = _i64(cu_seqlens)
    B = len(cu) - 1
    T, H, dk = k.shape
    dv = v.shape[-1]
    dev = k.device
    out_dtype = out_dtype or k.dtype
    if readout and o is None:
        o = torch.empty((T, H, dv), dtype=out_dtype, device=dev)
    if not readout:
        o = None
    if S_final is None:
        S_final = torch.empty((B, H, dv, dk), dtype=torch.float32, device=dev)
    flat, cu_ck = _flatten_ckpts(ckpt_pos, B)
    n_ck = 0 if cu_ck is None else int(cu_ck[-1])
    if ckpt_states is None and n_ck > 0:
        ckpt_states = torch.empty((n_ck, H, dv, dk), dtype=torch.float32, device=dev)
    ws = ws if ws is not None else _auto_ws(dev, algo, k, v, T, B)
    pr = _problem(cu, H, dk, dv, k.dtype, out_dtype, algo)
    rc = lib().gdn_prefill_ckpt(ctypes.byref(pr), _ptr(q if readout else None), _ptr(k), _ptr(v), _ptr(alpha),
                                _ptr(beta), _ptr(S0), _ptr(o), _ptr(S_final),
                                _p64(flat) if n_ck > 0 else None, _p64(cu_ck), _ptr(ckpt_states),
                                _ptr(ws), ws.numel(), _stream(stream, dev))
    _check(rc, "gdn_prefill_ckpt")
    return {"o": o, "S_final": S_final, "ckpt_states": ckpt_states}


def gdn_resume_from_ckpt(q, k, v, alpha, beta, cu_seqlens, ckpt_states, ckpt_pos, probes, *, S0=None,
                         readout: bool = True, out_dtype: Optional[torch.dtype] = None, S_out=None, o_out=None,
                         stream=None, ws: Optional[torch.Tensor] = None, algo: str = "auto"):
    """Resume at the probes' depths.  probes: list of (seq, depth).

    Returns dict(S_out=[P,H,dv,dk], o=[R,H,dv] or None, chosen=[P] positions c_j, offsets=[P+1])."""
    cu = _i64(cu_seqlens)
    B = len(cu) - 1
    T, H, dk = k.shape
    dv = v.shape[-1]
    dev = k.device
    out_dtype = out_dtype or k.dtype
    flat, cu_ck = _flatten_ckpts(ckpt_pos, B)
    n_ck = 0 if cu_ck is None else int(cu_ck[-1])
    P = len(probes)
    seqs = np.ascontiguousarray(np.asarray([int(s) for s, _ in probes], dtype=np.int32))
    deps = _i64(int(d) for _, d in probes)
    chosen = np.zeros(P, dtype=np.int64)
    offs = np.zeros(P + 1, dtype=np.int64)
    # first pass: host plan (no launch) to size the packed readout
    if readout and o_out is None:
        rows = 0
        for s, d in probes:
            lst = list(ckpt_pos[s]) if ckpt_pos is not None else []
            j = gdn_select_ckpt(lst, int(d))
            rows += int(d) - (0 if j < 0 else lst[j])
        o_out = torch.empty((max(rows, 0), H, dv), dtype=out_dtype, device=dev)
    if not readout:
        o_out = None
    if S_out is None:
        S_out = torch.empty((P, H, dv, dk), dtype=torch.float32, device=dev)
    ws = ws if ws is not None else _auto_ws(dev, algo, k, v, int(deps.sum()) if P else 0, P)
    pr = _problem(cu, H, dk, dv, k.dtype, out_dtype, algo)
    rc = lib().gdn_resume_from_ckpt(
        ctypes.byref(pr), _ptr(q if readout else None), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0),
        _ptr(ckpt_states), _p64(flat) if n_ck > 0 else None, _p64(cu_ck), P,
        seqs.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if P else None, _p64(deps) if P else None,
        _ptr(S_out), _ptr(o_out), _p64(chosen) if P else None, _p64(offs), _ptr(ws), ws.numel(),
        _stream(stream, dev))
    _check(rc, "gdn_resume_from_ckpt")
    return {"S_out": S_out, "o": o_out, "chosen": chosen.tolist(), "offsets": offs.tolist()}


def gdn_tail_replay(q, k, v, alpha, beta, cu_seqlens, m, r_num: int, r_den: int, *, S_a=None, readout: bool = False,
                    out_dtype: Optional[torch.dtype] = None, S_hat=None, S_exact=None, o=None, stream=None,
                    ws: Optional[torch.Tensor] = None, algo: str = "auto"):
    """Tail-Replay at matched lengths m (one per sequence).

    Returns dict(S_hat, S_exact or None, o or None, a=[B], k=[B])."""
    cu = _i64(cu_seqlens)
    B = len(cu) - 1
    T, H, dk = k.shape
    dv = v.shape[-1]
    dev = k.device
    out_dtype = out_dtype or k.dtype
    mm = _i64(m)
    if S_hat is None:
        S_hat = torch.empty((B, H, dv, dk), dtype=torch.float32, device=dev)
    if S_a is not None and S_exact is None:
        S_exact = torch.empty((B, H, dv, dk), dtype=torch.float32, device=dev)
    if readout and o is None:
        o = torch.zeros((T, H, dv), dtype=out_dtype, device=dev)
    if not readout:
        o = None
    a_out = np.zeros(B, dtype=np.int64)
    k_out = np.zeros(B, dtype=np.int64)
    twin = 2 if S_a is not None else 1
    ws = ws if ws is not None else _auto_ws(dev, algo, k, v, int(mm.sum()) * twin, B * twin)
    pr = _problem(cu, H, dk, dv, k.dtype, out_dtype, algo)
    rc = lib().gdn_tail_replay(ctypes.byref(pr), _ptr(q if readout else None), _ptr(k), _ptr(v), _ptr(alpha),
                               _ptr(beta), _p64(mm), r_num, r_den, _ptr(S_a), _ptr(S_hat),
                               _ptr(S_exact if S_a is not None else None), _ptr(o), _p64(a_out), _p64(k_out),
                               _ptr(ws), ws.numel(), _stream(stream, dev))
    _check(rc, "gdn_tail_replay")
    return {"S_hat": S_hat, "S_exact": S_exact if S_a is not None else None, "o": o, "a": a_out.tolist(),
            "k": k_out.tolist()}


def gdn_step(q, k, v, alpha, beta, cu_seqlens, *, prefill: Optional[dict] = None, resume: Optional[dict] = None,
             replay: Optional[dict] = None, out_dtype: Optional[torch.dtype] = None, stream=None,
             ws: Optional[torch.Tensor] = None, algo: str = "auto"):
    """One serving step in one launch: any of a prefill, resumes and tail replays over the same streams.

    prefill: dict(ckpt_pos=None, S0=None, readout=True, o=None, S_final=None, ckpt_states=None)
    resume:  dict(ckpt_states, ckpt_pos, probes, S0=None, readout=True, S_out=None, o_out=None); the
             checkpoints must come from an earlier call (this call's prefill may not write them)
    replay:  dict(m, r_num, r_den, S_a=None, readout=False, S_hat=None, S_exact=None, o=None)
    Returns dict(prefill=..., resume=..., replay=...), each as its own entry point returns it."""
    cu = _i64(cu_seqlens)
    B = len(cu) - 1
    T, H, dk = k.shape
    dv = v.shape[-1]
    dev = k.device
    out_dtype = out_dtype or k.dtype
    keep = []   # host arrays that must outlive the call
    res = {}
    pa = ra = ya = None
    tokens, ranges = 0, 0
    readout = False
    if prefill is not None:
        f = dict(prefill)
        rd = f.get("readout", True)
        o = f.get("o") if rd else None
        if rd and o is None:
            o = torch.empty((T, H, dv), dtype=out_dtype, device=dev)
        S_final = f.get("S_final")
        if S_final is None:
            S_final = torch.empty((B, H, dv, dk), dtype=torch.float32, device=dev)
        flat, cu_ck = _flatten_ckpts(f.get("ckpt_pos"), B)
        n_ck = 0 if cu_ck is None else int(cu_ck[-1])
        ck = f.get("ckpt_states")
        if ck is None and n_ck > 0:
            ck = torch.empty((n_ck, H, dv, dk), dtype=torch.float32, device=dev)
        keep += [flat, cu_ck]
        pa = _PrefillArgs(_ptr(f.get("S0")), _ptr(o), _ptr(S_final), _p64(flat) if n_ck > 0 else None, _p64(cu_ck),
                          _ptr(ck))
        res["prefill"] = {"o": o, "S_final": S_final, "ckpt_states": ck}
        readout = readout or rd
        tokens, ranges = tokens + T, ranges + B
    if resume is not None:
        f = dict(resume)
        rd = f.get("readout", True)
        probes = f["probes"]
        ckpt_pos = f["ckpt_pos"]
        flat, cu_ck = _flatten_ckpts(ckpt_pos, B)
        n_ck = 0 if cu_ck is None else int(cu_ck[-1])
        P = len(probes)
        seqs = np.ascontiguousarray(np.asarray([int(s) for s, _ in probes], dtype=np.int32))
        deps = _i64(int(d) for _, d in probes)
        chosen = np.zeros(P, dtype=np.int64)
        offs = np.zeros(P + 1, dtype=np.int64)
        o_out = f.get("o_out") if rd else None
        if rd and o_out is None:
            rows = 0
            for s, d in probes:
                lst = list(ckpt_pos[s]) if ckpt_pos is not None else []
                j = gdn_select_ckpt(lst, int(d))
                rows += int(d) - (0 if j < 0 else lst[j])
            o_out = torch.empty((max(rows, 0), H, dv), dtype=out_dtype, device=dev)
        S_out = f.get("S_out")
        if S_out is None:
            S_out = torch.empty((P, H, dv, dk), dtype=torch.float32, device=dev)
        keep += [flat, cu_ck, seqs, deps, chosen, offs]
        ra = _ResumeArgs(_ptr(f.get("S0")), _ptr(f["ckpt_states"]), _p64(flat) if n_ck > 0 else None, _p64(cu_ck), P,
                         seqs.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if P else None,
                         _p64(deps) if P else None, _ptr(S_out), _ptr(o_out), _p64(chosen) if P else None,
                         _p64(offs))
        res["resume"] = {"S_out": S_out, "o": o_out, "chosen": chosen, "offsets": offs}
        readout = readout or rd
        tokens, ranges = tokens + (int(deps.sum()) if P else 0), ranges + P
    if replay is not None:
        f = dict(replay)
        rd = f.get("readout", False)
        mm = _i64(f["m"])
        S_a = f.get("S_a")
        _, _, _, _, _, _, S_hat, S_exact, o = _replay_buffers(k, v, B, S_a, rd, out_dtype, f.get("S_hat"),
                                                              f.get("S_exact"), f.get("o"))
        a_out = np.zeros(B, dtype=np.int64)
        k_out = np.zeros(B, dtype=np.int64)
        keep += [mm, a_out, k_out]
        ya = _ReplayArgs(_p64(mm), int(f["r_num"]), int(f["r_den"]), _ptr(S_a), _ptr(S_hat),
                         _ptr(S_exact if S_a is not None else None), _ptr(o), _p64(a_out), _p64(k_out))
        res["replay"] = {"S_hat": S_hat, "S_exact": S_exact if S_a is not None else None, "o": o, "a": a_out,
                         "k": k_out}
        readout = readout or rd
        twin = 2 if S_a is not None else 1
        tokens, ranges = tokens + int(mm.sum()) * twin, ranges + B * twin
    ws = ws if ws is not None else _auto_ws(dev, algo, k, v, tokens, ranges)
    pr = _problem(cu, H, dk, dv, k.dtype, out_dtype, algo)
    rc = lib().gdn_step(ctypes.byref(pr), _ptr(q if readout else None), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                        ctypes.byref(pa) if pa is not None else None, ctypes.byref(ra) if ra is not None else None,
                        ctypes.byref(ya) if ya is not None else None, _ptr(ws), ws.numel(), _stream(stream, dev))
    _check(rc, "gdn_step")
    if "resume" in res:
        r = res["resume"]
        r["chosen"], r["offsets"] = r["chosen"].tolist(), r["offsets"].tolist()
    if "replay" in res:
        r = res["replay"]
        r["a"], r["k"] = r["a"].tolist(), r["k"].tolist()
    return res


def _replay_buffers(k, v, B, S_a, readout, out_dtype, S_hat, S_exact, o):
    T, H, dk = k.shape
    dv = v.shape[-1]
    dev = k.device
    out_dtype = out_dtype or k.dtype
    if S_hat is None:
        S_hat = torch.empty((B, H, dv, dk), dtype=torch.float32, device=dev)
    if S_a is not None and S_exact is None:
        S_exact = torch.empty((B, H, dv, dk), dtype=torch.float32, device=dev)
    if readout and o is None:
        o = torch.zeros((T, H, dv), dtype=out_dtype, device=dev)
    if not readout:
        o = None
    return T, H, dk, dv, dev, out_dtype, S_hat, S_exact, o


def gdn_tail_replay_k(q, k, v, alpha, beta, cu_seqlens, m, k_replay, *, S_a=None, readout: bool = False,
                      out_dtype: Optional[torch.dtype] = None, S_hat=None, S_exact=None, o=None, stream=None,
                      ws: Optional[torch.Tensor] = None, algo: str = "auto"):
    """Tail replay of the k_replay[b] tokens before m[b] of every sequence (zero initial state).

    Returns dict(S_hat, S_exact or None, o or None)."""
    cu = _i64(cu_seqlens)
    B = len(cu) - 1
    T, H, dk, dv, dev, out_dtype, S_hat, S_exact, o = _replay_buffers(k, v, B, S_a, readout, out_dtype, S_hat,
                                                                      S_exact, o)
    mm, kr = _i64(m), _i64(k_replay)
    ws = ws if ws is not None else _auto_ws(dev, algo, k, v, int(kr.sum()) + (int(mm.sum()) if S_a is not None else 0),
                                            B * (2 if S_a is not None else 1))
    pr = _problem(cu, H, dk, dv, k.dtype, out_dtype, algo)
    rc = lib().gdn_tail_replay_k(ctypes.byref(pr), _ptr(q if readout else None), _ptr(k), _ptr(v), _ptr(alpha),
                                 _ptr(beta), _p64(mm), _p64(kr), _ptr(S_a), _ptr(S_hat),
                                 _ptr(S_exact if S_a is not None else None), _ptr(o), _ptr(ws), ws.numel(),
                                 _stream(stream, dev))
    _check(rc, "gdn_tail_replay_k")
    return {"S_hat": S_hat, "S_exact": S_exact if S_a is not None else None, "o": o}


def gdn_tail_replay_overlap(q, k, v, alpha, beta, cu_seqlens, m, r_num: int, r_den: int, kv_host, kv_dev, *,
                            copy_stream, S_a=None, readout: bool = False, out_dtype: Optional[torch.dtype] = None,
                            S_hat=None, S_exact=None, o=None, stream=None, ws: Optional[torch.Tensor] = None,
                            algo: str = "auto"):
    """gdn_tail_replay with kv_host (pinned) copied into kv_dev on copy_stream beside the replay;
    `stream` waits for the copy afterwards.  Returns the gdn_tail_replay dict."""
    cu = _i64(cu_seqlens)
    B = len(cu) - 1
    T, H, dk, dv, dev, out_dtype, S_hat, S_exact, o = _replay_buffers(k, v, B, S_a, readout, out_dtype, S_hat,
                                                                      S_exact, o)
    nbytes = kv_host.numel() * kv_host.element_size()
    if kv_dev.numel() * kv_dev.element_size() != nbytes:
        raise ValueError("kv_host and kv_dev sizes differ")
    a_out = np.zeros(B, dtype=np.int64)
    k_out = np.zeros(B, dtype=np.int64)
    mm = _i64(m)
    twin = 2 if S_a is not None else 1
    ws = ws if ws is not None else _auto_ws(dev, algo, k, v, int(mm.sum()) * twin, B * twin)
    pr = _problem(cu, H, dk, dv, k.dtype, out_dtype, algo)
    rc = lib().gdn_tail_replay_overlap(ctypes.byref(pr), _ptr(q if readout else None), _ptr(k), _ptr(v),
                                       _ptr(alpha), _ptr(beta), _p64(mm), r_num, r_den, _ptr(S_a), _ptr(S_hat),
                                       _ptr(S_exact if S_a is not None else None), _ptr(o), _p64(a_out),
                                       _p64(k_out), ctypes.c_void_p(kv_host.data_ptr()),
                                       ctypes.c_void_p(kv_dev.data_ptr()), nbytes, _ptr(ws), ws.numel(),
                                       _stream(stream, dev), _stream(copy_stream, dev))
    _check(rc, "gdn_tail_replay_overlap")
    return {"S_hat": S_hat, "S_exact": S_exact if S_a is not None else None, "o": o, "a": a_out.tolist(),
            "k": k_out.tolist()}


def gdn_group_replay(h, weights, layers: int, heads: int, d_model: int, d_head: int, m: int, r_num: int,
                     r_den: int, *, exact: bool = True, stream=None, ws: Optional[torch.Tensor] = None):
    """In-group chained replay of one request (see the header).  h [m, d_model] fp32 on the GPU,
    weights flat fp32 on the GPU.  Returns dict(S_hat [layers, heads, d_head, d_head], S_exact or None, a, k)."""
    dev = h.device
    g = _Group(layers, heads, d_model, d_head)
    a_o, k_o = ctypes.c_int64(), ctypes.c_int64()
    _, kk = gdn_replay_plan(m, r_num, r_den)
    rows = m if exact else kk
    nbytes = lib().gdn_group_scratch_bytes(ctypes.byref(g), rows)
    scratch = torch.empty(max(int(nbytes) // 4, 4), dtype=torch.float32, device=dev)
    S_hat = torch.empty((layers, heads, d_head, d_head), dtype=torch.float32, device=dev)
    S_exact = torch.empty_like(S_hat) if exact else None
    ws = ws if ws is not None else workspace(dev)
    rc = lib().gdn_group_replay(ctypes.byref(g), _ptr(h), m, r_num, r_den, _ptr(weights), _ptr(S_hat), _ptr(S_exact),
                                ctypes.byref(a_o), ctypes.byref(k_o), _ptr(scratch), scratch.numel() * 4, _ptr(ws),
                                ws.numel(), _stream(stream, dev))
    _check(rc, "gdn_group_replay")
    return {"S_hat": S_hat, "S_exact": S_exact, "a": a_o.value, "k": k_o.value}


def gdn_adaptive_replay_plan(alpha, cu_seqlens, m, eps: float, rmax_num: int, rmax_den: int, H: int,
                             d_k: int = 128, d_v: int = 128, stream=None):
    """Per-sequence tail length from the gates (see the header): (k list, exact-recovery flags)."""
    cu = _i64(cu_seqlens)
    B = len(cu) - 1
    k_out = np.zeros(B, dtype=np.int64)
    ex = np.zeros(B, dtype=np.int32)
    pr = _problem(cu, H, d_k, d_v, torch.bfloat16, torch.bfloat16)
    rc = lib().gdn_adaptive_replay_plan(ctypes.byref(pr), _ptr(alpha), _p64(_i64(m)), ctypes.c_float(eps),
                                        rmax_num, rmax_den, _p64(k_out), ex.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                        _stream(stream, alpha.device))
    _check(rc, "gdn_adaptive_replay_plan")
    return k_out.tolist(), ex.tolist()
