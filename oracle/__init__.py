"""fp64 CPU oracle for the Gated DeltaNet state scan -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never does.  It shares no code with the CUDA path; the two
meet only in the seeded input generator (``synth``).

The arithmetic lives in ``gdn_oracle.c`` (plain double-precision loops).
This module marshals arguments and composes the three operations from the
pages out of one scan primitive:

* prefill with sparse checkpoints ("Sparse prefix caching in hybrid and
  recurrent LLM serving", section 3: exact states stored at c_1 < ... < c_M);
* resume from the deepest checkpoint at or below the overlap depth d and
  recompute c_j+1 .. d (same section);
* Tail-Replay ("Tail-Replay ..." notes page, sections 2.1-2.2): k = ceil(r m),
  a = m - k, zero state at a, run tokens a+1 .. m; optional exact twin from S_a;
* checkpoint placement (``oracle.placement``; "Sparse prefix caching ...",
  sections 3-5).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Callable, List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with the host C compiler (no CUDA)."""
    src = os.path.join(_HERE, "gdn_oracle.c")
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(src):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-ffp-contract=off", "-shared", "-o", tmp, src],
                   check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
            lib.gdn_oracle_replay_plan.argtypes = [i64, i32, i32, ctypes.POINTER(i64), ctypes.POINTER(i64)]
            lib.gdn_oracle_select_ckpt.argtypes = [vp, i32, i64, ctypes.POINTER(i32)]
            lib.gdn_oracle_scan.argtypes = [ctypes.c_int, ctypes.c_int, i64, vp, vp, vp, vp, vp, vp, vp, i32, vp,
                                            vp, vp]
            lib.gdn_oracle_place_dp.argtypes = [vp, i64, i32, vp, ctypes.POINTER(i64)]
            for f in ("gdn_oracle_replay_plan", "gdn_oracle_select_ckpt", "gdn_oracle_scan", "gdn_oracle_place_dp"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x) -> Optional[np.ndarray]:
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


# ------------------------------------------------------------------------------------------
# index work (exact integers)
# ------------------------------------------------------------------------------------------

def replay_plan(m: int, r_num: int, r_den: int):
    """(a, k): k = ceil(r m) with r = r_num / r_den, a = m - k (Tail-Replay, section 2.1)."""
    a, k = ctypes.c_int64(), ctypes.c_int64()
    if _load().gdn_oracle_replay_plan(m, r_num, r_den, ctypes.byref(a), ctypes.byref(k)) != 0:
        raise ValueError("invalid replay plan arguments")
    return a.value, k.value


def select_ckpt(c: Sequence[int], d: int) -> int:
    """0-based index of the deepest checkpoint c_i <= d, or -1 (Sparse prefix caching, section 3)."""
    arr = np.ascontiguousarray(np.asarray(list(c), dtype=np.int64))
    j = ctypes.c_int32()
    if _load().gdn_oracle_select_ckpt(_ptr(arr) if len(arr) else None, len(arr), d, ctypes.byref(j)) != 0:
        raise ValueError("invalid checkpoint selection arguments")
    return j.value


# ------------------------------------------------------------------------------------------
# the scan primitive
# ------------------------------------------------------------------------------------------

def scan(k, v, alpha, beta, S0=None, q=None, ckpt_pos: Sequence[int] = (), want_o: bool = True):
    """One (sequence, head) stream: k [n, dk], v [n, dv], alpha/beta [n], q [n, dk].

    Returns dict(o=[n, dv] or None, ckpt=[M, dv, dk], S=[dv, dk]) in float64."""
    k, v, alpha, beta = _f64(k), _f64(v), _f64(alpha), _f64(beta)
    n, dk = k.shape
    dv = v.shape[1]
    assert v.shape[0] == n and alpha.shape == (n,) and beta.shape == (n,)
    q = _f64(q) if (want_o and q is not None) else None
    S0a = _f64(S0)
    if S0a is not None:
        assert S0a.shape == (dv, dk)
    o = np.empty((n, dv), dtype=np.float64) if q is not None else None
    pos = np.ascontiguousarray(np.asarray(list(ckpt_pos), dtype=np.int64))
    ck = np.empty((len(pos), dv, dk), dtype=np.float64)
    S = np.empty((dv, dk), dtype=np.float64)
    rc = _load().gdn_oracle_scan(dk, dv, n, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0a), _ptr(o),
                                 len(pos), _ptr(pos) if len(pos) else None, _ptr(ck) if len(pos) else None, _ptr(S))
    if rc != 0:
        raise ValueError(f"oracle scan rejected its arguments (rc={rc})")
    return {"o": o, "ckpt": ck, "S": S}


# ------------------------------------------------------------------------------------------
# the three operations, composed from the primitive
# ------------------------------------------------------------------------------------------

def prefill(q, k, v, alpha, beta, S0=None, ckpt_pos: Sequence[int] = (), want_o: bool = True):
    """Full scan over 1..N with exact state dumps at the checkpoint positions."""
    return scan(k, v, alpha, beta, S0=S0, q=q, ckpt_pos=ckpt_pos, want_o=want_o)


def resume(q, k, v, alpha, beta, ckpt_states, ckpt_pos: Sequence[int], d: int, S0=None, want_o: bool = True):
    """Resume at overlap depth d from the deepest stored checkpoint c_j <= d.

    q/k/v/alpha/beta are the sequence's streams (at least d rows);
    ckpt_states[i] is the state after token ckpt_pos[i].  Returns dict with
    j (0-based, -1 = initial state), c (the chosen position, 0 for the initial
    state), S (state after token d) and o (readout of tokens c+1 .. d)."""
    j = select_ckpt(ckpt_pos, d)
    c = 0 if j < 0 else int(ckpt_pos[j])
    start = S0 if j < 0 else ckpt_states[j]
    sl = slice(c, d)
    r = scan(k[sl], v[sl], alpha[sl], beta[sl], S0=start, q=None if q is None else q[sl], want_o=want_o)
    return {"j": j, "c": c, "S": r["S"], "o": r["o"]}


def tail_replay(k, v, alpha, beta, m: int, r_num: int, r_den: int, S_a=None, q=None, want_o: bool = False):
    """Tail-Replay at matched length m: zero state at a = m - ceil(r m), run a+1..m.

    Streams are the sequence's own rows (at least m).  With S_a given, also run
    the exact twin from S_a over the same tokens.  Returns dict(a, k, S_hat,
    S_exact or None, o or None)."""
    a, kk = replay_plan(m, r_num, r_den)
    sl = slice(a, m)
    qq = None if q is None else q[sl]
    hat = scan(k[sl], v[sl], alpha[sl], beta[sl], S0=None, q=qq, want_o=want_o)
    ex = None
    if S_a is not None:
        ex = scan(k[sl], v[sl], alpha[sl], beta[sl], S0=S_a, q=None, want_o=False)["S"]
    return {"a": a, "k": kk, "S_hat": hat["S"], "S_exact": ex, "o": hat["o"]}


def run_many(jobs: List[Callable], threads: Optional[int] = None):
    """Run independent oracle jobs on a thread pool (the C loop releases the GIL)."""
    threads = threads or os.cpu_count() or 1
    if threads <= 1 or len(jobs) <= 1:
        return [j() for j in jobs]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(lambda f: f(), jobs))


def adaptive_replay_plan(alpha, cu_seqlens: Sequence[int], m: Sequence[int], eps: float, rmax_num: int,
                         rmax_den: int):
    """Adaptive tail length per request ("Tail-Replay" notes page, section 5, the proposed extension;
    the bound of section 2.3): k_b = the least k <= ceil(rmax m_b) such that the product of the last
    k gates is <= eps for every head, taken in fp32 with the newest gate first; when the budget is too
    short for some head, k_b = the budget and the request is flagged for exact recovery.

    alpha: [T, H] float32 (numpy or torch on the CPU).  Returns (k list, exact flags)."""
    a = np.asarray(alpha.cpu().numpy() if hasattr(alpha, "cpu") else alpha, dtype=np.float32)
    H = a.shape[1]
    e = np.float32(eps)
    ks, flags = [], []
    for b in range(len(cu_seqlens) - 1):
        _, K = replay_plan(int(m[b]), rmax_num, rmax_den)
        need, reached = 0, True
        if K == 0:
            reached = int(m[b]) == 0
        for h in range(H):
            if K == 0:
                break
            prod = np.float32(1.0)
            kh = None
            for i in range(1, K + 1):
                prod = np.float32(prod * a[cu_seqlens[b] + int(m[b]) - i, h])
                if prod <= e:
                    kh = i
                    break
            if kh is None:
                reached, kh = False, K
            need = max(need, kh)
        ks.append(need)
        flags.append(0 if reached else 1)
    return ks, flags
