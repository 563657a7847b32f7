"""In-group chained replay oracle -- TEST INFRASTRUCTURE (same rules as the rest of ``oracle``).

"Tail-Replay" notes page, section 2.2 step 3 and section 2.4: the linear-attention layers of a group
are replayed in sequence from zero states over the tail a+1..m; the first layer reads the group's exact
cached input hidden states and each later layer the previous layer's replayed outputs, so from the
second layer on the transitions and writes themselves differ from the full run and the replay error
obeys (section 2.3, right-multiplied layout)
    E_i = E_{i-1} T_i + S^_{i-1} (T_i - T^_i) + (b_i - b^_i),   T = alpha (I - beta k k^T), b = beta v k^T.
The group is synthetic (the pages fix no model): per layer and head q, k = unit-normalised projections,
v a projection, alpha = 1 - 0.1 sigmoid(w_a . h), beta = sigmoid(w_b . h); the next input is
h + W_o [o_1; ...; o_heads].  Everything here is fp64; the scans are the oracle's own.
"""
from __future__ import annotations

from typing import List

import numpy as np

from . import replay_plan, scan


def unpack(weights, layers: int, heads: int, d_model: int, d_head: int) -> List[dict]:
    w = np.asarray(weights.cpu().numpy() if hasattr(weights, "cpu") else weights, dtype=np.float64)
    Hd = heads * d_head
    out, o = [], 0
    for _ in range(layers):
        layer = {}
        for name, shape in (("Wq", (Hd, d_model)), ("Wk", (Hd, d_model)), ("Wv", (Hd, d_model)),
                            ("wa", (heads, d_model)), ("wb", (heads, d_model)), ("Wo", (d_model, Hd))):
            n = shape[0] * shape[1]
            layer[name] = w[o:o + n].reshape(shape)
            o += n
        out.append(layer)
    assert o == w.size
    return out


def project(h: np.ndarray, W: dict, heads: int, d_head: int):
    """q, k, v [rows, heads, d_head] and alpha, beta [rows, heads] of one layer."""
    R = h.shape[0]
    q = (h @ W["Wq"].T).reshape(R, heads, d_head)
    k = (h @ W["Wk"].T).reshape(R, heads, d_head)
    v = (h @ W["Wv"].T).reshape(R, heads, d_head)
    q = q / np.linalg.norm(q, axis=2, keepdims=True)
    k = k / np.linalg.norm(k, axis=2, keepdims=True)
    sig = lambda z: 1.0 / (1.0 + np.exp(-z))
    alpha = 1.0 - 0.1 * sig(h @ W["wa"].T)
    beta = sig(h @ W["wb"].T)
    return q, k, v, alpha, beta


def chain(h, Ws: List[dict], heads: int, d_head: int, keep_inputs: bool = False):
    """Run the group over the rows of h from zero states: per layer the final states [heads] and,
    with keep_inputs, the layer's (q, k, v, alpha, beta)."""
    h = np.asarray(h, dtype=np.float64)
    states, inputs = [], []
    for l, W in enumerate(Ws):
        q, k, v, a, b = project(h, W, heads, d_head)
        if keep_inputs:
            inputs.append((q, k, v, a, b))
        last = l + 1 == len(Ws)
        S_l, o_l = [], []
        for hh in range(heads):
            r = scan(k[:, hh], v[:, hh], a[:, hh], b[:, hh], q=None if last else q[:, hh], want_o=not last)
            S_l.append(np.asarray(r["S"]))
            if not last:
                o_l.append(np.asarray(r["o"]))
        states.append(S_l)
        if not last:
            o = np.stack(o_l, axis=1).reshape(h.shape[0], heads * d_head)
            h = h + o @ W["Wo"].T
    return states, inputs


def group_replay(h, weights, layers: int, heads: int, d_model: int, d_head: int, m: int, r_num: int, r_den: int,
                 exact: bool = True):
    """S_hat (and S_exact) [layers][heads] of one request, and the plan (a, k)."""
    Ws = unpack(weights, layers, heads, d_model, d_head)
    hh = np.asarray(h.cpu().numpy() if hasattr(h, "cpu") else h, dtype=np.float64)
    a, k = replay_plan(m, r_num, r_den)
    S_hat, _ = chain(hh[a:m], Ws, heads, d_head)
    S_ex = chain(hh[:m], Ws, heads, d_head)[0] if exact else None
    return {"S_hat": S_hat, "S_exact": S_ex, "a": a, "k": k}
