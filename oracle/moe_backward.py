"""fp64 CPU oracle of one DeepSeekMoE layer's backward pass (test
infrastructure only).

Source: "DeepSeek-V3 Technical Report" (the condensed report page).
  * DeepSeekMoE paragraph: the layer output is the shared experts' outputs
    plus the routed experts' outputs weighted by gates, the gates being the
    selected sigmoid affinities normalised among themselves.  The backward
    pass here is the chain rule of that forward, with the top-K selection
    held fixed (a choice is not differentiable) and the selection bias
    receiving no gradient (the auxiliary-loss-free paragraph uses it for
    choosing only).
  * Mixed precision framework paragraph (Figure 6): every linear has three
    GEMMs, Fprop, Dgrad and Wgrad; the DualPipe paragraph splits the MLP
    backward into "backward for input" and "backward for weights".  The
    functions below keep that split: inputs' gradients first, weights'
    gradients from the same intermediates.

Notation (per token t, selected set K_t, route scale rho):
    s_i   = sigmoid(u . e_i)               l_i = u . e_i  (the logit)
    g_i   = rho s_i / S,  S = sum_{j in K_t} s_j
    y     = sum_shared FFN(u) + sum_{i in K_t} g_i FFN_i(u)
    FFN   = W2 (silu(W1 u) * (W3 u))
Given dL/dy (``dout``):
    dL/dg_i  = dout . FFN_i(u)
    dL/ds_j  = (rho / S) (dL/dg_j - sum_i dL/dg_i s_i / S)     (j in K_t)
    dL/dl_j  = dL/ds_j s_j (1 - s_j)
    dL/de_j += dL/dl_j u ,  dL/du += dL/dl_j e_j
and through each FFN (a = W1 u, b = W3 u, h = silu(a) b, dy = g_i dout):
    dh = W2^T dy,  da = dh b silu'(a),  db = dh silu(a),
    silu'(a) = sigma(a) (1 + a (1 - sigma(a))),
    du += W1^T da + W3^T db,  dW1 += da u^T,  dW3 += db u^T,  dW2 += dy h^T.

Plain NumPy fp64, one expert at a time, no blocking and no fusion.
"""

from __future__ import annotations

import numpy as np

from .moe_oracle import _expert_weights, permute_rows, silu


def _sigma(a):
    a = np.asarray(a, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-a))


def swiglu_ffn_backward(u, w1, w3, w2, dy):
    """Gradients of one SwiGLU expert applied to the rows of ``u``.

    ``u`` [n, d]; ``w1``, ``w3`` [I, d]; ``w2`` [d, I]; ``dy`` [n, d] the
    gradient of the expert's output rows.  Returns a dict with ``du``
    [n, d], ``dw1``/``dw3`` [I, d], ``dw2`` [d, I] and the intermediates
    ``a``, ``b``, ``h``, ``dh``, ``da``, ``db``."""
    u = np.asarray(u, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    w1 = np.asarray(w1, dtype=np.float64)
    w3 = np.asarray(w3, dtype=np.float64)
    w2 = np.asarray(w2, dtype=np.float64)
    a = u @ w1.T
    b = u @ w3.T
    sig = _sigma(a)
    h = silu(a) * b
    dh = dy @ w2
    da = dh * b * (sig * (1.0 + a * (1.0 - sig)))
    db = dh * silu(a)
    return {
        "du": da @ w1 + db @ w3,
        "dw1": da.T @ u,
        "dw3": db.T @ u,
        "dw2": dy.T @ h,
        "a": a, "b": b, "h": h, "dh": dh, "da": da, "db": db,
    }


def gate_backward(s_sel, idx, route_scale, dgate):
    """Gradient of the normalised gates back to the selected logits.

    ``s_sel`` [T, E] the affinities the gates were made from, ``idx``
    [T, K] the fixed selection, ``dgate`` [T, K] = dL/dg for each selected
    slot.  Returns (ds [T, K], dlogit [T, K]) for the selected experts in
    slot order; unselected experts get no gradient."""
    s = np.take_along_axis(np.asarray(s_sel, dtype=np.float64), np.asarray(idx, np.int64), axis=1)
    dg = np.asarray(dgate, dtype=np.float64)
    S = s.sum(axis=1, keepdims=True)
    inner = (dg * s).sum(axis=1, keepdims=True) / S
    ds = (route_scale / S) * (dg - inner)
    return ds, ds * s * (1.0 - s)


def combine_backward(dout, y_perm, row_of_slot, gates):
    """Gradient of the gate-weighted combine.  For every slot (t, j), with
    r = row_of_slot[t, j]: the routed row's gradient dy_slot[t, j] =
    g[t, j] dout[t] (it belongs at permuted row r) and
    dgate[t, j] = dout[t] . y_perm[r].  ``y_perm`` may hold only the rows the
    slots name (any indexable).  Returns (dy_slot [T, K, d], dgate [T, K])."""
    dout = np.asarray(dout, dtype=np.float64)
    ros = np.asarray(row_of_slot, dtype=np.int64)
    gates = np.asarray(gates, dtype=np.float64)
    T, K = ros.shape
    dy_slot = np.zeros((T, K, dout.shape[1]))
    dgate = np.zeros((T, K))
    for t in range(T):
        for j in range(K):
            dgate[t, j] = float(np.dot(dout[t], np.asarray(y_perm[ros[t, j]], dtype=np.float64)))
            dy_slot[t, j] = gates[t, j] * dout[t]
    return dy_slot, dgate


def input_grad(dx_shared, dx_perm, row_of_slot, idx, dlogit, router_w):
    """dL/dx_t = dx_shared[t] + sum_j (dx_perm[row_of_slot[t, j]]
    + dlogit[t, j] e_{idx[t, j]}): the shared experts, the routed experts'
    input gradients brought back to their token, and the router's share
    through the logits l = x . e."""
    ros = np.asarray(row_of_slot, dtype=np.int64)
    idx = np.asarray(idx, dtype=np.int64)
    T, K = ros.shape
    rw = np.asarray(router_w, dtype=np.float64)
    d = rw.shape[1]
    dx = np.zeros((T, d)) if dx_shared is None else np.array(dx_shared, dtype=np.float64)
    for t in range(T):
        for j in range(K):
            dx[t] += np.asarray(dx_perm[ros[t, j]], dtype=np.float64) + dlogit[t, j] * rw[idx[t, j]]
    return dx


def router_weight_grad(x, idx, dlogit, n_experts):
    """dL/de_i = sum over the slots (t, j) with idx[t, j] = i of
    dlogit[t, j] x_t (unchosen experts get zero rows)."""
    x = np.asarray(x, dtype=np.float64)
    idx = np.asarray(idx, dtype=np.int64)
    T, K = idx.shape
    g = np.zeros((n_experts, x.shape[1]))
    for t in range(T):
        for j in range(K):
            g[idx[t, j]] += dlogit[t, j] * x[t]
    return g


def moe_layer_backward(x, router_w, w13, w2, ws13, ws2, fwd, dout, *, route_scale=1.0,
                       affinity32=None, y_perm=None):
    """Backward of one DeepSeekMoE layer in fp64, selection held fixed.

    ``fwd`` is the dict of ``moe_layer_forward`` for the same inputs (its
    ``topk_idx``, ``topk_w``, ``row_of_slot``, ``token_of_row``,
    ``offsets`` and ``y_perm``).  ``affinity32`` are the affinities the
    gates were made from (a device's fp32 ones when routing was taken from
    it); default the forward's own fp64 affinities rounded to float32.
    ``y_perm`` overrides the routed expert outputs used for dL/dg (e.g. a
    device's stored rows).

    Returns a dict: ``dy_perm`` [T K, d], ``dgate`` [T, K], ``dlogit``
    [T, K], ``dx_perm`` [T K, d] (routed experts' input gradients per
    permuted row), ``dx_shared`` [T, d] (or None), ``dx`` [T, d],
    ``drouter_w`` [E, d], ``dw13`` [E, 2I, d], ``dw2`` [E, d, I],
    ``dws13``/``dws2`` (or None), and ``h_perm`` [T K, I] (the routed
    SwiGLU outputs, kept for the weight gradients)."""
    x64 = np.asarray(x, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    rw = np.asarray(router_w, dtype=np.float64)
    T, d = x64.shape
    E = rw.shape[0]
    idx = np.asarray(fwd["topk_idx"], dtype=np.int64)
    K = idx.shape[1]
    gates = np.asarray(fwd["topk_w"], dtype=np.float64)
    ros = np.asarray(fwd["row_of_slot"], dtype=np.int64)
    offsets = np.asarray(fwd["offsets"], dtype=np.int64)
    yp = np.asarray(fwd["y_perm"] if y_perm is None else y_perm, dtype=np.float64)
    s_sel = (np.asarray(fwd["affinity"]).astype(np.float32) if affinity32 is None
             else np.asarray(affinity32, dtype=np.float32))

    # combine: out[t] = y_shared[t] + sum_j g[t, j] y_perm[row_of_slot[t, j]]
    dy_slot, dgate = combine_backward(dout, yp, ros, gates)
    dy_perm = np.zeros((T * K, d))
    for j in range(K):
        dy_perm[ros[:, j]] = dy_slot[:, j]

    # routed experts, one segment at a time
    x_perm = permute_rows(x64, fwd["token_of_row"])
    inter = np.asarray(w13[0]).shape[0] // 2
    dx_perm = np.zeros((T * K, d))
    h_perm = np.zeros((T * K, inter))
    dw13 = np.zeros((E, 2 * inter, d))
    dw2 = np.zeros((E, d, inter))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        w1, w3, w2e = _expert_weights(w13, w2, e)
        r = swiglu_ffn_backward(x_perm[lo:hi], w1, w3, w2e, dy_perm[lo:hi])
        dx_perm[lo:hi] = r["du"]
        h_perm[lo:hi] = r["h"]
        dw13[e, :inter] = r["dw1"]
        dw13[e, inter:] = r["dw3"]
        dw2[e] = r["dw2"]

    # shared experts see every token with gradient dout
    n_shared = 0 if ws13 is None else len(ws13)
    dx_shared = dws13 = dws2 = None
    if n_shared:
        dx_shared = np.zeros((T, d))
        dws13 = np.zeros((n_shared, 2 * inter, d))
        dws2 = np.zeros((n_shared, d, inter))
        for s in range(n_shared):
            w1, w3, w2s = _expert_weights(ws13, ws2, s)
            r = swiglu_ffn_backward(x64, w1, w3, w2s, dout)
            dx_shared += r["du"]
            dws13[s, :inter] = r["dw1"]
            dws13[s, inter:] = r["dw3"]
            dws2[s] = r["dw2"]

    # gates -> logits -> router weights and input
    _, dlogit = gate_backward(s_sel, idx, route_scale, dgate)
    dx = input_grad(dx_shared, dx_perm, ros, idx, dlogit, rw)
    drouter_w = router_weight_grad(x64, idx, dlogit, E)
    return {
        "dy_perm": dy_perm, "dgate": dgate, "dlogit": dlogit, "dx_perm": dx_perm,
        "dx_shared": dx_shared, "dx": dx, "drouter_w": drouter_w, "dw13": dw13,
        "dw2": dw2, "dws13": dws13, "dws2": dws2, "h_perm": h_perm,
    }
