"""fp64 CPU oracle of one DeepSeekMoE layer forward (test infrastructure only).

Source: "DeepSeek-V3 Technical Report" (the condensed report page).
  * DeepSeekMoE paragraph: the FFN output of token t is the sum of the
    shared experts' outputs plus the gate-weighted outputs of the K_r
    routed experts it selects; affinities are sigmoid(u_t . e_i) with e_i
    the centroid of routed expert i; gates are the selected affinities
    normalised among themselves.  (The display equation is missing from
    the extracted page; this module rebuilds it from the symbols the
    paragraph defines.)
  * Auxiliary-loss-free load balancing paragraph: a per-expert bias b_i is
    added to the affinity only to choose the top-K; the gate still comes
    from the unbiased affinity; after each step b_i moves down by gamma if
    expert i is overloaded over the whole batch and up by gamma otherwise;
    no token is dropped; routing is node-limited (at most M nodes).
  * Model hyper-parameters paragraph: 1 shared + 256 routed experts,
    intermediate 2048, 8 active, at most 4 nodes; gamma = 0.001.

Readings where the page is silent (each is listed in the design notes):
  * the residual u_t is not part of the returned FFN sum;
  * node-limited routing on one device becomes group-limited routing over
    contiguous blocks of E/G experts; a group is scored by the sum (fp32,
    descending order) of its top ``group_score_topn`` biased scores;
  * ordering is by descending fp32 value, ties broken by the lower index,
    for groups, experts and the within-group top-n;
  * the biased score is fl32(s + b) and is compared in fp32;
  * "overloaded" means load * E > T * K (strictly above the mean load);
    otherwise (equality included) the bias goes up;
  * gates are multiplied by a route scale rho (1 unless a config sets it);
  * every expert FFN is SwiGLU: W2 (silu(W1 u) * (W3 u));
  * rows inside an expert's segment are in ascending token order.

Everything here is deliberately plain: NumPy fp64, one expert at a time,
no blocking, no fusion.
"""

from __future__ import annotations

import numpy as np

# --------------------------------------------------------------------------
# Routing
# --------------------------------------------------------------------------


def sigmoid_affinity(u, centroids):
    """Token-to-expert affinity s[t, i] = 1 / (1 + exp(-u_t . e_i)) in fp64.

    DeepSeek-V3 Technical Report, DeepSeekMoE paragraph (sigmoid affinity
    with the expert centroid e_i).  ``u`` is [T, d], ``centroids`` is [E, d].
    """
    u = np.asarray(u, dtype=np.float64)
    e = np.asarray(centroids, dtype=np.float64)
    logits = u @ e.T
    with np.errstate(over="ignore"):  # exp(-l) = inf gives the exact limit 0
        return 1.0 / (1.0 + np.exp(-logits))


def biased_scores(s32, bias32):
    """Selection score fl32(s + b) (auxiliary-loss-free paragraph).

    The bias only steers the top-K choice; ``s32`` and ``bias32`` are
    converted to float32 and added in float32, exactly as a device would.
    """
    s32 = np.asarray(s32, dtype=np.float32)
    b32 = np.asarray(bias32, dtype=np.float32)
    return (s32 + b32[None, :]).astype(np.float32)


def _order_desc(values):
    """Indices of ``values`` (1-D) by descending value, ties by lower index."""
    # A stable sort of the negated values keeps equal keys in index order.
    return np.argsort(-values, kind="stable")


def group_scores(biased32, n_groups, topn):
    """Score of every expert group: fp32 sum of its ``topn`` largest biased
    scores, added in descending order.  Groups are contiguous blocks of
    E / n_groups experts (the single-device reading of node-limited
    routing).  Returns float32 [T, n_groups]."""
    T, E = biased32.shape
    per = E // n_groups
    topn = min(topn, per)
    out = np.zeros((T, n_groups), dtype=np.float32)
    for t in range(T):
        for g in range(n_groups):
            vals = biased32[t, g * per:(g + 1) * per]
            top = vals[_order_desc(vals)[:topn]]
            acc = np.float32(0.0)
            for v in top:
                acc = np.float32(acc + v)
            out[t, g] = acc
    return out


def select_experts(s32, bias32, n_groups, topk_groups, k, group_score_topn=2):
    """Group-limited top-K selection on biased scores.

    Auxiliary-loss-free paragraph (bias for selection only) and the
    node-limited routing sentence (tokens reach at most M of the groups).
    Steps, per token: biased score fl32(s + b); group scores; keep the
    ``topk_groups`` best groups; among the experts of those groups keep
    the ``k`` with the largest biased score.  Output [T, k] int32 is listed
    by descending biased score, ties by the lower expert index.
    """
    biased = biased_scores(s32, bias32)
    T, E = biased.shape
    per = E // n_groups
    gs = group_scores(biased, n_groups, group_score_topn)
    idx = np.zeros((T, k), dtype=np.int32)
    for t in range(T):
        kept_groups = _order_desc(gs[t])[:topk_groups]
        allowed = np.zeros(E, dtype=bool)
        for g in kept_groups:
            allowed[g * per:(g + 1) * per] = True
        cand = np.nonzero(allowed)[0]
        order = _order_desc(biased[t, cand])
        idx[t] = cand[order[:k]]
    return idx


def gating_weights(s, idx, route_scale=1.0):
    """Gate g[t, j] = rho * s[t, idx[t, j]] / sum_j' s[t, idx[t, j']] (fp64).

    DeepSeekMoE paragraph: normalisation among the selected (unbiased)
    affinities; the route scale rho multiplies the normalised gates.
    """
    s = np.asarray(s, dtype=np.float64)
    sel = np.take_along_axis(s, idx.astype(np.int64), axis=1)
    return route_scale * sel / sel.sum(axis=1, keepdims=True)


def expert_load(idx, n_experts):
    """Whole-batch load c_i = number of tokens routed to expert i."""
    counts = np.zeros(n_experts, dtype=np.int64)
    for e in idx.reshape(-1):
        counts[e] += 1
    return counts


def segment_layout(idx, n_experts):
    """Per-expert segments of the permuted rows (no token dropping).

    offsets[e] is the exclusive prefix sum of the loads; inside a segment the
    rows follow ascending token index.  row_of_slot[t, j] is the permuted
    row that holds token t's copy for its j-th selected expert and
    token_of_row[r] is the token that row r copies.
    """
    T, k = idx.shape
    counts = expert_load(idx, n_experts)
    offsets = np.zeros(n_experts + 1, dtype=np.int64)
    for e in range(n_experts):
        offsets[e + 1] = offsets[e] + counts[e]
    fill = offsets[:-1].copy()
    row_of_slot = np.zeros((T, k), dtype=np.int64)
    token_of_row = np.zeros(T * k, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            r = fill[e]
            fill[e] += 1
            row_of_slot[t, j] = r
            token_of_row[r] = t
    return counts, offsets, row_of_slot, token_of_row


def permute_rows(x, token_of_row):
    """Dispatch on one device: row r of the result is x[token_of_row[r]]."""
    return np.asarray(x)[np.asarray(token_of_row, dtype=np.int64)]


# --------------------------------------------------------------------------
# Experts
# --------------------------------------------------------------------------


def silu(a):
    """silu(a) = a / (1 + exp(-a)) in fp64."""
    a = np.asarray(a, dtype=np.float64)
    with np.errstate(over="ignore"):  # exp(-a) = inf gives the exact limit 0
        return a / (1.0 + np.exp(-a))


def swiglu_ffn(u, w1, w3, w2):
    """One expert FFN, SwiGLU: W2 (silu(W1 u) * (W3 u)) for every row of u.

    ``u`` [n, d]; ``w1``, ``w3`` [I, d] (gate and up projections); ``w2``
    [d, I].  Plain fp64 matrix products.
    """
    u = np.asarray(u, dtype=np.float64)
    a = u @ np.asarray(w1, dtype=np.float64).T
    b = u @ np.asarray(w3, dtype=np.float64).T
    h = silu(a) * b
    return h @ np.asarray(w2, dtype=np.float64).T


def _expert_weights(w13, w2, e):
    """Split expert e's stacked [2I, d] gate/up weights into W1 and W3.

    The stacked layout holds W1 in rows [0, I) and W3 in rows [I, 2I).
    ``w13`` and ``w2`` may be arrays or any indexable that returns one
    expert's weights (so that very large weight sets can be converted to
    fp64 one expert at a time)."""
    g = np.asarray(w13[e], dtype=np.float64)
    inter = g.shape[0] // 2
    return g[:inter], g[inter:], np.asarray(w2[e], dtype=np.float64)


def combine(y_shared, y_perm, row_of_slot, gates):
    """Gate-weighted combine: out[t] = y_shared[t] + sum_j g[t,j] y_perm[row].

    DeepSeekMoE paragraph (shared experts see every token; routed outputs
    enter weighted by their gates).  ``y_shared`` may be None (no shared
    expert).  fp64.
    """
    T, k = row_of_slot.shape
    d = y_perm.shape[1]
    out = np.zeros((T, d), dtype=np.float64)
    if y_shared is not None:
        out += np.asarray(y_shared, dtype=np.float64)
    for j in range(k):
        out += gates[:, j:j + 1] * np.asarray(y_perm, dtype=np.float64)[row_of_slot[:, j]]
    return out


def gate_of_row(row_of_slot, gates):
    """Gate of every permuted row: the row holding token t's copy for slot j
    carries g[t, j] (the weight of that expert's output in the DeepSeekMoE
    paragraph's sum).  With y_perm's rows multiplied by it, the combine is a
    plain sum: combine(y_shared, gate_of_row * y_perm, rows, 1) equals
    combine(y_shared, y_perm, rows, g)."""
    ros = np.asarray(row_of_slot)
    g = np.zeros(ros.size, dtype=np.float64)
    g[ros.reshape(-1)] = np.asarray(gates, dtype=np.float64).reshape(-1)
    return g


# --------------------------------------------------------------------------
# Auxiliary-loss-free bias update
# --------------------------------------------------------------------------


def bias_update(bias32, counts, n_tokens, k, gamma):
    """One step of the sign rule on the per-expert bias (fp32 state).

    Auxiliary-loss-free paragraph: at the end of a step, b_i goes down by
    gamma if expert i is overloaded over the whole batch, up by gamma
    otherwise.  Overloaded is read as c_i > T*K/E, compared in integers as
    c_i * E > T * K; the update is fl32(b_i -/+ fl32(gamma)).
    """
    b = np.asarray(bias32, dtype=np.float32).copy()
    E = b.shape[0]
    g32 = np.float32(gamma)
    for i in range(E):
        if int(counts[i]) * E > n_tokens * k:
            b[i] = np.float32(b[i] - g32)
        else:
            b[i] = np.float32(b[i] + g32)
    return b


def load_spread(counts):
    """Load-balance statistics of a whole-batch load vector."""
    c = np.asarray(counts, dtype=np.float64)
    mean = c.mean()
    return {
        "max_over_mean": float(c.max() / mean) if mean > 0 else 0.0,
        "cv": float(c.std() / mean) if mean > 0 else 0.0,
        "min": int(c.min()),
        "max": int(c.max()),
    }


def sequence_balance(affinity, topk_idx, seq_len, alpha=1e-4):
    """Sequence-wise balance statistic L_Bal = alpha * sum_i f_i P_i per
    sequence (auxiliary-loss-free paragraph: a complementary sequence-wise
    balance loss with a small factor; training hyper-parameters paragraph:
    alpha = 0.0001).  The pages do not define f_i and P_i; the reading here:
    for a sequence of L consecutive tokens,
        f_i = E / (K L) * #{(t, k) in the sequence: expert i chosen}
        P_i = (1 / L) * sum_t s_{i,t} / sum_j s_{j,t}
    so an even split of the selections gives f_i = 1.

    ``affinity`` [T, E] (the unbiased s), ``topk_idx`` [T, K]; T must be a
    multiple of ``seq_len``.  Returns (f [n_seq, E], P [n_seq, E],
    loss [n_seq]) in fp64."""
    s = np.asarray(affinity, dtype=np.float64)
    idx = np.asarray(topk_idx)
    T, E = s.shape
    K = idx.shape[1]
    assert T % seq_len == 0
    n = T // seq_len
    f = np.zeros((n, E))
    P = np.zeros((n, E))
    loss = np.zeros(n)
    for q in range(n):
        rows = range(q * seq_len, (q + 1) * seq_len)
        for t in rows:
            for e in idx[t]:
                f[q, int(e)] += 1.0
            P[q] += s[t] / s[t].sum()
        f[q] *= E / (K * seq_len)
        P[q] /= seq_len
        loss[q] = alpha * float(np.dot(f[q], P[q]))
    return f, P, loss


# --------------------------------------------------------------------------
# Whole layer
# --------------------------------------------------------------------------


def moe_layer_forward(x, router_w, bias, w13, w2, ws13, ws2, *, n_groups,
                      topk_groups, k, route_scale=1.0, group_score_topn=2,
                      affinity32=None, residual=False):
    """Forward of one DeepSeekMoE layer in fp64.

    ``x`` [T, d]; ``router_w`` [E, d] (the centroids e_i); ``bias`` [E];
    ``w13`` [E, 2I, d]; ``w2`` [E, d, I]; ``ws13`` [Ns, 2I, d] and
    ``ws2`` [Ns, d, I] for the shared experts (Ns may be 0 / None).

    Selection uses ``affinity32`` (float32 [T, E]) when given, so that a
    device's own fp32 affinities can be routed exactly; otherwise the
    oracle's fp64 affinities rounded to float32.  Gates always come from
    the affinities used for selection.  Returns a dict of every
    intermediate the layer exposes.
    """
    x64 = np.asarray(x, dtype=np.float64)
    T, d = x64.shape
    E = np.asarray(router_w).shape[0]
    s64 = sigmoid_affinity(x64, router_w)
    s_sel = s64.astype(np.float32) if affinity32 is None else np.asarray(affinity32, np.float32)
    idx = select_experts(s_sel, bias, n_groups, topk_groups, k, group_score_topn)
    gates = gating_weights(s_sel, idx, route_scale)
    counts, offsets, row_of_slot, token_of_row = segment_layout(idx, E)
    x_perm = permute_rows(x64, token_of_row)
    y_perm = np.zeros((T * k, d), dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            w1, w3, w2e = _expert_weights(w13, w2, e)
            y_perm[lo:hi] = swiglu_ffn(x_perm[lo:hi], w1, w3, w2e)
    y_shared = None
    n_shared = 0 if ws13 is None else len(ws13)
    if n_shared:
        y_shared = np.zeros((T, d), dtype=np.float64)
        for s in range(n_shared):
            w1, w3, w2s = _expert_weights(ws13, ws2, s)
            y_shared += swiglu_ffn(x64, w1, w3, w2s)
    out = combine(y_shared, y_perm, row_of_slot, gates)
    if residual:
        out = out + x64
    return {
        "affinity": s64, "topk_idx": idx, "topk_w": gates, "counts": counts,
        "offsets": offsets, "row_of_slot": row_of_slot,
        "token_of_row": token_of_row, "y_perm": y_perm, "y_shared": y_shared,
        "out": out,
    }


def moe_layer_tokens(x_rows, idx_rows, gates_rows, w13, w2, ws13, ws2):
    """Layer output for a few tokens whose routing is already known.

    Used to check very large layers on a sample of tokens: for every given
    token it sums the shared experts and its gate-weighted routed experts,
    converting each needed expert's weights to fp64 once.
    """
    x64 = np.asarray(x_rows, dtype=np.float64)
    n, d = x64.shape
    out = np.zeros((n, d), dtype=np.float64)
    n_shared = 0 if ws13 is None else len(ws13)
    for s in range(n_shared):
        w1, w3, w2s = _expert_weights(ws13, ws2, s)
        out += swiglu_ffn(x64, w1, w3, w2s)
    experts = sorted(set(int(e) for e in np.asarray(idx_rows).reshape(-1)))
    for e in experts:
        w1, w3, w2e = _expert_weights(w13, w2, e)
        rows, cols = np.nonzero(np.asarray(idx_rows) == e)
        y = swiglu_ffn(x64[rows], w1, w3, w2e)
        out[rows] += np.asarray(gates_rows, dtype=np.float64)[rows, cols][:, None] * y
    return out
