"""fp64 reference definitions of every step of the MoE layer (test infrastructure only).

Notation: T tokens, d model width, E experts, k experts per token, F expert FFN width,
r LoRA rank, s = alpha / r.  A *slot* is a (token t, rank j) pair, numbered ``t*k + j``;
rank 0 is the expert with the largest router logit.

Readings taken where the pages are silent (each one is listed in the design notes):

* router: ``L = x W_r^T + b`` with an fp32 W_r; softmax over all E experts; the top-k is
  chosen on the logits, ties going to the lower expert index; gates are the selected
  softmax probabilities renormalised to sum to one over the k selected experts.
* capacity: ``C = ceil(cf * T * k / E)`` with cf a rational; an infinite factor keeps
  every slot.  A slot is dropped when its expert already holds C earlier tokens
  ("arrival order" = ascending token index).  Dropped slots contribute nothing and the
  surviving gates are not renormalised again.
* expert network: SwiGLU, ``E_e(x) = W_d,e (silu(W_g,e x) * (W_u,e x))`` without biases,
  with a LoRA update on each of the three projections: ``W x + s B (A x)``.
* auxiliary loss: ``aux = E * sum_e f_e P_e`` with ``f_e`` the pre-drop fraction of slots
  routed to e and ``P_e`` the mean softmax probability of e.
* backward: the loss is ``<dy, y>`` with the routing decisions held fixed (no re-routing,
  per "Day-Level Adaptation ...", section 5: checkpoint boundaries avoid dynamic routing);
  the base weights and the router are frozen ("Adapting Trillion-Parameter MoE Models ...",
  section 3: tuning the routing gates disturbs load balance), so the gradients are dx and
  the LoRA factors.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "capacity",
    "router_logits",
    "softmax",
    "topk_select",
    "renormalised_gates",
    "route",
    "dispatch",
    "dispatch_remap",
    "permute",
    "silu",
    "lora_linear",
    "expert_forward",
    "combine",
    "aux_loss",
    "moe_forward",
    "moe_forward_fixed_routing",
    "expert_backward",
    "route_backward",
    "moe_backward",
]


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------------------
# Routing: "Adapting Trillion-Parameter MoE Models ...", section 2.1, equation 1 (g_i, TopK)
# and "Day-Level Adaptation ...", section 2.1 (Top-16 selection, capacity control).
# --------------------------------------------------------------------------------------

def capacity(T: int, k: int, E: int, cap_num: int, cap_den: int):
    """Per-expert capacity ``ceil(cf * T * k / E)`` with ``cf = cap_num / cap_den``.

    ``cap_den == 0`` means an infinite capacity factor and returns ``None`` (no clipping).
    Exact integer arithmetic ("Day-Level Adaptation ...", section 3.2: expert_capacity=1.25).
    """
    if cap_den == 0:
        return None
    num = cap_num * T * k
    den = cap_den * E
    return -(-num // den)


def router_logits(x, w_router, bias=None):
    """``L[t, e] = sum_c x[t, c] W_r[e, c] + b[e]`` in float64."""
    L = _f64(x) @ _f64(w_router).T
    if bias is not None:
        L = L + _f64(bias)[None, :]
    return L


def softmax(logits):
    """Row softmax over all experts, max-subtracted, float64."""
    L = _f64(logits)
    z = np.exp(L - L.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def topk_select(logits, k: int):
    """Indices of the k largest logits per row, ordered by (-logit, expert index).

    Sorting on the key (-L, e) puts larger logits first and breaks ties towards the lower
    expert index; a stable sort of -L over indices 0..E-1 is exactly that key.
    """
    L = _f64(logits)
    order = np.argsort(-L, axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def renormalised_gates(p, idx):
    """``g[t, j] = p[t, idx[t, j]] / sum_j' p[t, idx[t, j']]``."""
    psel = np.take_along_axis(_f64(p), idx, axis=1)
    return psel / psel.sum(axis=1, keepdims=True)


def route(logits, k: int):
    """Selection, softmax probabilities and renormalised gates for one batch of logits."""
    idx = topk_select(logits, k)
    p = softmax(logits)
    g = renormalised_gates(p, idx)
    return idx, g, p


# --------------------------------------------------------------------------------------
# Dispatch: capacity-clipped, arrival-ordered grouping of slots by expert ("Adapting
# Ultra-Large MoE Models ...", section 3.3: capacity factor, dropping, batch reshaping;
# "Trillion-Parameter MoE Model Training Adaptation ...", section 3 "Communication":
# tokens are permuted by routing result before the grouped matrix multiplications).
# --------------------------------------------------------------------------------------

def dispatch(idx, E: int, C):
    """Literal per-expert queues, filled by one pass over tokens then ranks.

    Returns a dict with
      counts    [E]   slots routed to each expert before any drop
      kept      [E]   min(counts, C)
      offsets   [E+1] exclusive scan of kept (segment starts of the permuted rows)
      pos       [T,k] arrival position of the slot in its expert's queue
      slot_row  [T*k] permuted row of each slot, -1 when dropped
      row_slot  [n_kept] slot held by each permuted row
      n_kept, n_dropped
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    queues = [[] for _ in range(E)]
    counts = np.zeros(E, dtype=np.int64)
    pos = np.zeros((T, k), dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            pos[t, j] = counts[e]
            counts[e] += 1
            if C is None or pos[t, j] < C:
                queues[e].append(t * k + j)
    kept = np.array([len(q) for q in queues], dtype=np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(kept)
    n_kept = int(offsets[E])
    slot_row = np.full(T * k, -1, dtype=np.int64)
    row_slot = np.zeros(n_kept, dtype=np.int64)
    for e in range(E):
        for q, slot in enumerate(queues[e]):
            slot_row[slot] = offsets[e] + q
            row_slot[offsets[e] + q] = slot
    return dict(counts=counts, kept=kept, offsets=offsets, pos=pos, slot_row=slot_row,
                row_slot=row_slot, n_kept=n_kept, n_dropped=T * k - n_kept)


def dispatch_remap(order, k: int, E: int, C, rounds: int):
    """Dispatch that remaps overflowing slots instead of dropping them at once.

    "Adapting Ultra-Large MoE Models ...", section 3.3: tokens beyond an expert's capacity
    are handled by remapping or dropping.  The pages give no mechanism; the rule taken:

    * ``order[t]`` lists token t's experts in preference order (the key (-logit, expert));
      its first k entries are the selection, slot j's alternatives are the entries
      j + k, j + 2k, ..., j + rounds * k (none of them selected, none shared by two slots).
    * Pass 0 is the plain dispatch: each expert takes the slots routed to it in arrival
      order (ascending token, then rank) while it holds fewer than C slots.
    * In round r = 1 .. rounds every slot still unplaced proposes its r-th alternative; each
      expert again takes the proposals in arrival order while it holds fewer than C slots.
    * Slots still unplaced after the last round are dropped.  A remapped slot keeps its gate.

    Within an expert the rows are in placement order (pass 0, then round 1, ...; arrival
    order inside a pass).  ``counts`` stays the pre-drop count of the original selection.
    Returns the dict of :func:`dispatch` plus ``slot_expert`` [T*k] (the expert a slot was
    placed on, -1 when dropped) and ``slot_pass`` [T*k] (the pass that placed it, -1).
    """
    order = np.asarray(order)
    T = order.shape[0]
    if order.shape[1] < (rounds + 1) * k:
        raise ValueError("order must list (rounds + 1) * k experts per token")
    held = [[] for _ in range(E)]
    slot_expert = np.full(T * k, -1, dtype=np.int64)
    slot_pass = np.full(T * k, -1, dtype=np.int64)
    pending = [(t, j) for t in range(T) for j in range(k)]   # arrival order
    for r in range(rounds + 1):
        rejected = []
        for t, j in pending:
            e = int(order[t, j + k * r])
            if C is None or len(held[e]) < C:
                held[e].append(t * k + j)
                slot_expert[t * k + j] = e
                slot_pass[t * k + j] = r
            else:
                rejected.append((t, j))
        pending = rejected
    counts = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            counts[int(order[t, j])] += 1
    kept = np.array([len(q) for q in held], dtype=np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(kept)
    n_kept = int(offsets[E])
    slot_row = np.full(T * k, -1, dtype=np.int64)
    row_slot = np.zeros(n_kept, dtype=np.int64)
    for e in range(E):
        for q, slot in enumerate(held[e]):
            slot_row[slot] = offsets[e] + q
            row_slot[offsets[e] + q] = slot
    return dict(counts=counts, kept=kept, offsets=offsets, slot_row=slot_row,
                row_slot=row_slot, n_kept=n_kept, n_dropped=T * k - n_kept,
                slot_expert=slot_expert, slot_pass=slot_pass)


def permute(x, row_slot, k: int):
    """``x_perm[row] = x[row_slot[row] // k]`` (the gather that feeds the grouped GEMM)."""
    x = np.asarray(x)
    return x[np.asarray(row_slot) // k]


# --------------------------------------------------------------------------------------
# Expert network with LoRA ("Adapting Trillion-Parameter MoE Models ...", section 3,
# equation 1: W' = W0 + (alpha/r) B A, applied as W0 x + s B (A x)).
# --------------------------------------------------------------------------------------

def silu(z):
    z = _f64(z)
    return z / (1.0 + np.exp(-z))


def lora_linear(X, W, A=None, B=None, s: float = 0.0):
    """Rows of ``X`` times ``(W + s B A)^T`` evaluated as ``X W^T + s (X A^T) B^T``."""
    out = _f64(X) @ _f64(W).T
    if A is not None:
        out = out + s * ((_f64(X) @ _f64(A).T) @ _f64(B).T)
    return out


def expert_forward(X, Wg, Wu, Wd, lora=None, s: float = 0.0):
    """SwiGLU expert on a block of rows.  ``lora`` is None or a dict with keys
    A_g, B_g, A_u, B_u, A_d, B_d for this expert.  Returns (a_g, a_u, h, o)."""
    L = lora or {}
    a_g = lora_linear(X, Wg, L.get("A_g"), L.get("B_g"), s)
    a_u = lora_linear(X, Wu, L.get("A_u"), L.get("B_u"), s)
    h = silu(a_g) * a_u
    o = lora_linear(h, Wd, L.get("A_d"), L.get("B_d"), s)
    return a_g, a_u, h, o


def _lora_of(lora, e):
    if lora is None:
        return None
    return {name: _f64(v)[e] for name, v in lora.items()}


def combine(o_rows, gates, slot_row, T: int, k: int):
    """``y[t] = sum_j g[t, j] o[slot_row[t*k+j]]`` over kept slots, summed in rank order."""
    d = o_rows.shape[1]
    y = np.zeros((T, d))
    g = _f64(gates)
    for t in range(T):
        for j in range(k):
            row = slot_row[t * k + j]
            if row >= 0:
                y[t] += g[t, j] * o_rows[row]
    return y


def aux_loss(counts, p, T: int, k: int, E: int):
    """``aux = E * sum_e f_e P_e``, ``f_e = counts_e / (T k)`` (pre-drop), ``P_e`` = mean p."""
    f = np.asarray(counts, dtype=np.float64) / float(T * k)
    P = _f64(p).mean(axis=0)
    return float(E * np.sum(f * P))


def _experts_forward(x_perm, offsets, Wg, Wu, Wd, lora, s):
    rows = x_perm.shape[0]
    F = Wg.shape[1]
    d = Wd.shape[1]
    a_g = np.zeros((rows, F))
    a_u = np.zeros((rows, F))
    h = np.zeros((rows, F))
    o = np.zeros((rows, d))
    E = len(offsets) - 1
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        a_g[lo:hi], a_u[lo:hi], h[lo:hi], o[lo:hi] = expert_forward(
            x_perm[lo:hi], _f64(Wg[e]), _f64(Wu[e]), _f64(Wd[e]), _lora_of(lora, e), s)
    return a_g, a_u, h, o


def moe_forward_fixed_routing(x, logits, idx, disp, Wg, Wu, Wd, lora=None, s=0.0):
    """Layer output for a given selection and dispatch, gates taken from ``logits``."""
    T, k = idx.shape
    p = softmax(logits)
    g = renormalised_gates(p, idx)
    x_perm = permute(_f64(x), disp["row_slot"], k)
    a_g, a_u, h, o = _experts_forward(x_perm, disp["offsets"], Wg, Wu, Wd, lora, s)
    y = combine(o, g, disp["slot_row"], T, k)
    return dict(y=y, p=p, gates=g, x_perm=x_perm, a_g=a_g, a_u=a_u, h=h, o=o)


def moe_forward(x, w_router, Wg, Wu, Wd, k, cap_num=0, cap_den=0, bias=None, lora=None,
                s=0.0, logits=None, remap_rounds=0):
    """The whole layer ``y = sum_{i in TopK(x)} g_i(x) E_i(x)``.

    When ``logits`` is given (e.g. the fp32 logits another implementation computed), the
    selection, gates and probabilities are taken from those logits instead of the fp64
    router product, so that integer decisions are made on identical inputs.
    ``remap_rounds`` > 0 remaps overflowing slots (:func:`dispatch_remap`) instead of
    dropping them; a slot's gate stays that of its original selection.
    """
    x = _f64(x)
    T = x.shape[0]
    E = Wg.shape[0]
    L = router_logits(x, w_router, bias) if logits is None else _f64(logits)
    idx = topk_select(L, k)
    C = capacity(T, k, E, cap_num, cap_den)
    if remap_rounds:
        disp = dispatch_remap(topk_select(L, (remap_rounds + 1) * k), k, E, C, remap_rounds)
    else:
        disp = dispatch(idx, E, C)
    out = moe_forward_fixed_routing(x, L, idx, disp, Wg, Wu, Wd, lora, s)
    out.update(logits=L, idx=idx, C=C, disp=disp,
               aux=aux_loss(disp["counts"], out["p"], T, k, E))
    return out


# --------------------------------------------------------------------------------------
# Backward of L = <dy, y> with routing fixed, base weights and router frozen
# ("Adapting Trillion-Parameter MoE Models ...", section 3: only adapter parameters take
# gradient updates; routing gates are not tuned).
# --------------------------------------------------------------------------------------

def _dsilu(z):
    sg = 1.0 / (1.0 + np.exp(-z))
    return sg * (1.0 + z * (1.0 - sg))


def expert_backward(X, dO, Wg, Wu, Wd, lora=None, s=0.0):
    """Gradients through one expert for a block of rows with upstream grad ``dO`` (w.r.t.
    the ungated expert output).  Returns dX and, when ``lora`` is given, the LoRA grads."""
    X = _f64(X)
    dO = _f64(dO)
    Lr = lora or {}
    a_g, a_u, h, _ = expert_forward(X, Wg, Wu, Wd, lora, s)
    grads = {}
    # down projection: o = h Wd^T + s (h A_d^T) B_d^T
    dh = dO @ _f64(Wd)
    if lora is not None:
        Ad, Bd = _f64(Lr["A_d"]), _f64(Lr["B_d"])
        v = dO @ Bd                        # [rows, r]  = dz B_d
        dh = dh + s * (v @ Ad)
        grads["B_d"] = s * dO.T @ (h @ Ad.T)     # [d, r]
        grads["A_d"] = s * v.T @ h               # [r, F]
    da_g = dh * a_u * _dsilu(a_g)
    da_u = dh * silu(a_g)
    dX = da_g @ _f64(Wg) + da_u @ _f64(Wu)
    if lora is not None:
        for nm, da in (("g", da_g), ("u", da_u)):
            A, B = _f64(Lr["A_" + nm]), _f64(Lr["B_" + nm])
            v = da @ B                           # [rows, r]
            dX = dX + s * (v @ A)
            grads["B_" + nm] = s * da.T @ (X @ A.T)  # [F, r]
            grads["A_" + nm] = s * v.T @ X           # [r, d]
    return dX, grads


def route_backward(p, idx, gates, dgate, kept_mask):
    """Gradient of the loss w.r.t. the router logits given d(loss)/d(gate).

    ``g = p_sel / sum(p_sel)`` so ``dp_i = (dg_i - sum_j g_j dg_j) / sum(p_sel)`` on the
    selection and 0 elsewhere; then the softmax Jacobian ``dL_e = p_e (dp_e - sum_i p_i dp_i)``.
    Dropped slots carry dg = 0 (they do not reach y).
    """
    p = _f64(p)
    T, k = idx.shape
    dg = _f64(dgate) * kept_mask
    psel = np.take_along_axis(p, idx, axis=1)
    S = psel.sum(axis=1, keepdims=True)
    dpsel = (dg - np.sum(gates * dg, axis=1, keepdims=True)) / S
    dp = np.zeros_like(p)
    np.put_along_axis(dp, idx, dpsel, axis=1)
    return p * (dp - np.sum(p * dp, axis=1, keepdims=True))


def moe_backward(fwd, x, dy, w_router, Wg, Wu, Wd, lora=None, s=0.0):
    """Gradients of ``<dy, y>`` for a forward produced by :func:`moe_forward`.

    Returns dict with dx (total), dx_expert, dx_gate, dgate [T,k], dlogits [T,E], and the
    LoRA gradients dA_g, dB_g, dA_u, dB_u, dA_d, dB_d stacked over experts.
    """
    x = _f64(x)
    dy = _f64(dy)
    idx = fwd["idx"]
    T, k = idx.shape
    E = Wg.shape[0]
    disp = fwd["disp"]
    slot_row, row_slot, offsets = disp["slot_row"], disp["row_slot"], disp["offsets"]
    g = fwd["gates"]
    o = fwd["o"]
    rows = len(row_slot)
    # combine backward: dO_row = g * dy[token], dgate = <dy[token], o_row>
    tok = row_slot // k
    g_row = g.reshape(-1)[row_slot]
    dO = g_row[:, None] * dy[tok]
    dgate = np.zeros((T, k))
    kept = np.zeros((T, k))
    for slot, row in enumerate(slot_row):
        if row >= 0:
            dgate[slot // k, slot % k] = float(dy[slot // k] @ o[row])
            kept[slot // k, slot % k] = 1.0
    x_perm = fwd["x_perm"]
    dx_perm = np.zeros((rows, x.shape[1]))
    grads = {}
    if lora is not None:
        for nm in ("A_g", "B_g", "A_u", "B_u", "A_d", "B_d"):
            grads[nm] = np.zeros(np.asarray(lora[nm]).shape)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        dX, ge = expert_backward(x_perm[lo:hi], dO[lo:hi], _f64(Wg[e]), _f64(Wu[e]),
                                 _f64(Wd[e]), _lora_of(lora, e), s)
        dx_perm[lo:hi] = dX
        for nm, v in ge.items():
            grads[nm][e] = v
    dx_expert = np.zeros_like(x)
    np.add.at(dx_expert, tok, dx_perm)
    dlogits = route_backward(fwd["p"], idx, g, dgate, kept)
    dx_gate = dlogits @ _f64(w_router)
    out = dict(dx=dx_expert + dx_gate, dx_expert=dx_expert, dx_gate=dx_gate, dgate=dgate,
               dlogits=dlogits, dx_perm=dx_perm, dO=dO)
    for nm, v in grads.items():
        out["d" + nm] = v
    return out
