"""Plain, slow, fp64 definition of what the fused MoE-LoRA expert layer computes.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the library. It shares no code, table or
helper with the CUDA path.

Sources (the pages describing vLLM's multi-LoRA serving for MoE models):

* "vLLM Multi-LoRA Serving for MoE Models" (agentlenshq.com), section
  "Multi-LoRA Serving for MoE Models": tokens are routed to experts; every
  expert has a gate_up and a down projection, and LoRA gives each projection a
  shrink op and an expand op.
* vLLM blog "multi-LoRA for MoE" (vllm.com.cn), section "Implementing
  multi-LoRA inference for MoE models in vLLM": each token goes to its top-k
  experts, whose outputs are summed with the routing weights; for a projection with
  base weight W (h_in x h_out) LoRA trains A (h_in x r) and B (r x h_out) and
  the output is y = xW + xAB; shrink is z = xA, expand is zB; each expert
  carries four LoRA ops (gate_up shrink/expand, down shrink/expand); tokens
  select an (expert, adapter) pair ("compound sparsity"). Fig. 1: hidden 4096,
  intermediate 11008, r = 32.

Readings where the pages are silent:

* Activation between the projections: SwiGLU, h = silu(gate) * up with
  silu(v) = v / (1 + exp(-v)); the gate_up output holds gate in columns
  [0, I) and up in [I, 2I). No bias, no clamp.
* LoRA scale is 1 (the pages write y = xW + xAB); callers fold alpha/r into B.
* Routing: the k largest logits per token (ties to the lower expert index,
  NaN counts as -inf); weights are the softmax over those k logits.
* Adapter id -1 means "base model only" for that token.
* Weights are stored transposed with respect to the pages' h_in x h_out
  notation, the reduction dimension innermost: W1 [E, 2I, H], W2 [E, H, I],
  A1 [L, E, r, H], B1 [L, E, 2I, r], A2 [L, E, r, I], B2 [L, E, H, r].
* A slot whose expert id or whose token's adapter id is out of range is
  dropped (contributes nothing) and flagged in an error word.
* Intermediates are kept in fp64 with no rounding.
* Adapters of different ranks (the pages give ranks "typically 16-64" but one r
  per serving instance): adapter l of rank r_l <= r is stored padded to r and uses
  the first r_l rows of A (of each slice) and the first r_l columns of B.
* Separate gate and up adapters (the pages describe one LoRA per projection and
  are silent on a gate_up projection split in two): A1 [L, E, 2r, H] stacks the
  gate and the up A, B1 [L, E, 2I, r] keeps gate rows first, and each half of
  the gate_up output takes its own z.
"""
from __future__ import annotations

import math
import numpy as np

ERR_EXPERT_RANGE = 1
ERR_ADAPTER_RANGE = 2


def as_f64(t) -> np.ndarray:
    """Exact fp64 copy of a torch tensor (bf16/fp32) or array."""
    if t is None:
        return None
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().to("cpu").to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)


def as_i64(t) -> np.ndarray:
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().to("cpu").to(torch.int64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.int64)


def silu(v):
    """silu(v) = v * sigmoid(v) = v / (1 + exp(-v))."""
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def swiglu(g: np.ndarray) -> np.ndarray:
    """gate_up output [n, 2I] -> silu(gate) * up, [n, I]."""
    I = g.shape[-1] // 2
    return silu(g[..., :I]) * g[..., I:]


# ----------------------------------------------------------------------------
# Routing: each token's top-k experts and their softmax weights.
# ----------------------------------------------------------------------------
def route_topk_softmax(logits, k: int):
    """Top-k experts per token and their softmax weights.

    ids[t] are the k largest logits of token t in decreasing order, equal
    logits ordered by the lower expert index, NaN treated as -inf; w[t] is the
    softmax over those k logits (fp64).
    """
    lg = as_f64(logits)
    T, E = lg.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    key = np.where(np.isnan(lg), -np.inf, lg)
    ids = np.argsort(-key, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(key, ids, axis=1)
    m = sel[:, :1]
    with np.errstate(invalid="ignore"):  # a row of only NaN/-inf logits has no weights (NaN)
        ex = np.exp(sel - m)
        w = ex / ex.sum(axis=1, keepdims=True)
    return ids.astype(np.int32), w


# ----------------------------------------------------------------------------
# Alignment: group token-slots by (expert, adapter) -- the compound sparsity.
# ----------------------------------------------------------------------------
def align(ids, token_adapter, E: int, L: int, bm_base: int, bm_lora: int) -> dict:
    """Sort slots s = t*k + j by the key (expert, adapter, s), adapter -1 first.

    Returns a dict with
      err           error bits (1: expert id out of range, 2: adapter id out of range)
      n_valid       number of slots kept
      sorted_slots  [S] kept slots in key order, then -1
      slot_row      [S] position of each slot in sorted_slots, -1 if dropped
      expert_begin  [E+1] first row of each expert (rows of expert e are
                    expert_begin[e] .. expert_begin[e+1]-1)
      tiles         [(e, row_begin, rows)] each expert's rows cut into chunks of
                    at most bm_base rows, in row order
      lora_blocks   [(row_begin, rows, e, l)] each (e, l >= 0) segment cut into
                    chunks of at most bm_lora rows, in row order
      row_expert, row_adapter  [n_valid] key of each sorted row
      n_lora_rows   rows with an adapter
    """
    ids = as_i64(ids)
    T, k = ids.shape
    S = T * k
    if token_adapter is None:
        ad = np.full(T, -1, dtype=np.int64)
    else:
        ad = as_i64(token_adapter)
    err = 0
    kept = []
    for s in range(S):
        t, j = divmod(s, k)
        e, l = int(ids[t, j]), int(ad[t])
        ok = True
        if not (0 <= e < E):
            err |= ERR_EXPERT_RANGE
            ok = False
        if not (-1 <= l < L):
            err |= ERR_ADAPTER_RANGE
            ok = False
        if ok:
            kept.append(s)

    def key(s):
        t, j = divmod(s, k)
        return (int(ids[t, j]), int(ad[t]), s)

    order = sorted(kept, key=key)
    n_valid = len(order)
    sorted_slots = np.full(S, -1, dtype=np.int64)
    slot_row = np.full(S, -1, dtype=np.int64)
    row_expert = np.zeros(n_valid, dtype=np.int64)
    row_adapter = np.zeros(n_valid, dtype=np.int64)
    for row, s in enumerate(order):
        sorted_slots[row] = s
        slot_row[s] = row
        row_expert[row], row_adapter[row], _ = key(s)

    counts = np.bincount(row_expert, minlength=E) if n_valid else np.zeros(E, dtype=np.int64)
    expert_begin = np.zeros(E + 1, dtype=np.int64)
    expert_begin[1:] = np.cumsum(counts)

    tiles = []
    for e in range(E):
        b0, b1 = int(expert_begin[e]), int(expert_begin[e + 1])
        for c in range(b0, b1, bm_base):
            tiles.append((e, c, min(bm_base, b1 - c)))

    lora_blocks = []
    row = 0
    while row < n_valid:
        e, l = int(row_expert[row]), int(row_adapter[row])
        end = row
        while end < n_valid and row_expert[end] == e and row_adapter[end] == l:
            end += 1
        if l >= 0:
            for c in range(row, end, bm_lora):
                lora_blocks.append((c, min(bm_lora, end - c), e, l))
        row = end

    return dict(err=err, n_valid=n_valid, sorted_slots=sorted_slots, slot_row=slot_row,
                expert_begin=expert_begin, tiles=tiles, lora_blocks=lora_blocks,
                row_expert=row_expert, row_adapter=row_adapter,
                n_lora_rows=int((row_adapter >= 0).sum()), T=T, k=k, S=S, E=E, L=L)


# ----------------------------------------------------------------------------
# The per-op definitions, on sorted rows.
# ----------------------------------------------------------------------------
def gather_rows(x, al: dict) -> np.ndarray:
    """xs[row] = x[token of sorted slot row]; [n_valid, H]."""
    X = as_f64(x)
    n = al["n_valid"]
    toks = al["sorted_slots"][:n] // al["k"]
    return X[toks]


def grouped_gemm(a_sorted, W, al: dict) -> np.ndarray:
    """Base expert projection (vLLM's fused_moe group GEMM): out[row] = a[row] W_e^T."""
    A = as_f64(a_sorted)
    Wf = W if isinstance(W, np.ndarray) and W.dtype == np.float64 else as_f64(W)
    n = al["n_valid"]
    out = np.zeros((n, Wf.shape[1]))
    eb = al["expert_begin"]
    for e in range(al["E"]):
        b0, b1 = int(eb[e]), int(eb[e + 1])
        if b1 > b0:
            out[b0:b1] = A[b0:b1] @ Wf[e].T
    return out


def rank_mask_A(A, adapter_ranks, rank: int):
    """A of adapters with their own ranks: adapter l keeps rows [0, r_l) of each slice of
    `rank` rows (r_l clamped to [0, rank]); the rows past r_l are zero."""
    Af = as_f64(A)
    if adapter_ranks is None:
        return Af
    Af = Af.copy()
    for l, rl in enumerate(as_i64(adapter_ranks)):
        rl = min(max(int(rl), 0), rank)
        for sl in range(Af.shape[2] // rank):
            Af[l, :, sl * rank + rl: (sl + 1) * rank] = 0.0
    return Af


def rank_mask_B(B, adapter_ranks):
    """B of adapters with their own ranks: adapter l keeps columns [0, r_l)."""
    Bf = as_f64(B)
    if adapter_ranks is None:
        return Bf
    Bf = Bf.copy()
    rank = Bf.shape[3]
    for l, rl in enumerate(as_i64(adapter_ranks)):
        Bf[l, :, :, min(max(int(rl), 0), rank):] = 0.0
    return Bf


def lora_shrink(X, A, al: dict, rows_are_slots: bool, adapter_ranks=None,
                rank: int = None) -> np.ndarray:
    """Shrink z = x A for every slot with an adapter; Z [S, r], zero elsewhere.

    rows_are_slots=False: the input row of slot s is token s // k of X [T, K].
    rows_are_slots=True:  the input row of slot s is its sorted row of X [n, K].
    adapter_ranks [L]: adapter l uses rows [0, r_l) of each slice of `rank` rows of A
    (default: all rows, one slice); z entries past r_l are zero.
    """
    Xf = as_f64(X)
    Af = rank_mask_A(A, adapter_ranks, as_f64(A).shape[2] if rank is None else rank)
    r = Af.shape[2]
    Z = np.zeros((al["S"], r))
    n = al["n_valid"]
    for row in range(n):
        l = int(al["row_adapter"][row])
        if l < 0:
            continue
        e = int(al["row_expert"][row])
        s = int(al["sorted_slots"][row])
        xin = Xf[row] if rows_are_slots else Xf[s // al["k"]]
        Z[s] = Af[l, e] @ xin
    return Z


def lora_delta_rows(Z, B, al: dict, slices: int = 1, adapter_ranks=None) -> np.ndarray:
    """Expand z B for each sorted row with an adapter; [n_valid, N], zero elsewhere.

    slices = 2 (separate gate and up adapters): z rows hold 2r values; output
    columns [0, N/2) take the first r with B rows [0, N/2), columns [N/2, N) the
    last r with B rows [N/2, N). adapter_ranks [L]: adapter l uses columns [0, r_l) of B.
    """
    Zf = as_f64(Z)
    Bf = rank_mask_B(B, adapter_ranks)
    n = al["n_valid"]
    N = Bf.shape[2]
    r = Bf.shape[3]
    D = np.zeros((n, N))
    for row in range(n):
        l = int(al["row_adapter"][row])
        if l < 0:
            continue
        e = int(al["row_expert"][row])
        s = int(al["sorted_slots"][row])
        if slices == 1:
            D[row] = Bf[l, e] @ Zf[s]
        else:
            D[row, : N // 2] = Bf[l, e, : N // 2] @ Zf[s, :r]
            D[row, N // 2:] = Bf[l, e, N // 2:] @ Zf[s, r: 2 * r]
    return D


def combine(O_rows, w, al: dict) -> np.ndarray:
    """Aggregate expert outputs: y[t] = sum_j w[t, j] * O[row of slot t*k+j]."""
    O = as_f64(O_rows)
    wf = as_f64(w)
    T, k = al["T"], al["k"]
    y = np.zeros((T, O.shape[1]))
    for t in range(T):
        for j in range(k):
            row = int(al["slot_row"][t * k + j])
            if row >= 0:
                y[t] += wf[t, j] * O[row]
    return y


def lora_expand_add(Z, B, al: dict, base_rows, epilogue: int, w=None,
                    adapter_ranks=None) -> np.ndarray:
    """Expand with the base add fused (vllm.com.cn, "Kernel optimizations").

    epilogue 0: base + zB                      [n_valid, N]
    epilogue 1: swiglu(base + zB)              [n_valid, N/2]
    epilogue 2: combine(base + zB, w)          [T, N]
    epilogue 3: as 1 with separate gate and up adapters (two z slices; see
                lora_delta_rows)              [n_valid, N/2]
    """
    G = as_f64(base_rows) + lora_delta_rows(Z, B, al, slices=2 if epilogue == 3 else 1,
                                            adapter_ranks=adapter_ranks)
    if epilogue == 0:
        return G
    if epilogue in (1, 3):
        return swiglu(G)
    if epilogue == 2:
        return combine(G, w, al)
    raise ValueError("epilogue must be 0, 1, 2 or 3")


# ----------------------------------------------------------------------------
# The whole layer.
# ----------------------------------------------------------------------------
def _slots_ok(ids, ad, E, L):
    e_ok = (ids >= 0) & (ids < E)
    l_ok = (ad >= -1) & (ad < L)
    return e_ok & l_ok[:, None]


def moe_lora_layer(x, W1, W2, ids, w, token_adapter=None, A1=None, B1=None, A2=None,
                   B2=None, gate_up_slices: int = 1, adapter_ranks=None) -> np.ndarray:
    """y[t] = sum_j w[t,j] * expert_{ids[t,j]}(x[t]) with the token's adapter.

    expert_e with adapter l (l = -1: none):
      g = x W1_e^T + (x A1_{l,e}^T) B1_{l,e}^T        gate_up with LoRA
      h = silu(g[:I]) * g[I:]                          SwiGLU
      o = h W2_e^T + (h A2_{l,e}^T) B2_{l,e}^T         down with LoRA
    gate_up_slices = 2: the gate and up projections carry separate adapters,
    A1 [L, E, 2r, H] (rows [0, r) gate, [r, 2r) up), B1 [L, E, 2I, r]:
      g[:I] += (x A1_{l,e}[:r]^T) B1_{l,e}[:I]^T,  g[I:] += (x A1_{l,e}[r:]^T) B1_{l,e}[I:]^T
    adapter_ranks [L]: adapter l has rank r_l <= r: it uses the first r_l rows of each
    slice of A1 and of A2 and the first r_l columns of B1 and B2 (stored padded to r).
    Slots that share (e, l) are stacked into one matrix product per group; the
    arithmetic per slot is unchanged. Weights may be torch tensors or fp64
    numpy arrays (the latter skip the per-call conversion).
    """
    X = as_f64(x)
    ids_ = as_i64(ids)
    wf = as_f64(w)
    T, k = ids_.shape
    E = W1.shape[0]
    L = 0 if A1 is None else A1.shape[0]
    ad = np.full(T, -1, dtype=np.int64) if token_adapter is None else as_i64(token_adapter)
    if L == 0:
        ad = np.full(T, -1, dtype=np.int64)  # no adapter resident: adapter ids carry no meaning
    ok = _slots_ok(ids_, ad, E, L)
    if adapter_ranks is not None and L > 0:
        rk = B2.shape[3]
        A1 = rank_mask_A(A1, adapter_ranks, rk)
        B1 = rank_mask_B(B1, adapter_ranks)
        A2 = rank_mask_A(A2, adapter_ranks, rk)
        B2 = rank_mask_B(B2, adapter_ranks)

    y = np.zeros((T, X.shape[1]))
    tt, jj = np.nonzero(ok)
    if tt.size == 0:
        return y
    ee = ids_[tt, jj]
    ll = ad[tt]
    keys = ee * (L + 1) + (ll + 1)
    cur_e, W1e, W2e = -1, None, None
    for key in np.unique(keys):  # ascending: all groups of one expert are adjacent
        sel = keys == key
        e, l = int(key // (L + 1)), int(key % (L + 1)) - 1
        if e != cur_e:
            cur_e, W1e, W2e = e, as_f64(W1[e]), as_f64(W2[e])
        ts, js = tt[sel], jj[sel]
        Xg = X[ts]
        g = Xg @ W1e.T
        if l >= 0 and gate_up_slices == 1:
            g = g + (Xg @ as_f64(A1[l, e]).T) @ as_f64(B1[l, e]).T
        elif l >= 0:
            A1le, B1le = as_f64(A1[l, e]), as_f64(B1[l, e])
            r1, I1 = A1le.shape[0] // 2, B1le.shape[0] // 2
            g[:, :I1] += (Xg @ A1le[:r1].T) @ B1le[:I1].T
            g[:, I1:] += (Xg @ A1le[r1:].T) @ B1le[I1:].T
        h = swiglu(g)
        o = h @ W2e.T
        if l >= 0:
            o = o + (h @ as_f64(A2[l, e]).T) @ as_f64(B2[l, e]).T
        np.add.at(y, ts, wf[ts, js][:, None] * o)
    return y


def moe_lora_layer_scalar(x, W1, W2, ids, w, token_adapter=None, A1=None, B1=None, A2=None,
                          B2=None) -> np.ndarray:
    """The same layer as explicit scalar loops over plain Python floats.

    Brute force for tiny shapes only; every sum is written out term by term.
    """
    X = as_f64(x).tolist()
    ids_ = as_i64(ids).tolist()
    wf = as_f64(w).tolist()
    W1f = as_f64(W1)
    W2f = as_f64(W2)
    E, twoI, H = W1f.shape
    I = twoI // 2
    L = 0 if A1 is None else A1.shape[0]
    r = 0 if A1 is None else A1.shape[2]
    W1l, W2l = W1f.tolist(), W2f.tolist()
    if L:
        A1l, B1l = as_f64(A1).tolist(), as_f64(B1).tolist()
        A2l, B2l = as_f64(A2).tolist(), as_f64(B2).tolist()
    T = len(X)
    k = len(ids_[0]) if T else 0
    ad = [-1] * T if (token_adapter is None or L == 0) else as_i64(token_adapter).tolist()
    y = [[0.0] * H for _ in range(T)]
    for t in range(T):
        l = ad[t]
        if not (-1 <= l < L):
            continue
        for j in range(k):
            e = ids_[t][j]
            if not (0 <= e < E):
                continue
            g = [0.0] * twoI
            for n in range(twoI):
                acc = 0.0
                for c in range(H):
                    acc += X[t][c] * W1l[e][n][c]
                g[n] = acc
            if l >= 0:
                z = [0.0] * r
                for q in range(r):
                    acc = 0.0
                    for c in range(H):
                        acc += X[t][c] * A1l[l][e][q][c]
                    z[q] = acc
                for n in range(twoI):
                    acc = 0.0
                    for q in range(r):
                        acc += z[q] * B1l[l][e][n][q]
                    g[n] += acc
            h = [0.0] * I
            for n in range(I):
                gate = g[n]
                # silu(gate) -> 0 as gate -> -inf; math.exp overflows below -709
                sg = gate / (1.0 + math.exp(-gate)) if gate > -700.0 else 0.0
                h[n] = sg * g[I + n]
            o = [0.0] * H
            for n in range(H):
                acc = 0.0
                for c in range(I):
                    acc += h[c] * W2l[e][n][c]
                o[n] = acc
            if l >= 0:
                z = [0.0] * r
                for q in range(r):
                    acc = 0.0
                    for c in range(I):
                        acc += h[c] * A2l[l][e][q][c]
                    z[q] = acc
                for n in range(H):
                    acc = 0.0
                    for q in range(r):
                        acc += z[q] * B2l[l][e][n][q]
                    o[n] += acc
            for n in range(H):
                y[t][n] += wf[t][j] * o[n]
    return np.array(y, dtype=np.float64).reshape(T, H)
