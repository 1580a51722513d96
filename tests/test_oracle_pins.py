"""Pins of the fp64 oracle to facts outside itself (CPU only).

Each pin checks the oracle against something it does not compute itself:
hand-worked values (tests/golden), closed forms, brute force by a different
algorithm, or textbook special cases. The planted-mistake tests at the end
show that a plausible error in the oracle trips at least one pin.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import moe_lora as om
from workloads import WORKLOAD_NAMES, make_layer_inputs, make_workload_inputs, make_workload_routing

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(1e-300, float(np.max(np.abs(b)))))


# ----------------------------------------------------------------------------
# pin functions (raise AssertionError when the oracle is wrong)
# ----------------------------------------------------------------------------
def _two_slice_weights(inp, seed):
    """Separate gate and up adapters for a workload, and the same map written as one
    adapter of rank 2r: A stacked, B block-diagonal (gate rows [B_g | 0], up rows
    [0 | B_u])."""
    rng = np.random.default_rng(seed)
    L, E, r, H = inp.A1.shape
    I2 = inp.B1.shape[2]
    A1s = torch.from_numpy(rng.standard_normal((L, E, 2 * r, H)) * 0.1)
    B1 = torch.from_numpy(rng.standard_normal((L, E, I2, r)) * 0.1)
    B1bd = torch.zeros((L, E, I2, 2 * r), dtype=torch.float64)
    B1bd[:, :, : I2 // 2, :r] = B1[:, :, : I2 // 2]
    B1bd[:, :, I2 // 2:, r:] = B1[:, :, I2 // 2:]
    return A1s, B1, B1bd



def pin_route_golden(golden_dir):
    with open(os.path.join(golden_dir, "route_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        lg = np.array([[float(v) for v in row] for row in c["logits"]], dtype=np.float32)
        ids, w = oracle.route_topk_softmax(torch.from_numpy(lg), c["k"])
        assert ids.tolist() == c["ids"], (ids.tolist(), c["ids"])
        np.testing.assert_allclose(w, np.array(c["w"]), rtol=0, atol=1e-15)


def pin_route_selection_bruteforce(seed=0):
    """Top-k by repeated selection of the maximum (a different algorithm)."""
    rng = np.random.default_rng(seed)
    for _ in range(30):
        T, E = int(rng.integers(1, 6)), int(rng.integers(1, 12))
        k = int(rng.integers(1, E + 1))
        lg = rng.integers(-3, 4, size=(T, E)).astype(np.float32)  # many ties
        ids, w = oracle.route_topk_softmax(torch.from_numpy(lg), k)
        for t in range(T):
            left = list(range(E))
            exp_ids = []
            for _j in range(k):
                best = left[0]
                for e in left[1:]:
                    if lg[t, e] > lg[t, best]:
                        best = e
                exp_ids.append(best)
                left.remove(best)
            assert ids[t].tolist() == exp_ids
            vals = [float(lg[t, e]) for e in exp_ids]
            den = sum(math.exp(v - vals[0]) for v in vals)
            for j in range(k):
                assert abs(w[t, j] - math.exp(vals[j] - vals[0]) / den) < 1e-15
            assert abs(w[t].sum() - 1.0) < 1e-15


def pin_align_golden(golden_dir):
    with open(os.path.join(golden_dir, "align_example.json")) as f:
        g = json.load(f)
    for c in g["cases"]:
        al = oracle.align(np.array(g["ids"]), np.array(g["token_adapter"]), g["E"], g["L"],
                          c["bm_base"], c["bm_lora"])
        assert al["err"] == 0
        assert al["sorted_slots"][: al["n_valid"]].tolist() == g["sorted_slots"]
        assert al["slot_row"].tolist() == g["slot_row"]
        assert al["expert_begin"].tolist() == g["expert_begin"]
        assert [list(t) for t in al["tiles"]] == c["tiles"]
        assert [list(b) for b in al["lora_blocks"]] == c["lora_blocks"]


def _align_bruteforce(ids, ad, E, L):
    """Bucket by explicit nested loops over expert, adapter, slot."""
    T, k = ids.shape
    order = []
    for e in range(E):
        for l in range(-1, L):
            for s in range(T * k):
                if ids[s // k, s % k] == e and ad[s // k] == l:
                    order.append(s)
    return order


def pin_align_bruteforce(seed=1):
    rng = np.random.default_rng(seed)
    for _ in range(40):
        T, k, E, L = (int(rng.integers(1, 5)), int(rng.integers(1, 4)),
                      int(rng.integers(1, 6)), int(rng.integers(0, 4)))
        ids = rng.integers(0, E, size=(T, k))
        ad = rng.integers(-1, L, size=T) if L > 0 else np.full(T, -1)
        bm_b, bm_l = int(rng.integers(1, 5)), int(rng.integers(1, 5))
        al = oracle.align(ids, ad, E, L, bm_b, bm_l)
        order = _align_bruteforce(ids, ad, E, L)
        assert al["sorted_slots"][: al["n_valid"]].tolist() == order
        assert al["n_valid"] == T * k
        for row, s in enumerate(order):
            assert al["slot_row"][s] == row
        # every LoRA row appears in exactly one block, blocks never straddle (e, l)
        covered = []
        for (rb, rows, e, l) in al["lora_blocks"]:
            assert 1 <= rows <= bm_l and l >= 0
            for row in range(rb, rb + rows):
                s = order[row]
                assert ids[s // k, s % k] == e and ad[s // k] == l
                covered.append(row)
        assert covered == [row for row, s in enumerate(order) if ad[s // k] >= 0]
        tcov = []
        for (e, rb, rows) in al["tiles"]:
            assert 1 <= rows <= bm_b
            for row in range(rb, rb + rows):
                s = order[row]
                assert ids[s // k, s % k] == e
                tcov.append(row)
        assert tcov == list(range(T * k))


def pin_align_invalid_ids():
    ids = np.array([[0, 5], [1, -1]])
    ad = np.array([0, 3])
    al = oracle.align(ids, ad, 4, 2, 4, 4)
    # slot 1 has expert 5 (bad); token 1 has adapter 3 (bad) -> slots 2, 3 dropped
    assert al["err"] == (om.ERR_EXPERT_RANGE | om.ERR_ADAPTER_RANGE)
    assert al["n_valid"] == 1 and al["sorted_slots"][0] == 0
    assert al["slot_row"].tolist() == [0, -1, -1, -1]


def pin_layer_scalar_vs_vectorised(inp):
    ids, w = oracle.route_topk_softmax(inp.logits, inp.k)
    ref = oracle.moe_lora_layer_scalar(inp.x, inp.W1, inp.W2, ids, w, inp.token_adapter,
                                       inp.A1, inp.B1, inp.A2, inp.B2)
    vec = oracle.moe_lora_layer(inp.x, inp.W1, inp.W2, ids, w, inp.token_adapter,
                                inp.A1, inp.B1, inp.A2, inp.B2)
    assert _rel(vec, ref) <= 1e-12, _rel(vec, ref)


def pin_dense_swiglu_mlp(seed=3):
    """E = 1, k = 1, w = 1, no adapter: the textbook gated MLP."""
    inp = make_layer_inputs(T=5, H=24, I=40, E=1, k=1, L=0, r=1, seed=seed)
    X = oracle.as_f64(inp.x)
    W1 = oracle.as_f64(inp.W1)[0]
    Wg, Wu = W1[:40], W1[40:]
    Wd = oracle.as_f64(inp.W2)[0]
    gate = X @ Wg.T
    expect = (gate * (1.0 / (1.0 + np.exp(-gate))) * (X @ Wu.T)) @ Wd.T
    ids = np.zeros((5, 1), dtype=np.int32)
    w = np.ones((5, 1))
    y = oracle.moe_lora_layer(inp.x, inp.W1, inp.W2, ids, w)
    assert _rel(y, expect) <= 1e-13


def pin_shrink_expand_dense(seed=4):
    """Shrink then expand equals x (A B) with A B formed densely (pages: y = xW + xAB)."""
    inp = make_layer_inputs(T=6, H=48, I=32, E=3, k=2, L=2, r=4, seed=seed,
                            adapters=[0, 1, 1, 0, 1, 0])
    ids, w = oracle.route_topk_softmax(inp.logits, inp.k)
    al = oracle.align(ids, inp.token_adapter, inp.E, inp.L, 4, 4)
    Z = oracle.lora_shrink(inp.x, inp.A1, al, rows_are_slots=False)
    D = oracle.lora_delta_rows(Z, inp.B1, al)
    X = oracle.as_f64(inp.x)
    A1 = oracle.as_f64(inp.A1)
    B1 = oracle.as_f64(inp.B1)
    for row in range(al["n_valid"]):
        s = int(al["sorted_slots"][row])
        e, l = int(al["row_expert"][row]), int(al["row_adapter"][row])
        dense = A1[l, e].T @ B1[l, e].T          # pages' A (h_in x r) times B (r x h_out)
        assert _rel(D[row], X[s // inp.k] @ dense) <= 1e-12


def pin_rank1_closed_form(seed=5):
    """r = 1: A = a^T, B = b gives delta = (x . a) b."""
    rng = np.random.default_rng(seed)
    H, N = 17, 9
    a = rng.standard_normal(H)
    b = rng.standard_normal(N)
    x = rng.standard_normal((3, H))
    A = a.reshape(1, 1, 1, H)
    B = b.reshape(1, 1, N, 1)
    ids = np.zeros((3, 1), dtype=np.int64)
    ad = np.zeros(3, dtype=np.int64)
    al = oracle.align(ids, ad, 1, 1, 8, 8)
    Z = oracle.lora_shrink(x, A, al, rows_are_slots=False)
    D = oracle.lora_delta_rows(Z, B, al)
    for t in range(3):
        dot = sum(float(x[t, c]) * float(a[c]) for c in range(H))
        assert _rel(D[al["slot_row"][t]], dot * b) <= 1e-13


def pin_lora_linearity(seed=6):
    inp = make_layer_inputs(T=6, H=32, I=24, E=2, k=2, L=2, r=4, seed=seed,
                            adapters=[0, 1, 1, 0, 1, 0])
    ids, w = oracle.route_topk_softmax(inp.logits, inp.k)
    al = oracle.align(ids, inp.token_adapter, inp.E, inp.L, 4, 4)
    Z = oracle.lora_shrink(inp.x, inp.A1, al, rows_are_slots=False)
    D1 = oracle.lora_delta_rows(Z, inp.B1, al)
    D2 = oracle.lora_delta_rows(Z, 2.0 * oracle.as_f64(inp.B1), al)
    assert _rel(D2, 2.0 * D1) <= 1e-15
    Zc = oracle.lora_shrink(inp.x, 4.0 * oracle.as_f64(inp.A1), al, rows_are_slots=False)
    Dc = oracle.lora_delta_rows(Zc, oracle.as_f64(inp.B1) / 4.0, al)
    assert _rel(Dc, D1) <= 1e-15


def pin_base_reductions(seed=7):
    """B = 0 or every adapter -1 leaves exactly the base MoE."""
    inp = make_layer_inputs(T=7, H=32, I=24, E=3, k=2, L=3, r=4, seed=seed)
    ids, w = oracle.route_topk_softmax(inp.logits, inp.k)
    base = oracle.moe_lora_layer(inp.x, inp.W1, inp.W2, ids, w)
    none = torch.full((inp.T,), -1, dtype=torch.int32)
    y_none = oracle.moe_lora_layer(inp.x, inp.W1, inp.W2, ids, w, none,
                                   inp.A1, inp.B1, inp.A2, inp.B2)
    assert np.array_equal(y_none, base)
    zB1 = torch.zeros_like(inp.B1)
    zB2 = torch.zeros_like(inp.B2)
    y_zero = oracle.moe_lora_layer(inp.x, inp.W1, inp.W2, ids, w, inp.token_adapter,
                                   inp.A1, zB1, inp.A2, zB2)
    assert _rel(y_zero, base) <= 1e-14
    y_lora = oracle.moe_lora_layer(inp.x, inp.W1, inp.W2, ids, w, inp.token_adapter,
                                   inp.A1, inp.B1, inp.A2, inp.B2)
    assert _rel(y_lora, base) > 1e-4  # the adapters are visible


def pin_permutation(seed=8):
    inp = make_layer_inputs(T=9, H=32, I=24, E=4, k=2, L=2, r=4, seed=seed)
    ids, w = oracle.route_topk_softmax(inp.logits, inp.k)
    y = oracle.moe_lora_layer(inp.x, inp.W1, inp.W2, ids, w, inp.token_adapter,
                              inp.A1, inp.B1, inp.A2, inp.B2)
    perm = np.random.default_rng(seed).permutation(inp.T)
    yp = oracle.moe_lora_layer(inp.x[perm], inp.W1, inp.W2, ids[perm], w[perm],
                               inp.token_adapter[perm], inp.A1, inp.B1, inp.A2, inp.B2)
    assert _rel(yp, y[perm]) <= 1e-14


def pin_per_op_chain(inp, bm_base=4, bm_lora=2):
    """gather -> base GEMM -> shrink/expand+SwiGLU -> down -> shrink/expand+combine."""
    ids, w = oracle.route_topk_softmax(inp.logits, inp.k)
    al = oracle.align(ids, inp.token_adapter, inp.E, inp.L, bm_base, bm_lora)
    xs = oracle.gather_rows(inp.x, al)
    G = oracle.grouped_gemm(xs, inp.W1, al)
    Z1 = oracle.lora_shrink(inp.x, inp.A1, al, rows_are_slots=False)
    h = oracle.lora_expand_add(Z1, inp.B1, al, G, epilogue=1)
    O = oracle.grouped_gemm(h, inp.W2, al)
    Z2 = oracle.lora_shrink(h, inp.A2, al, rows_are_slots=True)
    y = oracle.lora_expand_add(Z2, inp.B2, al, O, epilogue=2, w=w)
    ref = oracle.moe_lora_layer(inp.x, inp.W1, inp.W2, ids, w, inp.token_adapter,
                                inp.A1, inp.B1, inp.A2, inp.B2)
    assert _rel(y, ref) <= 1e-12
    # epilogue 0 then SwiGLU by hand equals epilogue 1
    G0 = oracle.lora_expand_add(Z1, inp.B1, al, G, epilogue=0)
    I = G0.shape[1] // 2
    assert _rel(G0[:, :I] / (1.0 + np.exp(-G0[:, :I])) * G0[:, I:], h) <= 1e-14


# ----------------------------------------------------------------------------
# tests
# ----------------------------------------------------------------------------
def test_route_golden(golden_dir):
    pin_route_golden(golden_dir)


def test_route_selection_bruteforce():
    pin_route_selection_bruteforce()


def test_align_golden(golden_dir):
    pin_align_golden(golden_dir)


def test_align_bruteforce():
    pin_align_bruteforce()


def test_align_invalid_ids():
    pin_align_invalid_ids()


@pytest.mark.parametrize("name", WORKLOAD_NAMES)
def test_align_invariants_on_workloads(name):
    lg, ad, c = make_workload_routing(name)
    ids, _ = oracle.route_topk_softmax(lg, c["k"])
    al = oracle.align(ids, ad, c["E"], c["L"], 64, 16)
    S = c["T"] * c["k"]
    n = al["n_valid"]
    assert n == S and al["err"] == 0
    ss = al["sorted_slots"][:n]
    assert sorted(ss.tolist()) == list(range(S))
    keys = [(int(al["row_expert"][i]), int(al["row_adapter"][i]), int(ss[i])) for i in range(n)]
    assert keys == sorted(keys)
    counts = np.bincount(ids.reshape(-1), minlength=c["E"])
    assert np.array_equal(np.diff(al["expert_begin"]), counts)
    lrows = sum(b[1] for b in al["lora_blocks"])
    assert lrows == al["n_lora_rows"] == int((ad.numpy() >= 0).sum()) * c["k"]


def test_layer_scalar_vs_vectorised_tiny_workload():
    pin_layer_scalar_vs_vectorised(make_workload_inputs("tiny"))


@pytest.mark.parametrize("seed", range(20))
def test_layer_scalar_vs_vectorised_random(seed):
    rng = np.random.default_rng(100 + seed)
    E = int(rng.integers(1, 5))
    inp = make_layer_inputs(T=int(rng.integers(1, 6)), H=int(rng.integers(1, 20)),
                            I=int(rng.integers(1, 12)), E=E, k=int(rng.integers(1, E + 1)),
                            L=int(rng.integers(0, 3)), r=int(rng.integers(1, 5)),
                            seed=200 + seed, lora_std=None)
    pin_layer_scalar_vs_vectorised(inp)


def pin_two_slice_gate_up(inp, seed):
    """Separate gate and up adapters equal one adapter of twice the rank with a stacked A
    and a block-diagonal B: the layer and the epilogue-3 expand against the (pinned)
    one-slice forms."""
    ids, w = oracle.route_topk_softmax(inp.logits, inp.k)
    A1s, B1, B1bd = _two_slice_weights(inp, seed)
    y2 = oracle.moe_lora_layer(inp.x, inp.W1, inp.W2, ids, w, inp.token_adapter, A1s, B1,
                               inp.A2, inp.B2, gate_up_slices=2)
    y1 = oracle.moe_lora_layer(inp.x, inp.W1, inp.W2, ids, w, inp.token_adapter, A1s, B1bd,
                               inp.A2, inp.B2)
    assert _rel(y2, y1) < 1e-12, _rel(y2, y1)
    al = oracle.align(torch.as_tensor(ids, dtype=torch.int32), inp.token_adapter, inp.E, inp.L, 16, 4)
    Z = oracle.lora_shrink(inp.x, A1s, al, rows_are_slots=False)
    G = np.random.default_rng(seed + 1).standard_normal((al["n_valid"], B1.shape[2]))
    h3 = oracle.lora_expand_add(Z, B1, al, G, epilogue=3)
    h1 = oracle.lora_expand_add(Z, B1bd, al, G, epilogue=1)
    assert _rel(h3, h1) < 1e-12, _rel(h3, h1)
    # a zero up adapter leaves the up half to the base output
    B1g = B1.clone()
    B1g[:, :, B1.shape[2] // 2:] = 0
    D = om.lora_delta_rows(Z, B1g, al, slices=2)
    assert np.all(D[:, B1.shape[2] // 2:] == 0)


@pytest.mark.parametrize("seed", range(3))
def test_two_slice_gate_up(seed):
    pin_two_slice_gate_up(make_layer_inputs(T=13, H=24, I=10, E=3, k=2, L=3, r=3,
                                            seed=400 + seed, adapters="uniform_with_none"), 500 + seed)


def test_planted_two_slice_swap(monkeypatch):
    """Feeding the up z to the gate columns (and the gate z to the up columns) trips the pin."""
    real = om.lora_delta_rows

    def swapped(Z, B, al, slices=1, adapter_ranks=None):
        if slices == 1:
            return real(Z, B, al, 1, adapter_ranks)
        Zf = np.array(om.as_f64(Z))
        r = om.as_f64(B).shape[3]
        Zs = Zf.copy()
        Zs[:, :r], Zs[:, r: 2 * r] = Zf[:, r: 2 * r], Zf[:, :r]
        return real(Zs, B, al, 2, adapter_ranks)

    monkeypatch.setattr(om, "lora_delta_rows", swapped)
    with pytest.raises(AssertionError):
        pin_two_slice_gate_up(make_layer_inputs(T=13, H=24, I=10, E=3, k=2, L=3, r=3, seed=400,
                                                adapters="uniform_with_none"), 500)


def pin_adapter_ranks(inp, ranks, slices=1, seed=0):
    """Adapters of their own ranks, by brute force over slots with truncated weights: adapter
    l of rank r_l uses A[:r_l] (per slice) and B[:, :r_l]. Checks the layer and the
    shrink / expand ops the GPU kernels are compared with."""
    X = om.as_f64(inp.x)
    W1, W2 = om.as_f64(inp.W1), om.as_f64(inp.W2)
    rng = np.random.default_rng(seed)
    r = inp.r
    A1 = torch.from_numpy(rng.standard_normal((inp.L, inp.E, slices * r, inp.H)) * 0.1)
    B1, A2, B2 = om.as_f64(inp.B1), om.as_f64(inp.A2), om.as_f64(inp.B2)
    ids, w = oracle.route_topk_softmax(inp.logits, inp.k)
    ad = om.as_i64(inp.token_adapter)
    A1f = om.as_f64(A1)
    I = W2.shape[2]
    y = np.zeros_like(X)
    for t in range(inp.T):
        for j in range(inp.k):
            e, l = int(ids[t, j]), int(ad[t])
            g = W1[e] @ X[t]
            if l >= 0:
                rl = int(ranks[l])
                if slices == 1:
                    g = g + B1[l, e][:, :rl] @ (A1f[l, e][:rl] @ X[t])
                else:
                    g[:I] += B1[l, e][:I, :rl] @ (A1f[l, e][:rl] @ X[t])
                    g[I:] += B1[l, e][I:, :rl] @ (A1f[l, e][r: r + rl] @ X[t])
            h = g[:I] / (1.0 + np.exp(-g[:I])) * g[I:]
            o = W2[e] @ h
            if l >= 0:
                o = o + B2[l, e][:, :rl] @ (A2[l, e][:rl] @ h)
            y[t] += float(w[t, j]) * o
    yo = oracle.moe_lora_layer(inp.x, inp.W1, inp.W2, ids, w, inp.token_adapter, A1, inp.B1,
                               inp.A2, inp.B2, gate_up_slices=slices,
                               adapter_ranks=torch.as_tensor(ranks))
    assert _rel(yo, y) < 1e-12, _rel(yo, y)
    # the ops: shrink z (zero past r_l) and the expand delta
    al = oracle.align(torch.as_tensor(ids, dtype=torch.int32), inp.token_adapter, inp.E, inp.L, 16, 4)
    Z = oracle.lora_shrink(inp.x, A1, al, False, adapter_ranks=torch.as_tensor(ranks), rank=r)
    Zb = np.zeros_like(Z)
    D = np.zeros((al["n_valid"], B1.shape[2]))
    for row in range(al["n_valid"]):
        l = int(al["row_adapter"][row])
        if l < 0:
            continue
        e, sl = int(al["row_expert"][row]), int(al["sorted_slots"][row])
        rl = int(ranks[l])
        for c in range(slices):
            Zb[sl, c * r: c * r + rl] = A1f[l, e][c * r: c * r + rl] @ X[sl // inp.k]
        if slices == 1:
            D[row] = B1[l, e][:, :rl] @ Zb[sl, :rl]
        else:
            D[row, :I] = B1[l, e][:I, :rl] @ Zb[sl, :rl]
            D[row, I:] = B1[l, e][I:, :rl] @ Zb[sl, r: r + rl]
    assert _rel(Z, Zb) < 1e-12, _rel(Z, Zb)
    Dq = om.lora_delta_rows(Zb, inp.B1, al, slices=slices, adapter_ranks=torch.as_tensor(ranks))
    assert _rel(Dq, D) < 1e-12, _rel(Dq, D)


@pytest.mark.parametrize("slices", [1, 2])
def test_adapter_ranks(slices):
    inp = make_layer_inputs(T=9, H=20, I=12, E=3, k=2, L=4, r=6, seed=600 + slices,
                            adapters="uniform_with_none")
    pin_adapter_ranks(inp, [6, 3, 0, 5], slices, seed=700 + slices)
    # full ranks reproduce the unranked oracle
    ids, w = oracle.route_topk_softmax(inp.logits, inp.k)
    y0 = oracle.moe_lora_layer(inp.x, inp.W1, inp.W2, ids, w, inp.token_adapter, inp.A1, inp.B1,
                               inp.A2, inp.B2)
    y1 = oracle.moe_lora_layer(inp.x, inp.W1, inp.W2, ids, w, inp.token_adapter, inp.A1, inp.B1,
                               inp.A2, inp.B2, adapter_ranks=torch.full((4,), 6))
    assert _rel(y1, y0) == 0.0


def test_planted_rank_off_by_one(monkeypatch):
    """Keeping one row too many of a truncated adapter trips the rank pin."""
    real = om.rank_mask_A

    def loose(A, adapter_ranks, rank):
        if adapter_ranks is None:
            return real(A, None, rank)
        return real(A, [min(int(v) + 1, rank) for v in om.as_i64(adapter_ranks)], rank)

    monkeypatch.setattr(om, "rank_mask_A", loose)
    inp = make_layer_inputs(T=9, H=20, I=12, E=3, k=2, L=4, r=6, seed=601, adapters="uniform_with_none")
    with pytest.raises(AssertionError):
        pin_adapter_ranks(inp, [6, 3, 0, 5], 1, seed=701)


def test_dense_swiglu_mlp():
    pin_dense_swiglu_mlp()


def test_shrink_expand_dense():
    pin_shrink_expand_dense()


def test_rank1_closed_form():
    pin_rank1_closed_form()


def test_lora_linearity():
    pin_lora_linearity()


def test_base_reductions():
    pin_base_reductions()


def test_permutation():
    pin_permutation()


@pytest.mark.parametrize("seed", range(3))
def test_per_op_chain(seed):
    pin_per_op_chain(make_layer_inputs(T=11, H=40, I=24, E=3, k=2, L=3, r=4, seed=300 + seed))


def test_even_k_fixture(golden_dir):
    with open(os.path.join(golden_dir, "even_k_example.json")) as f:
        g = json.load(f)
    bk, K = g["BLOCK_SIZE_K"], g["K"]
    assert -(-K // bk) == g["blocks"]
    assert g["blocks"] * bk - K == g["second_block_out_of_range"]
    assert (K % bk == 0) == g["even_k"]


# ----------------------------------------------------------------------------
# planted mistakes: each must trip at least one pin
# ----------------------------------------------------------------------------
def _trips(fn, *a):
    try:
        fn(*a)
    except (AssertionError, ValueError, IndexError):
        return True
    return False


def test_planted_gate_up_swap(monkeypatch):
    def bad(g):
        I = g.shape[-1] // 2
        return om.silu(g[..., I:]) * g[..., :I]
    monkeypatch.setattr(om, "swiglu", bad)
    assert _trips(pin_dense_swiglu_mlp)


def test_planted_sigmoid_for_silu(monkeypatch):
    monkeypatch.setattr(om, "silu", lambda v: 1.0 / (1.0 + np.exp(-v)))
    assert _trips(pin_dense_swiglu_mlp)


def test_planted_dropped_down_lora(monkeypatch):
    orig = om.moe_lora_layer

    def bad(x, W1, W2, ids, w, token_adapter=None, A1=None, B1=None, A2=None, B2=None):
        zero = None if B2 is None else torch.zeros_like(B2)
        return orig(x, W1, W2, ids, w, token_adapter, A1, B1, A2, zero)
    monkeypatch.setattr(om, "moe_lora_layer", bad)
    monkeypatch.setattr(oracle, "moe_lora_layer", bad)
    assert _trips(pin_per_op_chain, make_layer_inputs(T=11, H=40, I=24, E=3, k=2, L=3, r=4,
                                                      seed=301))


def test_planted_transposed_lora(monkeypatch):
    def bad(Z, B, al):
        Zf = om.as_f64(Z)
        Bf = om.as_f64(B)
        n = al["n_valid"]
        D = np.zeros((n, Bf.shape[2]))
        for row in range(n):
            l, e = int(al["row_adapter"][row]), int(al["row_expert"][row])
            if l >= 0:
                D[row] = Bf[e % Bf.shape[0], l % Bf.shape[1]] @ Zf[int(al["sorted_slots"][row])]
        return D
    monkeypatch.setattr(om, "lora_delta_rows", bad)
    monkeypatch.setattr(oracle, "lora_delta_rows", bad)
    assert _trips(pin_shrink_expand_dense)


def test_planted_wrong_tie_break(monkeypatch):
    def bad(logits, k):
        lg = om.as_f64(logits)
        ids = np.argsort(-lg[:, ::-1], axis=1, kind="stable")[:, :k]
        ids = lg.shape[1] - 1 - ids
        sel = np.take_along_axis(lg, ids, axis=1)
        ex = np.exp(sel - sel[:, :1])
        return ids.astype(np.int32), ex / ex.sum(axis=1, keepdims=True)
    monkeypatch.setattr(oracle, "route_topk_softmax", bad)
    assert _trips(pin_route_selection_bruteforce)


def test_planted_unstable_align(monkeypatch):
    orig = om.align

    def bad(ids, token_adapter, E, L, bm_base, bm_lora):
        al = orig(ids, token_adapter, E, L, bm_base, bm_lora)
        n = al["n_valid"]
        if n >= 2:  # reverse slot order inside the first (e, l) segment
            e0, l0 = al["row_expert"][0], al["row_adapter"][0]
            end = 0
            while end < n and al["row_expert"][end] == e0 and al["row_adapter"][end] == l0:
                end += 1
            al["sorted_slots"][:end] = al["sorted_slots"][:end][::-1].copy()
        return al
    monkeypatch.setattr(oracle, "align", bad)
    assert _trips(pin_align_bruteforce)


def test_planted_combine_weight_index(monkeypatch):
    def bad(O_rows, w, al):
        O = om.as_f64(O_rows)
        wf = om.as_f64(w)
        T, k = al["T"], al["k"]
        y = np.zeros((T, O.shape[1]))
        for t in range(T):
            for j in range(k):
                row = int(al["slot_row"][t * k + j])
                if row >= 0:
                    y[t] += wf[t, k - 1 - j] * O[row]
        return y
    monkeypatch.setattr(om, "combine", bad)
    assert _trips(pin_per_op_chain, make_layer_inputs(T=11, H=40, I=24, E=3, k=2, L=3, r=4,
                                                      seed=302))
