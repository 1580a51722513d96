"""Routing and alignment on the GPU: bit-exact against the oracle."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import WORKLOAD_NAMES, make_workload_routing

from gpu_util import dev, need_gpu

pytestmark = pytest.mark.gpu


def _check_align(m, ids, ad, E, L, bm_base, bm_lora):
    """Runs the GPU align and compares every array with the oracle, bit for bit."""
    ids_t = torch.as_tensor(np.asarray(ids), dtype=torch.int32)
    ad_t = None if ad is None else torch.as_tensor(np.asarray(ad), dtype=torch.int32)
    al = m.moe_lora_align(dev(ids_t), dev(ad_t), E, L, bm_base, bm_lora)
    ref = oracle.align(ids_t, ad_t, E, L, bm_base, bm_lora)
    h = al.header()
    n = ref["n_valid"]
    assert h["err"] == ref["err"]
    assert h["n_valid"] == n
    assert h["n_tiles"] == len(ref["tiles"])
    assert h["n_lora_blocks"] == len(ref["lora_blocks"])
    assert h["n_lora_rows"] == ref["n_lora_rows"]
    assert al.sorted_slots().cpu().numpy().tolist() == ref["sorted_slots"].tolist()
    assert al.slot_row().cpu().numpy().tolist() == ref["slot_row"].tolist()
    assert al.row_expert().cpu().numpy()[:n].tolist() == ref["row_expert"].tolist()
    assert al.row_adapter().cpu().numpy()[:n].tolist() == ref["row_adapter"].tolist()
    assert al.expert_begin().cpu().numpy().tolist() == ref["expert_begin"].tolist()
    tiles = al.tiles().cpu().numpy()[: h["n_tiles"], :3].tolist()
    assert tiles == [list(t) for t in ref["tiles"]]
    blocks = al.lora_blocks().cpu().numpy()[: h["n_lora_blocks"]].tolist()
    assert blocks == [list(b) for b in ref["lora_blocks"]]
    return al


# ---------------------------------------------------------------- routing
def test_route_golden_cases(golden_dir):
    m = need_gpu()
    with open(os.path.join(golden_dir, "route_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        lg = torch.tensor([[float(v) for v in row] for row in c["logits"]], dtype=torch.float32)
        ids, w = m.moe_topk_softmax(dev(lg), c["k"])
        assert ids.cpu().tolist() == c["ids"]
        np.testing.assert_allclose(w.cpu().numpy(), np.array(c["w"]), rtol=0, atol=1e-6)


@pytest.mark.parametrize("name", WORKLOAD_NAMES)
def test_route_workloads_bitexact_ids(name):
    m = need_gpu()
    lg, _, c = make_workload_routing(name)
    ids, w = m.moe_topk_softmax(dev(lg), c["k"])
    rid, rw = oracle.route_topk_softmax(lg, c["k"])
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=0, atol=2e-6)


@pytest.mark.parametrize("E,k", [(1, 1), (5, 3), (32, 32), (33, 4), (100, 8), (257, 2),
                                 (1024, 16)])
def test_route_ties_and_shapes(E, k):
    m = need_gpu()
    rng = np.random.default_rng(E * 100 + k)
    T = 37
    lg = rng.integers(-2, 3, size=(T, E)).astype(np.float32)  # many ties
    lg[3, :] = np.nan
    lg[4, ::2] = -np.inf
    lgt = torch.from_numpy(lg)
    ids, w = m.moe_topk_softmax(dev(lgt), k)
    rid, rw = oracle.route_topk_softmax(lgt, k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    fin = np.isfinite(rw).all(axis=1)
    np.testing.assert_allclose(w.cpu().numpy()[fin], rw[fin], rtol=0, atol=2e-6)


def test_route_empty():
    m = need_gpu()
    ids, w = m.moe_topk_softmax(torch.empty((0, 8), dtype=torch.float32, device="cuda"), 2)
    assert ids.shape == (0, 2)


# ---------------------------------------------------------------- align
@pytest.mark.parametrize("name", WORKLOAD_NAMES)
@pytest.mark.parametrize("bm_base,bm_lora", [(16, 16), (64, 1), (256, 7)])
def test_align_workloads(name, bm_base, bm_lora):
    m = need_gpu()
    lg, ad, c = make_workload_routing(name)
    ids, _ = oracle.route_topk_softmax(lg, c["k"])
    _check_align(m, ids, ad, c["E"], c["L"], bm_base, bm_lora)


def test_align_edge_cases():
    m = need_gpu()
    rng = np.random.default_rng(7)
    # every token adapter-free
    ids = rng.integers(0, 8, size=(40, 2))
    _check_align(m, ids, np.full(40, -1), 8, 4, 16, 16)
    # no adapter array at all
    _check_align(m, ids, None, 8, 0, 16, 16)
    # one expert
    _check_align(m, np.zeros((33, 1)), rng.integers(-1, 3, size=33), 1, 3, 16, 4)
    # one (expert, adapter) pair holds every slot; counts divisible by the tiles
    _check_align(m, np.full((64, 2), 3), np.full(64, 2), 4, 3, 32, 16)
    # a single token
    _check_align(m, np.array([[2, 0, 1]]), np.array([1]), 3, 2, 16, 1)
    # no tokens
    _check_align(m, np.zeros((0, 2)), np.zeros(0), 4, 2, 16, 16)
    # more slots than the shared-memory sort holds (global-memory sort path)
    T = 5000
    ids = np.stack([rng.permutation(16)[:4] for _ in range(T)])
    _check_align(m, ids, rng.integers(-1, 5, size=T), 16, 5, 64, 16)
    # many buckets: E * (L + 1) needs three radix digits
    ids = rng.integers(0, 256, size=(300, 2))
    _check_align(m, ids, rng.integers(-1, 255, size=300), 256, 255, 16, 3)


def test_align_out_of_range_ids_flagged_not_trapped():
    m = need_gpu()
    ids = np.array([[0, 5], [1, -1], [2, 3]])
    ad = np.array([0, 1, 9])
    al = _check_align(m, ids, ad, 4, 2, 16, 16)
    err = m.get_error(al.buf)
    assert err == 3  # expert and adapter range bits
    m.clear_error(al.buf)
    assert m.get_error(al.buf) == 0


def test_align_is_deterministic():
    m = need_gpu()
    lg, ad, c = make_workload_routing("gptoss20b_prefill")
    ids, _ = oracle.route_topk_softmax(lg, c["k"])
    ids_d = dev(torch.as_tensor(ids, dtype=torch.int32))
    a1 = m.moe_lora_align(ids_d, dev(ad), c["E"], c["L"], 256, 16)
    a2 = m.moe_lora_align(ids_d, dev(ad), c["E"], c["L"], 256, 16)
    torch.cuda.synchronize()
    n = a1.header()["n_valid"]
    assert torch.equal(a1.sorted_slots()[:n], a2.sorted_slots()[:n])


def test_align_multi_cta_cases():
    """From 2048 slots on, with at most half as many keys as slots, the align runs on many
    CTAs (local stable sorts of 512 slots, a scan of the (key, CTA) count table,
    placement): bit-exact with the oracle on a partial last CTA, keys needing two radix
    digits, out-of-range ids and adapters, one pair holding every slot, and bm_lora that
    does not divide the segments. Many keys over few slots stay on the one-CTA kernel."""
    m = need_gpu()
    rng = np.random.default_rng(11)
    # partial last CTA (S = 2050), adapters -1..3
    ids = np.stack([rng.permutation(8)[:2] for _ in range(1025)])
    _check_align(m, ids, rng.integers(-1, 4, size=1025), 8, 4, 16, 5)
    # two radix digits: E * (L + 1) + 1 = 1025 keys, S = 3000
    ids = rng.integers(0, 64, size=(1500, 2))
    _check_align(m, ids, rng.integers(-1, 15, size=1500), 64, 15, 32, 3)
    # many keys over few slots (65537 keys, S = 3000): the one-CTA kernel
    ids = rng.integers(0, 256, size=(1500, 2))
    _check_align(m, ids, rng.integers(-1, 255, size=1500), 256, 255, 32, 3)
    # out-of-range expert ids and adapters: slots dropped, bits set
    ids = rng.integers(0, 12, size=(700, 4))
    ids[rng.random(ids.shape) < 0.05] = 99
    ids[3, 1] = -2
    ad = rng.integers(-1, 6, size=700)
    ad[[5, 77]] = [6, -3]
    al = _check_align(m, ids, ad, 12, 6, 64, 16)
    assert m.get_error(al.buf) == 3
    # every slot in one (expert, adapter) pair: one long run across all CTAs
    _check_align(m, np.full((2048, 2), 1), np.full(2048, 0), 4, 2, 256, 16)
    # exactly four full CTAs, no adapters
    _check_align(m, rng.integers(0, 32, size=(512, 4)), None, 32, 0, 128, 16)


@pytest.mark.parametrize("S", [1, 3, 5, 127, 128, 129, 255, 256, 257, 510, 511, 512, 513, 600])
def test_align_rank_sort_sizes(S):
    """Up to 512 slots the one-CTA align places each word by its rank, with up to eight
    lanes sharing a word (8 up to 128 words, 4 up to 256, 2 up to 512) and the words
    padded to whole 16-byte groups; above, the radix sort. Bit-exact with the oracle at
    and around each boundary, at word counts with one to three padding words."""
    m = need_gpu()
    rng = np.random.default_rng(300 + S)
    ids = rng.integers(0, 7, size=(S, 1))
    _check_align(m, ids, rng.integers(-1, 3, size=S), 7, 3, 16, 4)


_ROUTED_SHAPES = {
    # 64 tokens, top-8 of 64 experts (two logits a lane): 512 slots, two lanes a word
    "k8_E64": dict(T=64, H=256, I=128, E=64, k=8, L=4, r=16),
    # 37 tokens, top-3 of 40 experts: 111 slots (one padding word), eight lanes a word
    "T37_k3_E40": dict(T=37, H=256, I=128, E=40, k=3, L=5, r=16),
}


@pytest.mark.parametrize("name", ["gptoss20b_decode", "tiny", "k8_E64", "T37_k3_E40"])
def test_align_routes_in_layer(name):
    """Up to 64 tokens the layer's one-CTA align routes the tokens itself (no route
    launch): the align tables it leaves at the start of the workspace -- the stable sort
    of the routed slots by (expert, adapter, slot), tiles and LoRA blocks -- equal the
    oracle's routing and alignment, bit for bit; so do the routing weights the combine
    read (y against the layer with the route kernel's ids and weights passed in)."""
    m = need_gpu()
    from workloads import make_layer_inputs, make_workload_inputs
    inp = (make_layer_inputs(seed=310 + len(name), **_ROUTED_SHAPES[name])
           if name in _ROUTED_SHAPES else make_workload_inputs(name))
    plan = m.moe_lora_layer_plan(inp.T, inp.k, inp.E, inp.L, inp.H, inp.I, inp.r)
    assert plan["route_in_align"] == 1, plan
    lora = dict(A1=dev(inp.A1), B1=dev(inp.B1), A2=dev(inp.A2), B2=dev(inp.B2))
    ws = m.new_workspace(inp.T, inp.k, inp.E, inp.L, inp.H, inp.I, inp.r)
    args = (dev(inp.x), dev(inp.W1), dev(inp.W2))
    y = m.moe_lora_layer(*args, logits=dev(inp.logits), k=inp.k, token_adapter=dev(inp.token_adapter),
                         workspace=ws, y_fp32=True, **lora)
    torch.cuda.synchronize()
    al = m.Align(ws, inp.T, inp.k, inp.E, inp.L, plan["bm_base"], plan["bm_lora"])
    ids, w = oracle.route_topk_softmax(inp.logits, inp.k)
    ids_t = torch.as_tensor(np.asarray(ids), dtype=torch.int32)
    ref = oracle.align(ids_t, inp.token_adapter, inp.E, inp.L, plan["bm_base"], plan["bm_lora"])
    h = al.header()
    n = ref["n_valid"]
    assert h["err"] == 0 and h["n_valid"] == n
    assert al.sorted_slots().cpu().numpy().tolist() == ref["sorted_slots"].tolist()
    assert al.expert_begin().cpu().numpy().tolist() == ref["expert_begin"].tolist()
    assert al.row_adapter().cpu().numpy()[:n].tolist() == ref["row_adapter"].tolist()
    blocks = al.lora_blocks().cpu().numpy()[: h["n_lora_blocks"]].tolist()
    assert blocks == [list(b) for b in ref["lora_blocks"]]
    # the same layer fed the route kernel's ids and weights: identical y
    rid, rw = m.moe_topk_softmax(dev(inp.logits), inp.k)
    y2 = m.moe_lora_layer(*args, topk_ids=rid, topk_w=rw, token_adapter=dev(inp.token_adapter),
                          y_fp32=True, **lora)
    assert torch.equal(y, y2)
