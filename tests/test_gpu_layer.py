"""The whole fused MoE-LoRA layer on the GPU against the fp64 oracle."""
import functools

import numpy as np
import pytest
import torch

import oracle
from workloads import WORKLOAD_NAMES, make_workload_inputs, make_layer_inputs

from gpu_util import LAYER_RTOL, Guarded, assert_close, dev, f64, need_gpu

pytestmark = pytest.mark.gpu


def run_layer(m, inp, y_fp32=False, adapters=True, B_zero=False, token_adapter=None, **kw):
    lora = {}
    if adapters and inp.L > 0:
        lora = dict(A1=dev(inp.A1), B1=dev(inp.B1), A2=dev(inp.A2), B2=dev(inp.B2))
        if B_zero:
            lora["B1"] = torch.zeros_like(lora["B1"])
            lora["B2"] = torch.zeros_like(lora["B2"])
    ta = inp.token_adapter if token_adapter is None else token_adapter
    y = Guarded((inp.T, inp.H), torch.float32 if y_fp32 else torch.bfloat16)
    m.moe_lora_layer(dev(inp.x), dev(inp.W1), dev(inp.W2), logits=dev(inp.logits), k=inp.k,
                     token_adapter=dev(ta), y=y.t, y_fp32=y_fp32, **lora, **kw)
    y.check()
    return y.t


def oracle_layer(inp, tokens=None, adapters=True, token_adapter=None):
    ids, w = oracle.route_topk_softmax(inp.logits, inp.k)
    ta = inp.token_adapter if token_adapter is None else token_adapter
    sel = slice(None) if tokens is None else tokens
    lora = (inp.A1, inp.B1, inp.A2, inp.B2) if adapters and inp.L > 0 else (None,) * 4
    return oracle.moe_lora_layer(inp.x[sel], inp.W1, inp.W2, ids[sel], w[sel], ta[sel], *lora)


_GPU_Y = {}
_REF_Y = {}


@functools.lru_cache(maxsize=1)
def _inputs(name):
    """A workload's inputs, drawn once for the consecutive tests that use them."""
    return make_workload_inputs(name)


def _workload_y(m, name, expand_mode):
    """The layer's y (bf16) on a workload, computed once per (workload, chain)."""
    key = (name, expand_mode)
    if key not in _GPU_Y:
        inp = _inputs(name)
        plan = m.moe_lora_layer_plan(inp.T, inp.k, inp.E, inp.L, inp.H, inp.I, inp.r,
                                     expand_mode=expand_mode)
        if expand_mode == 1:
            assert plan["fused_expand"] == 0
        _GPU_Y[key] = (run_layer(m, inp, expand_mode=expand_mode).cpu(), plan)
        torch.cuda.empty_cache()
    return _GPU_Y[key]


@pytest.mark.parametrize("expand_mode", [0, 1])
@pytest.mark.parametrize("name,chunk", [(n, c) for n in WORKLOAD_NAMES for c in
                                        (range(4) if n == "gptoss20b_prefill" else range(1))])
def test_layer_workloads(name, chunk, expand_mode):
    """All five workloads through the chain the library picks (expand fused into the grouped
    GEMMs where it applies) and through the chain with separate expand kernels, compared
    with the oracle on every token (the prefill workload's 4096 tokens in four chunks)."""
    m = need_gpu()
    inp = _inputs(name)
    y, plan = _workload_y(m, name, expand_mode)
    n_chunks = 4 if name == "gptoss20b_prefill" else 1
    per = (inp.T + n_chunks - 1) // n_chunks
    tokens = np.arange(chunk * per, min(inp.T, (chunk + 1) * per))
    key = (name, chunk)
    if key not in _REF_Y:
        _REF_Y[key] = oracle_layer(inp, tokens)
    assert_close(y[tokens], _REF_Y[key], LAYER_RTOL, f"{name} chunk {chunk} plan {plan}")


@pytest.mark.parametrize("expand_mode", [0, 1])
def test_dense_multi_lora_workload(expand_mode):
    """Dense multi-LoRA (one expert, top-1) at an 8B-class dense model's size: hidden 4096,
    intermediate 14336, 64 decode tokens over 8 adapters of rank 16 -- the workload the
    bench measures beside the five -- through both chains, every token against the oracle."""
    m = need_gpu()
    inp = _inputs("dense_4096_14336")
    y, plan = _workload_y(m, "dense_4096_14336", expand_mode)
    ref = oracle_layer(inp)
    assert_close(y, ref, LAYER_RTOL, f"dense plan {plan}")


def test_fused_chain_is_picked_where_it_applies():
    """The plan fuses the expand into the grouped GEMMs for the decode and prefill workloads
    (few rows per expert, or long (expert, adapter) runs), not for the 4096/11008 example
    (runs of about four rows: each run's adapter stages multiply a whole token tile) nor for
    separate gate and up adapters or per-adapter ranks, and never when asked for the
    separate kernels."""
    m = need_gpu()
    c = make_workload_inputs("paper_example_4096_11008")
    assert m.moe_lora_layer_plan(c.T, c.k, c.E, c.L, c.H, c.I, c.r)["fused_expand"] == 0
    for name in ("tiny", "gptoss20b_decode", "gptoss20b_prefill"):
        c = make_workload_inputs(name)
        args = (c.T, c.k, c.E, c.L, c.H, c.I, c.r)
        assert m.moe_lora_layer_plan(*args)["fused_expand"] == 1, name
        assert m.moe_lora_layer_plan(*args, expand_mode=1)["fused_expand"] == 0, name
        assert m.moe_lora_layer_plan(*args, gate_up_slices=2)["fused_expand"] == 0, name
        assert m.moe_lora_layer_plan(*args, adapter_ranks=True)["fused_expand"] == 0, name


@pytest.mark.parametrize("shape", ["r8_expert_major", "r24_expert_major", "r64_chunked",
                                   "r128_chunked", "tiles_many_runs", "persistent_r32",
                                   "base_only_tiles", "expert_major_k_tail",
                                   "dense_ksplit8_k_tail"])
def test_fused_expand_shapes(shape):
    """The fused chain on shapes that exercise its cases: ranks that need zero padding to a
    multiple of 16 (8, 24), ranks whose high and low z parts take separate 64-column chunks
    (64, 128), expert-major chunks, token tiles holding many adapter runs (one adapter per
    request of 64 tokens), persistent 128-row tiles, no adapters at all, and expert-major
    64-row chunks with a K tail, and one expert (dense) whose down GEMM splits its K range in
    eight shares of two k-blocks, the last with a 40-column tail. Every token is compared
    with the oracle and with the chain of separate expand kernels."""
    m = need_gpu()
    kw = {"r8_expert_major": dict(T=40, H=128, I=96, E=4, k=2, L=3, r=8),
          "r24_expert_major": dict(T=40, H=128, I=96, E=4, k=2, L=3, r=24),
          "r64_chunked": dict(T=60, H=256, I=192, E=5, k=2, L=4, r=64),
          "r128_chunked": dict(T=48, H=256, I=128, E=4, k=2, L=2, r=128),
          "tiles_many_runs": dict(T=1024, H=256, I=256, E=8, k=2, L=16, r=16,
                                  adapters="one_per_request16"),
          "persistent_r32": dict(T=700, H=128, I=256, E=4, k=2, L=3, r=32),
          "base_only_tiles": dict(T=300, H=256, I=192, E=4, k=2, L=0, r=16),
          # 64-row chunks (experts of more than 32 rows) and K = 200: the last 64-column
          # stage has 8 columns, the rest read as zeros
          "expert_major_k_tail": dict(T=64, H=200, I=96, E=4, k=2, L=3, r=16),
          "dense_ksplit8_k_tail": dict(T=20, H=256, I=1000, E=1, k=1, L=3, r=16)}[shape]
    inp = make_layer_inputs(seed=120 + len(shape), lora_std=None, **kw)
    plan = m.moe_lora_layer_plan(inp.T, inp.k, inp.E, inp.L, inp.H, inp.I, inp.r)
    assert plan["fused_expand"] == 1, plan
    y = run_layer(m, inp, y_fp32=True).cpu()
    y_sep = run_layer(m, inp, y_fp32=True, expand_mode=1).cpu()
    tokens = np.arange(inp.T) if inp.T <= 300 else np.arange(0, inp.T, 3)
    ref = oracle_layer(inp, tokens)
    assert_close(y[tokens], ref, LAYER_RTOL, f"fused {shape} {plan}")
    # the two chains differ only in fp32 summation order and where z is rounded
    assert_close(y, f64(y_sep), 1e-3, f"fused vs separate expand, {shape}")


@pytest.mark.parametrize("shape", ["odd_blocks_many_runs", "ragged_tiles_r32",
                                   "base_only", "r64_chunked_pairs", "one_tile"])
def test_fused_cta_pairs(shape):
    """256-row token tiles of the fused chain run on CTA pairs: one
    tcgen05.mma.cta_group::2 of M = 256 over two weight blocks, each CTA staging half of
    the tile's rows (split at half the MMA width, which follows the tile's rows). Shapes:
    an odd number of 64-feature gate_up blocks and of 128-row down blocks (the last
    pair's second CTA has no block), ragged last tiles of every expert, chunked rank-64
    z, no adapters, and a single tile shorter than the split. Every token against the
    oracle, and against the one-CTA MMAs."""
    m = need_gpu()
    kw = {"odd_blocks_many_runs": dict(T=1104, H=320, I=320, E=6, k=2, L=16, r=16,
                                       adapters="one_per_request16"),
          "ragged_tiles_r32": dict(T=900, H=384, I=224, E=5, k=3, L=5, r=32),
          "base_only": dict(T=700, H=256, I=192, E=4, k=2, L=0, r=16),
          "r64_chunked_pairs": dict(T=640, H=256, I=192, E=4, k=2, L=3, r=64),
          "one_tile": dict(T=300, H=128, I=64, E=2, k=1, L=2, r=16)}[shape]
    inp = make_layer_inputs(seed=300 + len(shape), lora_std=None, **kw)
    plan = m.moe_lora_layer_plan(inp.T, inp.k, inp.E, inp.L, inp.H, inp.I, inp.r)
    assert plan["fused_expand"] == 1 and plan["bm_base"] == 256, plan
    y = run_layer(m, inp, y_fp32=True).cpu()
    y1 = run_layer(m, inp, y_fp32=True, mma_pairs=-1).cpu()
    ref = oracle_layer(inp)
    assert_close(y, ref, LAYER_RTOL, f"pairs {shape} {plan}")
    assert_close(y1, ref, LAYER_RTOL, f"one CTA {shape} {plan}")
    # the same products in the same K order: only the accumulation hardware differs
    assert_close(y, f64(y1), 1e-4, f"pairs vs one CTA, {shape}")


def test_layer_error_word_clean_on_workload():
    m = need_gpu()
    inp = make_workload_inputs("gptoss20b_decode")
    ws = m.new_workspace(inp.T, inp.k, inp.E, inp.L, inp.H, inp.I, inp.r)
    run_layer(m, inp, workspace=ws)
    assert m.get_error(ws) == 0


def test_layer_amplified_adapters():
    """A, B ~ N(0, 1/fan_in): the low-rank term is as large as the base term, so the
    layer bound pins it."""
    m = need_gpu()
    for seed in range(3):
        inp = make_layer_inputs(T=24, H=128, I=96, E=6, k=2, L=3, r=16, seed=50 + seed,
                                lora_std=None)
        y = run_layer(m, inp, y_fp32=True).cpu()
        ref = oracle_layer(inp)
        base = oracle_layer(inp, adapters=False)
        assert np.abs(ref - base).max() > 0.3 * np.abs(ref).max()  # adapters matter here
        assert_close(y, ref, LAYER_RTOL, f"amplified seed {seed}")


def test_layer_lora_delta_matches_oracle():
    """With the workloads' own N(0, 0.02) adapters on the tiny layer the LoRA term is below
    the layer bound; check the GPU's delta y_lora - y_base against the oracle's directly."""
    m = need_gpu()
    inp = make_workload_inputs("tiny")
    y_l = run_layer(m, inp, y_fp32=True).cpu().double().numpy()
    y_b = run_layer(m, inp, y_fp32=True, adapters=False).cpu().double().numpy()
    d_gpu = y_l - y_b
    d_ref = oracle_layer(inp) - oracle_layer(inp, adapters=False)
    cos = float((d_gpu * d_ref).sum() / np.sqrt((d_gpu ** 2).sum() * (d_ref ** 2).sum()))
    assert cos >= 0.99, cos
    assert np.abs(d_gpu - d_ref).max() <= 0.1 * np.abs(d_ref).max()


@pytest.mark.parametrize("expand_mode", [1, 2])
def test_layer_base_reductions_bitwise(expand_mode):
    """Adapter -1 everywhere, or B = 0, give exactly the base-only output of the same chain
    (the separate expand kernels, or the expand fused into the grouped GEMMs)."""
    m = need_gpu()
    inp = make_workload_inputs("tiny")
    kw = dict(y_fp32=True, expand_mode=expand_mode)
    y_base = run_layer(m, inp, adapters=False, **kw)
    none = torch.full((inp.T,), -1, dtype=torch.int32)
    y_none = run_layer(m, inp, token_adapter=none, **kw)
    assert torch.equal(y_none, y_base)
    y_zero = run_layer(m, inp, B_zero=True, **kw)
    assert torch.equal(y_zero, y_base)


def test_layer_token_permutation():
    m = need_gpu()
    inp = make_layer_inputs(T=40, H=64, I=48, E=8, k=2, L=4, r=8, seed=60, lora_std=None)
    y = run_layer(m, inp, y_fp32=True).cpu()
    perm = torch.from_numpy(np.random.default_rng(1).permutation(inp.T))
    inp2 = make_layer_inputs(T=40, H=64, I=48, E=8, k=2, L=4, r=8, seed=60, lora_std=None)
    inp2.x = inp.x[perm].contiguous()
    inp2.logits = inp.logits[perm].contiguous()
    inp2.token_adapter = inp.token_adapter[perm].contiguous()
    y2 = run_layer(m, inp2, y_fp32=True).cpu()
    assert_close(y2, f64(y)[perm.numpy()], 1e-5, "permuted")


@pytest.mark.parametrize("T", [1, 7, 64, 513])
def test_layer_many_token_counts(T):
    """Back-to-back token counts: every size is a runtime argument (no per-size build)."""
    m = need_gpu()
    inp = make_layer_inputs(T=T, H=64, I=32, E=8, k=2, L=3, r=8, seed=70 + T, lora_std=None)
    y = run_layer(m, inp, y_fp32=True).cpu()
    tokens = np.arange(T) if T <= 64 else np.arange(0, T, 8)
    assert_close(y[tokens], oracle_layer(inp, tokens), LAYER_RTOL, f"T={T}")


def test_layer_dense_single_expert():
    """E = 1, k = 1: multi-LoRA on a dense gated MLP."""
    m = need_gpu()
    inp = make_layer_inputs(T=33, H=96, I=80, E=1, k=1, L=4, r=16, seed=80, lora_std=None)
    y = run_layer(m, inp, y_fp32=True).cpu()
    assert_close(y, oracle_layer(inp), LAYER_RTOL, "dense")


def test_layer_bad_adapter_ids_dropped_and_flagged():
    m = need_gpu()
    inp = make_layer_inputs(T=10, H=64, I=32, E=4, k=2, L=2, r=8, seed=90, lora_std=None)
    ta = inp.token_adapter.clone()
    ta[3] = 7
    ws = m.new_workspace(inp.T, inp.k, inp.E, inp.L, inp.H, inp.I, inp.r)
    y = run_layer(m, inp, y_fp32=True, token_adapter=ta, workspace=ws).cpu()
    assert m.get_error(ws) == 2
    ref = oracle_layer(inp, token_adapter=ta)
    assert np.all(ref[3] == 0.0) and torch.all(y[3] == 0)
    assert_close(y, ref, LAYER_RTOL, "bad adapter")


def test_layer_caller_routing_and_no_pdl():
    m = need_gpu()
    inp = make_layer_inputs(T=20, H=64, I=32, E=4, k=2, L=2, r=8, seed=91, lora_std=None)
    ids, w = oracle.route_topk_softmax(inp.logits, inp.k)
    y = torch.empty((inp.T, inp.H), dtype=torch.float32, device="cuda")
    m.moe_lora_layer(dev(inp.x), dev(inp.W1), dev(inp.W2),
                     topk_ids=dev(torch.as_tensor(ids, dtype=torch.int32)),
                     topk_w=dev(torch.as_tensor(w, dtype=torch.float32)),
                     token_adapter=dev(inp.token_adapter), A1=dev(inp.A1), B1=dev(inp.B1),
                     A2=dev(inp.A2), B2=dev(inp.B2), y=y, y_fp32=True, disable_pdl=True)
    assert_close(y.cpu(), oracle_layer(inp), LAYER_RTOL, "caller routing")


def test_layer_skewed_decode_multi_chunk():
    """Few rows per expert on average (the gate_up GEMM runs one CTA per expert and
    weight block) but Zipf-skewed: the top expert's rows span four chunks and some
    experts receive no token at all."""
    m = need_gpu()
    inp = make_layer_inputs(T=128, H=128, I=96, E=16, k=2, L=3, r=16, seed=95,
                            routing="zipf2.0", lora_std=None)
    ids, _ = oracle.route_topk_softmax(inp.logits, inp.k)
    counts = np.bincount(ids.reshape(-1), minlength=inp.E)
    assert counts.max() > 96 and (counts == 0).any()  # four chunks of 32; idle experts
    y = run_layer(m, inp, y_fp32=True).cpu()
    assert_close(y, oracle_layer(inp), LAYER_RTOL, "skewed decode")


def test_layers_chained_in_cuda_graph():
    """Three layers chained on one stream (layer i + 1 reads layer i's y, one shared
    workspace), captured in a CUDA graph with programmatic dependent launch across the
    layer boundaries: the replay reproduces the eager chain bit for bit, and the first
    layer matches the oracle."""
    m = need_gpu()
    inp = make_layer_inputs(T=24, H=256, I=192, E=8, k=2, L=3, r=16, seed=21,
                            adapters="uniform_with_none", lora_std=None)
    n = 3
    Ws = [(dev(torch.roll(inp.W1, i, 0)), dev(torch.roll(inp.W2, i, 0)),
           {nm: dev(torch.roll(getattr(inp, nm), i, 1)) for nm in ("A1", "B1", "A2", "B2")},
           dev(torch.roll(inp.logits, i, 1))) for i in range(n)]
    x = dev(inp.x)
    ta = dev(inp.token_adapter)
    ws = m.new_workspace(inp.T, inp.k, inp.E, inp.L, inp.H, inp.I, inp.r)
    ys = [torch.empty_like(x) for _ in range(n)]

    def chain():
        xin = x
        for (w1, w2, lo, lg), y in zip(Ws, ys):
            m.moe_lora_layer(xin, w1, w2, logits=lg, k=inp.k, token_adapter=ta, y=y,
                             workspace=ws, **lo)
            xin = y

    chain()
    torch.cuda.synchronize()
    eager = [y.clone() for y in ys]
    for y in ys:
        y.zero_()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        chain()
    torch.cuda.current_stream().wait_stream(side)
    for y in ys:
        y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for i in range(n):
        assert torch.equal(ys[i], eager[i]), f"layer {i}: graph replay differs from eager"
    assert m.get_error(ws) == 0
    ref = oracle_layer(inp)
    assert_close(eager[0].cpu(), ref, LAYER_RTOL, "first chained layer")


@pytest.mark.parametrize("shape", ["tiny", "decode", "prefill_like"])
def test_layer_two_slice_gate_up(shape):
    """Separate gate and up adapters (A1 [L, E, 2r, H]) through the whole layer: the gate_up
    shrink runs at rank 2r and the SwiGLU expand gives each half its own z."""
    m = need_gpu()
    if shape == "tiny":
        kw = dict(T=8, H=256, I=512, E=4, k=2, L=2, r=8, adapters="tiny")
    elif shape == "decode":
        kw = dict(T=64, H=512, I=384, E=32, k=4, L=8, r=32, adapters="round_robin_shuffled")
    else:
        kw = dict(T=1024, H=256, I=256, E=8, k=2, L=16, r=16, adapters="one_per_request16")
    inp = make_layer_inputs(seed=31, lora_std=None, **kw)
    rng = np.random.default_rng(32)
    A1s = torch.from_numpy(rng.standard_normal((inp.L, inp.E, 2 * inp.r, inp.H)).astype(np.float32)
                           * 0.05).to(torch.bfloat16)
    lora = dict(A1=dev(A1s), B1=dev(inp.B1), A2=dev(inp.A2), B2=dev(inp.B2))
    y = Guarded((inp.T, inp.H), torch.bfloat16)
    m.moe_lora_layer(dev(inp.x), dev(inp.W1), dev(inp.W2), logits=dev(inp.logits), k=inp.k,
                     token_adapter=dev(inp.token_adapter), y=y.t, gate_up_slices=2, **lora)
    y.check()
    ids, w = oracle.route_topk_softmax(inp.logits, inp.k)
    ref = oracle.moe_lora_layer(inp.x, inp.W1, inp.W2, ids, w, inp.token_adapter, A1s, inp.B1,
                                inp.A2, inp.B2, gate_up_slices=2)
    assert_close(y.t.cpu(), ref, LAYER_RTOL, f"two-slice gate_up, {shape}")


@pytest.mark.parametrize("shape", ["decode", "prefill_like", "stress_like"])
@pytest.mark.parametrize("slices", [1, 2])
def test_layer_adapter_ranks(shape, slices):
    """Adapters of their own ranks through the whole layer, with the padding of every A and B
    past an adapter's rank holding NaN (never used), one or two gate_up slices."""
    m = need_gpu()
    if shape == "decode":
        kw = dict(T=64, H=512, I=384, E=32, k=4, L=8, r=32, adapters="round_robin_shuffled")
    elif shape == "prefill_like":
        kw = dict(T=1024, H=256, I=256, E=8, k=2, L=16, r=16, adapters="one_per_request16")
    else:
        kw = dict(T=256, H=256, I=128, E=64, k=8, L=32, r=32, adapters="zipf1.1")
    inp = make_layer_inputs(seed=33, lora_std=None, **kw)
    r, L = kw["r"], kw["L"]
    ranks = [[r, 8, 0, r // 2, 5][l % 5] for l in range(L)]
    rng = np.random.default_rng(34)
    A1 = torch.from_numpy(rng.standard_normal((L, inp.E, slices * r, inp.H)).astype(np.float32)
                          * 0.05).to(torch.bfloat16)

    def poison(t, rank_dim_rows):
        t = t.clone()
        for l, rl in enumerate(ranks):
            if rank_dim_rows:
                for sl in range(t.shape[2] // r):
                    t[l, :, sl * r + rl: (sl + 1) * r] = float("nan")
            else:
                t[l, :, :, rl:] = float("nan")
        return t

    A1p, B1p = poison(A1, True), poison(inp.B1, False)
    A2p, B2p = poison(inp.A2, True), poison(inp.B2, False)
    rk = torch.as_tensor(ranks, dtype=torch.int32)
    ws = m.new_workspace(inp.T, inp.k, inp.E, L, inp.H, inp.I, r)
    y = Guarded((inp.T, inp.H), torch.bfloat16)
    m.moe_lora_layer(dev(inp.x), dev(inp.W1), dev(inp.W2), logits=dev(inp.logits), k=inp.k,
                     token_adapter=dev(inp.token_adapter), y=y.t, A1=dev(A1p), B1=dev(B1p),
                     A2=dev(A2p), B2=dev(B2p), gate_up_slices=slices, adapter_ranks=dev(rk),
                     workspace=ws)
    y.check()
    assert m.get_error(ws) == 0
    ids, w = oracle.route_topk_softmax(inp.logits, inp.k)
    tok = np.arange(min(inp.T, 64))
    ref = oracle.moe_lora_layer(inp.x[tok], inp.W1, inp.W2, ids[tok], w[tok], inp.token_adapter[tok],
                                A1p, B1p, A2p, B2p, gate_up_slices=slices, adapter_ranks=rk)
    assert not torch.isnan(y.t).any()
    assert_close(y.t.cpu()[tok], ref, LAYER_RTOL, f"ranked adapters, {shape}, slices={slices}")


def test_layer_adapter_rank_out_of_range_flagged():
    """A rank outside [0, r] is clamped and flagged in the error word."""
    m = need_gpu()
    inp = make_layer_inputs(T=8, H=128, I=128, E=4, k=2, L=2, r=8, seed=35, adapters="tiny")
    ws = m.new_workspace(inp.T, inp.k, inp.E, 2, inp.H, inp.I, 8)
    rk = torch.as_tensor([12, -1], dtype=torch.int32)
    y = run_layer(m, inp, workspace=ws, adapter_ranks=dev(rk))
    assert m.get_error(ws) & 0x8
    ids, w = oracle.route_topk_softmax(inp.logits, inp.k)
    ref = oracle.moe_lora_layer(inp.x, inp.W1, inp.W2, ids, w, inp.token_adapter, inp.A1, inp.B1,
                                inp.A2, inp.B2, adapter_ranks=torch.as_tensor([8, 0]))
    assert_close(y.cpu(), ref, LAYER_RTOL, "clamped ranks")


@pytest.mark.parametrize("name,with_adapter,y_fp32", [("tiny", True, True),
                                                      ("gptoss20b_decode", True, False),
                                                      ("gptoss20b_decode", False, False)])
def test_layer_host_staged(name, with_adapter, y_fp32):
    """moe_lora_layer_host: the inputs copied from one page-locked host block, the chain on
    the staged views, y copied back. Bit-identical to the device-pointer call on the same
    inputs (same kernels), and within tolerance of the oracle (the tiny workload on every
    token, the decode workload on a sample); without adapter ids the base MoE alone."""
    m = need_gpu()
    inp = make_workload_inputs(name)
    io = m.new_host_io(inp.T, inp.H, inp.E, with_adapter=with_adapter, y_fp32=y_fp32)
    io.x.copy_(inp.x)
    io.logits.copy_(inp.logits)
    if with_adapter:
        io.token_adapter.copy_(inp.token_adapter)
    lora = dict(A1=dev(inp.A1), B1=dev(inp.B1), A2=dev(inp.A2), B2=dev(inp.B2))
    W1, W2 = dev(inp.W1), dev(inp.W2)
    io.y_host.fill_(float("nan"))
    y_host = m.moe_lora_layer_host(io, W1, W2, k=inp.k, **lora)
    torch.cuda.synchronize()
    ta = dev(inp.token_adapter) if with_adapter else None
    y_dev = m.moe_lora_layer(dev(inp.x), W1, W2, logits=dev(inp.logits), k=inp.k,
                             token_adapter=ta, y_fp32=y_fp32, **lora).cpu()
    assert torch.equal(y_host, y_dev)
    tokens = np.arange(inp.T)
    no_adapter = np.full(inp.T, -1, dtype=np.int32)
    ref = oracle_layer(inp, tokens, token_adapter=None if with_adapter else no_adapter)
    assert_close(y_host[tokens], ref, LAYER_RTOL, f"host-staged {name}")


@pytest.mark.parametrize("y_fp32", [True, False])
def test_layer_output_any_alignment(y_fp32):
    """y is a caller buffer with no alignment rule: one offset by a single element (4- or
    2-byte aligned) takes the combine's scalar form instead of its 16-byte one, with the
    same sums in the same order, so the same bits."""
    m = need_gpu()
    inp = make_workload_inputs("gptoss20b_decode")
    dt = torch.float32 if y_fp32 else torch.bfloat16
    lora = dict(A1=dev(inp.A1), B1=dev(inp.B1), A2=dev(inp.A2), B2=dev(inp.B2))
    args = (dev(inp.x), dev(inp.W1), dev(inp.W2))
    kw = dict(logits=dev(inp.logits), k=inp.k, token_adapter=dev(inp.token_adapter),
              y_fp32=y_fp32, **lora)
    y = m.moe_lora_layer(*args, **kw)
    raw = torch.zeros(inp.T * inp.H + 1, dtype=dt, device="cuda")
    y_odd = raw[1:].view(inp.T, inp.H)
    assert y_odd.data_ptr() % 16 != 0
    m.moe_lora_layer(*args, y=y_odd, **kw)
    torch.cuda.synchronize()
    assert torch.equal(y, y_odd)
