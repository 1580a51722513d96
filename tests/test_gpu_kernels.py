"""Per-kernel parity on the GPU: gather, grouped GEMM, shrink, expand epilogues."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import make_layer_inputs

from gpu_util import (BF16_REL, KERNEL_RTOL, Guarded, assert_bf16_close, assert_close, dev, f64,
                      need_gpu)

pytestmark = pytest.mark.gpu


def _setup(T, H, I, E, k, L, r, seed, bm_base=16, bm_lora=16, adapters="uniform_with_none",
           routing="gaussian"):
    m = need_gpu()
    inp = make_layer_inputs(T=T, H=H, I=I, E=E, k=k, L=L, r=r, seed=seed, adapters=adapters,
                            routing=routing, lora_std=None)
    ids, w = oracle.route_topk_softmax(inp.logits, k)
    ids_t = torch.as_tensor(ids, dtype=torch.int32)
    al = m.moe_lora_align(dev(ids_t), dev(inp.token_adapter), E, L, bm_base, bm_lora)
    ref = oracle.align(ids_t, inp.token_adapter, E, L, bm_base, bm_lora)
    return m, inp, ids, w, al, ref


@pytest.mark.parametrize("H", [256, 136, 8, 1024, 1032, 2880])
def test_gather_exact(H):
    """Bit-exact row gather. A warp copies a segment of 128 16-byte chunks of a row: H = 1024
    is one full segment, 1032 adds a second segment of one chunk, 2880 three segments with a
    partial last one; H = 8 and 136 are single short segments."""
    m, inp, ids, w, al, ref = _setup(T=19, H=H, I=16, E=5, k=3, L=2, r=8, seed=1)
    xs = Guarded((al.S, H), torch.bfloat16)
    m.moe_gather_rows(dev(inp.x), al, out=xs.t)
    xs.check()
    n = ref["n_valid"]
    assert np.array_equal(f64(xs.t)[:n], oracle.gather_rows(inp.x, ref))


@pytest.mark.parametrize("bm_base", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("K,N", [(256, 1024), (136, 200), (64, 128)])
def test_grouped_gemm_vs_oracle(bm_base, K, N):
    """Several tiles per expert, ragged last tile, K tail (136 = 2*64 + 8), N tail (200)."""
    m, inp, ids, w, al, ref = _setup(T=150, H=K, I=N // 2, E=6, k=2, L=1, r=8, seed=2,
                                     bm_base=bm_base)
    xs = m.moe_gather_rows(dev(inp.x), al)
    out = Guarded((al.S, N), torch.float32, fill=float("nan"))
    m.moe_grouped_gemm(xs, dev(inp.W1), al, out=out.t)
    out.check()
    n = ref["n_valid"]
    expect = oracle.grouped_gemm(oracle.gather_rows(inp.x, ref), inp.W1, ref)
    assert_close(out.t[:n], expect, KERNEL_RTOL, f"gemm bm={bm_base} K={K} N={N}")
    assert torch.isnan(out.t[n:]).all()  # rows past n_valid untouched


def test_grouped_gemm_skewed_experts():
    """Zipf routing: one expert holds most rows (many tiles), others few or none."""
    m, inp, ids, w, al, ref = _setup(T=600, H=128, I=64, E=16, k=2, L=0, r=1, seed=3,
                                     bm_base=64, routing="zipf1.0", adapters="none")
    xs = m.moe_gather_rows(dev(inp.x), al)
    out = m.moe_grouped_gemm(xs, dev(inp.W1), al)
    expect = oracle.grouped_gemm(oracle.gather_rows(inp.x, ref), inp.W1, ref)
    assert_close(out[: ref["n_valid"]], expect, KERNEL_RTOL, "gemm zipf")


def test_grouped_gemm_full_size_sampled_rows():
    """The decode workload's gate_up shape (E=32, N=5760, K=2880) in the layer's tiling;
    every output row of a sample of rows against the oracle."""
    m = need_gpu()
    T, H, I, E, k = 64, 2880, 2880, 32, 4
    rng = np.random.default_rng(11)
    x = torch.from_numpy(rng.standard_normal((T, H), dtype=np.float32)).to(torch.bfloat16)
    W = torch.from_numpy((rng.standard_normal((E, 2 * I, H), dtype=np.float32) * 0.02)).to(
        torch.bfloat16)
    lg = torch.from_numpy(rng.standard_normal((T, E), dtype=np.float32))
    ids, _ = oracle.route_topk_softmax(lg, k)
    ids_t = torch.as_tensor(ids, dtype=torch.int32)
    bm = m.moe_lora_layer_tiles(T, k, E, 8, H, I, 32)[0]
    al = m.moe_lora_align(dev(ids_t), None, E, 0, bm, 16)
    ref = oracle.align(ids_t, None, E, 0, bm, 16)
    xs = m.moe_gather_rows(dev(x), al)
    out = m.moe_grouped_gemm(xs, dev(W), al).cpu()
    sample = rng.choice(ref["n_valid"], size=24, replace=False)
    X = f64(x)
    for row in sample:
        s = int(ref["sorted_slots"][row])
        e = int(ref["row_expert"][row])
        expect = f64(W[e]) @ X[s // k]
        assert_close(out[row], expect, KERNEL_RTOL, f"row {row}")


# ------------------------------------------------------------------ shrink
@pytest.mark.parametrize("K", [100, 136, 256, 2880])
@pytest.mark.parametrize("r", [1, 8, 16, 32, 64])
def test_shrink_vs_oracle(K, r):
    m, inp, ids, w, al, ref = _setup(T=90, H=K, I=8, E=3, k=2, L=3, r=r, seed=4, bm_lora=16)
    Z = Guarded((al.S, r), torch.float32, fill=0.0)
    m.lora_shrink(dev(inp.x), False, dev(inp.A1), al, out=Z.t)
    Z.check()
    expect = oracle.lora_shrink(inp.x, inp.A1, ref, rows_are_slots=False)
    assert_close(Z.t, expect, KERNEL_RTOL, f"shrink K={K} r={r}")


def test_shrink_even_k_example(golden_dir):
    """The pages' masking example: K = 100 with 64-wide K blocks leaves 28 dead lanes in the
    second block; the result must match the oracle exactly as for an even K."""
    with open(os.path.join(golden_dir, "even_k_example.json")) as f:
        g = json.load(f)
    K = g["K"]
    m, inp, ids, w, al, ref = _setup(T=33, H=K, I=8, E=2, k=2, L=2, r=16, seed=5, bm_lora=5)
    Z = m.lora_shrink(dev(inp.x), False, dev(inp.A1), al)
    assert_close(Z, oracle.lora_shrink(inp.x, inp.A1, ref, False), KERNEL_RTOL, "K=100")


@pytest.mark.parametrize("bm_lora", [1, 3, 16])
def test_shrink_rows_are_slots(bm_lora):
    m, inp, ids, w, al, ref = _setup(T=70, H=64, I=96, E=4, k=3, L=5, r=16, seed=6,
                                     bm_lora=bm_lora)
    n = ref["n_valid"]
    rng = np.random.default_rng(0)
    h = torch.from_numpy(rng.standard_normal((al.S, 96), dtype=np.float32)).to(torch.bfloat16)
    Z = m.lora_shrink(dev(h), True, dev(inp.A2), al)
    expect = oracle.lora_shrink(h[:n], inp.A2, ref, rows_are_slots=True)
    assert_close(Z, expect, KERNEL_RTOL, "shrink sorted rows")


def test_shrink_decode_shape():
    """The decode workload: one or two rows per (expert, adapter) pair, K = 2880, r = 32."""
    m, inp, ids, w, al, ref = _setup(T=64, H=2880, I=8, E=32, k=4, L=8, r=32, seed=7,
                                     adapters="round_robin_shuffled")
    Z = m.lora_shrink(dev(inp.x), False, dev(inp.A1), al)
    assert_close(Z, oracle.lora_shrink(inp.x, inp.A1, ref, False), KERNEL_RTOL, "decode")


# ------------------------------------------------------------------ expand
@pytest.mark.parametrize("r", [8, 5, 32])
@pytest.mark.parametrize("bm_lora", [1, 16])
def test_expand_add_inplace(r, bm_lora):
    m, inp, ids, w, al, ref = _setup(T=50, H=40, I=72, E=4, k=2, L=3, r=r, seed=8,
                                     bm_lora=bm_lora)
    n = ref["n_valid"]
    rng = np.random.default_rng(1)
    Zh = torch.from_numpy(rng.standard_normal((al.S, r))).to(torch.float32)
    G = torch.from_numpy(rng.standard_normal((al.S, 144))).to(torch.float32)
    base = Guarded((al.S, 144), torch.float32)
    base.t.copy_(G)
    m.lora_expand_add(dev(Zh), dev(inp.B1), al, 0, base.t)
    base.check()
    expect = oracle.lora_expand_add(Zh, inp.B1, ref, G[:n], epilogue=0)
    assert_close(base.t[:n], expect, KERNEL_RTOL, "expand epilogue 0")


@pytest.mark.parametrize("bm_base", [16, 64])
@pytest.mark.parametrize("r", [8, 32, 5, 0])
def test_expand_swiglu(bm_base, r):
    L = 3 if r else 0
    m, inp, ids, w, al, ref = _setup(T=80, H=40, I=72, E=4, k=2, L=L, r=max(r, 1), seed=9,
                                     bm_base=bm_base)
    n = ref["n_valid"]
    rng = np.random.default_rng(2)
    Zh = torch.from_numpy(rng.standard_normal((al.S, max(r, 1)))).to(torch.float32)
    G = torch.from_numpy(rng.standard_normal((al.S, 144))).to(torch.float32)
    h = Guarded((al.S, 72), torch.bfloat16)
    m.lora_expand_add(dev(Zh) if r else None, dev(inp.B1) if r else None, al, 1, dev(G),
                      out=h.t)
    h.check()
    if r:
        expect = oracle.lora_expand_add(Zh, inp.B1, ref, G[:n], epilogue=1)
    else:
        expect = oracle.swiglu(f64(G)[:n])
    assert_bf16_close(h.t[:n], expect, "expand epilogue 1")


@pytest.mark.parametrize("out_fp32", [True, False])
def test_expand_combine(out_fp32):
    m, inp, ids, w, al, ref = _setup(T=45, H=40, I=24, E=5, k=3, L=2, r=16, seed=10)
    n = ref["n_valid"]
    rng = np.random.default_rng(3)
    Zh = torch.from_numpy(rng.standard_normal((al.S, 16))).to(torch.float32)
    O = torch.from_numpy(rng.standard_normal((al.S, 40))).to(torch.float32)
    wt = torch.as_tensor(w, dtype=torch.float32)
    y = Guarded((45, 40), torch.float32 if out_fp32 else torch.bfloat16)
    m.lora_expand_add(dev(Zh), dev(inp.B2), al, 2, dev(O), out=y.t, out_fp32=out_fp32,
                      topk_w=dev(wt))
    y.check()
    expect = oracle.lora_expand_add(Zh, inp.B2, ref, O[:n], epilogue=2, w=wt)
    if out_fp32:
        assert_close(y.t, expect, KERNEL_RTOL, "combine fp32")
    else:
        assert_bf16_close(y.t, expect, "combine bf16")


def test_expand_swiglu_many_rows_per_cta():
    """Long (expert, adapter) segments: 16 sorted rows per CTA sharing B rows in registers,
    G fetched four rows at a time."""
    m, inp, ids, w, al, ref = _setup(T=2048, H=64, I=2048, E=2, k=1, L=2, r=16, seed=12,
                                     bm_base=256)
    n = ref["n_valid"]
    rng = np.random.default_rng(4)
    Zh = torch.from_numpy(rng.standard_normal((al.S, 16))).to(torch.float32)
    G = torch.from_numpy(rng.standard_normal((al.S, 4096), dtype=np.float32))
    h = m.lora_expand_add(dev(Zh), dev(inp.B1), al, 1, dev(G))
    expect = oracle.lora_expand_add(Zh, inp.B1, ref, G[:n], epilogue=1)
    assert_bf16_close(h[:n], expect, "expand epilogue 1, long segments")


@pytest.mark.parametrize("k", [1, 4])
def test_expand_combine_many_tokens_per_cta(k):
    """Several tokens per CTA in the fused down expand + combine."""
    m, inp, ids, w, al, ref = _setup(T=4096, H=256, I=16, E=8, k=k, L=3, r=16, seed=13)
    n = ref["n_valid"]
    rng = np.random.default_rng(5)
    Zh = torch.from_numpy(rng.standard_normal((al.S, 16))).to(torch.float32)
    O = torch.from_numpy(rng.standard_normal((al.S, 256), dtype=np.float32))
    wt = torch.as_tensor(w, dtype=torch.float32)
    y = m.lora_expand_add(dev(Zh), dev(inp.B2), al, 2, dev(O), out_fp32=True, topk_w=dev(wt))
    expect = oracle.lora_expand_add(Zh, inp.B2, ref, O[:n], epilogue=2, w=wt)
    assert_close(y, expect, KERNEL_RTOL, "combine, many tokens per CTA")


@pytest.mark.parametrize("r,T", [(16, 4096), (32, 2048), (64, 2048)])
def test_shrink_many_blocks(r, T):
    """Enough LoRA blocks that one CTA takes 16-64 ranks (prefill-like)."""
    m, inp, ids, w, al, ref = _setup(T=T, H=256, I=8, E=8, k=4, L=8, r=r, seed=14)
    Z = m.lora_shrink(dev(inp.x), False, dev(inp.A1), al)
    assert_close(Z, oracle.lora_shrink(inp.x, inp.A1, ref, False), KERNEL_RTOL, f"shrink r={r}")


@pytest.mark.parametrize("form", ["by_token", "sorted_rows", "ranked"])
@pytest.mark.parametrize("K,r", [(2880, 16), (2880, 32), (1032, 16), (1032, 24), (1032, 32)])
def test_shrink_pipelined(K, r, form):
    """Many blocks of up to 16 rows with long sums (prefill): the shrink that streams A and
    x through a ring of shared-memory stages by bulk copies. K = 1032 leaves an 8-column
    last stage; r = 24 half uses its second rank group's rows; adapters of their own ranks
    with NaN past them (never read); activations by token or in sorted-row order."""
    m, inp, ids, w, al, ref = _setup(T=3328, H=K, I=8, E=4, k=4, L=8, r=r, seed=31, bm_lora=16)
    assert len(ref["lora_blocks"]) > 4 * torch.cuda.get_device_properties(0).multi_processor_count
    if form == "sorted_rows":
        n = ref["n_valid"]
        rng = np.random.default_rng(3)
        h = torch.from_numpy(rng.standard_normal((al.S, K), dtype=np.float32)).to(torch.bfloat16)
        Z = m.lora_shrink(dev(h), True, dev(inp.A1), al)
        expect = oracle.lora_shrink(h[:n], inp.A1, ref, rows_are_slots=True)
    elif form == "ranked":
        ranks = [[8, 0, 5, 16, r][l % 5] for l in range(8)]
        A = _poison_A(inp.A1, ranks, r)
        rk = torch.as_tensor(ranks, dtype=torch.int32)
        Z = m.lora_shrink(dev(inp.x), False, dev(A), al, adapter_ranks=dev(rk))
        expect = oracle.lora_shrink(inp.x, A, ref, False, adapter_ranks=rk)
        assert not torch.isnan(Z).any()
    else:
        Z = m.lora_shrink(dev(inp.x), False, dev(inp.A1), al)
        expect = oracle.lora_shrink(inp.x, inp.A1, ref, False)
    assert_close(Z, expect, KERNEL_RTOL, f"pipelined shrink K={K} r={r} {form}")
    assert m.get_error(al.buf) == 0


@pytest.mark.parametrize("r", [32, 5])
def test_expand_short_segments(r):
    """Decode-like routing: about one row per (expert, adapter) pair; the SwiGLU expand walks
    rows and the down expand walks tokens (fused with the combine)."""
    m, inp, ids, w, al, ref = _setup(T=64, H=96, I=80, E=32, k=4, L=8, r=r, seed=15,
                                     adapters="round_robin_shuffled")
    n = ref["n_valid"]
    rng = np.random.default_rng(6)
    Zh = torch.from_numpy(rng.standard_normal((al.S, r))).to(torch.float32)
    G = torch.from_numpy(rng.standard_normal((al.S, 160), dtype=np.float32))
    h = m.lora_expand_add(dev(Zh), dev(inp.B1), al, 1, dev(G))
    assert_bf16_close(h[:n], oracle.lora_expand_add(Zh, inp.B1, ref, G[:n], epilogue=1),
                      "expand epilogue 1, short segments")
    O = torch.from_numpy(rng.standard_normal((al.S, 96), dtype=np.float32))
    wt = torch.as_tensor(w, dtype=torch.float32)
    y = m.lora_expand_add(dev(Zh), dev(inp.B2), al, 2, dev(O), out_fp32=True, topk_w=dev(wt))
    assert_close(y, oracle.lora_expand_add(Zh, inp.B2, ref, O[:n], epilogue=2, w=wt),
                 KERNEL_RTOL, "expand epilogue 2, short segments")


@pytest.mark.parametrize("r", [8, 16, 64])
@pytest.mark.parametrize("k", [1, 3, 4])
def test_expand_short_segment_forms(r, k):
    """About one row per (expert, adapter) pair: the SwiGLU expand takes one sorted row per
    CTA (all of a thread's loads issued before any is consumed) and the down expand walks
    tokens; ranks 8..64, k = 1..4 slots per token, ragged column tails (I = 300, H = 520)."""
    m, inp, ids, w, al, ref = _setup(T=48, H=520, I=300, E=32, k=k, L=8, r=r, seed=17,
                                     adapters="round_robin_shuffled")
    n = ref["n_valid"]
    rng = np.random.default_rng(7)
    Zh = torch.from_numpy(rng.standard_normal((al.S, r))).to(torch.float32)
    G = torch.from_numpy(rng.standard_normal((al.S, 600), dtype=np.float32))
    h = Guarded((al.S, 300), torch.bfloat16)
    m.lora_expand_add(dev(Zh), dev(inp.B1), al, 1, dev(G), out=h.t)
    h.check()
    assert_bf16_close(h.t[:n], oracle.lora_expand_add(Zh, inp.B1, ref, G[:n], epilogue=1),
                      "expand epilogue 1, one row per CTA")
    O = torch.from_numpy(rng.standard_normal((al.S, 520), dtype=np.float32))
    wt = torch.as_tensor(w, dtype=torch.float32)
    y = m.lora_expand_add(dev(Zh), dev(inp.B2), al, 2, dev(O), out_fp32=True, topk_w=dev(wt))
    assert_close(y, oracle.lora_expand_add(Zh, inp.B2, ref, O[:n], epilogue=2, w=wt),
                 KERNEL_RTOL, "expand epilogue 2, token walk")


@pytest.mark.parametrize("K", [136, 768, 2048])
@pytest.mark.parametrize("r", [32, 24])
def test_shrink_short_blocks_all_ranks(K, r):
    """Many short blocks (the many-adapter stress shape): one CTA takes all ranks of a block;
    K <= 832 stages the A slab in shared memory through asynchronous copies (K = 136: a
    partial last k-step), longer K loads two k-steps per batch into registers; r = 24 leaves
    the last rank tile partial."""
    m, inp, ids, w, al, ref = _setup(T=256, H=K, I=8, E=128, k=8, L=16, r=r, seed=18,
                                     bm_lora=8, adapters="zipf1.1")
    Z = Guarded((al.S, r), torch.float32, fill=0.0)
    m.lora_shrink(dev(inp.x), False, dev(inp.A1), al, out=Z.t)
    Z.check()
    assert_close(Z.t, oracle.lora_shrink(inp.x, inp.A1, ref, False), KERNEL_RTOL, f"K={K} r={r}")
    # the down shrink's form: rows addressed by sorted row
    n = ref["n_valid"]
    h = torch.from_numpy(np.random.default_rng(9).standard_normal((al.S, K), dtype=np.float32)).to(torch.bfloat16)
    Z2 = m.lora_shrink(dev(h), True, dev(inp.A1), al)
    assert_close(Z2, oracle.lora_shrink(h[:n], inp.A1, ref, rows_are_slots=True), KERNEL_RTOL,
                 f"sorted rows K={K} r={r}")


@pytest.mark.parametrize("K", [768, 136])
def test_shrink_short_blocks_fewer_items_than_ctas(K):
    """The short-K shrink's grid covers the host's block bound (~1000 here): with one adapter
    (a third of the tokens without one) only ~135 blocks are live, so most CTAs find no
    block and leave before any copy."""
    T = 128
    adapters = np.where(np.arange(T) % 3 == 0, -1, 0).astype(np.int32)
    m, inp, ids, w, al, ref = _setup(T=T, H=K, I=8, E=128, k=8, L=16, r=32, seed=23,
                                     bm_lora=8, adapters=adapters)
    assert len(ref["lora_blocks"]) < 304
    Z = Guarded((al.S, 32), torch.float32, fill=0.0)
    m.lora_shrink(dev(inp.x), False, dev(inp.A1), al, out=Z.t)
    Z.check()
    assert_close(Z.t, oracle.lora_shrink(inp.x, inp.A1, ref, False), KERNEL_RTOL, f"K={K}")


@pytest.mark.parametrize("I", [300, 302, 1024])
@pytest.mark.parametrize("r", [16, 64])
def test_expand_swiglu_long_segments_ragged(I, r):
    """Long (expert, adapter) segments take the tensor-core SwiGLU expand, whose G rows
    stream through a ring of asynchronous copies: a ragged last column tile (I = 300),
    I % 4 != 0 (302, the CUDA-core fallback) and two rank chunks (r = 64)."""
    m, inp, ids, w, al, ref = _setup(T=512, H=64, I=I, E=4, k=2, L=2, r=r, seed=19)
    n = ref["n_valid"]
    rng = np.random.default_rng(8)
    Zh = torch.from_numpy(rng.standard_normal((al.S, r))).to(torch.float32)
    G = torch.from_numpy(rng.standard_normal((al.S, 2 * I), dtype=np.float32))
    h = Guarded((al.S, I), torch.bfloat16)
    m.lora_expand_add(dev(Zh), dev(inp.B1), al, 1, dev(G), out=h.t)
    h.check()
    assert_bf16_close(h.t[:n], oracle.lora_expand_add(Zh, inp.B1, ref, G[:n], epilogue=1),
                      f"expand epilogue 1, long segments, I={I} r={r}")


@pytest.mark.parametrize("shape", ["short", "long", "long_ragged"])
@pytest.mark.parametrize("r", [5, 8, 32, 64])
def test_expand_two_slices(shape, r):
    """Epilogue 3: SwiGLU with separate gate and up adapters (z rows of 2r values, the up
    columns taking the second r), on each form of the expand: one row per CTA (short
    segments), the tensor-core block walk (long segments) and the CUDA-core row walk
    (I % 4 != 0, or r not a multiple of 8)."""
    if shape == "short":
        T, I, E, k, L = 48, 300, 32, 4, 8
        adapters = "round_robin_shuffled"
    else:
        T, I, E, k, L = 512, (300 if shape == "long" else 302), 4, 2, 2
        adapters = "uniform_with_none"
    m, inp, ids, w, al, ref = _setup(T=T, H=64, I=I, E=E, k=k, L=L, r=r, seed=20,
                                     adapters=adapters)
    n = ref["n_valid"]
    rng = np.random.default_rng(10)
    Zh = torch.from_numpy(rng.standard_normal((al.S, 2 * r))).to(torch.float32)
    G = torch.from_numpy(rng.standard_normal((al.S, 2 * I), dtype=np.float32))
    h = Guarded((al.S, I), torch.bfloat16)
    m.lora_expand_add(dev(Zh), dev(inp.B1), al, 3, dev(G), out=h.t)
    h.check()
    assert_bf16_close(h.t[:n], oracle.lora_expand_add(Zh, inp.B1, ref, G[:n], epilogue=3),
                      f"epilogue 3, {shape} segments, r={r}")


def _poison_A(A, ranks, rank):
    """A with the rows past each adapter's rank (per slice of `rank` rows) set to NaN."""
    A = A.clone()
    for l, rl in enumerate(ranks):
        for sl in range(A.shape[2] // rank):
            A[l, :, sl * rank + min(max(rl, 0), rank): (sl + 1) * rank] = float("nan")
    return A


def _poison_B(B, ranks):
    B = B.clone()
    for l, rl in enumerate(ranks):
        B[l, :, :, min(max(rl, 0), B.shape[3]):] = float("nan")
    return B


@pytest.mark.parametrize("case", ["decode", "stress_regs", "stress_smem", "prefill"])
def test_shrink_adapter_ranks(case):
    """Adapters of their own ranks (8, 0, 5, 16, full): the rows of A past an adapter's rank
    hold NaN and must never be used; z past the rank is 0. Every shrink form."""
    if case == "decode":
        kw = dict(T=64, H=2880, E=32, k=4, L=8, r=32, bm_lora=8, adapters="round_robin_shuffled")
    elif case == "stress_regs":
        kw = dict(T=256, H=2048, E=128, k=8, L=16, r=32, bm_lora=8, adapters="zipf1.1")
    elif case == "stress_smem":
        kw = dict(T=256, H=768, E=128, k=8, L=16, r=32, bm_lora=8, adapters="zipf1.1")
    else:
        kw = dict(T=1024, H=512, E=8, k=2, L=16, r=16, bm_lora=16, adapters="one_per_request16")
    m, inp, ids, w, al, ref = _setup(I=8, seed=22, **kw)
    r = kw["r"]
    ranks = [[8, 0, 5, 16, r][l % 5] for l in range(kw["L"])]
    A = _poison_A(inp.A1, ranks, r)
    rk = torch.as_tensor(ranks, dtype=torch.int32)
    Z = m.lora_shrink(dev(inp.x), False, dev(A), al, adapter_ranks=dev(rk))
    expect = oracle.lora_shrink(inp.x, A, ref, False, adapter_ranks=rk)
    assert not torch.isnan(Z).any()
    assert_close(Z, expect, KERNEL_RTOL, f"ranked shrink, {case}")
    assert m.get_error(al.buf) == 0


@pytest.mark.parametrize("epilogue", [0, 1, 2, 3])
@pytest.mark.parametrize("seg", ["short", "long"])
@pytest.mark.parametrize("r", [16, 64, 5])
def test_expand_adapter_ranks(epilogue, seg, r):
    """The expand with adapters of their own ranks: B columns past an adapter's rank hold NaN
    and must never be used (z there is arbitrary); every epilogue on the CUDA-core forms
    (short segments, r = 5) and the tensor-core forms (long segments)."""
    if seg == "short":
        T, H, I, E, k, L, adapters = 48, 96, 80, 32, 4, 8, "round_robin_shuffled"
    else:
        T, H, I, E, k, L, adapters = 512, 96, 80, 4, 2, 5, "uniform_with_none"
    m, inp, ids, w, al, ref = _setup(T=T, H=H, I=I, E=E, k=k, L=L, r=r, seed=23, adapters=adapters)
    n = ref["n_valid"]
    ranks = [[r, 0, min(8, r), 3, max(r - 1, 0)][l % 5] for l in range(L)]
    rk = torch.as_tensor(ranks, dtype=torch.int32)
    rng = np.random.default_rng(11)
    zc = 2 * r if epilogue == 3 else r
    Zh = torch.from_numpy(rng.standard_normal((al.S, zc))).to(torch.float32)
    if epilogue == 2:
        B = _poison_B(inp.B2, ranks)
        O = torch.from_numpy(rng.standard_normal((al.S, H), dtype=np.float32))
        wt = torch.as_tensor(w, dtype=torch.float32)
        y = m.lora_expand_add(dev(Zh), dev(B), al, 2, dev(O), out_fp32=True, topk_w=dev(wt),
                              adapter_ranks=dev(rk))
        expect = oracle.lora_expand_add(Zh, B, ref, O[:n], epilogue=2, w=wt, adapter_ranks=rk)
        assert_close(y, expect, KERNEL_RTOL, f"ranked epilogue 2, {seg}, r={r}")
        return
    B = _poison_B(inp.B1 if epilogue else inp.B2, ranks)
    N = B.shape[2]
    G = torch.from_numpy(rng.standard_normal((al.S, N), dtype=np.float32))
    out = m.lora_expand_add(dev(Zh), dev(B), al, epilogue, dev(G), adapter_ranks=dev(rk))
    expect = oracle.lora_expand_add(Zh, B, ref, G[:n], epilogue=epilogue, adapter_ranks=rk)
    if epilogue == 0:
        assert_close(out[:n], expect, KERNEL_RTOL, f"ranked epilogue 0, {seg}, r={r}")
    else:
        assert_bf16_close(out[:n], expect, f"ranked epilogue {epilogue}, {seg}, r={r}")
