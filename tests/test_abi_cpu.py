"""The C-ABI library on a machine without a GPU: it loads, exports every symbol
the header declares (and nothing else), sizes its buffers, and rejects invalid
arguments on the host before any CUDA call. No compute call is made here."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_lora.h")


@pytest.fixture(scope="session")
def L():
    from expert_adapter_gemms_gb300 import build as b
    if not os.path.exists(b.LIB_PATH):
        b.build()
    import expert_adapter_gemms_gb300 as m
    return m.lib()


def declared_symbols():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_LORA_API\s+[a-z_0-9 \*]+?\b([a-z_0-9]+)\(", txt)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ["moe_lora_align", "moe_grouped_gemm", "lora_shrink", "lora_expand_add",
              "moe_lora_layer", "moe_topk_softmax", "moe_lora_get_error"]:
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in declared_symbols():
        assert hasattr(L, n), n


def test_only_declared_symbols_are_exported(L):
    from expert_adapter_gemms_gb300 import LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("nm unavailable")
    exported = set()
    for line in out.stdout.splitlines():
        parts = line.split()
        if len(parts) == 3 and parts[1] in ("T", "W"):
            exported.add(parts[2])
    ours = {s for s in exported if s.startswith(("moe_", "lora_"))}
    assert ours == set(declared_symbols())


def test_no_runtime_compiler_linked():
    """Every kernel is compiled ahead of time for sm_103a: no JIT library is needed."""
    from expert_adapter_gemms_gb300 import LIB_PATH, build as b
    out = subprocess.run(["readelf", "-d", LIB_PATH], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("readelf unavailable")
    assert "nvrtc" not in out.stdout and "nvJitLink" not in out.stdout
    assert b.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings(L):
    import expert_adapter_gemms_gb300 as m
    assert m.status_string(0) == "ok"
    assert "workspace" in m.status_string(4)


def test_align_layout_and_sizes(L):
    import expert_adapter_gemms_gb300 as m
    for (T, k, E, Ln, bb, bl) in [(8, 2, 4, 2, 16, 16), (64, 4, 32, 8, 16, 16),
                                  (4096, 4, 32, 16, 256, 16), (256, 8, 128, 128, 32, 16),
                                  (0, 2, 4, 0, 16, 1), (5000, 4, 8, 3, 64, 7)]:
        offs = m.align_layout(T, k, E, Ln, bb, bl)
        S = T * k
        total = L.moe_lora_align_buffer_size(T, k, E, Ln, bb, bl)
        assert total == offs[11] > 0
        field_offs = [offs[i] for i in (0, 1, 2, 3, 4, 5, 6, 7, 10)]
        assert field_offs == sorted(field_offs)
        assert all(o % 256 == 0 for o in field_offs)
        assert offs[2] - offs[1] >= 4 * S
        max_tiles, max_blocks = offs[8], offs[9]
        assert max_tiles >= -(-S // bb) + min(E, S) - 1  # covers every expert's ragged tail
        assert max_blocks >= 1


def test_align_rejects_bad_tiles(L):
    assert L.moe_lora_align_buffer_size(8, 2, 4, 2, 24, 16) == 0     # bm_base not a multiple of 16
    assert L.moe_lora_align_buffer_size(8, 2, 4, 2, 512, 16) == 0    # bm_base too large
    assert L.moe_lora_align_buffer_size(8, 2, 4, 2, 16, 0) == 0
    assert L.moe_lora_align_buffer_size(8, 2, 4, 2, 16, 17) == 0
    assert L.moe_lora_align_buffer_size(-1, 2, 4, 2, 16, 16) == 0
    assert L.moe_lora_align_buffer_size(1 << 21, 4, 4, 2, 16, 16) == 0  # more than 1<<22 slots


def test_workspace_size(L):
    import expert_adapter_gemms_gb300 as m
    a = m.moe_lora_workspace_size(64, 4, 32, 8, 2880, 2880, 32)
    b = m.moe_lora_workspace_size(128, 4, 32, 8, 2880, 2880, 32)
    assert 0 < a < b
    # intermediates: xs, G, h, O (bf16/fp32) dominate
    S = 64 * 4
    assert a >= S * (2880 * 2 + 5760 * 4 + 2880 * 2 + 2880 * 4)
    assert m.moe_lora_workspace_size(64, 4, 32, 0, 2880, 2880, 0) < a
    assert m.moe_lora_workspace_size(64, 0, 32, 8, 2880, 2880, 32) == 0


def test_layer_tiles_heuristic(L):
    import expert_adapter_gemms_gb300 as m
    assert m.moe_lora_layer_tiles(64, 4, 32, 8, 2880, 2880, 32)[0] == 16
    assert m.moe_lora_layer_tiles(4096, 4, 32, 16, 2880, 2880, 16)[0] == 256
    assert m.moe_lora_layer_tiles(256, 8, 128, 128, 2048, 768, 32)[0] == 32
    for T in (1, 7, 64, 513, 4096):
        b, l = m.moe_lora_layer_tiles(T, 4, 32, 8, 2880, 2880, 32)
        assert b in (16, 32, 64, 128, 256) and 1 <= l <= 16


def test_expert_major_and_down_shares_heuristic(L):
    """Expert-major chunks where each expert's rows fit one chunk: up to 32 rows per expert
    on average, up to 64 where the count is exact (one expert: a dense layer); MoE at 48 or
    64 rows per expert keeps token tiles (an expert above the chunk would stream its
    weights once per chunk). The dense layer's down GEMM splits its K range into up to eight
    shares (each a partial output in the workspace), the MoE decode shape into two."""
    import expert_adapter_gemms_gb300 as m
    plan = m.moe_lora_layer_plan
    assert plan(64, 1, 1, 8, 4096, 14336, 16)["expert_major_rows"] == 64
    assert plan(64, 1, 1, 8, 4096, 14336, 16)["fused_expand"] == 1
    assert plan(65, 1, 1, 8, 4096, 14336, 16)["expert_major_rows"] == 0
    assert plan(64, 4, 32, 8, 2880, 2880, 32)["expert_major_rows"] == 32
    assert plan(256, 4, 32, 8, 2880, 2880, 32)["expert_major_rows"] == 64
    assert plan(384, 4, 32, 8, 2880, 2880, 32)["expert_major_rows"] == 0
    assert plan(512, 4, 32, 8, 2880, 2880, 32)["expert_major_rows"] == 0
    # the partial outputs: S H fp32 per share (8 for the dense 4096-wide layer, 2 at the
    # GPT-OSS decode shape), so the dense workspace grows by 6 S H 4 bytes over two shares
    S, H = 64, 4096
    dense = m.moe_lora_workspace_size(64, 1, 1, 8, 4096, 14336, 16)
    assert dense >= S * H * 4 * 8
    moe = m.moe_lora_workspace_size(64, 4, 32, 8, 2880, 2880, 32)
    assert 256 * 2880 * 4 * 2 < moe < 256 * 2880 * 4 * 8  # two shares, not eight


def test_host_validation_before_any_cuda_call(L):
    P = ctypes.c_void_p
    fake = P(0x1000)  # never dereferenced: every call below fails validation first
    assert L.moe_topk_softmax(fake, -1, 4, 2, fake, fake, None) == 1
    assert L.moe_topk_softmax(fake, 4, 4, 5, fake, fake, None) == 1       # k > E
    assert L.moe_topk_softmax(fake, 4, 2048, 2, fake, fake, None) == 2    # E > 1024
    assert L.moe_topk_softmax(None, 4, 4, 2, fake, fake, None) == 1       # null logits
    from expert_adapter_gemms_gb300._lib import AlignDesc
    bad = AlignDesc(None, 8, 2, 4, 2, 16, 16)
    assert L.moe_lora_align(fake, fake, ctypes.byref(bad), None) == 1     # null buffer
    odd = AlignDesc(0x1010, 8, 2, 4, 2, 16, 16)
    assert L.moe_lora_align(fake, fake, ctypes.byref(odd), None) == 1     # not 256-byte aligned
    tiles = AlignDesc(0x1000, 8, 2, 4, 2, 24, 16)
    assert L.moe_lora_align(fake, fake, ctypes.byref(tiles), None) == 2
    ok = AlignDesc(0x1000, 8, 2, 4, 2, 16, 16)
    assert L.moe_grouped_gemm(fake, fake, ctypes.byref(ok), 64, 100, fake, None) == 2  # K % 8
    assert L.moe_grouped_gemm(P(0x1008), fake, ctypes.byref(ok), 64, 64, fake, None) == 1
    assert L.lora_shrink(fake, 2, fake, ctypes.byref(ok), 64, 8, fake, None) == 1
    assert L.lora_shrink(fake, 0, fake, ctypes.byref(ok), 64, 300, fake, None) == 2
    assert L.lora_expand_add(fake, fake, ctypes.byref(ok), 64, 8, 4, fake, fake, 0, fake,
                             None) == 1  # epilogues are 0..3
    assert L.lora_expand_add(fake, fake, ctypes.byref(ok), 63, 8, 3, fake, fake, 0, fake,
                             None) == 1  # SwiGLU epilogues need an even N
    assert L.lora_expand_add(fake, fake, ctypes.byref(ok), 63, 8, 1, fake, fake, 0, fake,
                             None) == 1                                     # SwiGLU needs even N
    args = [fake, fake, None, None, None, 8, 256, 512, 4, 2, fake, fake, fake, fake, fake, fake,
            2, 8, fake, 0, P(0x100000), 1 << 30, None]
    a = list(args); a[6] = 100                                               # H % 8
    assert L.moe_lora_layer(*a) == 2
    a = list(args); a[2] = fake; a[3] = fake                                 # logits and ids
    assert L.moe_lora_layer(*a) == 1
    a = list(args); a[9] = 5                                                 # k > E
    assert L.moe_lora_layer(*a) == 1
    a = list(args); a[21] = 16                                               # workspace too small
    assert L.moe_lora_layer(*a) == 4
    a = list(args); a[14] = None                                             # L > 0 needs A2
    assert L.moe_lora_layer(*a) == 1
    a = list(args); a[5] = 0                                                 # T = 0: nothing to do
    assert L.moe_lora_layer(*a) == 0


def test_host_io_layout(L):
    """The host-staged call's block: x, logits, adapter ids, then y, each at a 256-byte
    aligned offset, back to back, and the input block ending where the last input ends."""
    off = (ctypes.c_int64 * 4)()
    ib, sb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    for T, H, E, wa, yf in [(64, 2880, 32, 1, 0), (5, 8, 3, 0, 1), (7, 24, 128, 1, 1)]:
        assert L.moe_lora_host_io_layout(T, H, E, wa, yf, off, ctypes.byref(ib),
                                         ctypes.byref(sb)) == 0
        sizes = [T * H * 2, T * E * 4, T * 4 if wa else 0, T * H * (4 if yf else 2)]
        used = [i for i in range(4) if i != 2 or wa]
        assert off[0] == 0 and (off[2] == -1) == (not wa)
        prev_end = 0
        for i in used:
            assert off[i] % 256 == 0 and off[i] >= prev_end and off[i] - prev_end < 256
            prev_end = off[i] + sizes[i]
        last_in = 2 if wa else 1
        assert ib.value == off[last_in] + sizes[last_in]
        assert sb.value == off[3] + sizes[3]
    assert L.moe_lora_host_io_layout(4, 8, 2, 2, 0, off, None, None) == 1   # with_adapter 0/1
    assert L.moe_lora_host_io_layout(4, 8, 2, 1, 0, None, None, None) == 1  # no offsets array


def test_host_staged_layer_validation(L):
    """moe_lora_layer_host checks its own arguments and the layer's before any copy."""
    P = ctypes.c_void_p
    fake = P(0x1000)
    args = [fake, fake, P(0x100000), 1 << 30, 1, 8, 256, 512, 4, 2, fake, fake, fake, fake, fake,
            fake, 2, 8, 0, P(0x200000), 1 << 30, None, None]
    a = list(args); a[0] = None                                              # no host block
    assert L.moe_lora_layer_host(*a) == 1
    a = list(args); a[2] = P(0x100010)                                       # staging alignment
    assert L.moe_lora_layer_host(*a) == 1
    a = list(args); a[3] = 1024                                              # staging too short
    assert L.moe_lora_layer_host(*a) == 4
    a = list(args); a[6] = 100                                               # H % 8
    assert L.moe_lora_layer_host(*a) == 2
    a = list(args); a[9] = 5                                                 # k > E
    assert L.moe_lora_layer_host(*a) == 1
    a = list(args); a[20] = 16                                               # workspace too small
    assert L.moe_lora_layer_host(*a) == 4
    a = list(args); a[4] = 3                                                 # with_adapter 0/1
    assert L.moe_lora_layer_host(*a) == 1
    a = list(args); a[5] = 0                                                 # T = 0: nothing to do
    assert L.moe_lora_layer_host(*a) == 0


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "expert_adapter_gemms_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in txt and "from oracle" not in txt, f


def test_chain_early_reads_come_from_completed_launches(L):
    """Under programmatic dependent launch some kernels read before their own wait: the
    shrinks read x or the gathered rows and the align tables, the grouped GEMMs the token
    tiles (and, fused, the gathered rows or h), the expand kernels G or O, B and the
    tables. The library checks each such read when it plans the chain (the producer at
    least two launches back, the launch in between triggering only after its own wait)
    and refuses a chain that breaks the rule; here every shape and option combination is
    planned and the number of checked reads is pinned per chain:
      fused, adapters: shrink1 <- align; GEMM1 <- gather, align; shrink2 <- align (its
        block, before prefetching A); GEMM2 <- GEMM1, align; combine <- align, route
        = 8 (7 where the align routes the tokens itself)
      separate expand, expert-major: shrink1 <- gather, align; expand1 <- GEMM1, align;
        shrink2 <- expand1, align; expand2 <- GEMM2, align, route = 9 (8 where the align
        routes the tokens itself: the weights then come from the align)
      separate expand, token tiles: + GEMM1 <- align, GEMM2 <- align, shrink1 by token
        (no gather) = 10
      no adapters: the GEMMs read token tiles early only in tile mode (the fused
        chain's combine reads the align's and the route's outputs early)."""
    import itertools
    import expert_adapter_gemms_gb300 as m
    shapes = [(8, 2, 4, 2, 256, 512, 8), (64, 4, 32, 8, 2880, 2880, 32),
              (4096, 4, 32, 16, 2880, 2880, 16), (512, 2, 8, 32, 4096, 11008, 64),
              (256, 8, 128, 128, 2048, 768, 32), (300, 2, 4, 0, 256, 192, 16)]
    for (T, k, E, Ln, H, I, r), mode, pdl, slices in itertools.product(
            shapes, (0, 1), (True, False), (1, 2)):
        p = m.moe_lora_layer_plan(T, k, E, Ln, H, I, r, expand_mode=mode, disable_pdl=not pdl,
                                  gate_up_slices=slices)
        if not pdl:
            assert p["early_reads"] == 0
            continue
        if Ln == 0:
            fused = 2 - p["route_in_align"]  # the combine's slot rows and weights
            assert p["early_reads"] == (fused if p["fused_expand"] else
                                        0 if p["expert_major_rows"] else 2), (T, mode, p)
        elif p["fused_expand"]:
            assert p["early_reads"] == 8 - p["route_in_align"], (T, mode, p)
        elif p["expert_major_rows"]:
            assert p["early_reads"] == 9 - p["route_in_align"], (T, mode, p)
        else:
            assert p["early_reads"] == 10 - p["route_in_align"], (T, mode, p)
