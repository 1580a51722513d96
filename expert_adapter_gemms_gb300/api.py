"""Python entry points with the C ABI's names, over torch tensors on the GPU.

Each function checks its tensors, allocates outputs (torch owns device memory)
and calls the library on the current stream; nothing here computes. Shapes and
layouts follow include/moe_lora.h.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

from . import _lib as L_
from ._lib import AlignDesc, LayerOpts, LayerPlan, check, lib, ptr, stream_handle


def _need(t: torch.Tensor, name: str, dtype, ndim: Optional[int] = None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device (there is no CPU path)")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def moe_topk_softmax(logits: torch.Tensor, k: int):
    """Top-k experts per token and softmax weights over the chosen logits."""
    _need(logits, "logits", torch.float32, 2)
    T, E = logits.shape
    ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    check(lib().moe_topk_softmax(ptr(logits), T, E, k, ptr(ids), ptr(w), stream_handle()),
          "moe_topk_softmax")
    return ids, w


def align_layout(T: int, k: int, E: int, L: int, bm_base: int, bm_lora: int) -> list:
    offs = (ctypes.c_int64 * L_.ALIGN_NFIELDS)()
    check(lib().moe_lora_align_layout(T, k, E, L, bm_base, bm_lora, offs), "moe_lora_align_layout")
    return list(offs)


@dataclass
class Align:
    """An align buffer (device) plus the host description the library needs."""
    buf: torch.Tensor
    T: int
    k: int
    E: int
    L: int
    bm_base: int
    bm_lora: int

    @property
    def S(self) -> int:
        return self.T * self.k

    def desc(self) -> AlignDesc:
        return AlignDesc(ptr(self.buf), self.T, self.k, self.E, self.L, self.bm_base, self.bm_lora)

    def _offsets(self):
        return align_layout(self.T, self.k, self.E, self.L, self.bm_base, self.bm_lora)

    def _i32(self, field: int, n: int) -> torch.Tensor:
        off = self._offsets()[field]
        return self.buf[off: off + 4 * n].view(torch.int32)

    def header(self) -> dict:
        h = self._i32(L_.AF_HEADER, 16).cpu().tolist()
        return dict(err=h[0] & 0xffffffff, n_valid=h[1], n_tiles=h[2], n_lora_blocks=h[3],
                    n_lora_rows=h[4])

    def sorted_slots(self):
        return self._i32(L_.AF_SORTED_SLOTS, self.S)

    def slot_row(self):
        return self._i32(L_.AF_SLOT_ROW, self.S)

    def row_expert(self):
        return self._i32(L_.AF_ROW_EXPERT, self.S)

    def row_adapter(self):
        return self._i32(L_.AF_ROW_ADAPTER, self.S)

    def expert_begin(self):
        return self._i32(L_.AF_EXPERT_BEGIN, self.E + 1)

    def tiles(self):
        o = self._offsets()
        return self._i32(L_.AF_TILES, 4 * o[L_.AF_MAX_TILES]).view(-1, 4)

    def lora_blocks(self):
        o = self._offsets()
        return self._i32(L_.AF_LORA_BLOCKS, 4 * o[L_.AF_MAX_LORA_BLOCKS]).view(-1, 4)


def new_align(T: int, k: int, E: int, L: int, bm_base: int, bm_lora: int,
              device="cuda") -> Align:
    n = lib().moe_lora_align_buffer_size(T, k, E, L, bm_base, bm_lora)
    if n == 0:
        raise L_.MoeLoraError(L_.ERR_UNSUPPORTED, "moe_lora_align_buffer_size")
    buf = torch.zeros(n, dtype=torch.uint8, device=device)
    return Align(buf, T, k, E, L, bm_base, bm_lora)


def moe_lora_align(ids: torch.Tensor, token_adapter: Optional[torch.Tensor], E: int, L: int,
                   bm_base: int = 64, bm_lora: int = 16, al: Optional[Align] = None) -> Align:
    """Stable (expert, adapter, slot) sort of the slots, tiles and LoRA blocks."""
    _need(ids, "ids", torch.int32, 2)
    T, k = ids.shape
    if token_adapter is not None:
        _need(token_adapter, "token_adapter", torch.int32, 1, (T,))
    if al is None:
        al = new_align(T, k, E, L, bm_base, bm_lora, ids.device)
    d = al.desc()
    check(lib().moe_lora_align(ptr(ids), ptr(token_adapter), ctypes.byref(d), stream_handle()),
          "moe_lora_align")
    return al


def get_error(buf: torch.Tensor) -> int:
    v = ctypes.c_uint32(0)
    st = lib().moe_lora_get_error(ptr(buf), stream_handle(), ctypes.byref(v))
    if st not in (L_.OK, L_.ERR_TIMEOUT):
        check(st, "moe_lora_get_error")
    return int(v.value)


def clear_error(buf: torch.Tensor) -> None:
    check(lib().moe_lora_clear_error(ptr(buf), stream_handle()), "moe_lora_clear_error")


def moe_gather_rows(x: torch.Tensor, al: Align, out: Optional[torch.Tensor] = None):
    _need(x, "x", torch.bfloat16, 2)
    H = x.shape[1]
    if out is None:
        out = torch.zeros((al.S, H), dtype=torch.bfloat16, device=x.device)
    _need(out, "out", torch.bfloat16, 2, (al.S, H))
    d = al.desc()
    check(lib().moe_gather_rows(ptr(x), ctypes.byref(d), H, ptr(out), stream_handle()),
          "moe_gather_rows")
    return out


def moe_grouped_gemm(a_sorted: torch.Tensor, W: torch.Tensor, al: Align,
                     out: Optional[torch.Tensor] = None):
    """out[row] = a_sorted[row] @ W[expert(row)].T for the sorted rows (fp32 out)."""
    _need(a_sorted, "a_sorted", torch.bfloat16, 2)
    _need(W, "W", torch.bfloat16, 3)
    E, N, K = W.shape
    if a_sorted.shape[1] != K or a_sorted.shape[0] != al.S or E != al.E:
        raise ValueError("shape mismatch between a_sorted, W and the align buffer")
    if out is None:
        out = torch.zeros((al.S, N), dtype=torch.float32, device=W.device)
    _need(out, "out", torch.float32, 2, (al.S, N))
    d = al.desc()
    check(lib().moe_grouped_gemm(ptr(a_sorted), ptr(W), ctypes.byref(d), N, K, ptr(out),
                                 stream_handle()), "moe_grouped_gemm")
    return out


def _with_ranks(d: AlignDesc, adapter_ranks: Optional[torch.Tensor], L: int) -> AlignDesc:
    if adapter_ranks is not None:
        _need(adapter_ranks, "adapter_ranks", torch.int32, 1, (L,))
        d.adapter_ranks = ptr(adapter_ranks)
    return d


def lora_shrink(X: torch.Tensor, rows_are_slots: bool, A: torch.Tensor, al: Align,
                out: Optional[torch.Tensor] = None, adapter_ranks: Optional[torch.Tensor] = None):
    """Z[s] = X[in(s)] @ A[l(s), e(s)].T for the slots with an adapter (fp32 out);
    adapter_ranks [L] int32 (device): adapter l uses the first r_l rows of A."""
    _need(X, "X", torch.bfloat16, 2)
    _need(A, "A", torch.bfloat16, 4)
    Ln, E, r, K = A.shape
    if X.shape[1] != K or E != al.E or Ln != al.L:
        raise ValueError("shape mismatch between X, A and the align buffer")
    if out is None:
        out = torch.zeros((al.S, r), dtype=torch.float32, device=X.device)
    _need(out, "out", torch.float32, 2, (al.S, r))
    d = _with_ranks(al.desc(), adapter_ranks, al.L)
    check(lib().lora_shrink(ptr(X), int(bool(rows_are_slots)), ptr(A), ctypes.byref(d), K, r,
                            ptr(out), stream_handle()), "lora_shrink")
    return out


def lora_expand_add(Z: torch.Tensor, B: Optional[torch.Tensor], al: Align, epilogue: int,
                    base: torch.Tensor, out: Optional[torch.Tensor] = None, out_fp32: bool = False,
                    topk_w: Optional[torch.Tensor] = None, N: Optional[int] = None,
                    adapter_ranks: Optional[torch.Tensor] = None):
    """Expand with the base add fused; epilogue 0 (in place), 1 (SwiGLU), 2 (combine),
    3 (SwiGLU with separate gate and up adapters: Z rows hold 2r values). adapter_ranks
    [L] int32 (device): adapter l uses the first r_l columns of B."""
    _need(base, "base", torch.float32, 2)
    Nb = base.shape[1]
    r = 0
    if B is not None:
        _need(B, "B", torch.bfloat16, 4)
        r = B.shape[3]
        if B.shape[2] != Nb or B.shape[1] != al.E or B.shape[0] != al.L:
            raise ValueError("shape mismatch between B, base and the align buffer")
        _need(Z, "Z", torch.float32, 2, (al.S, 2 * r if epilogue == 3 else r))
    dev = base.device
    if epilogue in (1, 3) and out is None:
        out = torch.zeros((al.S, Nb // 2), dtype=torch.bfloat16, device=dev)
    if epilogue == 2 and out is None:
        out = torch.zeros((al.T, Nb), dtype=torch.float32 if out_fp32 else torch.bfloat16,
                          device=dev)
    if epilogue == 2:
        _need(topk_w, "topk_w", torch.float32, 2, (al.T, al.k))
    d = _with_ranks(al.desc(), adapter_ranks, al.L)
    check(lib().lora_expand_add(ptr(Z) if B is not None else 0, ptr(B), ctypes.byref(d), Nb, r,
                                epilogue, ptr(base), ptr(out), int(out_fp32), ptr(topk_w),
                                stream_handle()), "lora_expand_add")
    return base if epilogue == 0 else out


def moe_lora_workspace_size(T: int, k: int, E: int, L: int, H: int, I: int, r: int) -> int:
    return int(lib().moe_lora_workspace_size(T, k, E, L, H, I, r))


def moe_lora_layer_tiles(T: int, k: int, E: int, L: int, H: int, I: int, r: int):
    b = ctypes.c_int32(0)
    l_ = ctypes.c_int32(0)
    check(lib().moe_lora_layer_tiles(T, k, E, L, H, I, r, ctypes.byref(b), ctypes.byref(l_)),
          "moe_lora_layer_tiles")
    return b.value, l_.value


def moe_lora_layer_plan(T: int, k: int, E: int, L: int, H: int, I: int, r: int, *,
                        bm_base: int = 0, bm_lora: int = 0, disable_pdl: bool = False,
                        gate_up_slices: int = 1, adapter_ranks: bool = False,
                        expand_mode: int = 0) -> dict:
    """How the layer runs this shape with these options: tiles, expert-major chunk rows,
    whether the expand is fused into the grouped GEMMs, and kernels per call."""
    opts = LayerOpts()
    opts.bm_base, opts.bm_lora, opts.disable_pdl = bm_base, bm_lora, int(disable_pdl)
    opts.gate_up_slices, opts.expand_mode = gate_up_slices, expand_mode
    if adapter_ranks:  # only whether an array is given matters to the plan
        opts.adapter_ranks = 1
    out = LayerPlan()
    check(lib().moe_lora_layer_plan(T, k, E, L, H, I, r, ctypes.byref(opts), ctypes.byref(out)),
          "moe_lora_layer_plan")
    return {f: getattr(out, f) for f, _ in LayerPlan._fields_}


def new_workspace(T: int, k: int, E: int, L: int, H: int, I: int, r: int, device="cuda"):
    n = moe_lora_workspace_size(T, k, E, L, H, I, r)
    if n == 0:
        raise L_.MoeLoraError(L_.ERR_UNSUPPORTED, "moe_lora_workspace_size")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    ws[:256].zero_()  # the sticky error word starts clear
    return ws


def _layer_weights(H: int, W1, W2, A1, B1, A2, B2, gate_up_slices: int):
    """Checks the layer's weights against hidden size H; returns (E, I, L, r)."""
    _need(W1, "W1", torch.bfloat16, 3)
    _need(W2, "W2", torch.bfloat16, 3)
    E, twoI, H1 = W1.shape
    I = twoI // 2
    if H1 != H or tuple(W2.shape) != (E, H, I):
        raise ValueError("W1/W2 shapes do not match x")
    Ln, r = 0, 0
    if gate_up_slices not in (1, 2):
        raise ValueError("gate_up_slices must be 1 or 2")
    if A1 is not None:
        _need(A1, "A1", torch.bfloat16, 4)
        Ln, _, r, _ = A1.shape
        if r % gate_up_slices:
            raise ValueError("A1 rows must hold gate_up_slices adapters of equal rank")
        r //= gate_up_slices
        _need(B1, "B1", torch.bfloat16, 4, (Ln, E, twoI, r))
        _need(A2, "A2", torch.bfloat16, 4, (Ln, E, r, I))
        _need(B2, "B2", torch.bfloat16, 4, (Ln, E, H, r))
    return E, I, Ln, r


def _layer_opts(Ln: int, bm_base: int, bm_lora: int, disable_pdl: bool, events,
                gate_up_slices: int, adapter_ranks, wait_limit_ns: int = 0,
                expand_mode: int = 0, mma_pairs: int = 0):
    """The layer options struct, and the event array it points to (keep it alive)."""
    opts = LayerOpts()
    opts.bm_base, opts.bm_lora, opts.disable_pdl = bm_base, bm_lora, int(disable_pdl)
    opts.gate_up_slices = gate_up_slices
    opts.wait_limit_ns = int(wait_limit_ns)
    opts.expand_mode = int(expand_mode)
    opts.mma_pairs = int(mma_pairs)
    if adapter_ranks is not None:
        _need(adapter_ranks, "adapter_ranks", torch.int32, 1, (Ln,))
        opts.adapter_ranks = ptr(adapter_ranks)
    ev_arr = None
    if events:
        ev_arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
        opts.num_events = len(events)
        opts.events = ctypes.cast(ev_arr, ctypes.POINTER(ctypes.c_void_p))
    return opts, ev_arr


def moe_lora_layer(x: torch.Tensor, W1: torch.Tensor, W2: torch.Tensor, *,
                   logits: Optional[torch.Tensor] = None, topk_ids: Optional[torch.Tensor] = None,
                   topk_w: Optional[torch.Tensor] = None, k: Optional[int] = None,
                   token_adapter: Optional[torch.Tensor] = None,
                   A1=None, B1=None, A2=None, B2=None, y: Optional[torch.Tensor] = None,
                   y_fp32: bool = False, workspace: Optional[torch.Tensor] = None,
                   bm_base: int = 0, bm_lora: int = 0, disable_pdl: bool = False,
                   events: Optional[Sequence] = None, gate_up_slices: int = 1,
                   adapter_ranks: Optional[torch.Tensor] = None,
                   wait_limit_ns: int = 0, expand_mode: int = 0,
                   mma_pairs: int = 0) -> torch.Tensor:
    """The whole fused MoE-LoRA layer; returns y [T, H]. gate_up_slices=2: separate gate
    and up adapters, A1 [L, E, 2r, H] (gate A rows first), B1 [L, E, 2I, r].
    adapter_ranks [L] int32 (device): adapter l has rank r_l <= r (weights padded to r).
    wait_limit_ns (tests of the give-up path): 0 default 4 s, < 0 give up at once.
    expand_mode: 0 the library picks, 1 the expand in kernels of its own, 2 the expand fused
    into the grouped GEMMs wherever it applies. mma_pairs: 0 the library picks (CTA pairs
    for the fused chain's 256-row token tiles), -1 one CTA per MMA."""
    _need(x, "x", torch.bfloat16, 2)
    T, H = x.shape
    E, I, Ln, r = _layer_weights(H, W1, W2, A1, B1, A2, B2, gate_up_slices)
    if logits is not None:
        _need(logits, "logits", torch.float32, 2, (T, E))
        if k is None:
            raise ValueError("k is required with logits")
    else:
        _need(topk_ids, "topk_ids", torch.int32, 2)
        k = topk_ids.shape[1]
        _need(topk_w, "topk_w", torch.float32, 2, (T, k))
    if token_adapter is not None:
        _need(token_adapter, "token_adapter", torch.int32, 1, (T,))
    if y is None:
        y = torch.empty((T, H), dtype=torch.float32 if y_fp32 else torch.bfloat16,
                        device=x.device)
    _need(y, "y", torch.float32 if y_fp32 else torch.bfloat16, 2, (T, H))
    if workspace is None:
        workspace = new_workspace(T, k, E, Ln, H, I, r, x.device)
    opts, _ev = _layer_opts(Ln, bm_base, bm_lora, disable_pdl, events, gate_up_slices,
                            adapter_ranks, wait_limit_ns, expand_mode, mma_pairs)
    check(lib().moe_lora_layer_ex(
        ptr(x), ptr(logits), ptr(topk_ids), ptr(topk_w), ptr(token_adapter), T, H, I, E, k,
        ptr(W1), ptr(W2), ptr(A1), ptr(B1), ptr(A2), ptr(B2), Ln, r, ptr(y), int(y_fp32),
        ptr(workspace), workspace.numel(), ctypes.byref(opts), stream_handle()),
        "moe_lora_layer")
    return y


def moe_lora_host_io_layout(T: int, H: int, E: int, with_adapter: bool = True,
                            y_fp32: bool = False) -> dict:
    """Byte offsets (x, logits, token_adapter or -1, y) of the host-staged layer call, the
    length of the host input block and of the device staging area."""
    off = (ctypes.c_int64 * 4)()
    ib, sb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    check(lib().moe_lora_host_io_layout(T, H, E, int(with_adapter), int(y_fp32), off,
                                        ctypes.byref(ib), ctypes.byref(sb)),
          "moe_lora_host_io_layout")
    return {"offsets": tuple(off), "in_bytes": ib.value, "staging_bytes": sb.value}


@dataclass
class HostIO:
    """Buffers of moe_lora_layer_host: the page-locked host input block, with views x [T, H]
    bf16, logits [T, E] fp32 and token_adapter [T] int32 (None without adapter ids) for the
    caller to fill; the page-locked host y; and the device staging area."""
    in_host: torch.Tensor
    y_host: torch.Tensor
    staging: torch.Tensor
    x: torch.Tensor
    logits: torch.Tensor
    token_adapter: Optional[torch.Tensor]
    T: int
    H: int
    E: int
    with_adapter: bool
    y_fp32: bool

    @property
    def in_bytes(self) -> int:
        return moe_lora_host_io_layout(self.T, self.H, self.E, self.with_adapter,
                                       self.y_fp32)["in_bytes"]


def new_host_io(T: int, H: int, E: int, with_adapter: bool = True, y_fp32: bool = False,
                device="cuda") -> HostIO:
    lay = moe_lora_host_io_layout(T, H, E, with_adapter, y_fp32)
    o = lay["offsets"]
    in_host = torch.zeros(max(lay["in_bytes"], 1), dtype=torch.uint8).pin_memory()

    def view(at, n, dt, shape):
        return in_host[at:at + n].view(dt).view(shape)

    x = view(o[0], T * H * 2, torch.bfloat16, (T, H))
    lg = view(o[1], T * E * 4, torch.float32, (T, E))
    ta = view(o[2], T * 4, torch.int32, (T,)) if with_adapter else None
    y_host = torch.empty((T, H), dtype=torch.float32 if y_fp32 else torch.bfloat16).pin_memory()
    staging = torch.empty(max(lay["staging_bytes"], 1), dtype=torch.uint8, device=device)
    return HostIO(in_host, y_host, staging, x, lg, ta, T, H, E, with_adapter, y_fp32)


def moe_lora_layer_host(io: HostIO, W1: torch.Tensor, W2: torch.Tensor, *, k: int,
                        A1=None, B1=None, A2=None, B2=None,
                        workspace: Optional[torch.Tensor] = None, bm_base: int = 0,
                        bm_lora: int = 0, disable_pdl: bool = False,
                        events: Optional[Sequence] = None, gate_up_slices: int = 1,
                        adapter_ranks: Optional[torch.Tensor] = None,
                        expand_mode: int = 0) -> torch.Tensor:
    """One step from host memory: copies io's input block to the device, runs the layer
    (routed from io.logits) and copies y back into io.y_host, all enqueued on the current
    stream. Returns io.y_host, valid once the stream has been synchronised."""
    T, H, E = io.T, io.H, io.E
    E1, I, Ln, r = _layer_weights(H, W1, W2, A1, B1, A2, B2, gate_up_slices)
    if E1 != E:
        raise ValueError("W1 has a different expert count than the host block's logits")
    if not io.in_host.is_pinned() or not io.y_host.is_pinned():
        raise ValueError("the host buffers must be page-locked (new_host_io allocates them so)")
    if workspace is None:
        workspace = new_workspace(T, k, E, Ln, H, I, r, io.staging.device)
    opts, _ev = _layer_opts(Ln, bm_base, bm_lora, disable_pdl, events, gate_up_slices,
                            adapter_ranks, expand_mode=expand_mode)
    check(lib().moe_lora_layer_host(
        ptr(io.in_host), ptr(io.y_host), ptr(io.staging), io.staging.numel(),
        int(io.with_adapter), T, H, I, E, k, ptr(W1), ptr(W2), ptr(A1), ptr(B1), ptr(A2),
        ptr(B2), Ln, r, int(io.y_fp32), ptr(workspace), workspace.numel(), ctypes.byref(opts),
        stream_handle()), "moe_lora_layer_host")
    return io.y_host
