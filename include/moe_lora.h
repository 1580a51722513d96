/*
 * moe_lora.h -- C ABI of the fused MoE-LoRA expert layer for NVIDIA GB300 (sm_103a).
 *
 * What the layer computes (vLLM blog "multi-LoRA for MoE", vllm.com.cn, section
 * "Implementing multi-LoRA inference for MoE models in vLLM"; and "vLLM Multi-LoRA
 * Serving for MoE Models", agentlenshq.com, section "Multi-LoRA Serving for MoE
 * Models"): each token is routed to its top-k experts; each expert applies a gate_up
 * projection, the gated activation and a down projection, and the experts' outputs
 * are summed with the routing weights. Multi-LoRA adds, per request, a low-rank adapter to both
 * projections: y = xW + (xA)B, where the shrink op is z = xA (h_in -> r) and the
 * expand op is zB (r -> h_out). Token routing and adapter selection together pick
 * an (expert, adapter) pair per token-slot ("compound sparsity").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All array pointers are DEVICE pointers owned by the caller. The library never
 *   allocates, frees or synchronises on the compute path; intermediates live in a
 *   caller-provided workspace or align buffer.
 * - Every call is asynchronous on the caller's stream and returns a status code
 *   (moe_lora_status below). Arguments are validated on the host before anything
 *   is launched; on error nothing is launched.
 * - bf16 arrays are passed as `const void*` holding IEEE bfloat16 bit patterns.
 * - Arrays are contiguous and row-major; base pointers of bf16 matrices read by
 *   the tensor-memory-accelerator path must be 16-byte aligned, and their row
 *   length (the reduction dimension) a multiple of 8 elements.
 * - Weight layouts keep the reduction dimension innermost (the transpose of the
 *   pages' h_in x h_out notation, as nn.Linear stores it):
 *       W1 [E, 2I, H]  gate_up (rows [0,I) gate, [I,2I) up)   W2 [E, H, I] down
 *       A1 [L, E, r, H]  B1 [L, E, 2I, r]  A2 [L, E, r, I]  B2 [L, E, H, r]
 *   LoRA scale is 1 (y = xW + xAB); fold any alpha/r into B. Adapters with a
 *   smaller rank are zero-padded to r.
 * - Slots: s = t*k + j for token t and routing choice j. A token's adapter id
 *   -1 means "base model only".
 * - Ids found out of range on the device never trap: the slot is dropped and a
 *   bit is set in a sticky device error word, read back with moe_lora_get_error.
 * - Kernels are chained with programmatic dependent launch on the caller's
 *   stream. Every size is a runtime argument: nothing is compiled or loaded per
 *   token count.
 */
#ifndef MOE_LORA_H_
#define MOE_LORA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_LORA_API __attribute__((visibility("default")))
#else
#define MOE_LORA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same underlying type as cudaStream_t; pass a CUDA stream handle (or 0). */
typedef struct CUstream_st* moe_lora_stream_t;

/* Status codes returned by every entry point. */
enum moe_lora_status {
  MOE_LORA_OK = 0,
  MOE_LORA_ERR_INVALID_ARG = 1,          /* null/misaligned pointer, negative size, k > E, ... */
  MOE_LORA_ERR_UNSUPPORTED = 2,          /* shape outside the documented limits, or not an sm_103 device */
  MOE_LORA_ERR_CUDA = 3,                 /* a CUDA runtime call or launch failed */
  MOE_LORA_ERR_WORKSPACE_TOO_SMALL = 4,  /* workspace/align buffer smaller than required */
  MOE_LORA_ERR_TIMEOUT = 5               /* reported by moe_lora_get_error when a bounded wait gave up */
};

/* Bits of the sticky device error word. */
#define MOE_LORA_DEVERR_EXPERT_RANGE 0x1u  /* an expert id outside [0, E): slot dropped */
#define MOE_LORA_DEVERR_ADAPTER_RANGE 0x2u /* an adapter id outside [-1, L): the token's slots dropped */
#define MOE_LORA_DEVERR_TIMEOUT 0x4u       /* a bounded wait inside a kernel gave up; results invalid */
#define MOE_LORA_DEVERR_RANK_RANGE 0x8u    /* an adapter rank outside [0, r]: clamped */

/* Human-readable name of a status code (static string). */
MOE_LORA_API const char* moe_lora_status_string(int status);

/* ---------------------------------------------------------------------------
 * Routing: the router picks each token's top-k experts.
 *
 * moe_topk_softmax: for each of T tokens, ids[t, 0..k) are the indices of the k
 * largest logits[t, :] in decreasing order (equal logits: lower index first; NaN
 * ranks below every number), and w[t, j] = exp(l_j - l_0) / sum_i exp(l_i - l_0)
 * over the chosen logits l_j (fp32). logits [T, E] fp32; ids [T, k] int32;
 * w [T, k] fp32. Requires 1 <= k <= E <= 1024 and k <= 32. T = 0 is a no-op.
 * ------------------------------------------------------------------------- */
MOE_LORA_API int moe_topk_softmax(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                     moe_lora_stream_t stream);

/* ---------------------------------------------------------------------------
 * Alignment: the compound sparsity of expert routing x adapter selection.
 *
 * Slots are stably sorted by the key (expert e, adapter l, slot s), l = -1 first.
 * The result lives in a caller-allocated "align buffer" described by
 * moe_lora_align_t. Its layout (byte offsets from moe_lora_align_layout):
 *   header        int32[64]: [0] error word (uint32, sticky, OR-ed), [1] n_valid,
 *                 [2] n_tiles, [3] n_lora_blocks, [4] n_lora_rows, [5..] echo of
 *                 T, k, E, L, bm_base, bm_lora
 *   sorted_slots  int32[S]    kept slots in key order, -1 after n_valid
 *   slot_row      int32[S]    sorted position of each slot, -1 if dropped
 *   row_expert    int32[S]    expert of each sorted row
 *   row_adapter   int32[S]    adapter of each sorted row (-1: none)
 *   expert_begin  int32[E+1]  rows of expert e are [expert_begin[e], expert_begin[e+1])
 *   tiles         int32[max_tiles][4]  {e, row_begin, rows, 0}: each expert's rows cut
 *                 into chunks of at most bm_base rows (the grouped GEMM's token tiles)
 *   lora_blocks   int32[max_lora_blocks][4] {row_begin, rows, e, l}: each (e, l >= 0)
 *                 segment cut into chunks of at most bm_lora rows
 *   then internal scratch (bucket counts and sort buffers).
 * Entries past the device-side counts are unspecified. Integer results are
 * bit-exact and deterministic.
 * Limits: S = T*k <= 1<<22, E*(L+1)+1 and S together fit 32 key bits,
 * bm_base a multiple of 16 in [16, 256], 1 <= bm_lora <= 16.
 * ------------------------------------------------------------------------- */
typedef struct moe_lora_align_t {
  void* buf;       /* device pointer to an align buffer of moe_lora_align_buffer_size bytes, 256-byte aligned */
  int32_t T;       /* tokens */
  int32_t k;       /* experts per token */
  int32_t E;       /* experts */
  int32_t L;       /* resident adapters (0: none) */
  int32_t bm_base; /* rows per grouped-GEMM token tile */
  int32_t bm_lora; /* rows per LoRA block */
  const int32_t* adapter_ranks; /* optional device array [L]: adapter l has rank r_l in [0, r]
                     and uses only the first r_l rows of each r-row slice of A and the
                     first r_l columns of B (storage stays padded to r); NULL: every
                     adapter has rank r. Used by lora_shrink and lora_expand_add (z
                     entries past r_l are written as 0); 16-byte groups wholly past r_l
                     are never read. Values outside [0, r] are clamped and flagged
                     (MOE_LORA_DEVERR_RANK_RANGE). The pages give one rank per serving
                     instance; per-adapter ranks are this library's extension. */
} moe_lora_align_t;

#define MOE_LORA_ALIGN_NFIELDS 12
/* Indices into the offsets array filled by moe_lora_align_layout. */
enum moe_lora_align_field {
  MOE_LORA_AF_HEADER = 0, MOE_LORA_AF_SORTED_SLOTS, MOE_LORA_AF_SLOT_ROW, MOE_LORA_AF_ROW_EXPERT,
  MOE_LORA_AF_ROW_ADAPTER, MOE_LORA_AF_EXPERT_BEGIN, MOE_LORA_AF_TILES, MOE_LORA_AF_LORA_BLOCKS,
  MOE_LORA_AF_MAX_TILES, MOE_LORA_AF_MAX_LORA_BLOCKS, MOE_LORA_AF_SCRATCH, MOE_LORA_AF_TOTAL_BYTES
};

/* Bytes of align buffer needed; 0 if the parameters are invalid. */
MOE_LORA_API size_t moe_lora_align_buffer_size(int T, int k, int E, int L, int bm_base, int bm_lora);

/* Fills offsets[MOE_LORA_ALIGN_NFIELDS] (byte offsets; MAX_* fields hold counts). Host only. */
MOE_LORA_API int moe_lora_align_layout(int T, int k, int E, int L, int bm_base, int bm_lora, int64_t* offsets);

/* ids [T, k] int32; token_adapter [T] int32 or NULL (all -1). Deterministic. Below 2048
 * slots (or with more buckets E*(L+1)+1 than half the slots) one CTA sorts every slot;
 * from 2048 slots three launches share the work: per-CTA stable sorts of 512-slot chunks,
 * one scan over the (key, chunk) count table, and a placement pass. */
MOE_LORA_API int moe_lora_align(const int32_t* ids, const int32_t* token_adapter, const moe_lora_align_t* al,
                   moe_lora_stream_t stream);

/* Copies the sticky error word of an align buffer (or of a layer workspace, whose
 * first bytes are its align buffer) to *err. Synchronises `stream`. */
MOE_LORA_API int moe_lora_get_error(const void* align_buf_or_workspace, moe_lora_stream_t stream, uint32_t* err);
/* Clears the sticky error word (asynchronous). */
MOE_LORA_API int moe_lora_clear_error(void* align_buf_or_workspace, moe_lora_stream_t stream);

/* ---------------------------------------------------------------------------
 * Gather: xs[row, :] = x[sorted_slots[row] / k, :] for the n_valid sorted rows.
 * x [T, H] bf16; xs [S, H] bf16 (rows past n_valid untouched).
 * ------------------------------------------------------------------------- */
MOE_LORA_API int moe_gather_rows(const void* x, const moe_lora_align_t* al, int H, void* xs,
                    moe_lora_stream_t stream);

/* ---------------------------------------------------------------------------
 * Base expert grouped GEMM (vLLM's fused_moe group GEMM, one GEMM per expert
 * over the tokens routed to it; vllm.com.cn, section "Implementing multi-LoRA
 * inference for MoE models in vLLM").
 *   out[row, n] = sum_c a[row, c] * W[e(row), n, c]   for row < n_valid
 * a [S, K] bf16 in sorted-row order; W [E, N, K] bf16; out [S, N] fp32 (rows past
 * n_valid untouched). bf16 in, fp32 accumulate on the tcgen05 tensor cores with
 * TMEM accumulators, operands staged by TMA. Requires K % 8 == 0, 16-byte aligned
 * a and W, N >= 1.
 * ------------------------------------------------------------------------- */
MOE_LORA_API int moe_grouped_gemm(const void* a, const void* W, const moe_lora_align_t* al, int N, int K,
                     float* out, moe_lora_stream_t stream);

/* ---------------------------------------------------------------------------
 * LoRA shrink z = xA for every slot whose token has an adapter (vllm.com.cn,
 * sections "Implementing ..." and "Kernel optimizations": r outputs, each a long
 * sum over h_in, so the sum over K is split across warps of a CTA).
 *   Z[s, i] = sum_c X[in(s), c] * A[l(s), e(s), i, c]
 * rows_are_slots = 0: in(s) = s / k, X is [T, K] (token activations).
 * rows_are_slots = 1: in(s) = slot_row[s], X is [S, K] (sorted rows, e.g. the
 *                     SwiGLU output feeding the down projection).
 * A [L, E, r, K] bf16; Z [S, r] fp32 (slots without adapter untouched).
 * With al->adapter_ranks, adapter l uses rows [0, r_l) of A and Z[s, i >= r_l] = 0.
 * Any K >= 1 and 1 <= r <= 256; K % 8 == 0 with 16-byte aligned X and A takes the
 * 128-bit load path, and K % 32 == 0 also drops the bounds masks (EVEN_K).
 * Deterministic (fixed-order reductions, no atomics).
 * ------------------------------------------------------------------------- */
MOE_LORA_API int lora_shrink(const void* X, int rows_are_slots, const void* A, const moe_lora_align_t* al,
                int K, int r, float* Z, moe_lora_stream_t stream);

/* ---------------------------------------------------------------------------
 * LoRA expand with the base add fused in (vllm.com.cn, section "Kernel
 * optimizations": the LoRA result is added to the base output inside the expand
 * kernel), plus the layer's epilogues:
 *   delta[row, n] = sum_i Z[s, i] * B[l, e, n, i]      (rows with an adapter)
 *   epilogue 0: base[row, n] += delta[row, n]           in place, fp32 [S, N]
 *   epilogue 1: out[row, n] = silu(g) * u with g = base[row, n] + delta[row, n],
 *               u = base[row, N/2 + n] + delta[row, N/2 + n]; out [S, N/2] bf16,
 *               every valid row (with or without adapter). N must be even.
 *   epilogue 2: out[t, n] = sum_j w[t, j] * (base[row(t,j), n] + delta[row(t,j), n]),
 *               j in increasing order; out [T, N] bf16 (out_fp32 = 0) or fp32.
 *               base is only read.
 *   epilogue 3: as epilogue 1 with separate gate and up adapters: Z rows hold 2r
 *               values, columns [0, N/2) take z[0, r) and B rows [0, N/2), columns
 *               [N/2, N) take z[r, 2r) and B rows [N/2, N); B stays [L, E, N, r].
 * Z [S, r] fp32 ([S, 2r] for epilogue 3); B [L, E, N, r] bf16 (NULL or L = 0: no
 * adapter term). With al->adapter_ranks, adapter l uses columns [0, r_l) of B only.
 * topk_w [T, k] fp32 (epilogue 2 only). Requires L < 65535. Deterministic.
 * ------------------------------------------------------------------------- */
MOE_LORA_API int lora_expand_add(const float* Z, const void* B, const moe_lora_align_t* al, int N, int r,
                    int epilogue, float* base, void* out, int out_fp32, const float* topk_w,
                    moe_lora_stream_t stream);

/* ---------------------------------------------------------------------------
 * The whole layer, as one of two chains of launches (moe_lora_layer_plan says which):
 *   route (if logits != NULL) -> align -> gather -> gate_up grouped GEMM ->
 *   gate_up shrink -> gate_up expand + SwiGLU -> down grouped GEMM -> down shrink
 *   -> down expand + weighted top-k combine;
 * or, with the expand fused into the grouped GEMMs by concatenation along K
 * (y = xW + zB = [x | z][W | B]^T for the rows of each adapter):
 *   route -> align -> gather -> gate_up shrink -> gate_up GEMM + expand + SwiGLU ->
 *   down shrink -> down GEMM + expand -> weighted top-k combine.
 * x [T, H] bf16. Routing: either logits [T, E] fp32 (topk_ids/topk_w NULL) or
 * caller-provided topk_ids [T, k] int32 and topk_w [T, k] fp32 (logits NULL).
 * token_adapter [T] int32 or NULL. LoRA weights may be NULL with L = 0 (base MoE).
 * y [T, H]: bf16 (y_fp32 = 0) or fp32. workspace: moe_lora_workspace_size bytes,
 * 256-byte aligned; its first bytes are the layer's align buffer (error word).
 * Requires H % 8 == 0, I % 8 == 0, 1 <= k <= min(E, 32), E <= 1024, L < 65535.
 * ------------------------------------------------------------------------- */
MOE_LORA_API size_t moe_lora_workspace_size(int T, int k, int E, int L, int H, int I, int r);

MOE_LORA_API int moe_lora_layer(const void* x, const float* logits, const int32_t* topk_ids,
                   const float* topk_w, const int32_t* token_adapter, int T, int H, int I, int E,
                   int k, const void* W1, const void* W2, const void* A1, const void* B1,
                   const void* A2, const void* B2, int L, int r, void* y, int y_fp32,
                   void* workspace, size_t workspace_bytes, moe_lora_stream_t stream);

/* Optional controls for moe_lora_layer_ex (zero-initialise, then set fields). */
typedef struct moe_lora_layer_opts {
  int32_t bm_base;      /* grouped-GEMM token tile; 0 = heuristic */
  int32_t bm_lora;      /* LoRA block rows; 0 = heuristic */
  int32_t disable_pdl;  /* 1: plain stream-ordered launches */
  int32_t num_events;   /* length of `events` (0: none) */
  void** events;        /* cudaEvent_t handles recorded on `stream` before each stage and
                           after the last: [0] route, [1] align (at few tokens the align
                           routes them itself: [0] and [1] mark the same point), [2]
                           gather, then for the
                           chain with a separate expand: [3] gate_up GEMM, [4] gate_up
                           shrink, [5] gate_up expand+SwiGLU, [6] down GEMM, [7] down shrink,
                           [8] down expand+combine; for the fused chain
                           (moe_lora_layer_plan_t.fused_expand): [3] gate_up shrink, [4]
                           gate_up GEMM with expand+SwiGLU, [5] empty, [6] down shrink, [7]
                           down GEMM with expand, [8] combine; [9] end */
  const int32_t* adapter_ranks; /* optional device array [L] of per-adapter ranks (see
                           moe_lora_align_t.adapter_ranks); NULL: every adapter has rank r */
  int32_t gate_up_slices; /* 0 or 1: one adapter over the fused gate_up output (A1
                           [L,E,r,H]); 2: separate gate and up adapters, A1 [L,E,2r,H]
                           with the gate A in rows [0,r) and the up A in [r,2r), B1
                           [L,E,2I,r] unchanged: gate columns take the gate z, up columns
                           the up z (lora_expand_add epilogue 3). The pages describe one
                           adapter per projection and are silent on a split gate_up. */
  int32_t expand_mode;  /* 0: the library picks; 1: the expand in kernels of its own (after
                           each grouped GEMM); 2: the fused chain (the expand as extra K-steps
                           of the grouped GEMMs, SwiGLU in the gate_up GEMM's epilogue)
                           wherever it applies: one adapter rank (no adapter_ranks), one
                           gate_up slice, r % 8 == 0, and shapes whose shifted z buffers stay
                           small (they grow with E * L). The library picks the fused chain
                           where it applies and pays: with adapters, at few rows per expert or
                           at (expert, adapter) runs of 16 rows or more on average; without,
                           with token tiles. Both chains compute the same function; their
                           results differ in fp32 summation order only. */
  int64_t wait_limit_ns; /* for tests of the give-up path: the wall-time limit of the grouped
                           GEMMs' main-loop mbarrier waits (and of the short-K shrink's slab
                           wait). 0: the default, 4 s; < 0: give up at the first unsuccessful
                           poll. A wait that gives up sets MOE_LORA_DEVERR_TIMEOUT; the CTA then
                           drains its own copies and tensor-core work (those waits keep the 4 s
                           limit), frees its tensor memory and exits, and that launch's
                           results are invalid. */
  int32_t mma_pairs;    /* fused chain with 256-row token tiles: 0 = the library's choice
                           (pairs of CTAs, each job one tcgen05.mma.cta_group::2 of M = 256
                           over two 128-row weight blocks, each CTA staging half the token
                           rows); -1 = one CTA per 128-row weight block. Same results up to
                           fp32 summation order. */
} moe_lora_layer_opts;

#define MOE_LORA_LAYER_NUM_STAGES 9

MOE_LORA_API int moe_lora_layer_ex(const void* x, const float* logits, const int32_t* topk_ids,
                      const float* topk_w, const int32_t* token_adapter, int T, int H, int I,
                      int E, int k, const void* W1, const void* W2, const void* A1,
                      const void* B1, const void* A2, const void* B2, int L, int r, void* y,
                      int y_fp32, void* workspace, size_t workspace_bytes,
                      const moe_lora_layer_opts* opts, moe_lora_stream_t stream);

/* ---------------------------------------------------------------------------
 * One serving step with its per-step inputs and its output in host memory: the
 * same layer as moe_lora_layer_ex, routed from logits, with the copies in and out
 * issued by the library on the same stream. The pages describe the device-side
 * computation only; this call stages it for a caller whose batch arrives in host
 * memory (the router logits and adapter ids of a decode step, for instance).
 *
 * moe_lora_host_io_layout (host only) gives the byte offsets, each 256-byte aligned:
 *   offsets[0] x [T, H] bf16, offsets[1] logits [T, E] fp32,
 *   offsets[2] token_adapter [T] int32 (with_adapter = 1; else -1),
 *   offsets[3] y [T, H] bf16 (y_fp32 = 0) or fp32.
 * The caller's host input block holds x, logits and (with_adapter) the adapter ids
 * at offsets[0..2] and is *in_bytes long; the device staging area, *staging_bytes
 * long, holds the same inputs plus y at offsets[3].
 *
 * moe_lora_layer_host enqueues on `stream`, in order: one cudaMemcpyAsync of the
 * whole input block (in_bytes) into `staging`; the layer on the staged views
 * (moe_lora_layer_ex with logits routing; token_adapter NULL when with_adapter = 0;
 * weights, workspace and opts as there); one cudaMemcpyAsync of y into y_host
 * (T*H*2 bytes, or T*H*4 with y_fp32). It returns without waiting: synchronise the
 * stream before reading y_host or rewriting in_host. Page-locked host memory keeps
 * both copies asynchronous; pageable memory works but the copies then synchronise
 * with the host. staging: device memory, 256-byte aligned, at least staging_bytes.
 * Errors: every argument, the layer's included, is checked before anything is
 * copied or launched (MOE_LORA_ERR_WORKSPACE_TOO_SMALL for a short staging area).
 * ------------------------------------------------------------------------- */
MOE_LORA_API int moe_lora_host_io_layout(int T, int H, int E, int with_adapter, int y_fp32,
                                         int64_t* offsets, size_t* in_bytes,
                                         size_t* staging_bytes);

MOE_LORA_API int moe_lora_layer_host(const void* in_host, void* y_host, void* staging,
                                     size_t staging_bytes, int with_adapter, int T, int H, int I,
                                     int E, int k, const void* W1, const void* W2, const void* A1,
                                     const void* B1, const void* A2, const void* B2, int L, int r,
                                     int y_fp32, void* workspace, size_t workspace_bytes,
                                     const moe_lora_layer_opts* opts, moe_lora_stream_t stream);

/* Tile sizes the layer picks for a shape (host only): bm_base, bm_lora. */
MOE_LORA_API int moe_lora_layer_tiles(int T, int k, int E, int L, int H, int I, int r, int32_t* bm_base,
                         int32_t* bm_lora);

/* How moe_lora_layer_ex runs a shape with the given options (NULL: defaults); host only.
 *   bm_base, bm_lora      the align's token tile and LoRA block rows
 *   expert_major_rows     > 0: each grouped-GEMM CTA takes one (expert, 128-row weight block)
 *                         and all of the expert's rows in chunks of this many (few rows per
 *                         expert); 0: token tiles of bm_base rows
 *   fused_expand          1: the LoRA expand runs as extra K-steps of the grouped GEMMs
 *                         (y = [x | z][W | B]^T per adapter run of a tile; the gate_up GEMM
 *                         writes the SwiGLU output directly, the down GEMM its rows, then a
 *                         combine kernel); 0: the expand in kernels of its own
 *   launches              kernels one call launches when routed from logits (one fewer with
 *                         caller-provided ids)
 *   early_reads           (kernel, earlier step) pairs where a kernel reads that step's
 *                         output before its own griddepcontrol.wait (programmatic dependent
 *                         launch). The plan checks each: the producer is at least two launches
 *                         back and the launch in between triggers its dependents only after its
 *                         own wait, so the producer has completed when the reader starts; a
 *                         chain that broke this would be refused (MOE_LORA_ERR_UNSUPPORTED).
 *   route_in_align        1: routed from logits, the one-CTA align routes the tokens itself
 *                         (up to 64 tokens, 64 experts): no separate route launch */
typedef struct moe_lora_layer_plan_t {
  int32_t bm_base;
  int32_t bm_lora;
  int32_t expert_major_rows;
  int32_t fused_expand;
  int32_t launches;
  int32_t early_reads;
  int32_t route_in_align;
} moe_lora_layer_plan_t;

MOE_LORA_API int moe_lora_layer_plan(int T, int k, int E, int L, int H, int I, int r,
                                     const moe_lora_layer_opts* opts, moe_lora_layer_plan_t* plan);

/* ---------------------------------------------------------------------------
 * moe_lora_layer_noalloc: the same layer as moe_lora_layer for callers that cannot
 * allocate device memory -- e.g. a serving engine that has reserved nearly all HBM
 * for weights and KV cache and hands out only its own buffers, a plugin interface
 * that passes inputs and outputs but no allocator, or a latency-critical path
 * where cudaMalloc/cudaFree may synchronise the device. The pages describe no such
 * entry point; it has no counterpart there.
 * Arguments are moe_lora_layer's without the workspace; intermediates live in a
 * 64 MiB array in device global memory held by the library (every GPU that loads
 * it keeps the 64 MiB until the process exits). Shapes whose
 * moe_lora_workspace_size exceeds 64 MiB return MOE_LORA_ERR_WORKSPACE_TOO_SMALL
 * and launch nothing. err_out: optional device pointer that receives this call's
 * device error word (MOE_LORA_DEVERR_* bits; cleared at the start of each call).
 * The function allocates nothing. All calls on a device share the array and it
 * keeps the last call's contents: calls that overlap on the GPU race, so order
 * them on one stream. The first call on each device looks up the array's device
 * address; make that first call before any stream capture. The address belongs to
 * the device's current context: after that context is re-created (cudaDeviceReset)
 * the next call looks it up again.
 * ------------------------------------------------------------------------- */
MOE_LORA_API int moe_lora_layer_noalloc(const void* x, const float* logits,
                                        const int32_t* topk_ids, const float* topk_w,
                                        const int32_t* token_adapter, int T, int H, int I, int E,
                                        int k, const void* W1, const void* W2, const void* A1,
                                        const void* B1, const void* A2, const void* B2, int L,
                                        int r, void* y, int y_fp32, uint32_t* err_out,
                                        moe_lora_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_LORA_H_ */
