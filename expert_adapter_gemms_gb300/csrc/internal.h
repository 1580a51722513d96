// Host-side launchers shared between the translation units of the library.
#pragma once

#include "common.cuh"

namespace moe_lora {

int check_route_args(const float* logits, int T, int E, int k, const int32_t* ids, const float* w);
int launch_topk_softmax(const float* logits, int T, int E, int k, int* ids, float* w,
                        cudaStream_t stream, bool pdl);

// The one-CTA align routing the tokens itself (few tokens): ids and w are written by the
// same launch. align_can_route tells where it applies.
constexpr int kAlignRouteMaxTokens = 64;
bool align_can_route(const AlignLayout& a, int T, int E);
int launch_route_align(const float* logits, int* ids, float* w, const int* token_adapter,
                       const moe_lora_align_t* al, const AlignLayout& a, cudaStream_t stream,
                       bool pdl);
int launch_align(const int* ids, const int* token_adapter, const moe_lora_align_t* al,
                 const AlignLayout& a, cudaStream_t stream, bool pdl);

int launch_gather(const void* x, const moe_lora_align_t* al, const AlignLayout& a, int H,
                  void* xs, cudaStream_t stream, bool pdl, bool trigger_first);

// bf16 tensor map over `rank` (2 or 3) dimensions, innermost first (dims[0] contiguous),
// byte strides of dimensions 1.. in strides_bytes, box `box` (box[0] x 2 bytes equal to the
// swizzle width), zero fill out of bounds. Host only; no device work.
int make_tmap_bf16(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                   const uint64_t* strides_bytes, const uint32_t* box,
                   CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);

// silu(v) = v / (1 + exp(-v)) with the hardware exponential and a reciprocal-based
// divide (CUDA's __expf, __fdividef): a few fp32 ulps, far below the bf16 rounding of the
// SwiGLU output; for v below about -87 it returns 0 where the exact form gives a value
// under 1e-36.
__device__ __forceinline__ float silu_fast(float v) { return __fdividef(v, 1.f + __expf(-v)); }

// Tensor maps are built on the host for every call (cheap; no device work).
int launch_grouped_gemm(const void* a_sorted, const void* W, const moe_lora_align_t* al,
                        const AlignLayout& a, int N, int K, float* out, cudaStream_t stream,
                        bool pdl);

int launch_shrink(const void* X, int rows_are_slots, const void* A, const moe_lora_align_t* al,
                  const AlignLayout& a, int K, int r, float* Z, cudaStream_t stream, bool pdl);

// ---- the shifted z buffer of the fused expand (fused_gemm.cu) ----
// z of sorted row j of pair (e, l) is row j + (e L + l + 1) gap, as bf16 high parts in
// columns [0, r) and the bf16 remainders in [lo_off, lo_off + r); columns [r, rp16) of each
// half are zero, and so are the gap rows before and after every pair written.
struct ZPadLayout {
  int rp16;      // rank rounded up to 16
  int zw;        // row width (bf16 elements, a multiple of 64)
  int lo_off;    // first column of the low parts
  int zk;        // > 0: high and low share one 64-column row (zk K16 steps each)
  int zchunks;   // LoRA stages per adapter run in a token tile
  int gap;       // zero rows between pairs (>= the fused GEMM's token tile)
  int64_t rows;  // rows of the buffer
};
ZPadLayout zpad_layout(int S, int E, int L, int r, int gap);

// Where a shrink publishes z: Z [S, r] fp32 by slot (p == nullptr), or the shifted buffer.
struct ZPadOut {
  __nv_bfloat16* p;
  int zw, lo_off, rp16, gap, L;
  const int* row_expert;
  const int* row_adapter;
};

// The fused expand: the grouped GEMM over sorted rows a_sorted [S, K] and W [E, N_w, K]
// with, for rows with an adapter, the K-steps of z (the shifted buffer) against B
// [L, E, N_w, r]. glu: N_w = 2I and out is h [S, I] bf16 = silu(gate) * up; else out is
// [S, N_w] fp32. B or zpad null (or L = 0): the base GEMM only. `early`: everything but z
// may be read before griddepcontrol.wait.
// ksplit > 1 (expert-major down form): the K range in ksplit shares, each CTA writing its
// own partial output at out + share * S * N (the combine sums them).
// pairs: 256-row token tiles run on CTA pairs (tcgen05.mma.cta_group::2, M = 256 over two
// weight blocks).
int launch_fused_gemm(const void* a_sorted, const void* W, const void* B, const void* zpad,
                      const ZPadLayout& zl, const moe_lora_align_t* al, const AlignLayout& a,
                      int N_w, int K, int r, bool glu, void* out, cudaStream_t stream, bool pdl,
                      bool early, int expert_major_bn, unsigned long long wait_ns, int ksplit = 1,
                      bool pairs = true);

// y[t] = sum_j w[t, j] O[row(t, j)] (j ascending) over O [S, N] fp32 by sorted row; with
// nparts > 1, O holds nparts partial outputs part_stride elements apart, summed in order.
// early: the slot rows and the weights are read before griddepcontrol.wait.
int launch_combine(const float* O, const float* topk_w, const moe_lora_align_t* al,
                   const AlignLayout& a, int N, void* y, int y_fp32, cudaStream_t stream, bool pdl,
                   int nparts = 1, size_t part_stride = 0, bool early = false);

int launch_expand(const float* Z, const void* B, const moe_lora_align_t* al, const AlignLayout& a,
                  int N, int r, int epilogue, float* base, void* out, int out_fp32,
                  const float* topk_w, cudaStream_t stream, bool pdl);

// Variants for the layer chain: with `early`, a kernel reads data produced two or
// more launches back before its griddepcontrol.wait (valid because every kernel
// of the library triggers its dependents only after its own wait).
// r: ranks per row of A (2 r_slice with separate gate and up adapters); rs: ranks per
// slice, the unit that al->adapter_ranks truncates.
int launch_shrink_impl(const void* X, int rows_are_slots, const void* A,
                       const moe_lora_align_t* al, const AlignLayout& a, int K, int r, int rs,
                       float* Z, cudaStream_t stream, bool pdl, bool early,
                       unsigned long long wait_ns = kWaitLimitNs, const ZPadOut* zpad = nullptr,
                       int flags = 0);
// flags of launch_shrink_impl: every CTA resident at once; the block table is two or more
// launches old, so each CTA reads its block and prefetches its rows of A into L2 before its
// wait (for a shrink whose activations come from its immediate predecessor)
enum { kShrinkOneWave = 1, kShrinkPrefetchA = 2 };
// expert_major_bn > 0: one CTA per (expert, weight block) taking the expert's rows in
// chunks of that many rows (16..256), which lets the weights stream before the align
// tables exist; 0: one CTA per (token tile of bm_base rows, weight block).
// wait_ns: limit of the main-loop mbarrier waits (the shrink's short-K slab wait too);
// the waits that drain copies and MMAs before a CTA exits always use kWaitLimitNs.
int launch_grouped_gemm_impl(const void* a_sorted, const void* W, const moe_lora_align_t* al,
                             const AlignLayout& a, int N, int K, float* out, cudaStream_t stream,
                             bool pdl, bool early, int expert_major_bn,
                             unsigned long long wait_ns = kWaitLimitNs);
int launch_expand_impl(const float* Z, const void* B, const moe_lora_align_t* al,
                       const AlignLayout& a, int N, int r, int epilogue, float* base, void* out,
                       int out_fp32, const float* topk_w, cudaStream_t stream, bool pdl,
                       bool early);

// ---- adapters of their own ranks (moe_lora_align_t.adapter_ranks) ----
// Rank of adapter l, clamped to [0, r]; an out-of-range value sets
// MOE_LORA_DEVERR_RANK_RANGE. ranks is a caller input (read-only path).
__device__ __forceinline__ int adapter_rank(const int* ranks, int l, int r, const int* hdr) {
  if (!ranks) return r;
  const int v = __ldg(ranks + l);
  if (v >= 0 && v <= r) return v;
  if (hdr) set_dev_error(const_cast<int*>(hdr), MOE_LORA_DEVERR_RANK_RANGE);
  return v < 0 ? 0 : r;
}
// The first v (0..8) bf16 of a 16-byte group; the rest zeroed.
__device__ __forceinline__ uint4 keep_first_bf16(uint4 u, int v) {
  uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (2 * i >= v) w[i] = 0u;
    else if (2 * i + 1 >= v) w[i] &= 0xFFFFu;
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
// 16-byte group g (ranks 8g .. 8g+7) of a B row when the adapter uses rv ranks: groups
// wholly past rv are not read. The entries of a partial group past rv are cleared
// with b_tail where the group is consumed, not here: a select right at the load would
// make every load wait for its own result before the next one is issued.
__device__ __forceinline__ uint4 b_group(const uint4* row, int g, int rv) {
  if (8 * g >= rv) return make_uint4(0, 0, 0, 0);
  return __ldg(row + g);
}
// Clears the entries past rv of a group whose first rank is k0.
__device__ __forceinline__ uint4 b_tail(uint4 u, int k0, int rv) {
  return k0 + 8 > rv ? keep_first_bf16(u, rv - k0) : u;
}
// Rows base .. base + 63 of A (ranks numbered across slices of rs rows): bit i set when
// row base + i lies within the first rl rows of its slice. Two modulos and two ballots per
// warp (every lane of the warp must call it).
__device__ __forceinline__ unsigned long long rank_row_mask(int base, int rs, int rl) {
  const int lane = threadIdx.x & 31;
  const unsigned lo = __ballot_sync(0xffffffffu, (base + lane) % rs < rl);
  const unsigned hi = __ballot_sync(0xffffffffu, (base + 32 + lane) % rs < rl);
  return (unsigned long long)lo | ((unsigned long long)hi << 32);
}

}  // namespace moe_lora
