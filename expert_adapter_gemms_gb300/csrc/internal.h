// Host-side launchers shared between the translation units of the library.
#pragma once

#include "common.cuh"

namespace moe_lora {

int check_route_args(const float* logits, int T, int E, int k, const int32_t* ids, const float* w);
int launch_topk_softmax(const float* logits, int T, int E, int k, int* ids, float* w,
                        cudaStream_t stream, bool pdl);

int launch_align(const int* ids, const int* token_adapter, const moe_lora_align_t* al,
                 const AlignLayout& a, cudaStream_t stream, bool pdl);

int launch_gather(const void* x, const moe_lora_align_t* al, const AlignLayout& a, int H,
                  void* xs, cudaStream_t stream, bool pdl, bool trigger_first);

// Tensor maps are built on the host for every call (cheap; no device work).
int launch_grouped_gemm(const void* a_sorted, const void* W, const moe_lora_align_t* al,
                        const AlignLayout& a, int N, int K, float* out, cudaStream_t stream,
                        bool pdl);

int launch_shrink(const void* X, int rows_are_slots, const void* A, const moe_lora_align_t* al,
                  const AlignLayout& a, int K, int r, float* Z, cudaStream_t stream, bool pdl);

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
                       float* Z, cudaStream_t stream, bool pdl, bool early);
// expert_major_bn > 0: one CTA per (expert, weight block) taking the expert's rows in
// chunks of that many rows (16..256), which lets the weights stream before the align
// tables exist; 0: one CTA per (token tile of bm_base rows, weight block).
int launch_grouped_gemm_impl(const void* a_sorted, const void* W, const moe_lora_align_t* al,
                             const AlignLayout& a, int N, int K, float* out, cudaStream_t stream,
                             bool pdl, bool early, int expert_major_bn);
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
