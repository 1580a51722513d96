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
int launch_shrink_impl(const void* X, int rows_are_slots, const void* A,
                       const moe_lora_align_t* al, const AlignLayout& a, int K, int r, float* Z,
                       cudaStream_t stream, bool pdl, bool early);
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

}  // namespace moe_lora
