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
                  void* xs, cudaStream_t stream, bool pdl);

// Tensor maps are built on the host for every call (cheap; no device work).
int launch_grouped_gemm(const void* a_sorted, const void* W, const moe_lora_align_t* al,
                        const AlignLayout& a, int N, int K, float* out, cudaStream_t stream,
                        bool pdl);

int launch_shrink(const void* X, int rows_are_slots, const void* A, const moe_lora_align_t* al,
                  const AlignLayout& a, int K, int r, float* Z, cudaStream_t stream, bool pdl);

int launch_expand(const float* Z, const void* B, const moe_lora_align_t* al, const AlignLayout& a,
                  int N, int r, int epilogue, float* base, void* out, int out_fp32,
                  const float* topk_w, cudaStream_t stream, bool pdl);

}  // namespace moe_lora
