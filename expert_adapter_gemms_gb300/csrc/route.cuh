// Router top-k + softmax of one token by one warp (the router picks each token's top-k
// experts; vllm.com.cn, section "Implementing multi-LoRA inference for MoE models in
// vLLM"): the k largest logits (ties to the lower expert id, NaN below every number),
// then the softmax over the chosen values. Shared by the routing kernel
// and the one-CTA align that routes for itself, so both give the same bits.
#pragma once

#include "common.cuh"

namespace moe_lora {

// The token's E logits (lrow) as this lane holds them: experts lane, lane+32, ...,
// lane+32(V-1); past E: -inf (never chosen, see topk_softmax_select).
template <int V>
__device__ __forceinline__ void topk_softmax_load(const float* __restrict__ lrow, int E, float (&v)[V]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? __ldcg(lrow + e) : -INFINITY;
  }
}

// The order of a logit as an unsigned key: a larger number gets a larger key, -0 and +0 the
// same one, and every key of a number (-inf included) is above 0, the key of an expert
// already chosen or out of range.
__device__ __forceinline__ uint32_t topk_order_key(float x) {
  if (x == 0.f) x = 0.f;
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The choice from loaded logits for TB tokens at once: token b (tok[b] >= 0) writes choice
// j < k to ids[tok[b] k + j] and w[tok[b] k + j] (and, given, ids_copy[tok[b] k + j]).
// Choice j is the largest key not chosen before (one warp-wide integer max) and, among the
// experts holding it, the lowest id (one ballot per value a lane holds): the k largest
// logits with ties to the lower expert id, NaN below every number. Running TB tokens side
// by side lets their dependent steps overlap.
template <int V, int TB>
__device__ __forceinline__ void topk_softmax_select(const float (&vin)[TB][V], const int (&tok)[TB],
                                                    int E, int k, int* __restrict__ ids,
                                                    float* __restrict__ w,
                                                    int* ids_copy = nullptr) {
  const int lane = threadIdx.x & 31;
  float v[TB][V];
  uint32_t key[TB][V];  // 0: chosen already or out of range
#pragma unroll
  for (int b = 0; b < TB; ++b) {
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = lane + 32 * i;
      float x = vin[b][i];
      if (isnan(x)) x = -INFINITY;  // NaN ranks below every number
      v[b][i] = x;
      key[b][i] = e < E ? topk_order_key(x) : 0u;
    }
  }
  float sel_val[TB];
  int sel_id[TB];
#pragma unroll
  for (int b = 0; b < TB; ++b) {
    sel_val[b] = 0.f;
    sel_id[b] = 0;
  }
  for (int j = 0; j < k; ++j) {
    uint32_t m[TB];
#pragma unroll
    for (int b = 0; b < TB; ++b) {
      uint32_t lm = key[b][0];
#pragma unroll
      for (int i = 1; i < V; ++i) lm = max(lm, key[b][i]);
      m[b] = __reduce_max_sync(0xffffffffu, lm);
    }
#pragma unroll
    for (int b = 0; b < TB; ++b) {
      // the lowest id e = lane + 32 i holding the maximum: the lowest i first, then lane
      int win = -1;
      float wv = 0.f;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const unsigned bal = __ballot_sync(0xffffffffu, key[b][i] == m[b]);
        if (win < 0 && bal) {
          const int src = __ffs(bal) - 1;
          win = src + 32 * i;
          wv = __shfl_sync(0xffffffffu, v[b][i], src);
        }
      }
#pragma unroll
      for (int i = 0; i < V; ++i)
        if (win == lane + 32 * i) key[b][i] = 0u;
      if (lane == j) {
        sel_val[b] = wv;
        sel_id[b] = win;
      }
    }
  }
  float ex[TB], sum[TB];
#pragma unroll
  for (int b = 0; b < TB; ++b) {
    const float m = __shfl_sync(0xffffffffu, sel_val[b], 0);
    ex[b] = lane < k ? expf(sel_val[b] - m) : 0.f;
    sum[b] = ex[b];
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) {
#pragma unroll
    for (int b = 0; b < TB; ++b) sum[b] += __shfl_xor_sync(0xffffffffu, sum[b], off);
  }
#pragma unroll
  for (int b = 0; b < TB; ++b) {
    if (tok[b] >= 0 && lane < k) {
      ids[(size_t)tok[b] * k + lane] = sel_id[b];
      w[(size_t)tok[b] * k + lane] = ex[b] / sum[b];
      if (ids_copy) ids_copy[(size_t)tok[b] * k + lane] = sel_id[b];
    }
  }
}

// One token: its logits lrow; lane j < k writes choice j to ids_row[j] and w_row[j].
template <int V>
__device__ __forceinline__ void topk_softmax_token(const float* __restrict__ lrow, int E, int k,
                                                   int* __restrict__ ids_row,
                                                   float* __restrict__ w_row) {
  float v[1][V];
  const int tok[1] = {0};
  topk_softmax_load<V>(lrow, E, v[0]);
  topk_softmax_select<V, 1>(v, tok, E, k, ids_row, w_row);
}

}  // namespace moe_lora
