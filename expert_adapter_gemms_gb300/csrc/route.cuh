// Router top-k + softmax of one token by one warp (the router picks each token's top-k
// experts; vllm.com.cn, section "Implementing multi-LoRA inference for MoE models in
// vLLM"): the k largest logits (ties to the lower expert id, NaN below every number),
// then the softmax over the chosen values. Shared by the routing kernel
// and the one-CTA align that routes for itself, so both give the same bits.
#pragma once
#include <climits>

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

// The choice from loaded logits for TB tokens at once: token b (tok[b] >= 0) writes choice
// j < k to ids[tok[b] k + j] and w[tok[b] k + j] (and, given, ids_copy[tok[b] k + j]).
// Each token takes exactly the steps of a single token; running TB of them side by side
// lets their dependent shuffle chains overlap.
template <int V, int TB>
__device__ __forceinline__ void topk_softmax_select(const float (&vin)[TB][V], const int (&tok)[TB],
                                                    int E, int k, int* __restrict__ ids,
                                                    float* __restrict__ w,
                                                    int* ids_copy = nullptr) {
  const int lane = threadIdx.x & 31;
  float v[TB][V];
  uint32_t taken[TB];  // bit i: expert lane + 32 i chosen already or out of range
#pragma unroll
  for (int b = 0; b < TB; ++b) {
    taken[b] = 0;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = lane + 32 * i;
      float x = vin[b][i];
      if (e < E) {
        if (isnan(x)) x = -INFINITY;  // NaN ranks below every number
      } else {
        taken[b] |= 1u << i;
      }
      v[b][i] = x;
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
    float bv[TB];
    int bi[TB];
#pragma unroll
    for (int b = 0; b < TB; ++b) {
      bv[b] = -INFINITY;
      bi[b] = INT_MAX;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int e = lane + 32 * i;
        if (!((taken[b] >> i) & 1u) && (v[b][i] > bv[b] || (v[b][i] == bv[b] && e < bi[b]))) {
          bv[b] = v[b][i];
          bi[b] = e;
        }
      }
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
#pragma unroll
      for (int b = 0; b < TB; ++b) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv[b], off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi[b], off);
        if (ov > bv[b] || (ov == bv[b] && oi < bi[b])) {
          bv[b] = ov;
          bi[b] = oi;
        }
      }
    }
#pragma unroll
    for (int b = 0; b < TB; ++b) {
      if ((bi[b] & 31) == lane) taken[b] |= 1u << (bi[b] >> 5);
      if (lane == j) {
        sel_val[b] = bv[b];
        sel_id[b] = bi[b];
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
