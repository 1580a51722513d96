// LoRA expand zB with the base-output add fused in (vllm.com.cn, section
// "Kernel optimizations": the LoRA result is added to the base output inside the
// expand kernel to save launches), and the layer's epilogues: SwiGLU between the
// projections and the routing-weighted top-k combine after the down projection
// (the router "aggregates" the experts' outputs; section "Implementing multi-LoRA
// inference for MoE models in vLLM").
//
// Each thread owns one output column n, so the rows of B_{l,e} (r contiguous
// bf16, 128-bit loads) and the base output are read coalesced across the warp;
// the block's z rows are staged in shared memory and broadcast. Sums over the
// rank run in a fixed order: deterministic.
#include "internal.h"

namespace moe_lora {

constexpr int kExpandThreads = 256;
constexpr int kMaxBmLora = 16;
constexpr int kSwigluRowChunk = 32;

// dot(z[0..r), B row) with the B row read 8 bf16 at a time when aligned.
template <bool kVecB>
__device__ __forceinline__ float dot_zb(const float* zs, const __nv_bfloat16* brow, int r) {
  float acc = 0.f;
  if (kVecB) {
    const uint4* b4 = reinterpret_cast<const uint4*>(brow);
    for (int i = 0; i < r; i += 8) {
      const uint4 u = __ldg(b4 + (i >> 3));
      acc = fmaf(zs[i + 0], bf16_lo(u.x), acc);
      acc = fmaf(zs[i + 1], bf16_hi(u.x), acc);
      acc = fmaf(zs[i + 2], bf16_lo(u.y), acc);
      acc = fmaf(zs[i + 3], bf16_hi(u.y), acc);
      acc = fmaf(zs[i + 4], bf16_lo(u.z), acc);
      acc = fmaf(zs[i + 5], bf16_hi(u.z), acc);
      acc = fmaf(zs[i + 6], bf16_lo(u.w), acc);
      acc = fmaf(zs[i + 7], bf16_hi(u.w), acc);
    }
  } else {
    for (int i = 0; i < r; ++i) acc = fmaf(zs[i], __bfloat162float(brow[i]), acc);
  }
  return acc;
}

// epilogue 0: base[row, n] += z[s] . B[l, e, n, :] over the rows of each LoRA block.
template <bool kVecB>
__global__ void __launch_bounds__(kExpandThreads)
    expand_add_kernel(const float* __restrict__ Z, const __nv_bfloat16* __restrict__ B,
                      const int* __restrict__ hdr, const int4* __restrict__ blocks,
                      const int* __restrict__ sorted_slots, int N, int r, int E,
                      float* __restrict__ base) {
  extern __shared__ float zs[];  // [rows][r]
  pdl_wait();
  const int nb = hdr[HDR_NBLOCKS];
  const int b = blockIdx.x;
  if (b >= nb) return;
  pdl_trigger();
  const int4 blk = blocks[b];
  const int row0 = blk.x, rows = blk.y, e = blk.z, l = blk.w;
  for (int i = threadIdx.x; i < rows * r; i += blockDim.x) {
    const int m = i / r, c = i - m * r;
    zs[i] = Z[(size_t)sorted_slots[row0 + m] * r + c];
  }
  __syncthreads();
  const int n = blockIdx.y * kExpandThreads + threadIdx.x;
  if (n >= N) return;
  const __nv_bfloat16* brow = B + (((size_t)l * E + e) * N + n) * (size_t)r;
  float acc[kMaxBmLora];
  if (kVecB) {
    // read the B row once, apply it to every row of the block
#pragma unroll
    for (int m = 0; m < kMaxBmLora; ++m) acc[m] = 0.f;
    const uint4* b4 = reinterpret_cast<const uint4*>(brow);
    for (int i = 0; i < r; i += 8) {
      const uint4 u = __ldg(b4 + (i >> 3));
      const float bv[8] = {bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y),
                           bf16_lo(u.z), bf16_hi(u.z), bf16_lo(u.w), bf16_hi(u.w)};
#pragma unroll
      for (int m = 0; m < kMaxBmLora; ++m) {
        if (m < rows) {
          const float* z = zs + m * r + i;
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[m] = fmaf(z[j], bv[j], acc[m]);
        }
      }
    }
  } else {
#pragma unroll
    for (int m = 0; m < kMaxBmLora; ++m) acc[m] = m < rows ? dot_zb<false>(zs + m * r, brow, r) : 0.f;
  }
#pragma unroll
  for (int m = 0; m < kMaxBmLora; ++m)
    if (m < rows) base[(size_t)(row0 + m) * N + n] += acc[m];
}

// epilogue 1: h[row, n] = silu(g) * u over every row of each token tile, with
// g = G[row, n] + z.B[l, e, n], u = G[row, I + n] + z.B[l, e, I + n].
template <bool kVecB>
__global__ void __launch_bounds__(kExpandThreads)
    expand_swiglu_kernel(const float* __restrict__ Z, const __nv_bfloat16* __restrict__ B,
                         const int* __restrict__ hdr, const int4* __restrict__ tiles,
                         const int* __restrict__ sorted_slots, const int* __restrict__ row_adapter,
                         int I, int r, int E, const float* __restrict__ G,
                         __nv_bfloat16* __restrict__ h) {
  extern __shared__ float zs[];  // [kSwigluRowChunk][r]
  __shared__ int s_l[kSwigluRowChunk];
  pdl_wait();
  const int nt = hdr[HDR_NTILES];
  if ((int)blockIdx.x >= nt) return;
  pdl_trigger();
  const int4 tile = tiles[blockIdx.x];
  const int e = tile.x, row0 = tile.y, rows = tile.z;
  const int n = blockIdx.y * kExpandThreads + threadIdx.x;
  const size_t twoI = 2 * (size_t)I;
  for (int c0 = 0; c0 < rows; c0 += kSwigluRowChunk) {
    const int cr = min(kSwigluRowChunk, rows - c0);
    __syncthreads();
    if (threadIdx.x < cr) s_l[threadIdx.x] = B ? row_adapter[row0 + c0 + threadIdx.x] : -1;
    __syncthreads();
    if (B) {
      for (int i = threadIdx.x; i < cr * r; i += blockDim.x) {
        const int m = i / r, c = i - m * r;
        zs[i] = s_l[m] >= 0 ? Z[(size_t)sorted_slots[row0 + c0 + m] * r + c] : 0.f;
      }
    }
    __syncthreads();
    if (n < I) {
      for (int m = 0; m < cr; ++m) {
        const int row = row0 + c0 + m;
        float g = G[(size_t)row * twoI + n];
        float u = G[(size_t)row * twoI + I + n];
        const int l = s_l[m];
        if (l >= 0) {
          const __nv_bfloat16* bl = B + ((size_t)l * E + e) * twoI * (size_t)r;
          g += dot_zb<kVecB>(zs + m * r, bl + (size_t)n * r, r);
          u += dot_zb<kVecB>(zs + m * r, bl + (size_t)(I + n) * r, r);
        }
        const float sg = g / (1.f + expf(-g));
        h[(size_t)row * I + n] = __float2bfloat16_rn(sg * u);
      }
    }
  }
}

// Weighted top-k combine: y[t, n] = sum_j w[t, j] * O[row(t, j), n], j ascending.
template <bool kOutF32>
__global__ void __launch_bounds__(kExpandThreads)
    combine_kernel(const float* __restrict__ O, const float* __restrict__ w,
                   const int* __restrict__ slot_row, int T, int k, int N, void* __restrict__ y) {
  pdl_wait();
  pdl_trigger();
  const int n = blockIdx.y * kExpandThreads + threadIdx.x;
  if (n >= N) return;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    float acc = 0.f;
    for (int j = 0; j < k; ++j) {
      const int row = slot_row[(size_t)t * k + j];
      if (row >= 0) acc = fmaf(w[(size_t)t * k + j], O[(size_t)row * N + n], acc);
    }
    if (kOutF32) static_cast<float*>(y)[(size_t)t * N + n] = acc;
    else static_cast<__nv_bfloat16*>(y)[(size_t)t * N + n] = __float2bfloat16_rn(acc);
  }
}

int launch_expand(const float* Z, const void* B, const moe_lora_align_t* al, const AlignLayout& a,
                  int N, int r, int epilogue, float* base, void* out, int out_fp32,
                  const float* topk_w, cudaStream_t stream, bool pdl) {
  if (a.S == 0) return MOE_LORA_OK;
  AlignView v = align_view(al->buf, a);
  const auto* Bp = (al->L > 0) ? static_cast<const __nv_bfloat16*>(B) : nullptr;
  const bool vecB = (r % 8 == 0) && aligned16(B);
  int st = MOE_LORA_OK;
  if (epilogue == 0 || epilogue == 2) {
    if (Bp) {
      const dim3 grid(a.max_blocks, ceil_div(N, kExpandThreads));
      const size_t smem = (size_t)kMaxBmLora * r * sizeof(float);
      st = vecB ? launch_pdl(expand_add_kernel<true>, grid, kExpandThreads, smem, stream, pdl, Z,
                             Bp, (const int*)v.hdr, (const int4*)v.blocks,
                             (const int*)v.sorted_slots, N, r, al->E, base)
                : launch_pdl(expand_add_kernel<false>, grid, kExpandThreads, smem, stream, pdl, Z,
                             Bp, (const int*)v.hdr, (const int4*)v.blocks,
                             (const int*)v.sorted_slots, N, r, al->E, base);
      if (st != MOE_LORA_OK) return st;
    }
    if (epilogue == 2) {
      int bx = al->T < 65535 ? al->T : 65535;
      const dim3 grid(bx, ceil_div(N, kExpandThreads));
      st = out_fp32 ? launch_pdl(combine_kernel<true>, grid, kExpandThreads, 0, stream, pdl,
                                 (const float*)base, topk_w, (const int*)v.slot_row, al->T, al->k,
                                 N, out)
                    : launch_pdl(combine_kernel<false>, grid, kExpandThreads, 0, stream, pdl,
                                 (const float*)base, topk_w, (const int*)v.slot_row, al->T, al->k,
                                 N, out);
    }
    return st;
  }
  if (epilogue == 1) {
    const int I = N / 2;
    const dim3 grid(a.max_tiles, ceil_div(I, kExpandThreads));
    const size_t smem = (size_t)kSwigluRowChunk * r * sizeof(float);
    auto* hp = static_cast<__nv_bfloat16*>(out);
    return vecB ? launch_pdl(expand_swiglu_kernel<true>, grid, kExpandThreads, smem, stream, pdl,
                             Z, Bp, (const int*)v.hdr, (const int4*)v.tiles,
                             (const int*)v.sorted_slots, (const int*)v.row_adapter, I, r, al->E,
                             (const float*)base, hp)
                : launch_pdl(expand_swiglu_kernel<false>, grid, kExpandThreads, smem, stream, pdl,
                             Z, Bp, (const int*)v.hdr, (const int4*)v.tiles,
                             (const int*)v.sorted_slots, (const int*)v.row_adapter, I, r, al->E,
                             (const float*)base, hp);
  }
  return MOE_LORA_ERR_INVALID_ARG;
}

}  // namespace moe_lora

extern "C" int lora_expand_add(const float* Z, const void* B, const moe_lora_align_t* al, int N,
                               int r, int epilogue, float* base, void* out, int out_fp32,
                               const float* topk_w, moe_lora_stream_t stream) {
  using namespace moe_lora;
  AlignLayout a;
  int st = check_align(al, &a);
  if (st != MOE_LORA_OK) return st;
  if (N < 1 || epilogue < 0 || epilogue > 2) return MOE_LORA_ERR_INVALID_ARG;
  if (al->L > 0 && (r < 1 || r > 256)) return r < 1 ? MOE_LORA_ERR_INVALID_ARG : MOE_LORA_ERR_UNSUPPORTED;
  if (epilogue == 1 && N % 2 != 0) return MOE_LORA_ERR_INVALID_ARG;
  if (a.S > 0) {
    if (!base) return MOE_LORA_ERR_INVALID_ARG;
    if (al->L > 0 && (!Z || !B)) return MOE_LORA_ERR_INVALID_ARG;
    if (epilogue != 0 && !out) return MOE_LORA_ERR_INVALID_ARG;
    if (epilogue == 2 && !topk_w) return MOE_LORA_ERR_INVALID_ARG;
  }
  if ((st = check_device()) != MOE_LORA_OK) return st;
  return launch_expand(Z, B, al, a, N, r, epilogue, base, out, out_fp32, topk_w,
                       reinterpret_cast<cudaStream_t>(stream), true);
}
