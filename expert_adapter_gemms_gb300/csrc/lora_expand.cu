// LoRA expand zB with the base-output add fused in (vllm.com.cn, section
// "Kernel optimizations": the LoRA result is added to the base output inside the
// expand kernel to save launches), and the layer's epilogues: SwiGLU between the
// projections and the routing-weighted top-k combine after the down projection
// (the router "aggregates" the experts' outputs; section "Implementing multi-LoRA
// inference for MoE models in vLLM").
//
// The expand is a stream: every touched B_{l,e} (N x r bf16) is read, each output
// element needs r multiply-adds. Threads own output columns, so B rows (r
// contiguous bf16, 128-bit loads) and base rows are read coalesced across a warp,
// and every thread issues all its loads before it consumes any. z rows are staged
// in shared memory and broadcast. Sums over the rank run in a fixed order:
// deterministic.
//
// Launch ordering: every kernel of the library triggers its dependents only after
// its own griddepcontrol.wait, so when a kernel starts, everything launched two or
// more steps earlier has completed. With `early` set (the layer sets it where it
// holds), a kernel reads such older data -- B weights, align tables, the base
// output of the GEMM two launches back -- before its own wait, and waits only for
// the z produced by its immediate predecessor.
#include <atomic>
#include "internal.h"

namespace moe_lora {

constexpr int kExpandThreads = 256;
constexpr int kMaxBmLora = 16;
constexpr int kMaxRegRank = 64;  // ranks held in registers; larger r reads B from L1
constexpr int kGStages = 6;     // tiles of G in flight per warp in the tensor-core SwiGLU expand
// bytes of the z staging area (bf16 high parts and remainders, 16 rows) for KC rank chunks
__host__ __device__ constexpr size_t zsmem_bytes(int KC) { return (size_t)2 * 16 * 32 * KC * 2; }

__device__ __forceinline__ void fma8(float& acc, const float* z, uint4 u) {
  acc = fmaf(z[0], bf16_lo(u.x), acc);
  acc = fmaf(z[1], bf16_hi(u.x), acc);
  acc = fmaf(z[2], bf16_lo(u.y), acc);
  acc = fmaf(z[3], bf16_hi(u.y), acc);
  acc = fmaf(z[4], bf16_lo(u.z), acc);
  acc = fmaf(z[5], bf16_hi(u.z), acc);
  acc = fmaf(z[6], bf16_lo(u.w), acc);
  acc = fmaf(z[7], bf16_hi(u.w), acc);
}

// 16-byte asynchronous copy global -> shared at L2 (coherent with earlier launches);
// `valid` false zero-fills the destination without reading the source.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// dot(z[0..r), B row) reading the B row from memory (any r, any alignment when !kVec).
template <bool kVec>
__device__ __forceinline__ float dot_zb_mem(const float* zs, const __nv_bfloat16* brow, int r) {
  float acc = 0.f;
  if (kVec) {
    const uint4* b4 = reinterpret_cast<const uint4*>(brow);
    for (int i = 0; i < r; i += 8) fma8(acc, zs + i, __ldg(b4 + (i >> 3)));
  } else {
    for (int i = 0; i < r; ++i) acc = fmaf(zs[i], __bfloat162float(brow[i]), acc);
  }
  return acc;
}

// ----------------------------------------------------------------------------
// epilogue 0: base[row, n] += z[s] . B[l, e, n, :] over the rows of each LoRA
// block; two columns per thread, B rows loaded once per block.
// ----------------------------------------------------------------------------
template <int RV>  // r / 8 when the B rows sit in registers (r % 8 == 0, r <= 64); 0 otherwise
__global__ void __launch_bounds__(kExpandThreads)
    expand_add_kernel(const float* __restrict__ Z, const __nv_bfloat16* __restrict__ B,
                      const int* __restrict__ hdr, const int4* __restrict__ blocks,
                      const int* __restrict__ sorted_slots, int N, int r, int E,
                      float* __restrict__ base, int early, const int* __restrict__ ranks) {
  extern __shared__ float zs[];  // [rows][r]
  if (!early) pdl_wait();
  const int nb = __ldcg(hdr + HDR_NBLOCKS);
  const int b = blockIdx.x;
  if (b >= nb) {
    if (early) pdl_wait();
    return;
  }
  const int4 blk = __ldcg(blocks + b);
  const int row0 = blk.x, rows = blk.y, e = blk.z, l = blk.w;
  const int n0 = blockIdx.y * (2 * kExpandThreads) + threadIdx.x;
  const int n1 = n0 + kExpandThreads;
  const __nv_bfloat16* bl = B + ((size_t)l * E + e) * (size_t)N * r;
  const int rl = adapter_rank(ranks, l, r, hdr);  // B columns past it are not used
  uint4 b0[RV > 0 ? RV : 1], b1[RV > 0 ? RV : 1];
  if (RV > 0) {
#pragma unroll
    for (int i = 0; i < RV; ++i) {
      b0[i] = n0 < N ? b_group(reinterpret_cast<const uint4*>(bl + (size_t)n0 * r), i, rl) : make_uint4(0, 0, 0, 0);
      b1[i] = n1 < N ? b_group(reinterpret_cast<const uint4*>(bl + (size_t)n1 * r), i, rl) : make_uint4(0, 0, 0, 0);
    }
  }
  if (early) pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i < rows * r; i += blockDim.x) {
    const int m = i / r, c = i - m * r;
    zs[i] = __ldcg(Z + (size_t)__ldcg(sorted_slots + row0 + m) * r + c);
  }
  __syncthreads();
  float acc0[kMaxBmLora], acc1[kMaxBmLora];
#pragma unroll
  for (int m = 0; m < kMaxBmLora; ++m) {
    acc0[m] = 0.f;
    acc1[m] = 0.f;
    if (m < rows) {
      if (RV > 0) {
#pragma unroll
        for (int i = 0; i < RV; ++i) {
          fma8(acc0[m], zs + m * r + 8 * i, b_tail(b0[i], 8 * i, rl));
          fma8(acc1[m], zs + m * r + 8 * i, b_tail(b1[i], 8 * i, rl));
        }
      } else {
        if (n0 < N) acc0[m] = dot_zb_mem<false>(zs + m * r, bl + (size_t)n0 * r, rl);
        if (n1 < N) acc1[m] = dot_zb_mem<false>(zs + m * r, bl + (size_t)n1 * r, rl);
      }
    }
  }
#pragma unroll
  for (int m = 0; m < kMaxBmLora; ++m) {
    if (m < rows) {
      float* o = base + (size_t)(row0 + m) * N;
      if (n0 < N) o[n0] += acc0[m];
      if (n1 < N) o[n1] += acc1[m];
    }
  }
}

// ----------------------------------------------------------------------------
// epilogue 1, row walk (short (expert, adapter) segments, e.g. decode; and ranks
// that are not a multiple of 8): h[row, n] = silu(g) * u for every valid row, with
//   g = G[row, n] + z.B[l, e, n],  u = G[row, I + n] + z.B[l, e, I + n].
// A CTA owns `rows_per_cta` consecutive sorted rows and 256 columns. With one row
// per CTA (short (expert, adapter) segments, e.g. decode) every load of a thread
// -- the G pair and both B rows -- is in flight at once, before the wait for z.
// With more rows (long segments, e.g. prefill) rows sorted by (e, l) share the B
// row pair, which stays in registers, and G is fetched four rows at a time.
// ----------------------------------------------------------------------------
template <int RV>
__global__ void __launch_bounds__(kExpandThreads)
    expand_swiglu_rows_kernel(const float* __restrict__ Z, const __nv_bfloat16* __restrict__ B,
                         const int* __restrict__ hdr, const int* __restrict__ sorted_slots,
                         const int* __restrict__ row_expert, const int* __restrict__ row_adapter,
                         int I, int r, int E, const float* __restrict__ G,
                         __nv_bfloat16* __restrict__ h, int rows_per_cta, int early,
                         int zstride, int zu_off, const int* __restrict__ ranks) {
  // z rows: zstride floats (r, or 2r with separate gate and up adapters); the gate
  // columns take z[0, r), the up columns z[zu_off, zu_off + r)
  extern __shared__ float zs[];  // [rows_per_cta][zstride]
  __shared__ int s_key[64];      // e * 65536 + (l + 1), or -1 without adapter
  __shared__ int s_slot[64];
  if (!early) pdl_wait();
  const int n_valid = __ldcg(hdr + HDR_NVALID);
  const int r0 = blockIdx.x * rows_per_cta;
  if (r0 >= n_valid) {
    if (early) pdl_wait();
    return;
  }
  const int rows = min(rows_per_cta, n_valid - r0);
  const int n = blockIdx.y * kExpandThreads + threadIdx.x;
  const bool col = n < I;
  const size_t twoI = 2 * (size_t)I;
  if (threadIdx.x < rows) {
    const int row = r0 + threadIdx.x;
    const int l = B ? __ldcg(row_adapter + row) : -1;
    s_key[threadIdx.x] = l < 0 ? -1 : __ldcg(row_expert + row) * 65536 + l + 1;
    s_slot[threadIdx.x] = __ldcg(sorted_slots + row);
  }
  __syncthreads();
  uint4 bg[RV > 0 ? RV : 1], bu[RV > 0 ? RV : 1];
  int cur = -1, cur_rl = r;
  auto load_b = [&](int key) {
    const int e = key >> 16, l = (key & 0xffff) - 1;
    const __nv_bfloat16* bl = B + ((size_t)l * E + e) * twoI * (size_t)r;
    cur_rl = adapter_rank(ranks, l, r, hdr);  // B columns past it are not used
#pragma unroll
    for (int i = 0; i < RV; ++i) {
      bg[i] = b_group(reinterpret_cast<const uint4*>(bl + (size_t)n * r), i, cur_rl);
      bu[i] = b_group(reinterpret_cast<const uint4*>(bl + (size_t)(I + n) * r), i, cur_rl);
    }
  };
  // G values are fetched four rows at a time; the first batch and the first B rows
  // are older than the predecessor and go out before the wait
  constexpr int RB = 4;
  float gv[RB], uv[RB];
  auto load_g = [&](int m0) {
#pragma unroll
    for (int q = 0; q < RB; ++q) {
      gv[q] = 0.f;
      uv[q] = 0.f;
      if (col && m0 + q < rows) {
        gv[q] = __ldcg(G + (size_t)(r0 + m0 + q) * twoI + n);
        uv[q] = __ldcg(G + (size_t)(r0 + m0 + q) * twoI + I + n);
      }
    }
  };
  if (early) {
    load_g(0);
    if (col && RV > 0 && s_key[0] >= 0) {
      load_b(s_key[0]);
      cur = s_key[0];
    }
    pdl_wait();
  }
  pdl_trigger();
  if (!early) load_g(0);
  if (B) {
    for (int i = threadIdx.x; i < rows * zstride; i += blockDim.x) {
      const int m = i / zstride, c = i - m * zstride;
      zs[i] = s_key[m] >= 0 ? __ldcg(Z + (size_t)s_slot[m] * zstride + c) : 0.f;
    }
  }
  __syncthreads();
  if (!col) return;
  for (int m0 = 0; m0 < rows; m0 += RB) {
    if (m0 > 0) load_g(m0);
#pragma unroll
    for (int q = 0; q < RB; ++q) {
      const int m = m0 + q;
      if (m >= rows) break;
      const int key = s_key[m];
      float g = gv[q], u = uv[q];
      if (key >= 0) {
        if (RV > 0) {
          if (key != cur) {
            load_b(key);
            cur = key;
          }
#pragma unroll
          for (int i = 0; i < RV; ++i) {
            fma8(g, zs + m * zstride + 8 * i, b_tail(bg[i], 8 * i, cur_rl));
            fma8(u, zs + m * zstride + zu_off + 8 * i, b_tail(bu[i], 8 * i, cur_rl));
          }
        } else {
          const int e = key >> 16, l = (key & 0xffff) - 1;
          const __nv_bfloat16* bl = B + ((size_t)l * E + e) * twoI * (size_t)r;
          const int rl = adapter_rank(ranks, l, r, hdr);
          g += dot_zb_mem<false>(zs + m * zstride, bl + (size_t)n * r, rl);
          u += dot_zb_mem<false>(zs + m * zstride + zu_off, bl + (size_t)(I + n) * r, rl);
        }
      }
      h[(size_t)(r0 + m) * I + n] = __float2bfloat16_rn(silu_fast(g) * u);
    }
  }
}

// ----------------------------------------------------------------------------
// epilogue 2: y[t, n] = sum_j w[t, j] * (O[row(t,j), n] + z[t k + j] . B[l, e_j, n, :]),
// j ascending, one thread per column, `tokens_per_cta` tokens per CTA. O values,
// B rows, routing weights and align tables are all older than the predecessor
// (the down shrink) and the first slot's are fetched before the wait; only z
// waits. The next slot's O value and B rows are fetched while the current slot
// is reduced.
// ----------------------------------------------------------------------------
template <int RV, bool kOutF32>
__global__ void __launch_bounds__(kExpandThreads)
    expand_combine_kernel(const float* __restrict__ Z, const __nv_bfloat16* __restrict__ B,
                          const int* __restrict__ slot_row, const int* __restrict__ row_expert,
                          const int* __restrict__ row_adapter, const float* __restrict__ w,
                          int T, int k, int N, int r, int E, const float* __restrict__ O,
                          void* __restrict__ y, int tokens_per_cta, int early,
                          const int* __restrict__ ranks) {
  extern __shared__ float zs[];  // [tokens_per_cta * k][r]
  __shared__ int s_row[256], s_key[256];
  __shared__ float s_w[256];
  if (!early) pdl_wait();
  const int t0 = blockIdx.x * tokens_per_cta;
  const int nt = min(tokens_per_cta, T - t0);
  const int ns = nt * k;  // slots of this CTA (the host keeps tokens_per_cta * k <= 256)
  for (int i = threadIdx.x; i < ns; i += blockDim.x) {
    const size_t s = (size_t)t0 * k + i;
    const int row = __ldcg(slot_row + s);
    int key = -1;
    if (row >= 0 && B) {
      const int l = __ldcg(row_adapter + row);
      if (l >= 0) key = __ldcg(row_expert + row) * 65536 + l + 1;
    }
    s_row[i] = row;
    s_key[i] = key;
    s_w[i] = __ldcg(w + s);
  }
  __syncthreads();
  const int n = blockIdx.y * kExpandThreads + threadIdx.x;
  const bool col = n < N;
  auto brow = [&](int key) {
    const int e = key >> 16, l = (key & 0xffff) - 1;
    return B + (((size_t)l * E + e) * N + n) * (size_t)r;
  };
  uint4 bcur[RV > 0 ? RV : 1], bnext[RV > 0 ? RV : 1];
  auto load_slot = [&](int q, float& o, uint4 (&bv)[RV > 0 ? RV : 1]) {
    if (s_row[q] >= 0) o = __ldcg(O + (size_t)s_row[q] * N + n);
    if (RV > 0 && s_key[q] >= 0) {
      const uint4* p = reinterpret_cast<const uint4*>(brow(s_key[q]));
      const int rl = adapter_rank(ranks, (s_key[q] & 0xffff) - 1, r, nullptr);
#pragma unroll
      for (int i = 0; i < RV; ++i) bv[i] = b_group(p, i, rl);
    }
  };
  float o_cur = 0.f;
  if (early && col && ns > 0) load_slot(0, o_cur, bcur);
  if (early) pdl_wait();
  pdl_trigger();
  if (B) {
    for (int i = threadIdx.x; i < ns * r; i += blockDim.x) {
      const int q = i / r, c = i - q * r;
      zs[i] = s_key[q] >= 0 ? __ldcg(Z + ((size_t)t0 * k + q) * r + c) : 0.f;
    }
  }
  __syncthreads();
  if (!col) return;
  if (!early && ns > 0) load_slot(0, o_cur, bcur);
  for (int ti = 0; ti < nt; ++ti) {
    float acc = 0.f;
    for (int j = 0; j < k; ++j) {
      const int q = ti * k + j;
      float o_next = 0.f;
      if (q + 1 < ns) load_slot(q + 1, o_next, bnext);
      if (s_row[q] >= 0) {
        float o = o_cur;
        if (s_key[q] >= 0) {
          if (RV > 0) {
            const int rl = adapter_rank(ranks, (s_key[q] & 0xffff) - 1, r, nullptr);
#pragma unroll
            for (int i = 0; i < RV; ++i) fma8(o, zs + q * r + 8 * i, b_tail(bcur[i], 8 * i, rl));
          } else {
            o += dot_zb_mem<false>(zs + q * r, brow(s_key[q]), adapter_rank(ranks, (s_key[q] & 0xffff) - 1, r, nullptr));
          }
        }
        acc = fmaf(s_w[q], o, acc);
      }
      o_cur = o_next;
#pragma unroll
      for (int i = 0; i < (RV > 0 ? RV : 1); ++i) bcur[i] = bnext[i];
    }
    const size_t yi = (size_t)(t0 + ti) * N + n;
    if (kOutF32) static_cast<float*>(y)[yi] = acc;
    else static_cast<__nv_bfloat16*>(y)[yi] = __float2bfloat16_rn(acc);
  }
}

// ----------------------------------------------------------------------------
// epilogue 1, one sorted row per CTA (short (expert, adapter) segments: decode, or
// many adapters): the same arithmetic as the row walk above, but a thread's loads
// do not wait on one another. The row's align tables, the G pair and then the B
// rows are all issued before anything is consumed, and no thread waits at a
// barrier for another thread's table reads; the one barrier stages z (r floats)
// after the B rows are in flight.
// ----------------------------------------------------------------------------
// kTwo: separate gate and up adapters (two z slices); kRanked: adapters of their own ranks
template <int RV, bool kTwo, bool kRanked>
__global__ void __launch_bounds__(kExpandThreads)
    expand_swiglu_row1_kernel(const float* __restrict__ Z, const __nv_bfloat16* __restrict__ B,
                              const int* __restrict__ hdr, const int* __restrict__ sorted_slots,
                              const int* __restrict__ row_expert,
                              const int* __restrict__ row_adapter, int I, int r, int E,
                              const float* __restrict__ G, __nv_bfloat16* __restrict__ h,
                              int early, int zstride, int zu_off, const int* __restrict__ ranks) {
  if (!early) pdl_wait();
  const int row = blockIdx.x;
  const int n = blockIdx.y * kExpandThreads + threadIdx.x;
  const int lane = threadIdx.x & 31;
  const bool col = n < I;
  const size_t twoI = 2 * (size_t)I;
  // rows past n_valid exist (the tables and G have S rows); their values are unused
  const int n_valid = __ldcg(hdr + HDR_NVALID);
  const int l = B ? __ldcg(row_adapter + row) : -1;
  const int e = __ldcg(row_expert + row);
  const int slot = __ldcg(sorted_slots + row);
  float g = 0.f, u = 0.f;
  if (col) {
    g = __ldcg(G + (size_t)row * twoI + n);
    u = __ldcg(G + (size_t)row * twoI + I + n);
  }
  const bool active = row < n_valid;
  const bool lora = active && l >= 0;  // uniform over the CTA
  const int rl = kRanked && lora ? adapter_rank(ranks, l, r, hdr) : r;  // B columns past it unused
  uint4 bg[RV], bu[RV];
#pragma unroll
  for (int i = 0; i < RV; ++i) bg[i] = bu[i] = make_uint4(0, 0, 0, 0);
  if (lora && col) {
    const __nv_bfloat16* bl = B + ((size_t)l * E + e) * twoI * (size_t)r;
    const uint4* pg = reinterpret_cast<const uint4*>(bl + (size_t)n * r);
    const uint4* pu = reinterpret_cast<const uint4*>(bl + (size_t)(I + n) * r);
#pragma unroll
    for (int i = 0; i < RV; ++i) {
      bg[i] = b_group(pg, i, rl);
      bu[i] = b_group(pu, i, rl);
    }
  }
  if (early) pdl_wait();
  pdl_trigger();
  if (!active) return;
  if (lora) {
    // z (r = 8 RV floats) is read once per warp, one or two values per lane, and
    // broadcast with shuffles: no shared-memory staging, no barrier
    // (the up columns' z sits zu_off floats further when gate and up have separate adapters)
    constexpr int ZL = RV > 4 ? 2 : 1;
    float zl[ZL], zul[ZL];
    const float* zrow = Z + (size_t)slot * zstride;
#pragma unroll
    for (int j = 0; j < ZL; ++j) {
      const int i = lane + 32 * j;
      zl[j] = i < 8 * RV ? __ldcg(zrow + i) : 0.f;
      zul[j] = kTwo && i < 8 * RV ? __ldcg(zrow + zu_off + i) : 0.f;
    }
    // every lane takes part in the shuffles (lanes past the last column included)
#pragma unroll
    for (int i = 0; i < RV; ++i) {
      float zv[8], zw[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        zv[c] = __shfl_sync(0xffffffffu, zl[(8 * i + c) >> 5], (8 * i + c) & 31);
        zw[c] = kTwo ? __shfl_sync(0xffffffffu, zul[(8 * i + c) >> 5], (8 * i + c) & 31) : zv[c];
      }
      fma8(g, zv, kRanked ? b_tail(bg[i], 8 * i, rl) : bg[i]);
      fma8(u, zw, kRanked ? b_tail(bu[i], 8 * i, rl) : bu[i]);
    }
  }
  if (col) h[(size_t)row * I + n] = __float2bfloat16_rn(silu_fast(g) * u);
}

// ----------------------------------------------------------------------------
// Tensor-core expand of one LoRA block (at most 16 rows of one (e, l) segment):
//   D[m, n] = sum_i z[m, i] * B[l, e, n, i]
// with mma.sync m16n8k16: the block's rows on M (padded to 16), 8 output columns
// on N, the rank on K, fp32 accumulation. z is held as a bf16 pair (high part and
// the bf16 rounding of the remainder), so z . B = z_hi . B + z_lo . B keeps the
// fp32 z to about 2^-16 relative; B is bf16 already. Each lane loads 16 bytes of
// the B row of column n0 + lane/4 at k = 32c + 8(lane%4); both operands feed
// those 8 consecutive k to the fragment slots through the same permutation (the
// shrink's scheme), which leaves the sums unchanged.
// One CTA takes a whole block: its z fragments stay in registers while the warps
// sweep the output columns 8 at a time, each tile's B fragments and base values
// fetched while the previous tile is reduced.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// z rows of a block in shared memory as bf16 high parts [16][r_pad] followed by the
// bf16 remainders [16][r_pad]; rows >= rows and ranks >= r are zero.
__device__ __forceinline__ void stage_z_split(__nv_bfloat16* zb, const float* __restrict__ Z,
                                              const int* __restrict__ sorted_slots, int row0,
                                              int rows, int r, int r_pad, int zstride = -1,
                                              int zoff = 0) {
  if (zstride < 0) zstride = r;  // z rows of zstride floats; this slice starts at zoff
  for (int i = threadIdx.x; i < 16 * r_pad; i += blockDim.x) {
    const int m = i / r_pad, c = i - m * r_pad;
    float v = 0.f;
    if (m < rows && c < r) v = __ldcg(Z + (size_t)__ldcg(sorted_slots + row0 + m) * zstride + zoff + c);
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    zb[i] = hi;
    zb[16 * r_pad + i] = __float2bfloat16_rn(v - __bfloat162float(hi));
  }
}

// This lane's z fragments, chunk c: [part][c] = {row lane/4, row lane/4 + 8} x 8 k.
template <int KC>
struct ZFrag {
  uint4 a[2][KC], b[2][KC];
  __device__ __forceinline__ void load(const __nv_bfloat16* zb, int r_pad) {
    const int lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
#pragma unroll
    for (int part = 0; part < 2; ++part)
#pragma unroll
      for (int c = 0; c < KC; ++c) {
        const __nv_bfloat16* zp = zb + part * 16 * r_pad + 32 * c + 8 * q;
        a[part][c] = *reinterpret_cast<const uint4*>(zp + gid * r_pad);
        b[part][c] = *reinterpret_cast<const uint4*>(zp + (gid + 8) * r_pad);
      }
  }
};

// The B fragment of chunk c for this lane (zeros past the adapter's rank rv or the last
// column; 16-byte groups wholly past rv are not read).
__device__ __forceinline__ uint4 b_frag(const __nv_bfloat16* brow, int c, int rv) {
  const int k0 = 32 * c + 8 * (threadIdx.x & 3);
  if (!brow || k0 >= rv) return make_uint4(0, 0, 0, 0);
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(brow + k0));
  return u;  // entries past rv of a partial group: cleared with b_frag_mask where consumed
}
// Per-lane AND masks that clear a fragment's entries past rv (all ones unless this lane's
// 8-rank group of chunk c is the partial one); built once per block, applied with and4.
__device__ __forceinline__ uint4 b_frag_mask(int c, int rv) {
  const int v = rv - (32 * c + 8 * (threadIdx.x & 3));
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) w[i] = 2 * i + 1 < v ? 0xFFFFFFFFu : (2 * i < v ? 0x0000FFFFu : 0u);
  return make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ uint4 and4(uint4 a, uint4 m) {
  return make_uint4(a.x & m.x, a.y & m.y, a.z & m.z, a.w & m.w);
}

template <int KC>
__device__ __forceinline__ void block_mma(float (&acc)[4], const ZFrag<KC>& z, const uint4 (&bf)[KC]) {
  acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
#pragma unroll
  for (int part = 0; part < 2; ++part)
#pragma unroll
    for (int c = 0; c < KC; ++c) {
      mma_bf16_16816(acc, z.a[part][c].x, z.b[part][c].x, z.a[part][c].y, z.b[part][c].y,
                     bf[c].x, bf[c].y);
      mma_bf16_16816(acc, z.a[part][c].z, z.b[part][c].z, z.a[part][c].w, z.b[part][c].w,
                     bf[c].z, bf[c].w);
    }
}

// epilogue 1 with tensor cores. CTAs [0, max_blocks): one LoRA block each, all
// columns; CTAs beyond: (token tile, 512-column chunk) pairs applying the plain
// SwiGLU to the tile's rows without adapter.
// kTwo: separate gate and up adapters (two z slices); kRanked: adapters of their own ranks
template <int KC, bool kTwo, bool kRanked>
__global__ void __launch_bounds__(kExpandThreads)
    expand_swiglu_mma_kernel(const float* __restrict__ Z, const __nv_bfloat16* __restrict__ B,
                             const int* __restrict__ hdr, const int4* __restrict__ blocks,
                             const int4* __restrict__ tiles, const int* __restrict__ sorted_slots,
                             const int* __restrict__ row_adapter, int I, int r, int E,
                             const float* __restrict__ G, __nv_bfloat16* __restrict__ h,
                             int max_blocks, int col_chunks, int early, int zstride, int zu_off,
                             const int* __restrict__ ranks) {
  constexpr int kWarps = kExpandThreads / 32;
  constexpr int kChunk = 2 * kExpandThreads;  // columns per plain-SwiGLU CTA
  __shared__ int s_flag[256];
  __shared__ int s_any;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __nv_bfloat16* zb = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  const int r_pad = 32 * KC;
  const size_t twoI = 2 * (size_t)I;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
  if (!early) pdl_wait();
  if ((int)blockIdx.x < max_blocks * col_chunks) {
    const int b = blockIdx.x / col_chunks, chunk = blockIdx.x - b * col_chunks;
    if (!B || b >= __ldcg(hdr + HDR_NBLOCKS)) {
      if (early) pdl_wait();
      return;
    }
    const int4 blk = __ldcg(blocks + b);
    const int row0 = blk.x, rows = blk.y, e = blk.z, l = blk.w;
    const __nv_bfloat16* bl = B + ((size_t)l * E + e) * twoI * (size_t)r;
    const int rl = kRanked ? adapter_rank(ranks, l, r, hdr) : r;  // z and B past it unused
    uint4 bmask[KC];
#pragma unroll
    for (int c = 0; c < KC; ++c) bmask[c] = kRanked ? b_frag_mask(c, rl) : make_uint4(0, 0, 0, 0);
    // this CTA's 8-column tiles: [t_begin, t_end)
    const int all_tiles = (I + 7) / 8;
    const int per = (all_tiles + col_chunks - 1) / col_chunks;
    const int t_begin = chunk * per;
    const int ntiles = min(all_tiles, t_begin + per);
    // B fragments of a tile go to registers one tile ahead; the G values of the block's
    // rows (the largest stream: fp32 rows of the gate_up GEMM) go through a per-warp
    // ring of kGStages tiles in shared memory with asynchronous copies, so each warp
    // keeps several KB of G in flight without spending registers on it. A tile's G
    // part is [16 rows][8 columns] fp32 for gate and for up: lane -> (row lane / 2,
    // columns 4 (lane % 2) .. +3), one 16-byte copy per part.
    // B fragments two tiles ahead: the warp's tiles alternate between two register sets
    uint4 bg0[KC], bu0[KC], bg1[KC], bu1[KC];
    auto fetch_b = [&](int t, uint4 (&bg)[KC], uint4 (&bu)[KC]) {
      if (t >= ntiles) return;
      const int nl = t * 8 + gid;
#pragma unroll
      for (int c = 0; c < KC; ++c) {
        bg[c] = b_frag(nl < I ? bl + (size_t)nl * r : nullptr, c, rl);
        bu[c] = b_frag(nl < I ? bl + (size_t)(I + nl) * r : nullptr, c, rl);
      }
    };
    // shared memory: z of the gate columns, z of the up columns, then the G ring
    float* gring = reinterpret_cast<float*>(smem_raw + 2 * zsmem_bytes(KC)) + warp * (kGStages * 256);
    auto fetch_g = [&](int t, int stage) {
      if (t < ntiles) {
        const int m = lane >> 1, c4 = (lane & 1) * 4;
        const int n = t * 8 + c4;
        const bool ok = m < rows && n < I;
        const float* src = ok ? G + (size_t)(row0 + m) * twoI + n : G;
        float* dst = gring + stage * 256 + m * 8 + c4;
        cp_async16(dst, src, ok);
        cp_async16(dst + 128, ok ? src + I : G, ok);
      }
      cp_async_commit();  // one group per stage, empty or not
    };
    int t = t_begin + warp;
#pragma unroll
    for (int d = 0; d < kGStages - 1; ++d) fetch_g(t + d * kWarps, d);
    fetch_b(t, bg0, bu0);
    fetch_b(t + kWarps, bg1, bu1);
    if (early) pdl_wait();
    pdl_trigger();
    __nv_bfloat16* zbu = zb + zsmem_bytes(KC) / sizeof(__nv_bfloat16);
    stage_z_split(zb, Z, sorted_slots, row0, rows, rl, r_pad, zstride, 0);
    if (kTwo) stage_z_split(zbu, Z, sorted_slots, row0, rows, rl, r_pad, zstride, zu_off);
    __syncthreads();
    ZFrag<KC> z, z2;
    z.load(zb, r_pad);
    if (kTwo) z2.load(zbu, r_pad);
    const ZFrag<KC>& zu = kTwo ? z2 : z;
    // tile t (the j-th of this warp) from the register set (bg, bu), which then takes tile
    // t + 2 kWarps
    auto tile = [&](int t, int j, uint4 (&bg)[KC], uint4 (&bu)[KC]) {
      fetch_g(t + (kGStages - 1) * kWarps, (j + kGStages - 1) % kGStages);
      cp_async_wait<kGStages - 1>();  // this tile's copies have landed
      __syncwarp();                   // ... every lane's
      uint4 tg[KC], tu[KC];
#pragma unroll
      for (int c = 0; c < KC; ++c) {
        tg[c] = bg[c];
        tu[c] = bu[c];
      }
      fetch_b(t + 2 * kWarps, bg, bu);  // B two tiles ahead in flight
      if (kRanked) {
#pragma unroll
        for (int c = 0; c < KC; ++c) {  // entries past the adapter's rank
          tg[c] = and4(tg[c], bmask[c]);
          tu[c] = and4(tu[c], bmask[c]);
        }
      }
      float dg[4], du[4];
      block_mma<KC>(dg, z, tg);
      block_mma<KC>(du, zu, tu);
      const int n = t * 8 + 2 * q;
      const float* gs = gring + (j % kGStages) * 256;
      if (n < I) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int m = gid + 8 * half;
          if (m >= rows) continue;
          const float2 gv = *reinterpret_cast<const float2*>(gs + m * 8 + 2 * q);
          const float2 uv = *reinterpret_cast<const float2*>(gs + 128 + m * 8 + 2 * q);
          const float g0 = gv.x + dg[2 * half], g1 = gv.y + dg[2 * half + 1];
          const float u0 = uv.x + du[2 * half], u1 = uv.y + du[2 * half + 1];
          __nv_bfloat162 o;
          o.x = __float2bfloat16_rn(silu_fast(g0) * u0);
          o.y = __float2bfloat16_rn(silu_fast(g1) * u1);
          *reinterpret_cast<__nv_bfloat162*>(h + (size_t)(row0 + m) * I + n) = o;
        }
      }
      __syncwarp();  // the stage is read by every lane before it is refilled
    };
    for (int j = 0; t < ntiles; t += 2 * kWarps, j += 2) {
      tile(t, j, bg0, bu0);
      if (t + kWarps < ntiles) tile(t + kWarps, j + 1, bg1, bu1);
    }
    cp_async_wait<0>();
  } else {
    // adapter-free rows of one token tile: plain SwiGLU, two columns per thread
    const int nch = (I + kChunk - 1) / kChunk;
    const int idx = blockIdx.x - max_blocks * col_chunks;
    const int ti = idx / nch, ch = idx - ti * nch;
    if (ti >= __ldcg(hdr + HDR_NTILES)) {
      if (early) pdl_wait();
      return;
    }
    const int4 tile = __ldcg(tiles + ti);
    const int row0 = tile.y, rows = tile.z;  // rows <= 256
    if (threadIdx.x == 0) s_any = 0;
    __syncthreads();
    if ((int)threadIdx.x < rows) {  // which rows need the plain SwiGLU (no adapter)
      const int f = B ? (__ldcg(row_adapter + row0 + threadIdx.x) < 0) : 1;
      s_flag[threadIdx.x] = f;
      if (f) s_any = 1;
    }
    __syncthreads();
    if (early) pdl_wait();
    pdl_trigger();
    const int n = ch * kChunk + 2 * threadIdx.x;
    if (!s_any || n >= I) return;
    for (int m = 0; m < rows; ++m) {
      if (!s_flag[m]) continue;  // a LoRA-block CTA owns it
      const size_t gr = (size_t)(row0 + m) * twoI;
      const float2 g = __ldcg(reinterpret_cast<const float2*>(G + gr + n));
      const float2 u = __ldcg(reinterpret_cast<const float2*>(G + gr + I + n));
      __nv_bfloat162 o;
      o.x = __float2bfloat16_rn(silu_fast(g.x) * u.x);
      o.y = __float2bfloat16_rn(silu_fast(g.y) * u.y);
      *reinterpret_cast<__nv_bfloat162*>(h + (size_t)(row0 + m) * I + n) = o;
    }
  }
}

// epilogue 0 (and the block-walk half of epilogue 2) with tensor cores:
// base[row, n..n+1] += D for the rows of each LoRA block. A warp takes its column
// tiles TB at a time: the B fragments and base values of all TB tiles are loaded
// before any is reduced, so each warp keeps several KB of the read-modify-write
// in flight (base is two or more launches old: with `early` the first batch goes
// out before the wait).
template <int KC, bool kRanked>  // kRanked: adapters of their own ranks
__global__ void __launch_bounds__(kExpandThreads)
    expand_add_mma_kernel(const float* __restrict__ Z, const __nv_bfloat16* __restrict__ B,
                          const int* __restrict__ hdr, const int4* __restrict__ blocks,
                          const int* __restrict__ sorted_slots, int N, int r, int E,
                          float* __restrict__ base, int col_chunks, int early,
                          const int* __restrict__ ranks) {
  constexpr int kWarps = kExpandThreads / 32;
  constexpr int TB = 8 / KC > 1 ? 8 / KC : 1;  // tiles per batch
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __nv_bfloat16* zb = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  const int r_pad = 32 * KC;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, q = lane & 3;
  if (!early) pdl_wait();
  const int b = blockIdx.x / col_chunks, chunk = blockIdx.x - b * col_chunks;
  const int nb = __ldcg(hdr + HDR_NBLOCKS);
  const int4 blk = __ldcg(blocks + b);  // in bounds: the grid covers the host's block bound
  if (b >= nb) {
    if (early) pdl_wait();
    return;
  }
  const int row0 = blk.x, rows = blk.y, e = blk.z, l = blk.w;
  const __nv_bfloat16* bl = B + ((size_t)l * E + e) * (size_t)N * r;
  const int rl = kRanked ? adapter_rank(ranks, l, r, hdr) : r;  // z and B past it unused
  uint4 bmask[KC];
#pragma unroll
  for (int c = 0; c < KC; ++c) bmask[c] = kRanked ? b_frag_mask(c, rl) : make_uint4(0, 0, 0, 0);
  const int all_tiles = (N + 7) / 8;
  const int per = (all_tiles + col_chunks - 1) / col_chunks;
  const int t_begin = chunk * per;
  const int ntiles = min(all_tiles, t_begin + per);
  uint4 bf[TB][KC];
  float2 ov[TB][2];
  auto fetch = [&](int t0) {
#pragma unroll
    for (int j = 0; j < TB; ++j) {
      const int t = t0 + j * kWarps;
      const int nl = t * 8 + gid, n = t * 8 + 2 * q;
      const bool tv = t < ntiles;
#pragma unroll
      for (int c = 0; c < KC; ++c)
        bf[j][c] = b_frag(tv && nl < N ? bl + (size_t)nl * r : nullptr, c, rl);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int m = gid + 8 * half;
        ov[j][half] = make_float2(0.f, 0.f);
        if (tv && n < N && m < rows)
          ov[j][half] = __ldcg(reinterpret_cast<const float2*>(base + (size_t)(row0 + m) * N + n));
      }
    }
  };
  int t0 = t_begin + warp;
  if (early && t0 < ntiles) fetch(t0);
  if (early) pdl_wait();
  pdl_trigger();
  stage_z_split(zb, Z, sorted_slots, row0, rows, rl, r_pad, r, 0);
  __syncthreads();
  ZFrag<KC> z;
  z.load(zb, r_pad);
  if (!early && t0 < ntiles) fetch(t0);
  for (; t0 < ntiles; t0 += TB * kWarps) {
#pragma unroll
    for (int j = 0; j < TB; ++j) {
      const int t = t0 + j * kWarps;
      const int n = t * 8 + 2 * q;
      if (t >= ntiles || n >= N) continue;
      float d[4];
      uint4 bt[KC];
#pragma unroll
      for (int c = 0; c < KC; ++c) bt[c] = kRanked ? and4(bf[j][c], bmask[c]) : bf[j][c];
      block_mma<KC>(d, z, bt);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int m = gid + 8 * half;
        if (m >= rows) continue;
        float2 v = ov[j][half];
        v.x += d[2 * half];
        v.y += d[2 * half + 1];
        *reinterpret_cast<float2*>(base + (size_t)(row0 + m) * N + n) = v;
      }
    }
    if (t0 + TB * kWarps < ntiles) fetch(t0 + TB * kWarps);
  }
}

// ----------------------------------------------------------------------------
// Weighted top-k combine after an in-place expand over LoRA blocks:
//   y[t, n] = sum_j w[t, j] * O[row(t, j), n], j ascending.
// The CTA's slot rows and weights are staged in shared memory first (with `early`,
// before the wait: the align and the routing are two or more launches back); then each
// thread issues the O values of all of a token's slots (eight at a time) before
// it sums them, in j order.
// ----------------------------------------------------------------------------
template <bool kOutF32>
__global__ void __launch_bounds__(kExpandThreads)
    combine_kernel(const float* __restrict__ O, const float* __restrict__ w,
                   const int* __restrict__ slot_row, int T, int k, int N, void* __restrict__ y,
                   int tokens_per_cta, int nparts, size_t part_stride, int early) {
  constexpr int KM = 8;
  __shared__ int s_row[kExpandThreads];
  __shared__ float s_w[kExpandThreads];
  if (!early) {
    pdl_wait();
    pdl_trigger();
  }
  const int t0 = blockIdx.x * tokens_per_cta;
  const int t1 = min(T, t0 + tokens_per_cta);
  const int ns = (t1 - t0) * k;  // the host keeps tokens_per_cta * k <= 256
  for (int i = threadIdx.x; i < ns; i += blockDim.x) {
    s_row[i] = __ldcg(slot_row + (size_t)t0 * k + i);
    s_w[i] = __ldcg(w + (size_t)t0 * k + i);
  }
  if (early) {
    pdl_wait();
    pdl_trigger();
  }
  __syncthreads();
  const int n = blockIdx.y * kExpandThreads + threadIdx.x;
  if (n >= N) return;
  for (int t = t0; t < t1; ++t) {
    const int q0 = (t - t0) * k;
    float acc = 0.f;
    for (int j0 = 0; j0 < k; j0 += KM) {
      float o[KM];
#pragma unroll
      for (int j = 0; j < KM; ++j) {
        o[j] = 0.f;
        if (j0 + j < k) {
          const int row = s_row[q0 + j0 + j];
          if (row >= 0) {
            o[j] = __ldcg(O + (size_t)row * N + n);
            for (int pp = 1; pp < nparts; ++pp)  // partial outputs of a split K range
              o[j] += __ldcg(O + pp * part_stride + (size_t)row * N + n);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < KM; ++j)
        if (j0 + j < k && s_row[q0 + j0 + j] >= 0) acc = fmaf(s_w[q0 + j0 + j], o[j], acc);
    }
    if (kOutF32) static_cast<float*>(y)[(size_t)t * N + n] = acc;
    else static_cast<__nv_bfloat16*>(y)[(size_t)t * N + n] = __float2bfloat16_rn(acc);
  }
}

// The same combine, four columns per thread: 16-byte loads of O, and the loads of eight
// consecutive slots (two tokens at k = 4) in flight before they are summed -- per element
// the same products in the same order as above, so the same bits. N % 4 == 0 and y
// aligned for 16-byte (fp32) or 8-byte (bf16) stores.
template <bool kOutF32>
__global__ void __launch_bounds__(kExpandThreads)
    combine4_kernel(const float* __restrict__ O, const float* __restrict__ w,
                    const int* __restrict__ slot_row, int T, int k, int N, void* __restrict__ y,
                    int tokens_per_cta, int nparts, size_t part_stride, int early) {
  constexpr int KM = 8;
  __shared__ int s_row[kExpandThreads];
  __shared__ float s_w[kExpandThreads];
  if (!early) {
    pdl_wait();
    pdl_trigger();
  }
  const int t0 = blockIdx.x * tokens_per_cta;
  const int t1 = min(T, t0 + tokens_per_cta);
  const int ns = (t1 - t0) * k;  // the host keeps tokens_per_cta * k <= 256
  for (int i = threadIdx.x; i < ns; i += blockDim.x) {
    s_row[i] = __ldcg(slot_row + (size_t)t0 * k + i);
    s_w[i] = __ldcg(w + (size_t)t0 * k + i);
  }
  if (early) {
    pdl_wait();
    pdl_trigger();
  }
  __syncthreads();
  const int n = 4 * (blockIdx.y * kExpandThreads + threadIdx.x);
  if (n >= N) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int q0 = 0; q0 < ns; q0 += KM) {
    float4 o[KM];
#pragma unroll
    for (int i = 0; i < KM; ++i) {
      o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      const int row = q0 + i < ns ? s_row[q0 + i] : -1;
      if (row >= 0) {
        o[i] = __ldcg(reinterpret_cast<const float4*>(O + (size_t)row * N + n));
        for (int pp = 1; pp < nparts; ++pp) {  // partial outputs of a split K range
          const float4 v = __ldcg(reinterpret_cast<const float4*>(O + pp * part_stride + (size_t)row * N + n));
          o[i].x += v.x;
          o[i].y += v.y;
          o[i].z += v.z;
          o[i].w += v.w;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < KM; ++i) {
      const int q = q0 + i;
      if (q >= ns) break;
      if (s_row[q] >= 0) {
        const float wq = s_w[q];
        acc.x = fmaf(wq, o[i].x, acc.x);
        acc.y = fmaf(wq, o[i].y, acc.y);
        acc.z = fmaf(wq, o[i].z, acc.z);
        acc.w = fmaf(wq, o[i].w, acc.w);
      }
      if ((q + 1) % k == 0) {  // the token's last slot
        const size_t at = (size_t)(t0 + q / k) * N + n;
        if (kOutF32) {
          *reinterpret_cast<float4*>(static_cast<float*>(y) + at) = acc;
        } else {
          const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
          const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
          uint2 u;
          u.x = *reinterpret_cast<const uint32_t*>(&lo);
          u.y = *reinterpret_cast<const uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(y) + at) = u;
        }
        acc = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------
template <template <int> class K, typename... Args>
static int launch_rv(int rv, dim3 grid, size_t smem, cudaStream_t stream, bool pdl,
                     Args... args) {
  switch (rv) {
    case 1: return launch_pdl(K<1>::fn, grid, kExpandThreads, smem, stream, pdl, args...);
    case 2: return launch_pdl(K<2>::fn, grid, kExpandThreads, smem, stream, pdl, args...);
    case 4: return launch_pdl(K<4>::fn, grid, kExpandThreads, smem, stream, pdl, args...);
    case 8: return launch_pdl(K<8>::fn, grid, kExpandThreads, smem, stream, pdl, args...);
    default: return launch_pdl(K<0>::fn, grid, kExpandThreads, smem, stream, pdl, args...);
  }
}
template <int RV> struct AddK { static constexpr auto fn = expand_add_kernel<RV>; };
template <int RV> struct SwigluK { static constexpr auto fn = expand_swiglu_rows_kernel<RV>; };

// r / 8 when the B rows can sit in registers with 128-bit loads, else 0.
static int reg_ranks(int r, const void* B) {
  if (r % 8 != 0 || r > kMaxRegRank || !aligned16(B)) return 0;
  const int rv = r / 8;
  return (rv == 1 || rv == 2 || rv == 4 || rv == 8) ? rv : 0;
}

int launch_expand_impl(const float* Z, const void* B, const moe_lora_align_t* al,
                       const AlignLayout& a, int N, int r, int epilogue_in, float* base, void* out,
                       int out_fp32, const float* topk_w, cudaStream_t stream, bool pdl,
                       bool early) {
  if (a.S == 0) return MOE_LORA_OK;
  // epilogue 3 is epilogue 1 with separate gate and up adapters: z rows of 2r floats,
  // the up columns taking the second r
  const int epilogue = epilogue_in == 3 ? 1 : epilogue_in;
  const int zstride = epilogue_in == 3 ? 2 * r : r, zu_off = epilogue_in == 3 ? r : 0;
  AlignView v = align_view(al->buf, a);
  const int* ranks = al->L > 0 ? al->adapter_ranks : nullptr;
  const auto* Bp = (al->L > 0) ? static_cast<const __nv_bfloat16*>(B) : nullptr;
  const int rv = Bp ? reg_ranks(r, B) : 1;
  const int rr = Bp ? r : 0;
  const int sms = num_sms();
  const int ea = early ? 1 : 0;
  // tensor-core block expand: B rows of r % 8 == 0 ranks, 16-byte aligned, column pairs
  const int kc = (r + 31) / 32;
  const bool mma_ok = Bp && r % 8 == 0 && aligned16(B) && kc <= 8 &&
                      (reinterpret_cast<uintptr_t>(base) & 7u) == 0 &&
                      (epilogue == 1 ? (N / 2) % 2 == 0 : N % 2 == 0);
  const int kcp = kc <= 1 ? 1 : kc <= 2 ? 2 : kc <= 4 ? 4 : 8;
  const size_t zsmem = (size_t)2 * 16 * 32 * kcp * sizeof(__nv_bfloat16);  // z high + remainder
  // column chunks per LoRA block: enough CTAs to cover the SMs a few times over when
  // blocks are few (the device count is at most max_blocks; assume about half)
  auto chunks_for = [&](int cols) {
    const int tiles8 = ceil_div(cols, 8);
    const int est = a.max_blocks / 2 > 0 ? a.max_blocks / 2 : 1;
    int c = ceil_div(4 * sms, est);
    const int cap = tiles8 / (2 * (kExpandThreads / 32)) > 0 ? tiles8 / (2 * (kExpandThreads / 32)) : 1;
    return c < 1 ? 1 : c > cap ? cap : c;
  };
  auto add_mma = [&](dim3) {
    const int cc = chunks_for(N);
    const dim3 grid(a.max_blocks * cc);
    auto go = [&](auto kern) {
      return launch_pdl(kern, grid, kExpandThreads, zsmem, stream, pdl, Z, Bp, (const int*)v.hdr,
                        (const int4*)v.blocks, (const int*)v.sorted_slots, N, r, al->E, base, cc,
                        ea, ranks);
    };
    switch (kcp * 2 + (ranks ? 1 : 0)) {
      case 2: return go(expand_add_mma_kernel<1, false>);
      case 3: return go(expand_add_mma_kernel<1, true>);
      case 4: return go(expand_add_mma_kernel<2, false>);
      case 5: return go(expand_add_mma_kernel<2, true>);
      case 8: return go(expand_add_mma_kernel<4, false>);
      case 9: return go(expand_add_mma_kernel<4, true>);
      case 16: return go(expand_add_mma_kernel<8, false>);
      default: return go(expand_add_mma_kernel<8, true>);
    }
  };
  if (epilogue == 0 && mma_ok) return add_mma(dim3(a.max_blocks));
  const bool short_segments = (int64_t)a.S <= 2 * (int64_t)al->E * (al->L > 0 ? al->L : 1);
  // epilogue 1 with tensor cores also streams G through 16-byte asynchronous copies:
  // G 16-byte aligned and I % 4 == 0
  const bool g_ok = aligned16(base) && (N / 2) % 4 == 0;
  if (epilogue == 1 && !short_segments && ((mma_ok && g_ok) || (!Bp && (N / 2) % 2 == 0))) {
    const int I = N / 2;
    const int cc = chunks_for(I);
    const dim3 grid(a.max_blocks * cc + a.max_tiles * ceil_div(I, 2 * kExpandThreads));
    const size_t smem1 = Bp ? 2 * zsmem + (size_t)(kExpandThreads / 32) * kGStages * 256 * sizeof(float) : 0;
    static std::atomic<uint64_t> configured[kMaxDevices];  // every instance, once per context
    const int cst = once_per_context(configured, [] {
      const int lim = (int)(2 * zsmem_bytes(8) + (size_t)(kExpandThreads / 32) * kGStages * 256 * sizeof(float));
      const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
#define ML_SWIGLU_ATTR(KC_)                                                                  \
  ML_CHECK_CUDA(cudaFuncSetAttribute(expand_swiglu_mma_kernel<KC_, false, false>, attr, lim)); \
  ML_CHECK_CUDA(cudaFuncSetAttribute(expand_swiglu_mma_kernel<KC_, true, false>, attr, lim));  \
  ML_CHECK_CUDA(cudaFuncSetAttribute(expand_swiglu_mma_kernel<KC_, false, true>, attr, lim));  \
  ML_CHECK_CUDA(cudaFuncSetAttribute(expand_swiglu_mma_kernel<KC_, true, true>, attr, lim));
      ML_SWIGLU_ATTR(1) ML_SWIGLU_ATTR(2) ML_SWIGLU_ATTR(4) ML_SWIGLU_ATTR(8)
#undef ML_SWIGLU_ATTR
      return MOE_LORA_OK;
    });
    if (cst != MOE_LORA_OK) return cst;
    auto go = [&](auto kern) -> int {
      return launch_pdl(kern, grid, kExpandThreads, smem1, stream, pdl, Z, Bp,
                        (const int*)v.hdr, (const int4*)v.blocks, (const int4*)v.tiles,
                        (const int*)v.sorted_slots, (const int*)v.row_adapter, I, r, al->E,
                        (const float*)base, static_cast<__nv_bfloat16*>(out), a.max_blocks, cc,
                        ea, Bp ? zstride : 0, Bp ? zu_off : 0, ranks);
    };
    const bool two = Bp && zu_off != 0, rk = Bp && ranks;
    switch ((Bp ? kcp : 1) * 4 + (two ? 2 : 0) + (rk ? 1 : 0)) {
      case 4: return go(expand_swiglu_mma_kernel<1, false, false>);
      case 5: return go(expand_swiglu_mma_kernel<1, false, true>);
      case 6: return go(expand_swiglu_mma_kernel<1, true, false>);
      case 7: return go(expand_swiglu_mma_kernel<1, true, true>);
      case 8: return go(expand_swiglu_mma_kernel<2, false, false>);
      case 9: return go(expand_swiglu_mma_kernel<2, false, true>);
      case 10: return go(expand_swiglu_mma_kernel<2, true, false>);
      case 11: return go(expand_swiglu_mma_kernel<2, true, true>);
      case 16: return go(expand_swiglu_mma_kernel<4, false, false>);
      case 17: return go(expand_swiglu_mma_kernel<4, false, true>);
      case 18: return go(expand_swiglu_mma_kernel<4, true, false>);
      case 19: return go(expand_swiglu_mma_kernel<4, true, true>);
      case 32: return go(expand_swiglu_mma_kernel<8, false, false>);
      case 33: return go(expand_swiglu_mma_kernel<8, false, true>);
      case 34: return go(expand_swiglu_mma_kernel<8, true, false>);
      default: return go(expand_swiglu_mma_kernel<8, true, true>);
    }
  }
  if (epilogue == 0) {
    if (!Bp) return MOE_LORA_OK;
    const dim3 grid(a.max_blocks, ceil_div(N, 2 * kExpandThreads));
    const size_t smem = (size_t)kMaxBmLora * r * sizeof(float);
    return launch_rv<AddK>(rv, grid, smem, stream, pdl, Z, Bp, (const int*)v.hdr,
                           (const int4*)v.blocks, (const int*)v.sorted_slots, N, r, al->E, base,
                           ea, ranks);
  }
  if (epilogue == 1) {
    const int I = N / 2;
    const int ncol = ceil_div(I, kExpandThreads);
    // rows per CTA ~ the mean (expert, adapter) segment length, so that a CTA's rows
    // share B rows; but enough CTAs to cover the SMs a few times over
    const int64_t segs = (int64_t)al->E * (al->L + 1);
    int rpc = 1;
    while (rpc < 64 && (int64_t)rpc * 2 * segs <= a.S) rpc *= 2;
    while (rpc > 1 && (int64_t)ceil_div(a.S, rpc) * ncol < 4 * sms) rpc /= 2;
    auto* hp = static_cast<__nv_bfloat16*>(out);
    if (rpc == 1 && Bp && rv >= 1 && aligned16(Z)) {
      const dim3 g1(a.S, ncol);
      auto go = [&](auto kern) {
        return launch_pdl(kern, g1, kExpandThreads, 0, stream, pdl, Z, Bp, (const int*)v.hdr,
                          (const int*)v.sorted_slots, (const int*)v.row_expert,
                          (const int*)v.row_adapter, I, r, al->E, (const float*)base, hp, ea,
                          zstride, zu_off, ranks);
      };
      switch (rv * 4 + (zu_off != 0 ? 2 : 0) + (ranks ? 1 : 0)) {
        case 4: return go(expand_swiglu_row1_kernel<1, false, false>);
        case 5: return go(expand_swiglu_row1_kernel<1, false, true>);
        case 6: return go(expand_swiglu_row1_kernel<1, true, false>);
        case 7: return go(expand_swiglu_row1_kernel<1, true, true>);
        case 8: return go(expand_swiglu_row1_kernel<2, false, false>);
        case 9: return go(expand_swiglu_row1_kernel<2, false, true>);
        case 10: return go(expand_swiglu_row1_kernel<2, true, false>);
        case 11: return go(expand_swiglu_row1_kernel<2, true, true>);
        case 16: return go(expand_swiglu_row1_kernel<4, false, false>);
        case 17: return go(expand_swiglu_row1_kernel<4, false, true>);
        case 18: return go(expand_swiglu_row1_kernel<4, true, false>);
        case 19: return go(expand_swiglu_row1_kernel<4, true, true>);
        case 32: return go(expand_swiglu_row1_kernel<8, false, false>);
        case 33: return go(expand_swiglu_row1_kernel<8, false, true>);
        case 34: return go(expand_swiglu_row1_kernel<8, true, false>);
        default: return go(expand_swiglu_row1_kernel<8, true, true>);
      }
    }
    const dim3 grid(ceil_div(a.S, rpc), ncol);
    const int zs_rows = Bp ? zstride : 0;
    const size_t smem = (size_t)rpc * zs_rows * sizeof(float);
    return launch_rv<SwigluK>(rv, grid, smem, stream, pdl, Z, Bp, (const int*)v.hdr,
                              (const int*)v.sorted_slots, (const int*)v.row_expert,
                              (const int*)v.row_adapter, I, r, al->E, (const float*)base, hp,
                              rpc, ea, zs_rows, Bp ? zu_off : 0, ranks);
  }
  if (epilogue == 2 && Bp && (int64_t)a.S >= 2 * (int64_t)al->E * al->L) {
    // several rows per (expert, adapter) pair: apply each B row once per LoRA block
    // (in place on the base output), then combine
    int st;
    if (mma_ok) {
      st = add_mma(dim3(a.max_blocks));
    } else {
      const dim3 grid(a.max_blocks, ceil_div(N, 2 * kExpandThreads));
      const size_t smem = (size_t)kMaxBmLora * r * sizeof(float);
      st = launch_rv<AddK>(rv, grid, smem, stream, pdl, Z, Bp, (const int*)v.hdr,
                           (const int4*)v.blocks, (const int*)v.sorted_slots, N, r, al->E, base,
                           ea, ranks);
    }
    if (st != MOE_LORA_OK) return st;
    return launch_combine(base, topk_w, al, a, N, out, out_fp32, stream, pdl);
  }
  if (epilogue == 2) {
    const int ncol = ceil_div(N, kExpandThreads);
    int tpc = 1;
    while (tpc < 8 && (int64_t)ceil_div(al->T, tpc * 2) * ncol >= 4 * sms &&
           tpc * 2 * al->k <= 256 && (int64_t)tpc * 2 * al->k * rr * 4 <= 32 * 1024)
      tpc *= 2;
    const dim3 grid(ceil_div(al->T, tpc), ncol);
    const size_t smem = (size_t)tpc * al->k * rr * sizeof(float);
    auto go = [&](auto kern) {
      return launch_pdl(kern, grid, kExpandThreads, smem, stream, pdl, Z, Bp,
                        (const int*)v.slot_row, (const int*)v.row_expert,
                        (const int*)v.row_adapter, topk_w, al->T, al->k, N, r, al->E,
                        (const float*)base, out, tpc, ea, ranks);
    };
    if (out_fp32) {
      switch (rv) {
        case 1: return go(expand_combine_kernel<1, true>);
        case 2: return go(expand_combine_kernel<2, true>);
        case 4: return go(expand_combine_kernel<4, true>);
        case 8: return go(expand_combine_kernel<8, true>);
        default: return go(expand_combine_kernel<0, true>);
      }
    }
    switch (rv) {
      case 1: return go(expand_combine_kernel<1, false>);
      case 2: return go(expand_combine_kernel<2, false>);
      case 4: return go(expand_combine_kernel<4, false>);
      case 8: return go(expand_combine_kernel<8, false>);
      default: return go(expand_combine_kernel<0, false>);
    }
  }
  return MOE_LORA_ERR_INVALID_ARG;
}

int launch_combine(const float* O, const float* topk_w, const moe_lora_align_t* al,
                   const AlignLayout& a, int N, void* y, int y_fp32, cudaStream_t stream, bool pdl,
                   int nparts, size_t part_stride, bool early) {
  if (a.S == 0 || al->T == 0) return MOE_LORA_OK;
  const int ea = early ? 1 : 0;
  AlignView v = align_view(al->buf, a);
  const int sms = num_sms();
  // four columns a thread where the row width and y's address allow 16-byte (8-byte) access
  const uintptr_t ya = reinterpret_cast<uintptr_t>(y);
  const bool vec = N % 4 == 0 && (ya % (y_fp32 ? 16 : 8)) == 0 &&
                   reinterpret_cast<uintptr_t>(O) % 16 == 0 && part_stride % 4 == 0;
  // tokens per CTA: as many as keep about four CTAs per SM busy (at most 8, and the CTA's
  // slots within the 256-entry shared tables)
  const int ncol = ceil_div(N, kExpandThreads * (vec ? 4 : 1));
  int tpc = 1;
  while (tpc < 8 && (int64_t)ceil_div(al->T, tpc * 2) * ncol >= 4 * sms &&
         tpc * 2 * al->k <= kExpandThreads)
    tpc *= 2;
  if (tpc * al->k > kExpandThreads) return MOE_LORA_ERR_UNSUPPORTED;
  const dim3 g2(ceil_div(al->T, tpc), ncol);
  if (vec)
    return y_fp32 ? launch_pdl(combine4_kernel<true>, g2, kExpandThreads, 0, stream, pdl, O, topk_w,
                               (const int*)v.slot_row, al->T, al->k, N, y, tpc, nparts, part_stride, ea)
                  : launch_pdl(combine4_kernel<false>, g2, kExpandThreads, 0, stream, pdl, O, topk_w,
                               (const int*)v.slot_row, al->T, al->k, N, y, tpc, nparts, part_stride, ea);
  return y_fp32 ? launch_pdl(combine_kernel<true>, g2, kExpandThreads, 0, stream, pdl, O, topk_w,
                             (const int*)v.slot_row, al->T, al->k, N, y, tpc, nparts, part_stride, ea)
                : launch_pdl(combine_kernel<false>, g2, kExpandThreads, 0, stream, pdl, O, topk_w,
                             (const int*)v.slot_row, al->T, al->k, N, y, tpc, nparts, part_stride, ea);
}

int launch_expand(const float* Z, const void* B, const moe_lora_align_t* al, const AlignLayout& a,
                  int N, int r, int epilogue, float* base, void* out, int out_fp32,
                  const float* topk_w, cudaStream_t stream, bool pdl) {
  return launch_expand_impl(Z, B, al, a, N, r, epilogue, base, out, out_fp32, topk_w, stream, pdl,
                            false);
}

}  // namespace moe_lora

extern "C" int lora_expand_add(const float* Z, const void* B, const moe_lora_align_t* al, int N,
                               int r, int epilogue, float* base, void* out, int out_fp32,
                               const float* topk_w, moe_lora_stream_t stream) {
  using namespace moe_lora;
  AlignLayout a;
  int st = check_align(al, &a);
  if (st != MOE_LORA_OK) return st;
  if (N < 1 || epilogue < 0 || epilogue > 3) return MOE_LORA_ERR_INVALID_ARG;
  if (al->L > 0 && (r < 1 || r > 256)) return r < 1 ? MOE_LORA_ERR_INVALID_ARG : MOE_LORA_ERR_UNSUPPORTED;
  if (al->L >= 65535 || al->E >= 32768) return MOE_LORA_ERR_UNSUPPORTED;  // packed (e, l) keys
  if ((epilogue == 1 || epilogue == 3) && N % 2 != 0) return MOE_LORA_ERR_INVALID_ARG;
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
