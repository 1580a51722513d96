// LoRA shrink z = xA per (expert, adapter) block (vllm.com.cn, sections
// "Implementing multi-LoRA inference for MoE models in vLLM" and "Kernel
// optimizations").
//
// The shrink has few outputs (r per row) and long sums (K = h_in), and at decode
// a block holds one or two rows, so the kernel is a stream of A_{l,e} at HBM
// speed. One CTA takes one LoRA block and one group of 8*NT ranks; its 8 warps
// split the K sum (split-K inside the CTA) and reduce their partials through
// shared memory in a fixed warp order, so results are deterministic and no
// cross-CTA atomics are needed. Each warp walks K in 32-wide steps; every lane
// issues one 128-bit load per operand row and the products are formed with
// mma.sync m16n8k16 (bf16 in, fp32 accumulate): the block's rows on M (padded
// to 16), ranks on N. Which k a lane feeds to which fragment slot is permuted
// identically for both operands, which leaves the dot products unchanged while
// keeping every load 16 bytes wide. Masks on K are compiled out when
// K % 32 == 0 (the EVEN_K specialisation); K % 8 != 0 or unaligned bases fall
// back to element loads.
#include <atomic>
#include <algorithm>

#include "internal.h"

namespace moe_lora {

constexpr int kShrinkWarps = 8;

// kCoherent: the row may have been written by an earlier launch (activations), so it
// is read at L2 (ld.global.cg); weights take the read-only path.
template <bool kVec, bool kEvenK, bool kCoherent = false>
__device__ __forceinline__ uint4 load8_bf16(const __nv_bfloat16* p, int kofs, int K) {
  uint4 r = make_uint4(0u, 0u, 0u, 0u);
  if (p == nullptr) return r;
  if (kVec) {
    if (kEvenK || kofs < K) {
      const uint4* q = reinterpret_cast<const uint4*>(p + kofs);
      r = kCoherent ? __ldcg(q) : __ldg(q);
    }
  } else {
    const unsigned short* q = reinterpret_cast<const unsigned short*>(p);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = (kofs + 2 * i < K) ? __ldcg(q + kofs + 2 * i) : 0u;
      const uint32_t hi = (kofs + 2 * i + 1 < K) ? __ldcg(q + kofs + 2 * i + 1) : 0u;
      w[i] = lo | (hi << 16);
    }
    r = make_uint4(w[0], w[1], w[2], w[3]);
  }
  return r;
}

__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// z of (sorted row, rank) of pair (e, l) into the shifted buffer of the fused expand: the
// bf16 rounding of v and the bf16 rounding of the remainder.
__device__ __forceinline__ void zpad_put(const ZPadOut& o, int row, int e, int l, int rank, float v) {
  const size_t at = ((size_t)row + ((size_t)e * o.L + l + 1) * o.gap) * o.zw;
  const __nv_bfloat16 hi = __float2bfloat16_rn(v);
  o.p[at + rank] = hi;
  o.p[at + o.lo_off + rank] = __float2bfloat16_rn(v - __bfloat162float(hi));
}

// Run by the CTA of rank group 0 of a LoRA block: the zero columns [r, rp16) of its rows
// in both halves and, for the first (last) block of its pair, the `gap` zero rows before
// (after) the pair, which a fused-expand tile reads for its rows of other pairs. When the
// rows just before belong to the pair of the previous key, that pair's trailing gap is
// this pair's leading gap (the shifts differ by one gap): it is written once, there.
__device__ void zpad_extras(const ZPadOut& o, const int* hdr, int row0, int rows, int e, int l,
                            int r) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const size_t shift = ((size_t)e * o.L + l + 1) * o.gap;
  const __nv_bfloat16 zero = __ushort_as_bfloat16((unsigned short)0);
  const int pad = o.rp16 - r;
  for (int i = tid; i < rows * pad; i += nt) {
    const int m = i / pad, c = r + (i - m * pad);
    const size_t at = ((size_t)row0 + m + shift) * o.zw;
    o.p[at + c] = zero;
    o.p[at + o.lo_off + c] = zero;
  }
  const int n_valid = __ldcg(hdr + HDR_NVALID);
  const int end = row0 + rows;
  bool first = true;
  if (row0 > 0) {
    const int pe = __ldcg(o.row_expert + row0 - 1), pl = __ldcg(o.row_adapter + row0 - 1);
    // a new pair starts here; its leading gap is written unless the previous pair is the
    // previous key's (whose trailing gap it is)
    first = (pe != e || pl != l) && !(pl >= 0 && pe * o.L + pl + 1 == e * o.L + l);
  }
  const bool last = end >= n_valid || __ldcg(o.row_expert + end) != e ||
                    __ldcg(o.row_adapter + end) != l;
  const int groups = o.gap * (o.zw / 8);  // 16-byte groups of `gap` rows
  const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
  if (first) {
    uint4* q = reinterpret_cast<uint4*>(o.p + ((size_t)row0 + shift - o.gap) * o.zw);
    for (int i = tid; i < groups; i += nt) q[i] = z4;
  }
  if (last) {
    uint4* q = reinterpret_cast<uint4*>(o.p + ((size_t)end + shift) * o.zw);
    for (int i = tid; i < groups; i += nt) q[i] = z4;
  }
}

template <int NT, int U, bool kVec, bool kEvenK, bool kSmallM>
__global__ void __launch_bounds__(kShrinkWarps * 32, !kSmallM ? 1 : NT == 1 ? 5 : NT == 4 ? 2 : 1)
    lora_shrink_kernel(const __nv_bfloat16* __restrict__ X, int rows_are_slots,
                       const __nv_bfloat16* __restrict__ A, const int* __restrict__ hdr,
                       const int4* __restrict__ blocks, const int* __restrict__ sorted_slots, int k,
                       int K, int r, int E, float* __restrict__ Z, int ngroups, int early,
                       const int* __restrict__ ranks, int rs, const ZPadOut zo, int prefetch) {
  constexpr int R = 8 * NT;  // ranks per CTA
  constexpr int XB = kSmallM ? 1 : U;  // kSmallM: blocks of at most 8 rows, no second row set
  constexpr int RM = kSmallM ? 8 : 16;  // rows of the reduction buffer
  __shared__ float red[kShrinkWarps][RM][R + 1];

  // With `early` every input was produced two or more launches back (see
  // lora_expand.cu on launch ordering): compute first, wait only before publishing.
  // With `prefetch` only the block table is that old: the CTA reads its block and pulls
  // its rows of A into L2 before waiting for the activations.
  const bool tables_early = early || prefetch;
  if (!tables_early) pdl_wait();
  // The block count and this CTA's descriptor are read together: the grid covers the
  // host's bound on the block count, so blocks + b is in bounds either way.
  const int b = blockIdx.x / ngroups;
  const int g = blockIdx.x - b * ngroups;
  const int nb = __ldcg(hdr + HDR_NBLOCKS);
  const int4 blk = __ldcg(blocks + b);
  if (b >= nb) {
    if (tables_early) pdl_wait();
    return;
  }
  if (prefetch && !early) {
    // weights never depend on a launch: this CTA's rows of A head for L2 while the
    // predecessor drains (rank rows g R .. g R + R - 1, one bulk prefetch per row)
    if (kVec && threadIdx.x < R && g * R + (int)threadIdx.x < r)
      bulk_prefetch_l2(A + (((size_t)blk.w * E + blk.z) * r + g * R + threadIdx.x) * K,
                       (uint32_t)K * 2u);
    pdl_wait();
  }
  if (!early) pdl_trigger();
  const int row0 = blk.x, rows = blk.y, e = blk.z, l = blk.w;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, q = lane & 3;
  // the slot of the first z element this thread stores, fetched with the operands
  const int slot0 = (int)threadIdx.x < rows * R ? __ldcg(sorted_slots + row0 + threadIdx.x / R) : 0;

  const __nv_bfloat16* Ab = A + ((size_t)l * E + e) * (size_t)r * K;
  // rank rows past the adapter's own rank (per slice of rs rows) are not read: their z is 0
  const int rl = adapter_rank(ranks, l, rs, hdr);
  const unsigned long long vmask = rank_row_mask(g * R, rs, rl);  // R <= 64 rows
  const __nv_bfloat16* ap[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int rank = g * R + nt * 8 + gid;
    ap[nt] = rank < r && ((vmask >> (nt * 8 + gid)) & 1ull) ? Ab + (size_t)rank * K : nullptr;
  }
  const __nv_bfloat16* x0 = nullptr;
  const __nv_bfloat16* x1 = nullptr;
  if (gid < rows) {
    const int row = row0 + gid;
    x0 = X + (size_t)(rows_are_slots ? row : __ldcg(sorted_slots + row) / k) * K;
  }
  if (!kSmallM && gid + 8 < rows) {
    const int row = row0 + gid + 8;
    x1 = X + (size_t)(rows_are_slots ? row : __ldcg(sorted_slots + row) / k) * K;
  }

  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

  // Batches of U k-steps per warp; the next batch's loads are in flight while the
  // current batch is reduced (two register buffers, used alternately).
  const int nsteps = (K + 31) >> 5;
  struct Batch {
    uint4 xa[U], xb[XB], av[U][NT];
  };
  auto load = [&](Batch& bt, int st0) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int st = st0 + u * kShrinkWarps;
      const bool ok = st < nsteps;
      const int k0 = st * 32 + q * 8;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        bt.av[u][nt] = ok ? load8_bf16<kVec, kEvenK>(ap[nt], k0, K) : make_uint4(0, 0, 0, 0);
      bt.xa[u] = ok ? load8_bf16<kVec, kEvenK, true>(x0, k0, K) : make_uint4(0, 0, 0, 0);
      if (!kSmallM)
        bt.xb[kSmallM ? 0 : u] = ok ? load8_bf16<kVec, kEvenK, true>(x1, k0, K) : make_uint4(0, 0, 0, 0);
    }
  };
  auto reduce = [&](const Batch& bt) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint4 xb = kSmallM ? make_uint4(0, 0, 0, 0) : bt.xb[kSmallM ? 0 : u];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma_16816(acc[nt], bt.xa[u].x, xb.x, bt.xa[u].y, xb.y, bt.av[u][nt].x, bt.av[u][nt].y);
        mma_16816(acc[nt], bt.xa[u].z, xb.z, bt.xa[u].w, xb.w, bt.av[u][nt].z, bt.av[u][nt].w);
      }
    }
  };
  constexpr int STRIDE = U * kShrinkWarps;
  Batch b0, b1;
  int st = warp;
  if (st < nsteps) load(b0, st);
  while (st < nsteps) {
    if (st + STRIDE < nsteps) load(b1, st + STRIDE);
    reduce(b0);
    st += STRIDE;
    if (st >= nsteps) break;
    if (st + STRIDE < nsteps) load(b0, st + STRIDE);
    reduce(b1);
    st += STRIDE;
  }

  // accumulator fragment: c0,c1 -> (row gid, ranks 2q, 2q+1); c2,c3 -> (row gid+8, ...)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    red[warp][gid][nt * 8 + 2 * q] = acc[nt][0];
    red[warp][gid][nt * 8 + 2 * q + 1] = acc[nt][1];
    if (!kSmallM) {  // rows 8..15 (empty with blocks of at most 8 rows)
      red[warp][(gid + 8) % RM][nt * 8 + 2 * q] = acc[nt][2];
      red[warp][(gid + 8) % RM][nt * 8 + 2 * q + 1] = acc[nt][3];
    }
  }
  __syncthreads();
  if (early) {
    pdl_wait();
    pdl_trigger();
  }
  for (int idx = threadIdx.x; idx < rows * R; idx += blockDim.x) {
    const int m = idx / R, c = idx - m * R;
    const int rank = g * R + c;
    if (rank >= r) continue;
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kShrinkWarps; ++w) sum += red[w][m][c];
    if (zo.p) {
      zpad_put(zo, row0 + m, e, l, rank, sum);
    } else {
      const int slot = idx == (int)threadIdx.x ? slot0 : __ldcg(sorted_slots + row0 + m);
      Z[(size_t)slot * r + rank] = sum;
    }
  }
  if (zo.p && g == 0) zpad_extras(zo, hdr, row0, rows, e, l, r);
}

// ----------------------------------------------------------------------------
// Short K, short blocks, all ranks of a block in one CTA (the many-adapter shape's
// down shrink: K = 768, r = 32, thousands of blocks of one or two rows). Register
// loads cap the bytes a CTA keeps in flight and, at 124 registers, the CTAs per SM;
// here the block's A slab (8 NT rows x K) lands in shared memory through one bulk copy
// per rank row (the copy engine, not the load/store path), only the activation
// fragments sit in registers, and four CTAs fit an SM. The same mma.sync products and
// fixed-order warp reduction (done in the slab's space once the products are formed)
// as the kernel above.
// ----------------------------------------------------------------------------
// One contiguous global -> shared copy by the bulk-copy (TMA) engine, completing on an
// mbarrier; both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

constexpr int kShortUMax = 4;  // k-steps per warp: K <= 8 warps x 4 x 32 = 1024

// bytes per shared-memory row of A: at least K bf16, == 64 (mod 128) so that the rows
// of a fragment load fall in alternate bank halves
inline int short_astride(int K) { return (K * 2 + 127) / 128 * 128 + 64; }

template <int NT, bool kEvenK, bool kRanked>  // kRanked: adapters of their own ranks
__global__ void __launch_bounds__(kShrinkWarps * 32, 4)
    lora_shrink_smem_kernel(const __nv_bfloat16* __restrict__ X, int rows_are_slots,
                            const __nv_bfloat16* __restrict__ A, const int* __restrict__ hdr,
                            const int4* __restrict__ blocks, const int* __restrict__ sorted_slots,
                            int k, int K, int r, int E, float* __restrict__ Z, int ngroups,
                            int early, int astride, const int* __restrict__ ranks, int rs,
                            unsigned long long wait_ns, const ZPadOut zo) {
  constexpr int R = 8 * NT;
  static_assert(R == 32, "one rank row per lane of warp 0");
  extern __shared__ __align__(16) uint8_t sA[];  // [R][astride] bytes; reused for the reduction
  __shared__ uint64_t bar;                       // the slab's copies complete here
  if (!early) pdl_wait();
  const int b = blockIdx.x / ngroups;
  const int g = blockIdx.x - b * ngroups;
  const int nb = __ldcg(hdr + HDR_NBLOCKS);
  const int4 blk = __ldcg(blocks + b);  // in bounds: the grid covers the host's block bound
  if (b >= nb) {
    if (early) pdl_wait();
    return;
  }
  if (!early) pdl_trigger();
  const int row0 = blk.x, rows = min(blk.y, 8), e = blk.z, l = blk.w;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, q = lane & 3;
  const int slot0 = (int)threadIdx.x < rows * R ? __ldcg(sorted_slots + row0 + threadIdx.x / R) : 0;
  // the slab: rank rows g R .. g R + nr - 1, 16 bytes per copy
  const int nr = min(R, r - g * R);
  // rows past the adapter's rank (per slice) are not read
  const unsigned long long vmask =
      kRanked ? rank_row_mask(g * R, rs, adapter_rank(ranks, l, rs, hdr)) : ~0ull;  // R <= 64 rows
  // one bulk copy per rank row (2K bytes: K % 8 == 0 and 16-byte aligned bases, checked
  // on the host), issued by lane rho of warp 0 and completing on one mbarrier
  const __nv_bfloat16* Ab = A + (((size_t)l * E + e) * r + (size_t)g * R) * K;
  if (warp == 0) {
    if (lane == 0) {
      mbar_init(&bar, 1);
      fence_barrier_init();
    }
    __syncwarp();
    const bool take = lane < nr && ((vmask >> lane) & 1ull);
    const unsigned tk = __ballot_sync(0xffffffffu, take);
    if (lane == 0) mbar_arrive_expect_tx(&bar, (uint32_t)__popc(tk) * (uint32_t)(2 * K));
    __syncwarp();
    if (take) bulk_g2s(sA + (size_t)lane * astride, Ab + (size_t)lane * K, (uint32_t)(2 * K), &bar);
  }
  // activation fragments of this warp's k-steps (rows gid < rows)
  const int nsteps = (K + 31) >> 5;
  const __nv_bfloat16* x0 = nullptr;
  if (gid < rows) {
    const int row = row0 + gid;
    x0 = X + (size_t)(rows_are_slots ? row : __ldcg(sorted_slots + row) / k) * K;
  }
  uint4 xa[kShortUMax];
#pragma unroll
  for (int u = 0; u < kShortUMax; ++u) {
    const int st = warp + kShrinkWarps * u;
    const int k0 = st * 32 + q * 8;
    xa[u] = make_uint4(0, 0, 0, 0);
    if (x0 && st < nsteps && (kEvenK || k0 < K)) xa[u] = __ldcg(reinterpret_cast<const uint4*>(x0 + k0));
  }
  __syncthreads();  // the barrier is initialised before any thread waits on it
  const bool landed = mbar_wait_bounded(&bar, 0, wait_ns);
  if (__syncthreads_or(!landed)) {  // a thread gave up: the CTA records it and writes nothing
    if (threadIdx.x == 0) set_dev_error(const_cast<int*>(hdr), MOE_LORA_DEVERR_TIMEOUT);
    mbar_wait_bounded(&bar, 0);  // the slab's copies land before the CTA exits
    return;
  }
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
  for (int u = 0; u < kShortUMax; ++u) {
    const int st = warp + kShrinkWarps * u;
    if (st >= nsteps) break;
    const int k0 = st * 32 + q * 8;
    const bool kin = kEvenK || k0 < K;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int rho = nt * 8 + gid;
      uint4 av = make_uint4(0, 0, 0, 0);
      if (rho < nr && ((vmask >> rho) & 1ull) && kin)
        av = *reinterpret_cast<const uint4*>(sA + (size_t)rho * astride + k0 * 2);
      mma_16816(acc[nt], xa[u].x, 0u, xa[u].y, 0u, av.x, av.y);
      mma_16816(acc[nt], xa[u].z, 0u, xa[u].w, 0u, av.z, av.w);
    }
  }
  __syncthreads();  // every warp is done with the slab
  float (*red)[8][R + 1] = reinterpret_cast<float (*)[8][R + 1]>(sA);  // [warp][row][rank]
  // accumulator fragment: c0, c1 -> (row gid, ranks 2q, 2q+1); rows 8..15 are empty
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    red[warp][gid][nt * 8 + 2 * q] = acc[nt][0];
    red[warp][gid][nt * 8 + 2 * q + 1] = acc[nt][1];
  }
  __syncthreads();
  if (early) {
    pdl_wait();
    pdl_trigger();
  }
  for (int idx = threadIdx.x; idx < rows * R; idx += blockDim.x) {
    const int m = idx / R, c = idx - m * R;
    const int rank = g * R + c;
    if (rank >= r) continue;
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kShrinkWarps; ++w) sum += red[w][m][c];
    if (zo.p) {
      zpad_put(zo, row0 + m, e, l, rank, sum);
    } else {
      const int slot = idx == (int)threadIdx.x ? slot0 : __ldcg(sorted_slots + row0 + m);
      Z[(size_t)slot * r + rank] = sum;
    }
  }
  if (zo.p && g == 0) zpad_extras(zo, hdr, row0, rows, e, l, r);
}

// ----------------------------------------------------------------------------
// Long K, blocks of up to 16 rows, many blocks (prefill): the register kernel above keeps
// about 128 bytes a thread in flight, too little to cover the latency of a K = 2880 sum.
// Here the block's rank rows of A and its x rows go through a ring of shared-memory
// stages (256 columns, 512 bytes a row) filled by 16-byte asynchronous copies
// (cp.async: the load path, no registers held while in flight; the bulk-copy engine
// was measured slower for these 512-byte pieces), three stages ahead; eight warps form the
// same mma.sync products from shared memory (warp w takes k-step w of each stage) and the
// partials are reduced in warp order. Rows past the block and rank rows
// past the adapter's rank are not copied: their stale stage contents only reach outputs
// that are not stored (masked ranks are written as zero).
// ----------------------------------------------------------------------------
constexpr int kPipeKC = 256;                  // columns per stage
constexpr int kPipeRow = kPipeKC * 2 + 64;    // bytes per stage row: == 64 (mod 128)
constexpr int kPipeWarps = 8;  // one 32-column k-step of each stage a warp
constexpr int kPipeStages = 4;
__host__ __device__ constexpr size_t pipe_smem(int R) {
  return (size_t)kPipeStages * (R + 16) * kPipeRow + (R + 16) * sizeof(void*);
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src))
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int NT, bool kRanked>
__global__ void __launch_bounds__(kPipeWarps * 32, NT <= 2 ? 3 : 2)
    lora_shrink_pipe_kernel(const __nv_bfloat16* __restrict__ X, int rows_are_slots,
                            const __nv_bfloat16* __restrict__ A, const int* __restrict__ hdr,
                            const int4* __restrict__ blocks, const int* __restrict__ sorted_slots,
                            int k, int K, int r, int E, float* __restrict__ Z, int ngroups,
                            int early, const int* __restrict__ ranks, int rs, const ZPadOut zo,
                            int prefetch) {
  constexpr int R = 8 * NT;
  constexpr int NS = kPipeStages;
  constexpr int ROWS = R + 16;  // stage rows: R rank rows of A, then 16 x rows
  constexpr int GROUPS = kPipeKC / 8;  // 16-byte pieces per stage row
  extern __shared__ __align__(128) uint8_t smem[];
  const __nv_bfloat16** s_src =
      reinterpret_cast<const __nv_bfloat16**>(smem + (size_t)NS * ROWS * kPipeRow);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, q = lane & 3;

  const bool tables_early = early || prefetch;
  if (!tables_early) pdl_wait();
  const int b = blockIdx.x / ngroups;
  const int g = blockIdx.x - b * ngroups;
  const int nb = __ldcg(hdr + HDR_NBLOCKS);
  const int4 blk = __ldcg(blocks + b);  // in bounds: the grid covers the host's block bound
  if (b >= nb) {
    if (tables_early) pdl_wait();
    return;
  }
  const int row0 = blk.x, rows = min(blk.y, 16), e = blk.z, l = blk.w;
  const __nv_bfloat16* Ab = A + (((size_t)l * E + e) * r + (size_t)g * R) * K;
  const int nr = min(R, r - g * R);  // rank rows of this group
  const unsigned long long vmask =
      kRanked ? rank_row_mask(g * R, rs, adapter_rank(ranks, l, rs, hdr)) : ~0ull;
  if (prefetch && !early) {  // weights never depend on a launch: A heads for L2 first
    if (threadIdx.x < nr && ((vmask >> threadIdx.x) & 1ull))
      bulk_prefetch_l2(Ab + (size_t)threadIdx.x * K, (uint32_t)K * 2u);
    pdl_wait();
  }
  if (!early) pdl_trigger();
  // each stage row's source (null: not copied)
  for (int i = threadIdx.x; i < ROWS; i += blockDim.x) {
    const __nv_bfloat16* src = nullptr;
    if (i < R) {
      if (i < nr && ((vmask >> i) & 1ull)) src = Ab + (size_t)i * K;
    } else if (i - R < rows) {
      const int row = row0 + i - R;
      src = X + (size_t)(rows_are_slots ? row : __ldcg(sorted_slots + row) / k) * K;
    }
    s_src[i] = src;
  }
  __syncthreads();

  const int nchunks = (K + kPipeKC - 1) / kPipeKC;
  // Lane q copies the 16-byte group q of stage rows warp, warp + 8, ... (a warp moves one
  // whole 512-byte row a step); the rows' sources stay in registers for every chunk.
  static_assert(GROUPS == 32, "one 16-byte group of a stage row a lane");
  constexpr int NPC = (ROWS + kPipeWarps - 1) / kPipeWarps;
  const __nv_bfloat16* psrc[NPC];
#pragma unroll
  for (int u = 0; u < NPC; ++u) {
    const int i = warp + u * kPipeWarps;
    const __nv_bfloat16* src = i < ROWS ? s_src[i] : nullptr;
    psrc[u] = src ? src + lane * 8 : nullptr;
  }
  auto issue = [&](int c) {  // chunk c into its stage (an empty group past the last chunk)
    if (c < nchunks) {
      uint8_t* st = smem + (size_t)(c % NS) * ROWS * kPipeRow + lane * 16;
      const int c0 = c * kPipeKC;
      if (c0 + lane * 8 < K) {
#pragma unroll
        for (int u = 0; u < NPC; ++u)
          if (psrc[u]) cp_async16(st + (size_t)(warp + u * kPipeWarps) * kPipeRow, psrc[u] + c0);
      }
    }
    cp_async_commit();
  };
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
  for (int c = 0; c < NS - 1; ++c) issue(c);
  for (int c = 0; c < nchunks; ++c) {
    cp_async_wait<NS - 2>();  // this thread's copies of chunk c have landed
    __syncthreads();          // everyone's have; and every warp is done with chunk c - 1
    issue(c + NS - 1);        // into chunk c - 1's stage
    const uint8_t* st = smem + (size_t)(c % NS) * ROWS * kPipeRow;
    const int cols = min(kPipeKC, K - c * kPipeKC);
#pragma unroll
    for (int h = 0; h < kPipeKC / 32 / kPipeWarps; ++h) {
      const int s0 = (warp + kPipeWarps * h) * 32;  // the warp's k-step in the stage
      if (s0 >= cols) continue;  // the whole warp: mma.sync needs all of its lanes
      // K % 8 == 0: a lane's 16-byte group is wholly in or out; out, it feeds zeros
      const int k0 = s0 + q * 8;
      const bool kin = k0 < cols;
      const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
      const uint4 xa = kin ? *reinterpret_cast<const uint4*>(st + (size_t)(R + gid) * kPipeRow + k0 * 2) : z4;
      const uint4 xb = kin ? *reinterpret_cast<const uint4*>(st + (size_t)(R + gid + 8) * kPipeRow + k0 * 2) : z4;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint4 av = kin ? *reinterpret_cast<const uint4*>(st + (size_t)(nt * 8 + gid) * kPipeRow + k0 * 2) : z4;
        mma_16816(acc[nt], xa.x, xb.x, xa.y, xb.y, av.x, av.y);
        mma_16816(acc[nt], xa.z, xb.z, xa.w, xb.w, av.z, av.w);
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();  // every warp is done with the stages
  // reduce the warps' partials in warp order, in the first stage
  float (*red)[16][R + 1] = reinterpret_cast<float (*)[16][R + 1]>(smem);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    red[warp][gid][nt * 8 + 2 * q] = acc[nt][0];
    red[warp][gid][nt * 8 + 2 * q + 1] = acc[nt][1];
    red[warp][gid + 8][nt * 8 + 2 * q] = acc[nt][2];
    red[warp][gid + 8][nt * 8 + 2 * q + 1] = acc[nt][3];
  }
  __syncthreads();
  if (early) {
    pdl_wait();
    pdl_trigger();
  }
  for (int idx = threadIdx.x; idx < rows * R; idx += blockDim.x) {
    const int m = idx / R, c = idx - m * R;
    const int rank = g * R + c;
    if (rank >= r) continue;
    float sum = 0.f;
    if ((vmask >> c) & 1ull) {
#pragma unroll
      for (int w = 0; w < kPipeWarps; ++w) sum += red[w][m][c];
    }
    if (zo.p) {
      zpad_put(zo, row0 + m, e, l, rank, sum);
    } else {
      Z[(size_t)__ldcg(sorted_slots + row0 + m) * r + rank] = sum;
    }
  }
  if (zo.p && g == 0) zpad_extras(zo, hdr, row0, rows, e, l, r);
}

template <int NT>
static int launch_shrink_pipe(const __nv_bfloat16* X, int rows_are_slots, const __nv_bfloat16* A,
                              const AlignView& v, int max_blocks, int k, int K, int r, int E,
                              float* Z, cudaStream_t stream, bool pdl, int early,
                              const int* ranks, int rs, const ZPadOut& zo, int prefetch) {
  constexpr int R = 8 * NT;
  const int ngroups = ceil_div(r, R);
  const int64_t grid = (int64_t)max_blocks * ngroups;
  if (grid > 0x7fffffff) return MOE_LORA_ERR_UNSUPPORTED;
  const size_t smem = pipe_smem(R);
  static std::atomic<uint64_t> configured[kMaxDevices];
  const int cst = once_per_context(configured, [smem] {
    const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
    ML_CHECK_CUDA(cudaFuncSetAttribute(lora_shrink_pipe_kernel<NT, false>, attr, (int)smem));
    ML_CHECK_CUDA(cudaFuncSetAttribute(lora_shrink_pipe_kernel<NT, true>, attr, (int)smem));
    return MOE_LORA_OK;
  });
  if (cst != MOE_LORA_OK) return cst;
  auto go = [&](auto kern) {
    return launch_pdl(kern, dim3((unsigned)grid), kPipeWarps * 32, smem, stream, pdl, X,
                      rows_are_slots, A, (const int*)v.hdr, (const int4*)v.blocks,
                      (const int*)v.sorted_slots, k, K, r, E, Z, ngroups, early, ranks, rs, zo,
                      prefetch);
  };
  return ranks ? go(lora_shrink_pipe_kernel<NT, true>) : go(lora_shrink_pipe_kernel<NT, false>);
}

template <int NT, int U>
static int launch_shrink_nt(const __nv_bfloat16* X, int rows_are_slots, const __nv_bfloat16* A,
                            const AlignView& v, int max_blocks, int k, int K, int r, int E,
                            float* Z, bool vec, cudaStream_t stream, bool pdl, int early,
                            bool small_m, const int* ranks, int rs, const ZPadOut& zo,
                            int prefetch) {
  const int ngroups = ceil_div(r, 8 * NT);
  const int64_t grid = (int64_t)max_blocks * ngroups;
  if (grid > 0x7fffffff) return MOE_LORA_ERR_UNSUPPORTED;
  const dim3 g((unsigned)grid);
  auto args = [&](auto kern) {
    return launch_pdl(kern, g, kShrinkWarps * 32, 0, stream, pdl, X, rows_are_slots, A,
                      (const int*)v.hdr, (const int4*)v.blocks, (const int*)v.sorted_slots, k, K,
                      r, E, Z, ngroups, early, ranks, rs, zo, prefetch);
  };
  if (small_m) {
    if (vec && K % 32 == 0) return args(lora_shrink_kernel<NT, U, true, true, true>);
    if (vec) return args(lora_shrink_kernel<NT, U, true, false, true>);
    return args(lora_shrink_kernel<NT, U, false, false, true>);
  }
  if (vec && K % 32 == 0) return args(lora_shrink_kernel<NT, U, true, true, false>);
  if (vec) return args(lora_shrink_kernel<NT, U, true, false, false>);
  return args(lora_shrink_kernel<NT, U, false, false, false>);
}

int launch_shrink_impl(const void* X, int rows_are_slots, const void* A,
                       const moe_lora_align_t* al, const AlignLayout& a, int K, int r, int rs,
                       float* Z, cudaStream_t stream, bool pdl, bool early,
                       unsigned long long wait_ns, const ZPadOut* zpad, int flags) {
  const int* ranks = al->adapter_ranks;
  if (a.S == 0 || al->L == 0) return MOE_LORA_OK;
  const ZPadOut zo = zpad ? *zpad : ZPadOut{};
  const int pf = (flags & kShrinkPrefetchA) ? 1 : 0;
  AlignView v = align_view(al->buf, a);
  const auto* Xp = static_cast<const __nv_bfloat16*>(X);
  const auto* Ap = static_cast<const __nv_bfloat16*>(A);
  const bool vec = (K % 8 == 0) && aligned16(X) && aligned16(A);
  const int ea = early ? 1 : 0;
  // Few blocks (decode): one 8-rank group per CTA to spread the A stream over
  // many CTAs. Many blocks (prefill): all ranks in one CTA so that X is read once.
  const int blocks_est = a.max_blocks;
  const int sms = num_sms();
  // long sums over many blocks of up to 16 rows (prefill): the pipelined kernel
  if (vec && al->bm_lora > 8 && K >= 1024 && r <= 32 &&
      (int64_t)blocks_est * ceil_div(r, 16) > 4 * (int64_t)sms) {
    if (r <= 16)
      return launch_shrink_pipe<2>(Xp, rows_are_slots, Ap, v, a.max_blocks, al->k, K, r, al->E, Z,
                                   stream, pdl, ea, ranks, rs, zo, pf);
    return launch_shrink_pipe<4>(Xp, rows_are_slots, Ap, v, a.max_blocks, al->k, K, r, al->E, Z,
                                 stream, pdl, ea, ranks, rs, zo, pf);
  }
  int nt;
  if ((int64_t)blocks_est * ceil_div(r, 8) <= 8 * sms) nt = 1;
  else if (r <= 16) nt = 2;
  else if (r <= 32) nt = 4;
  else nt = 8;
  if (flags & kShrinkOneWave) {
    // every CTA resident at once (the launch bounds' CTAs per SM), so that the next kernel
    // of the chain launches as soon as these have passed their wait -- where some choice
    // of ranks per CTA (at most the adapter's) allows it; else the choice above stands
    const bool sm8 = al->bm_lora <= 8;
    for (int c : {1, 2, 4, 8}) {
      const int per_sm = !sm8 ? 1 : c == 1 ? 5 : c == 4 ? 2 : 1;
      if (8 * c > ((r + 7) & ~7) * 2) break;
      if ((int64_t)blocks_est * ceil_div(r, 8 * c) <= (int64_t)sms * per_sm) {
        nt = c;
        break;
      }
    }
  }
  switch (nt) {
    case 1: return launch_shrink_nt<1, 2>(Xp, rows_are_slots, Ap, v, a.max_blocks, al->k, K, r, al->E, Z, vec, stream, pdl, ea, al->bm_lora <= 8, ranks, rs, zo, pf);
    case 2: return launch_shrink_nt<2, 2>(Xp, rows_are_slots, Ap, v, a.max_blocks, al->k, K, r, al->E, Z, vec, stream, pdl, ea, al->bm_lora <= 8, ranks, rs, zo, pf);
    case 4:  // short blocks: two k-steps per batch, still two CTAs per SM
      if (al->bm_lora <= 8 && vec && K <= 32 * kShrinkWarps * kShortUMax &&
          32 * short_astride(K) <= 56 * 1024) {  // short K: the slab in shared memory
        const int astride = short_astride(K);
        // the reduction reuses the slab: [8 warps][8 rows][33] floats at least
        const size_t smem = std::max((size_t)32 * astride, (size_t)kShrinkWarps * 8 * 33 * sizeof(float));
        const int ngroups = ceil_div(r, 32);
        const int64_t grid = (int64_t)a.max_blocks * ngroups;
        if (grid > 0x7fffffff) return MOE_LORA_ERR_UNSUPPORTED;
        static std::atomic<uint64_t> configured[kMaxDevices];  // every instance, once per context
        const int cst = once_per_context(configured, [] {
          const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
          ML_CHECK_CUDA(cudaFuncSetAttribute(lora_shrink_smem_kernel<4, true, false>, attr, 56 * 1024));
          ML_CHECK_CUDA(cudaFuncSetAttribute(lora_shrink_smem_kernel<4, false, false>, attr, 56 * 1024));
          ML_CHECK_CUDA(cudaFuncSetAttribute(lora_shrink_smem_kernel<4, true, true>, attr, 56 * 1024));
          ML_CHECK_CUDA(cudaFuncSetAttribute(lora_shrink_smem_kernel<4, false, true>, attr, 56 * 1024));
          return MOE_LORA_OK;
        });
        if (cst != MOE_LORA_OK) return cst;
        auto go = [&](auto kern) -> int {
          return launch_pdl(kern, dim3((unsigned)grid), kShrinkWarps * 32, smem, stream, pdl, Xp,
                            rows_are_slots, Ap, (const int*)v.hdr, (const int4*)v.blocks,
                            (const int*)v.sorted_slots, al->k, K, r, al->E, Z, ngroups, ea, astride,
                            ranks, rs, wait_ns, zo);
        };
        if (ranks)
          return K % 32 == 0 ? go(lora_shrink_smem_kernel<4, true, true>) : go(lora_shrink_smem_kernel<4, false, true>);
        return K % 32 == 0 ? go(lora_shrink_smem_kernel<4, true, false>) : go(lora_shrink_smem_kernel<4, false, false>);
      }
      if (al->bm_lora <= 8)
        return launch_shrink_nt<4, 2>(Xp, rows_are_slots, Ap, v, a.max_blocks, al->k, K, r, al->E, Z, vec, stream, pdl, ea, true, ranks, rs, zo, pf);
      return launch_shrink_nt<4, 1>(Xp, rows_are_slots, Ap, v, a.max_blocks, al->k, K, r, al->E, Z, vec, stream, pdl, ea, false, ranks, rs, zo, pf);
    default: return launch_shrink_nt<8, 1>(Xp, rows_are_slots, Ap, v, a.max_blocks, al->k, K, r, al->E, Z, vec, stream, pdl, ea, al->bm_lora <= 8, ranks, rs, zo, pf);
  }
}

int launch_shrink(const void* X, int rows_are_slots, const void* A, const moe_lora_align_t* al,
                  const AlignLayout& a, int K, int r, float* Z, cudaStream_t stream, bool pdl) {
  return launch_shrink_impl(X, rows_are_slots, A, al, a, K, r, r, Z, stream, pdl, false);
}

}  // namespace moe_lora

extern "C" int lora_shrink(const void* X, int rows_are_slots, const void* A,
                           const moe_lora_align_t* al, int K, int r, float* Z,
                           moe_lora_stream_t stream) {
  using namespace moe_lora;
  AlignLayout a;
  int st = check_align(al, &a);
  if (st != MOE_LORA_OK) return st;
  if (K < 1 || r < 1 || (rows_are_slots != 0 && rows_are_slots != 1)) return MOE_LORA_ERR_INVALID_ARG;
  if (r > 256) return MOE_LORA_ERR_UNSUPPORTED;
  if (a.S > 0 && al->L > 0 && (!X || !A || !Z)) return MOE_LORA_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_LORA_OK) return st;
  return launch_shrink(X, rows_are_slots, A, al, a, K, r, Z, reinterpret_cast<cudaStream_t>(stream),
                       true);
}
