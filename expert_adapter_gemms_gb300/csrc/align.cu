// Alignment of token-slots by (expert, adapter): the "compound sparsity" of
// expert routing and adapter selection (vllm.com.cn, section "Implementing
// multi-LoRA inference for MoE models in vLLM"; agentlenshq.com, section
// "Multi-LoRA Serving for MoE Models").
//
// One CTA of 1024 threads. Each slot s gets the packed word (key << slot_bits) | s
// with key = e * (L + 1) + (l + 1) (dropped slots use the last bucket). A stable
// least-significant-digit radix sort on the key bits (8-bit digits, per-warp
// digit histograms, ranks from __match_any_sync) keeps equal keys in slot
// order, so the result is the unique stable order: deterministic and bit-exact.
// Bucket counts give the expert and (expert, adapter) segment boundaries, from
// which the grouped-GEMM token tiles and the LoRA blocks are cut.
#include "common.cuh"

namespace moe_lora {

constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr int kSmemSortMaxSlots = 16384;

// Exclusive scan of one int per thread across the CTA; returns the prefix and
// writes the total to *total. `tmp` holds kAlignWarps + 1 ints.
__device__ __forceinline__ int block_exclusive_scan(int v, int* tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += u;
  }
  if (lane == 31) tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int x = tmp[lane];
    int xi = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, xi, off);
      if (lane >= off) xi += u;
    }
    tmp[lane] = xi - x;  // exclusive prefix of warp totals
    if (lane == 31) tmp[kAlignWarps] = xi;
  }
  __syncthreads();
  const int r = tmp[warp] + incl - v;
  *total = tmp[kAlignWarps];
  __syncthreads();
  return r;
}

// Exclusive scan of a global int array in place-free form: out[i] = sum in[0..i).
__device__ void block_scan_array(const int* in, int* out, int n, int* tmp) {
  const int chunk = (n + kAlignThreads - 1) / kAlignThreads;
  const int b = threadIdx.x * chunk;
  const int e = min(n, b + chunk);
  int s = 0;
  for (int i = b; i < e; ++i) s += in[i];
  int total;
  int run = block_exclusive_scan(s, tmp, &total);
  for (int i = b; i < e; ++i) {
    const int x = in[i];
    out[i] = run;
    run += x;
  }
}

__global__ void __launch_bounds__(kAlignThreads, 1)
    align_kernel(const int* __restrict__ ids, const int* __restrict__ token_adapter, AlignView v,
                 int T, int k, int E, int L, int bm_base, int bm_lora, int S, int nbuckets,
                 int key_bits, int slot_bits, int smem_sort) {
  extern __shared__ __align__(16) int smem[];
  int* hist = smem;                       // [256 digits][32 warps]
  int* tmp = smem + 256 * kAlignWarps;    // scan scratch
  __shared__ unsigned int s_err;
  __shared__ int s_nvalid, s_ntiles, s_nblocks, s_nlora;

  uint32_t* bufA = smem_sort ? reinterpret_cast<uint32_t*>(smem + 256 * kAlignWarps + 64) : v.sort0;
  uint32_t* bufB = smem_sort ? bufA + S : v.sort1;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int drop = nbuckets - 1;
  const uint32_t smask = (slot_bits >= 32) ? 0xffffffffu : ((1u << slot_bits) - 1u);

  pdl_wait();
  if (tid == 0) s_err = 0u;
  for (int i = tid; i < nbuckets; i += kAlignThreads) v.bucket_count[i] = 0;
  __syncthreads();

  // 1. keys and bucket counts
  for (int s = tid; s < S; s += kAlignThreads) {
    const int t = s / k;
    const int e = ids[s];
    const int l = token_adapter ? token_adapter[t] : -1;
    unsigned int bad = 0;
    if (e < 0 || e >= E) bad |= MOE_LORA_DEVERR_EXPERT_RANGE;
    if (l < -1 || l >= L) bad |= MOE_LORA_DEVERR_ADAPTER_RANGE;
    int key = drop;
    if (bad) atomicOr(&s_err, bad);
    else key = e * (L + 1) + (l + 1);
    bufA[s] = (static_cast<uint32_t>(key) << slot_bits) | static_cast<uint32_t>(s);
    atomicAdd(&v.bucket_count[key], 1);
  }
  __syncthreads();

  // 2. stable LSD radix sort on the key bits
  uint32_t* src = bufA;
  uint32_t* dst = bufB;
  const int chunk = (S + kAlignWarps - 1) / kAlignWarps;
  const int wb = min(S, warp * chunk), we = min(S, wb + chunk);
  for (int shift = slot_bits; shift < slot_bits + key_bits; shift += 8) {
    for (int d = lane; d < 256; d += 32) hist[d * kAlignWarps + warp] = 0;
    __syncwarp();
    for (int base = wb; base < we; base += 32) {
      const int i = base + lane;
      const bool act = i < we;
      const unsigned mask = __ballot_sync(0xffffffffu, act);
      if (act) {
        const int d = (src[i] >> shift) & 255;
        const unsigned peers = __match_any_sync(mask, d);
        if (lane == __ffs(peers) - 1) hist[d * kAlignWarps + warp] += __popc(peers);
      }
      __syncwarp();
    }
    __syncthreads();
    {  // exclusive scan over (digit, warp) in digit-major order: 8 entries per thread
      int loc[8];
      int s = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        loc[q] = hist[tid * 8 + q];
        s += loc[q];
      }
      int total;
      int run = block_exclusive_scan(s, tmp, &total);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        hist[tid * 8 + q] = run;
        run += loc[q];
      }
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int base = wb; base < we; base += 32) {
      const int i = base + lane;
      const bool act = i < we;
      const unsigned mask = __ballot_sync(0xffffffffu, act);
      int d = 0;
      unsigned peers = 0;
      if (act) {
        const uint32_t x = src[i];
        d = (x >> shift) & 255;
        peers = __match_any_sync(mask, d);
        dst[hist[d * kAlignWarps + warp] + __popc(peers & lt)] = x;
      }
      __syncwarp();
      if (act && lane == __ffs(peers) - 1) hist[d * kAlignWarps + warp] += __popc(peers);
      __syncwarp();
    }
    __syncthreads();
    uint32_t* sw = src;
    src = dst;
    dst = sw;
  }

  // 3. sorted rows
  const int n_valid = S - v.bucket_count[drop];
  for (int i = tid; i < S; i += kAlignThreads) {
    const uint32_t x = src[i];
    const int s = static_cast<int>(x & smask);
    const int key = static_cast<int>(x >> slot_bits);
    if (key == drop) {
      v.sorted_slots[i] = -1;
      v.slot_row[s] = -1;
    } else {
      const int e = key / (L + 1), l = key % (L + 1) - 1;
      v.sorted_slots[i] = s;
      v.slot_row[s] = i;
      v.row_expert[i] = e;
      v.row_adapter[i] = l;
    }
  }
  // 4. segment starts
  block_scan_array(v.bucket_count, v.bucket_start, nbuckets, tmp);
  __syncthreads();
  for (int e = tid; e <= E; e += kAlignThreads) v.expert_begin[e] = v.bucket_start[e * (L + 1)];
  __syncthreads();

  // 5. token tiles (per expert, bm_base rows) and LoRA blocks (per (e, l>=0), bm_lora rows)
  {
    const int c = (n_valid + kAlignThreads - 1) / kAlignThreads;
    const int b = tid * c, en = min(n_valid, b + c);
    int nt = 0, nb = 0, nl = 0;
    for (int i = b; i < en; ++i) {
      const int e = v.row_expert[i], l = v.row_adapter[i];
      if ((i - v.expert_begin[e]) % bm_base == 0) ++nt;
      if (l >= 0) {
        ++nl;
        if ((i - v.bucket_start[e * (L + 1) + l + 1]) % bm_lora == 0) ++nb;
      }
    }
    int tot_t, tot_b, tot_l;
    int ti = block_exclusive_scan(nt, tmp, &tot_t);
    int bi = block_exclusive_scan(nb, tmp, &tot_b);
    block_exclusive_scan(nl, tmp, &tot_l);
    for (int i = b; i < en; ++i) {
      const int e = v.row_expert[i], l = v.row_adapter[i];
      const int eb = v.expert_begin[e];
      if ((i - eb) % bm_base == 0) v.tiles[ti++] = make_int4(e, i, min(bm_base, v.expert_begin[e + 1] - i), 0);
      if (l >= 0) {
        const int key = e * (L + 1) + l + 1;
        const int sb = v.bucket_start[key];
        if ((i - sb) % bm_lora == 0)
          v.blocks[bi++] = make_int4(i, min(bm_lora, sb + v.bucket_count[key] - i), e, l);
      }
    }
    if (tid == 0) {
      s_nvalid = n_valid;
      s_ntiles = tot_t;
      s_nblocks = tot_b;
      s_nlora = tot_l;
    }
  }
  __syncthreads();
  if (tid == 0) {
    if (s_err) atomicOr(reinterpret_cast<unsigned int*>(v.hdr + HDR_ERR), s_err);
    v.hdr[HDR_NVALID] = s_nvalid;
    v.hdr[HDR_NTILES] = s_ntiles;
    v.hdr[HDR_NBLOCKS] = s_nblocks;
    v.hdr[HDR_NLORAROWS] = s_nlora;
    v.hdr[HDR_T] = T;
    v.hdr[HDR_K] = k;
    v.hdr[HDR_E] = E;
    v.hdr[HDR_L] = L;
    v.hdr[HDR_BMB] = bm_base;
    v.hdr[HDR_BML] = bm_lora;
  }
  pdl_trigger();
}

static size_t align_smem_bytes(int S, bool smem_sort) {
  size_t b = (size_t)(256 * kAlignWarps + 64) * 4;
  if (smem_sort) b += (size_t)2 * S * 4;
  return b;
}

int launch_align(const int* ids, const int* token_adapter, const moe_lora_align_t* al,
                 const AlignLayout& a, cudaStream_t stream, bool pdl) {
  AlignView v = align_view(al->buf, a);
  const bool smem_sort = a.S <= kSmemSortMaxSlots;
  const size_t smem = align_smem_bytes(a.S, smem_sort);
  static int configured[64] = {0};
  int dev = 0;
  ML_CHECK_CUDA(cudaGetDevice(&dev));
  if (dev < 64 && !configured[dev]) {
    ML_CHECK_CUDA(cudaFuncSetAttribute(align_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)align_smem_bytes(kSmemSortMaxSlots, true)));
    configured[dev] = 1;
  }
  return launch_pdl(align_kernel, 1, kAlignThreads, smem, stream, pdl, ids, token_adapter, v,
                    al->T, al->k, al->E, al->L, al->bm_base, al->bm_lora, a.S, a.nbuckets,
                    a.key_bits, a.slot_bits, smem_sort ? 1 : 0);
}

}  // namespace moe_lora

extern "C" size_t moe_lora_align_buffer_size(int T, int k, int E, int L, int bm_base, int bm_lora) {
  moe_lora::AlignLayout a = moe_lora::align_layout(T, k, E, L, bm_base, bm_lora);
  return a.valid ? (size_t)a.off[MOE_LORA_AF_TOTAL_BYTES] : 0;
}

extern "C" int moe_lora_align_layout(int T, int k, int E, int L, int bm_base, int bm_lora,
                                     int64_t* offsets) {
  if (!offsets) return MOE_LORA_ERR_INVALID_ARG;
  moe_lora::AlignLayout a = moe_lora::align_layout(T, k, E, L, bm_base, bm_lora);
  if (!a.valid) return MOE_LORA_ERR_UNSUPPORTED;
  for (int i = 0; i < MOE_LORA_ALIGN_NFIELDS; ++i) offsets[i] = a.off[i];
  return MOE_LORA_OK;
}

extern "C" int moe_lora_align(const int32_t* ids, const int32_t* token_adapter,
                              const moe_lora_align_t* al, moe_lora_stream_t stream) {
  using namespace moe_lora;
  AlignLayout a;
  int st = check_align(al, &a);
  if (st != MOE_LORA_OK) return st;
  if (a.S > 0 && !ids) return MOE_LORA_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_LORA_OK) return st;
  return launch_align(ids, token_adapter, al, a, reinterpret_cast<cudaStream_t>(stream), true);
}
