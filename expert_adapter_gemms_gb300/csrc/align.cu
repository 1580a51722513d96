// Alignment of token-slots by (expert, adapter): the "compound sparsity" of
// expert routing and adapter selection (vllm.com.cn, section "Implementing
// multi-LoRA inference for MoE models in vLLM"; agentlenshq.com, section
// "Multi-LoRA Serving for MoE Models").
//
// One CTA (256 threads up to 4096 slots, 1024 beyond). Each slot s gets the
// packed word (key << slot_bits) | s with key = e * (L + 1) + (l + 1) (dropped
// slots use the last bucket). A stable least-significant-digit radix sort on the
// key bits (8-bit digits, per-warp digit histograms, ranks inside a warp from
// eight ballots) keeps equal keys in slot order, so the result is the unique
// stable order: deterministic and bit-exact. Bucket starts, read off the sorted
// keys, give the expert and (expert, adapter) segment boundaries, from which the
// grouped-GEMM token tiles and the LoRA blocks are cut. Working state (bucket counts and starts, the
// sort buffers) stays in shared memory whenever it fits; only results go out.
#include "common.cuh"

namespace moe_lora {

constexpr int kSmemSortMaxSlots = 16384;
constexpr size_t kAlignSmemBudget = 200 * 1024;

// Exclusive scan of one int per thread across the CTA; returns the prefix and
// writes the total to *total. `tmp` holds NW + 1 ints.
template <int NW>
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
    const int x = lane < NW ? tmp[lane] : 0;
    int xi = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, xi, off);
      if (lane >= off) xi += u;
    }
    if (lane < NW) tmp[lane] = xi - x;  // exclusive prefix of warp totals
    if (lane == 31) tmp[NW] = xi;
  }
  __syncthreads();
  const int r = tmp[warp] + incl - v;
  *total = tmp[NW];
  __syncthreads();
  return r;
}

// Lanes of `mask` whose 8-bit digit equals this lane's: the AND over the digit's
// bits of each bit's ballot (or its complement).
__device__ __forceinline__ unsigned digit_peers(unsigned mask, int d) {
  unsigned peers = mask;
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const unsigned bb = __ballot_sync(mask, (d >> b) & 1);
    peers &= ((d >> b) & 1) ? bb : ~bb;
  }
  return peers;
}

// Shared-memory plan of one align launch (host and device agree through this).
struct AlignSmem {
  int hist_off, tmp_off, bcount_off, bstart_off, sort_off;  // in ints
  size_t bytes;
  bool smem_buckets, smem_sort;
};

__host__ __device__ inline AlignSmem align_smem_plan(int S, int nbuckets, int nthreads) {
  AlignSmem p;
  const int nw = nthreads / 32;
  p.hist_off = 0;
  p.tmp_off = 256 * (nw + 1);
  int o = p.tmp_off + 64;
  const size_t sort_b = (size_t)2 * S * 4;
  const size_t bucket_b = (size_t)2 * nbuckets * 4;
  p.smem_sort = S <= kSmemSortMaxSlots;
  const size_t base = (size_t)o * 4 + (p.smem_sort ? sort_b : 0);
  p.smem_buckets = base + bucket_b <= kAlignSmemBudget;
  p.bcount_off = o;
  p.bstart_off = o + (p.smem_buckets ? nbuckets : 0);
  o = p.bstart_off + (p.smem_buckets ? nbuckets : 0);
  p.sort_off = o;
  p.bytes = (size_t)o * 4 + (p.smem_sort ? sort_b : 0);
  return p;
}

template <int NT>
__global__ void __launch_bounds__(NT, 1)
    align_kernel(const int* __restrict__ ids, const int* __restrict__ token_adapter, AlignView v,
                 int T, int k, int E, int L, int bm_base, int bm_lora, int S, int nbuckets,
                 int key_bits, int slot_bits) {
  constexpr int NW = NT / 32;
  extern __shared__ __align__(16) int smem[];
  const AlignSmem plan = align_smem_plan(S, nbuckets, NT);
  // [256 digits][NW warps + 1]: the pad puts a warp's different digits in different banks
  constexpr int HS = NW + 1;
  int* hist = smem + plan.hist_off;
  int* tmp = smem + plan.tmp_off;
  int* bcount = plan.smem_buckets ? smem + plan.bcount_off : v.bucket_count;
  int* bstart = plan.smem_buckets ? smem + plan.bstart_off : v.bucket_start;
  uint32_t* bufA = plan.smem_sort ? reinterpret_cast<uint32_t*>(smem + plan.sort_off) : v.sort0;
  uint32_t* bufB = plan.smem_sort ? bufA + S : v.sort1;
  __shared__ unsigned int s_err;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int drop = nbuckets - 1;
  const uint32_t smask = (slot_bits >= 32) ? 0xffffffffu : ((1u << slot_bits) - 1u);

  // the next launch waits before reading any of this launch's results
  pdl_trigger();
  pdl_wait();
  if (tid == 0) s_err = 0u;
  __syncthreads();

  // 1. keys (the loads of four slots go out together)
  for (int s0 = tid; s0 < S; s0 += 4 * NT) {
    int ev[4], lv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int s = s0 + u * NT;
      ev[u] = 0;
      lv[u] = -1;
      if (s < S) {
        ev[u] = __ldcg(ids + s);
        if (token_adapter) lv[u] = __ldcg(token_adapter + s / k);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int s = s0 + u * NT;
      if (s >= S) break;
      const int e = ev[u], l = lv[u];
      unsigned int bad = 0;
      if (e < 0 || e >= E) bad |= MOE_LORA_DEVERR_EXPERT_RANGE;
      if (l < -1 || l >= L) bad |= MOE_LORA_DEVERR_ADAPTER_RANGE;
      int key = drop;
      if (bad) atomicOr(&s_err, bad);
      else key = e * (L + 1) + (l + 1);
      bufA[s] = (static_cast<uint32_t>(key) << slot_bits) | static_cast<uint32_t>(s);
    }
  }
  __syncthreads();

  // 2. stable LSD radix sort on the key bits (8-bit digits)
  uint32_t* src = bufA;
  uint32_t* dst = bufB;
  const int chunk = (S + NW - 1) / NW;
  const int wb = min(S, warp * chunk), we = min(S, wb + chunk);
  const unsigned lt = (1u << lane) - 1u;
  for (int shift = slot_bits; shift < slot_bits + key_bits; shift += 8) {
    for (int d = lane; d < 256; d += 32) hist[d * HS + warp] = 0;
    __syncwarp();
    for (int base = wb; base < we; base += 32) {
      const int i = base + lane;
      const bool act = i < we;
      const unsigned mask = __ballot_sync(0xffffffffu, act);
      if (act) {
        const int d = (src[i] >> shift) & 255;
        const unsigned peers = digit_peers(mask, d);
        if (lane == __ffs(peers) - 1) hist[d * HS + warp] += __popc(peers);
      }
      __syncwarp();
    }
    __syncthreads();
    {  // exclusive scan over (digit, warp) in digit-major order
      constexpr int PER = 256 * NW / NT;
      int loc[PER];
      int s = 0;
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const int pidx = tid * PER + q;  // (digit, warp) in digit-major order
        loc[q] = hist[(pidx / NW) * HS + pidx % NW];
        s += loc[q];
      }
      int total;
      int run = block_exclusive_scan<NW>(s, tmp, &total);
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const int pidx = tid * PER + q;
        hist[(pidx / NW) * HS + pidx % NW] = run;
        run += loc[q];
      }
    }
    __syncthreads();
    for (int base = wb; base < we; base += 32) {
      const int i = base + lane;
      const bool act = i < we;
      const unsigned mask = __ballot_sync(0xffffffffu, act);
      int d = 0;
      unsigned peers = 0;
      if (act) {
        const uint32_t x = src[i];
        d = (x >> shift) & 255;
        peers = digit_peers(mask, d);
        dst[hist[d * HS + warp] + __popc(peers & lt)] = x;
      }
      __syncwarp();
      if (act && lane == __ffs(peers) - 1) hist[d * HS + warp] += __popc(peers);
      __syncwarp();
    }
    __syncthreads();
    uint32_t* sw = src;
    src = dst;
    dst = sw;
  }

  // 3. segment starts: bucket c starts at the first sorted word with key >= c
  //    (bucket order is expert-major, adapter -1 first); each sorted position
  //    fills the starts of the buckets between its predecessor's key and its own,
  //    so every bucket is written once; counts are differences.
  for (int i = tid; i <= S; i += NT) {
    const int kp = i == 0 ? -1 : static_cast<int>(src[i - 1] >> slot_bits);
    const int kc = i == S ? nbuckets - 1 : static_cast<int>(src[i] >> slot_bits);
    for (int c = kp + 1; c <= kc; ++c) bstart[c] = i;
  }
  __syncthreads();
  for (int c = tid; c < nbuckets; c += NT)
    bcount[c] = (c + 1 < nbuckets ? bstart[c + 1] : S) - bstart[c];
  __syncthreads();
  const int n_valid = bstart[drop];

  // 4. sorted rows, expert starts. slot_row is the inverse permutation: with the sort in
  //    shared memory it is built in the free sort buffer and then written out coalesced.
  int* inv = plan.smem_sort ? reinterpret_cast<int*>(dst) : nullptr;
  for (int i = tid; i < S; i += NT) {
    const uint32_t x = src[i];
    const int s = static_cast<int>(x & smask);
    const int key = static_cast<int>(x >> slot_bits);
    if (key == drop) {
      v.sorted_slots[i] = -1;
      if (inv) inv[s] = -1;
      else v.slot_row[s] = -1;
    } else {
      const int e = key / (L + 1), l = key % (L + 1) - 1;
      v.sorted_slots[i] = s;
      if (inv) inv[s] = i;
      else v.slot_row[s] = i;
      v.row_expert[i] = e;
      v.row_adapter[i] = l;
    }
  }
  for (int e = tid; e <= E; e += NT) v.expert_begin[e] = bstart[e * (L + 1)];
  __syncthreads();  // the inverse permutation (and global bucket arrays) complete
  if (inv)
    for (int s = tid; s < S; s += NT) v.slot_row[s] = inv[s];

  // 5. token tiles (per expert, bm_base rows) and LoRA blocks (per (e, l>=0), bm_lora rows),
  //    numbered in sorted-row order. Each warp takes a contiguous range of rows and its lanes
  //    consecutive rows; ballots order the starts inside the warp, a block scan across warps.
  const int per_w = ((n_valid + NW - 1) / NW + 31) & ~31;
  const int wb5 = min(n_valid, warp * per_w), we5 = min(n_valid, wb5 + per_w);
  auto starts = [&](int i, int& e, int& l, int& key, bool& ft, bool& fb, bool& fl) {
    ft = fb = fl = false;
    e = l = key = 0;
    if (i >= we5) return;
    key = static_cast<int>(src[i] >> slot_bits);
    e = key / (L + 1);
    l = key % (L + 1) - 1;
    ft = (i - bstart[e * (L + 1)]) % bm_base == 0;
    if (l >= 0) {
      fl = true;
      fb = (i - bstart[key]) % bm_lora == 0;
    }
  };
  int nt = 0, nb = 0, nl = 0;
  for (int base = wb5; base < we5; base += 32) {
    int e, l, key;
    bool ft, fb, fl;
    starts(base + lane, e, l, key, ft, fb, fl);
    nt += __popc(__ballot_sync(0xffffffffu, ft));
    nb += __popc(__ballot_sync(0xffffffffu, fb));
    nl += __popc(__ballot_sync(0xffffffffu, fl));
  }
  int tot_t, tot_b, tot_l;
  int ti = __shfl_sync(0xffffffffu, block_exclusive_scan<NW>(lane == 0 ? nt : 0, tmp, &tot_t), 0);
  int bi = __shfl_sync(0xffffffffu, block_exclusive_scan<NW>(lane == 0 ? nb : 0, tmp, &tot_b), 0);
  block_exclusive_scan<NW>(lane == 0 ? nl : 0, tmp, &tot_l);
  for (int base = wb5; base < we5; base += 32) {
    const int i = base + lane;
    int e, l, key;
    bool ft, fb, fl;
    starts(i, e, l, key, ft, fb, fl);
    const unsigned bt = __ballot_sync(0xffffffffu, ft), bb = __ballot_sync(0xffffffffu, fb);
    if (ft)
      v.tiles[ti + __popc(bt & lt)] = make_int4(e, i, min(bm_base, bstart[(e + 1) * (L + 1)] - i), 0);
    if (fb) {
      const int sb = bstart[key];
      v.blocks[bi + __popc(bb & lt)] = make_int4(i, min(bm_lora, sb + bcount[key] - i), e, l);
    }
    ti += __popc(bt);
    bi += __popc(bb);
  }
  if (tid == 0) {
    if (s_err) atomicOr(reinterpret_cast<unsigned int*>(v.hdr + HDR_ERR), s_err);
    v.hdr[HDR_NVALID] = n_valid;
    v.hdr[HDR_NTILES] = tot_t;
    v.hdr[HDR_NBLOCKS] = tot_b;
    v.hdr[HDR_NLORAROWS] = tot_l;
    v.hdr[HDR_T] = T;
    v.hdr[HDR_K] = k;
    v.hdr[HDR_E] = E;
    v.hdr[HDR_L] = L;
    v.hdr[HDR_BMB] = bm_base;
    v.hdr[HDR_BML] = bm_lora;
  }
}

template <int NT>
static int launch_align_t(const int* ids, const int* token_adapter, const moe_lora_align_t* al,
                          const AlignLayout& a, cudaStream_t stream, bool pdl) {
  AlignView v = align_view(al->buf, a);
  const AlignSmem plan = align_smem_plan(a.S, a.nbuckets, NT);
  static int configured[64] = {0};
  int dev = 0;
  ML_CHECK_CUDA(cudaGetDevice(&dev));
  if (dev < 64 && !configured[dev]) {
    ML_CHECK_CUDA(cudaFuncSetAttribute(align_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)(kAlignSmemBudget + 16 * 1024)));
    configured[dev] = 1;
  }
  return launch_pdl(align_kernel<NT>, 1, NT, plan.bytes, stream, pdl, ids, token_adapter, v,
                    al->T, al->k, al->E, al->L, al->bm_base, al->bm_lora, a.S, a.nbuckets,
                    a.key_bits, a.slot_bits);
}

int launch_align(const int* ids, const int* token_adapter, const moe_lora_align_t* al,
                 const AlignLayout& a, cudaStream_t stream, bool pdl) {
  // few slots: a small CTA keeps the many barriers of the sort cheap
  if (a.S <= 4096) return launch_align_t<256>(ids, token_adapter, al, a, stream, pdl);
  return launch_align_t<1024>(ids, token_adapter, al, a, stream, pdl);
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
