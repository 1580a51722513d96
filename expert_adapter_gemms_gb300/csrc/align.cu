// Alignment of token-slots by (expert, adapter): the "compound sparsity" of
// expert routing and adapter selection (vllm.com.cn, section "Implementing
// multi-LoRA inference for MoE models in vLLM"; agentlenshq.com, section
// "Multi-LoRA Serving for MoE Models").
//
// One CTA of 1024 threads (up to a few thousand slots). Each slot s gets the
// packed word (key << slot_bits) | s with key = e * (L + 1) + (l + 1) (dropped
// slots use the last bucket). A stable least-significant-digit radix sort on the
// key bits (8-bit digits, per-warp digit histograms, ranks inside a warp from
// eight ballots) keeps equal keys in slot order, so the result is the unique
// stable order: deterministic and bit-exact. Bucket starts, read off the sorted
// keys, give the expert and (expert, adapter) segment boundaries, from which the
// grouped-GEMM token tiles and the LoRA blocks are cut. Working state (bucket counts and starts, the
// sort buffers) stays in shared memory whenever it fits; only results go out.
// Up to kRankSortMaxSlots slots the words are placed by rank instead of the radix sort, and
// a layer at few tokens has this CTA route the tokens first (one launch fewer).
#include <atomic>

#include "internal.h"
#include "route.cuh"

namespace moe_lora {

constexpr int kSmemSortMaxSlots = 16384;
constexpr size_t kAlignSmemBudget = 200 * 1024;
constexpr int kRankSortMaxSlots = 512;

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

// Stable least-significant-digit radix sort of the n words in a (n fits a and b) on
// bits [lo, lo + nbits), 8-bit digits; returns the buffer that holds the result. Each
// warp owns a contiguous range of words; per-warp digit histograms (padded rows, so a
// warp's different digits fall in different banks) give every (digit, warp) its
// output offset, and a lane's rank among same-digit lanes of its warp comes from eight
// ballots. All NT threads call it; hist holds 256 * (NT / 32 + 1) ints, tmp NT / 32 + 1.
template <int NT>
__device__ uint32_t* block_radix_sort(uint32_t* a, uint32_t* b, int n, int lo, int nbits, int* hist,
                                      int* tmp) {
  constexpr int NW = NT / 32, HS = NW + 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* src = a;
  uint32_t* dst = b;
  const int chunk = (n + NW - 1) / NW;
  const int wb = min(n, warp * chunk), we = min(n, wb + chunk);
  const unsigned lt = (1u << lane) - 1u;
  for (int shift = lo; shift < lo + nbits; shift += 8) {
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
  return src;
}

// The words are unique ((key, slot) with distinct slots), so the stable key order of the
// radix sort is their ascending order, and a word's place is the number of smaller words:
// for a few hundred words one pass of broadcast shared-memory reads per thread, without
// the radix sort's barriers. The same result, bit for bit. P lanes of a warp share a word
// (as many as the threads allow, up to 8), each counting over every P-th 16-byte group of
// words (P consecutive groups per step: one wavefront), and add their counts with
// shuffles inside the group. The buffer is padded to whole groups with all-ones words,
// which are smaller than no word.
template <int NT, int P>
__device__ void rank_place(const uint32_t* a, uint32_t* b, int n) {
  const int lane = threadIdx.x & 31, part = lane & (P - 1);
  const unsigned group = ((1u << P) - 1u) << (lane & ~(P - 1));  // the word's P lanes
  const uint4* a4 = reinterpret_cast<const uint4*>(a);
  const int n4 = (n + 3) >> 2;
  for (int i = threadIdx.x / P; i < n; i += NT / P) {  // the same i for a group's lanes
    const uint32_t x = a[i];
    int pos = 0;
#pragma unroll 4
    for (int q = part; q < n4; q += P) {
      const uint4 y = a4[q];
      pos += (y.x < x ? 1 : 0) + (y.y < x ? 1 : 0) + (y.z < x ? 1 : 0) + (y.w < x ? 1 : 0);
    }
#pragma unroll
    for (int o = 1; o < P; o <<= 1) pos += __shfl_xor_sync(group, pos, o);
    if (part == 0) b[pos] = x;
  }
}
template <int NT>
__device__ uint32_t* block_rank_sort(const uint32_t* a, uint32_t* b, int n) {
  if (8 * n <= NT) rank_place<NT, 8>(a, b, n);
  else if (4 * n <= NT) rank_place<NT, 4>(a, b, n);
  else if (2 * n <= NT) rank_place<NT, 2>(a, b, n);
  else rank_place<NT, 1>(a, b, n);
  __syncthreads();
  return b;
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
  const int S4 = (S + 3) & ~3;  // each sort buffer in whole 16-byte groups
  const size_t sort_b = (size_t)2 * S4 * 4;
  const size_t bucket_b = (size_t)2 * nbuckets * 4;
  p.smem_sort = S <= kSmemSortMaxSlots;
  const size_t base = (size_t)o * 4 + (p.smem_sort ? sort_b : 0);
  p.smem_buckets = base + bucket_b <= kAlignSmemBudget;
  p.bcount_off = o;
  p.bstart_off = o + (p.smem_buckets ? nbuckets : 0);
  o = p.bstart_off + (p.smem_buckets ? nbuckets : 0);
  o = (o + 3) & ~3;
  p.sort_off = o;
  p.bytes = (size_t)o * 4 + (p.smem_sort ? sort_b : 0);
  return p;
}

// V > 0: route first (logits [T, E], V experts a lane): ids and w are written here and
// the keys read the ids back (ids then points at that buffer).
template <int NT, int V>
__global__ void __launch_bounds__(NT, 1)
    align_kernel(const int* __restrict__ ids, const int* __restrict__ token_adapter, AlignView v,
                 int T, int k, int E, int L, int bm_base, int bm_lora, int S, int nbuckets,
                 int key_bits, int slot_bits, const float* __restrict__ logits,
                 float* __restrict__ w_out) {
  constexpr int NW = NT / 32;
  extern __shared__ __align__(16) int smem[];
  const AlignSmem plan = align_smem_plan(S, nbuckets, NT);
  int* hist = smem + plan.hist_off;  // [256 digits][NW warps + 1]
  int* tmp = smem + plan.tmp_off;
  int* bcount = plan.smem_buckets ? smem + plan.bcount_off : v.bucket_count;
  int* bstart = plan.smem_buckets ? smem + plan.bstart_off : v.bucket_start;
  uint32_t* bufA = plan.smem_sort ? reinterpret_cast<uint32_t*>(smem + plan.sort_off) : v.sort0;
  uint32_t* bufB = plan.smem_sort ? bufA + ((S + 3) & ~3) : v.sort1;
  __shared__ unsigned int s_err;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int drop = nbuckets - 1;
  const uint32_t smask = (slot_bits >= 32) ? 0xffffffffu : ((1u << slot_bits) - 1u);

  // the next launch waits before reading any of this launch's results
  pdl_trigger();
  pdl_wait();
  if (tid == 0) s_err = 0u;
  // routing here: the adapter ids of this thread's first four slots, in flight with the
  // logits
  int lv0[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int s = tid + u * NT;
    lv0[u] = V > 0 && token_adapter && s < S ? __ldcg(token_adapter + s / k) : -1;
  }
  // routed here: the ids also stay in shared memory for the keys (T k <= 64 * 32 slots)
  __shared__ int s_rid[V > 0 ? kAlignRouteMaxTokens * 32 : 1];
  if constexpr (V > 0) {  // 0. routing, one warp per token: TB of a warp's tokens at
    // once (64 tokens in one round), their logits in flight and their selections side by side
    constexpr int TB = NT >= 1024 ? 2 : 8;
    int* ids_out = const_cast<int*>(ids);
    for (int t0 = warp; t0 < T; t0 += NW * TB) {
      float lv[TB][V];
      int tok[TB];
#pragma unroll
      for (int b = 0; b < TB; ++b) {
        const int t = t0 + b * NW;
        tok[b] = t < T ? t : -1;
        if (t < T) topk_softmax_load<V>(logits + (size_t)t * E, E, lv[b]);
        else
#pragma unroll
          for (int i = 0; i < V; ++i) lv[b][i] = -INFINITY;
      }
      topk_softmax_select<V, TB>(lv, tok, E, k, ids_out, w_out, s_rid);
    }
  }
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
        if constexpr (V > 0) ev[u] = s_rid[s];
        else ev[u] = __ldcg(ids + s);
        if (V > 0 && s0 == tid) lv[u] = lv0[u];
        else if (token_adapter) lv[u] = __ldcg(token_adapter + s / k);
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
  if (plan.smem_sort && tid < ((S + 3) & ~3) - S) bufA[S + tid] = 0xffffffffu;  // group padding
  __syncthreads();

  // 2. stable LSD radix sort on the key bits (8-bit digits)
  uint32_t* src = plan.smem_sort && S <= kRankSortMaxSlots
                      ? block_rank_sort<NT>(bufA, bufB, S)
                      : block_radix_sort<NT>(bufA, bufB, S, slot_bits, key_bits, hist, tmp);
  uint32_t* dst = src == bufA ? bufB : bufA;
  const unsigned lt = (1u << lane) - 1u;

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
  int tot_t, tot_b, tot_l, ti, bi;
  if (S < 1024) {  // the three counts (each <= S) in 10-bit fields of one scan
    int tot;
    const int pre = __shfl_sync(
        0xffffffffu, block_exclusive_scan<NW>(lane == 0 ? nt | nb << 10 | nl << 20 : 0, tmp, &tot), 0);
    ti = pre & 1023;
    bi = (pre >> 10) & 1023;
    tot_t = tot & 1023;
    tot_b = (tot >> 10) & 1023;
    tot_l = tot >> 20;
  } else {
    ti = __shfl_sync(0xffffffffu, block_exclusive_scan<NW>(lane == 0 ? nt : 0, tmp, &tot_t), 0);
    bi = __shfl_sync(0xffffffffu, block_exclusive_scan<NW>(lane == 0 ? nb : 0, tmp, &tot_b), 0);
    block_exclusive_scan<NW>(lane == 0 ? nl : 0, tmp, &tot_l);
  }
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

// ----------------------------------------------------------------------------
// Multi-CTA align (many slots): the one-CTA kernel above runs its sort on one SM;
// here the same unique stable order comes from three launches.
//  local: CTA c takes slots [c C, (c + 1) C) (C = kAlignChunk), computes their keys,
//         sorts them stably with the block radix sort, and records for each word its
//         rank among the CTA's words of the same key and, per key, the CTA's count
//         in counts[c][key].
//  scan:  one CTA turns the count table, read in (key, CTA) order, into exclusive
//         offsets: the first sorted position of CTA c's words of each key. Bucket
//         starts, expert starts, token tiles, LoRA blocks and the header follow
//         from the per-key totals.
//  place: word i of CTA c goes to offsets[c][key] + its rank.
// Keys ordered by (key, CTA, rank within the CTA) are ordered by (key, slot), since the
// CTAs hold increasing slot ranges and each CTA's sort is stable.
// ----------------------------------------------------------------------------
template <int NT>
__global__ void __launch_bounds__(NT)
    align_local_kernel(const int* __restrict__ ids, const int* __restrict__ token_adapter,
                       AlignView v, int k, int E, int L, int S, int nbuckets, int key_bits,
                       int slot_bits, int ctas) {
  constexpr int NW = NT / 32, C = kAlignChunk, PT = C / NT;
  __shared__ uint32_t bufA[C], bufB[C];
  __shared__ int hist[256 * (NW + 1)];
  __shared__ int tmp[NW + 1];
  __shared__ int head[C];
  __shared__ unsigned int s_err;
  // the next launch waits before reading any of this launch's results
  pdl_trigger();
  pdl_wait();
  const int c = blockIdx.x, tid = threadIdx.x;
  const int s0 = c * C, n = min(C, S - s0);
  const int drop = nbuckets - 1;
  if (tid == 0) s_err = 0u;
  int* cnt_c = v.counts + (size_t)c * nbuckets;  // this CTA's row of the count table
  for (int b = tid; b < nbuckets; b += NT) cnt_c[b] = 0;
  int ev[PT], lv[PT];
#pragma unroll
  for (int u = 0; u < PT; ++u) {
    const int i = tid + u * NT;
    ev[u] = 0;
    lv[u] = -1;
    if (i < n) {
      ev[u] = __ldcg(ids + s0 + i);
      if (token_adapter) lv[u] = __ldcg(token_adapter + (s0 + i) / k);
    }
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < PT; ++u) {
    const int i = tid + u * NT;
    if (i >= n) break;
    const int e = ev[u], l = lv[u];
    unsigned int bad = 0;
    if (e < 0 || e >= E) bad |= MOE_LORA_DEVERR_EXPERT_RANGE;
    if (l < -1 || l >= L) bad |= MOE_LORA_DEVERR_ADAPTER_RANGE;
    int key = drop;
    if (bad) atomicOr(&s_err, bad);
    else key = e * (L + 1) + (l + 1);
    bufA[i] = (static_cast<uint32_t>(key) << slot_bits) | static_cast<uint32_t>(s0 + i);
  }
  __syncthreads();
  const uint32_t* srt = block_radix_sort<NT>(bufA, bufB, n, slot_bits, key_bits, hist, tmp);
  // rank within the key run: the run's first index by an inclusive max-scan of run heads
  for (int i = tid; i < C; i += NT)
    head[i] = (i < n && (i == 0 || (srt[i] >> slot_bits) != (srt[i - 1] >> slot_bits))) ? i : 0;
  __syncthreads();
  for (int off = 1; off < C; off <<= 1) {
    int hv[PT];
#pragma unroll
    for (int u = 0; u < PT; ++u) {
      const int i = tid + u * NT;
      hv[u] = i >= off ? max(head[i], head[i - off]) : head[i];
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < PT; ++u) head[tid + u * NT] = hv[u];
    __syncthreads();
  }
  for (int i = tid; i < n; i += NT) {
    const uint32_t w = srt[i];
    const int key = static_cast<int>(w >> slot_bits);
    const int rank = i - head[i];
    v.sort0[s0 + i] = w;
    v.sort1[s0 + i] = static_cast<uint32_t>(rank);
    if (i == n - 1 || (srt[i + 1] >> slot_bits) != static_cast<uint32_t>(key))
      cnt_c[key] = rank + 1;  // the run's last word holds its length
  }
  if (tid == 0 && s_err) atomicOr(reinterpret_cast<unsigned int*>(v.hdr + HDR_ERR), s_err);
}

template <int NT>
__global__ void __launch_bounds__(NT)
    align_scan_kernel(AlignView v, int T, int k, int E, int L, int bm_base, int bm_lora, int S,
                      int nbuckets, int ctas) {
  constexpr int NW = NT / 32;
  __shared__ int tmp[NW + 1];
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x;
  // 1. exclusive scan of the count table in (key, CTA) order, in place. The table is
  //    stored CTA-major ([ctas][nbuckets]); a tile of NT keys is read one key per thread
  //    (coalesced across threads for each CTA row), totalled per key, scanned across
  //    the tile with the carry of the tiles before, and written back as offsets.
  int carry = 0;
  for (int b0 = 0; b0 < nbuckets; b0 += NT) {
    const int b = b0 + tid;
    int tot = 0;
    if (b < nbuckets) {
#pragma unroll 8
      for (int c = 0; c < ctas; ++c) tot += __ldcg(v.counts + (size_t)c * nbuckets + b);
    }
    int tile_total;
    int run = carry + block_exclusive_scan<NW>(tot, tmp, &tile_total);
    if (b < nbuckets) {
      v.bucket_start[b] = run;
      v.bucket_count[b] = tot;
      // sixteen counts are loaded before their offsets are stored (a load after a store
      // that may alias it would wait for it: one round trip per CTA)
      constexpr int CB = 16;
      for (int c0 = 0; c0 < ctas; c0 += CB) {
        int cnt[CB];
#pragma unroll
        for (int u = 0; u < CB; ++u)
          cnt[u] = c0 + u < ctas ? __ldcg(v.counts + (size_t)(c0 + u) * nbuckets + b) : 0;
#pragma unroll
        for (int u = 0; u < CB; ++u) {
          if (c0 + u < ctas) {
            v.counts[(size_t)(c0 + u) * nbuckets + b] = run;
            run += cnt[u];
          }
        }
      }
    }
    carry += tile_total;
  }
  __syncthreads();
  // 2. expert starts
  for (int e = tid; e <= E; e += NT) v.expert_begin[e] = __ldcg(v.bucket_start + (size_t)e * (L + 1));
  __syncthreads();
  const int n_valid = __ldcg(v.bucket_start + nbuckets - 1);
  // 3. token tiles: each expert's rows in chunks of bm_base, experts in order
  const int pe = (E + NT - 1) / NT;
  const int e0 = min(E, tid * pe), e1 = min(E, e0 + pe);
  int nt = 0;
  for (int e = e0; e < e1; ++e) {
    const int rows = __ldcg(v.expert_begin + e + 1) - __ldcg(v.expert_begin + e);
    nt += (rows + bm_base - 1) / bm_base;
  }
  int tot_t;
  int ti = block_exclusive_scan<NW>(nt, tmp, &tot_t);
  for (int e = e0; e < e1; ++e) {
    const int rb = __ldcg(v.expert_begin + e), rows = __ldcg(v.expert_begin + e + 1) - rb;
    for (int j = 0; j * bm_base < rows; ++j)
      v.tiles[ti++] = make_int4(e, rb + j * bm_base, min(bm_base, rows - j * bm_base), 0);
  }
  // 4. LoRA blocks: each (e, l >= 0) bucket's rows in chunks of bm_lora, buckets in order
  const int pb = (nbuckets + NT - 1) / NT;
  const int q0 = min(nbuckets, tid * pb), q1 = min(nbuckets, q0 + pb);
  int nb = 0, nl = 0;
  for (int b = q0; b < q1; ++b) {
    if (b % (L + 1) == 0) continue;  // adapter -1 (and the dropped-slot bucket)
    const int cnt = __ldcg(v.bucket_count + b);
    nb += (cnt + bm_lora - 1) / bm_lora;
    nl += cnt;
  }
  int tot_b, tot_l;
  int bi = block_exclusive_scan<NW>(nb, tmp, &tot_b);
  block_exclusive_scan<NW>(nl, tmp, &tot_l);
  for (int b = q0; b < q1; ++b) {
    if (b % (L + 1) == 0) continue;
    const int e = b / (L + 1), l = b % (L + 1) - 1;
    const int rb = __ldcg(v.bucket_start + b), cnt = __ldcg(v.bucket_count + b);
    for (int j = 0; j * bm_lora < cnt; ++j)
      v.blocks[bi++] = make_int4(rb + j * bm_lora, min(bm_lora, cnt - j * bm_lora), e, l);
  }
  if (tid == 0) {
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
__global__ void __launch_bounds__(NT)
    align_place_kernel(AlignView v, int L, int S, int nbuckets, int slot_bits, int ctas) {
  constexpr int C = kAlignChunk;
  pdl_trigger();
  pdl_wait();
  const int c = blockIdx.x;
  const int s0 = c * C, n = min(C, S - s0);
  const int drop = nbuckets - 1;
  const uint32_t smask = (slot_bits >= 32) ? 0xffffffffu : ((1u << slot_bits) - 1u);
  for (int i = threadIdx.x; i < n; i += NT) {
    const uint32_t w = __ldcg(v.sort0 + s0 + i);
    const int rank = static_cast<int>(__ldcg(v.sort1 + s0 + i));
    const int key = static_cast<int>(w >> slot_bits);
    const int s = static_cast<int>(w & smask);
    const int pos = __ldcg(v.counts + (size_t)c * nbuckets + key) + rank;
    if (key == drop) {
      v.sorted_slots[pos] = -1;
      v.slot_row[s] = -1;
    } else {
      v.sorted_slots[pos] = s;
      v.slot_row[s] = pos;
      v.row_expert[pos] = key / (L + 1);
      v.row_adapter[pos] = key % (L + 1) - 1;
    }
  }
}

template <int NT, int V>
static int launch_align_t(const int* ids, const int* token_adapter, const moe_lora_align_t* al,
                          const AlignLayout& a, cudaStream_t stream, bool pdl,
                          const float* logits = nullptr, float* w = nullptr) {
  AlignView v = align_view(al->buf, a);
  const AlignSmem plan = align_smem_plan(a.S, a.nbuckets, NT);
  static std::atomic<uint64_t> configured[kMaxDevices];
  int st = once_per_context(configured, [] {
    ML_CHECK_CUDA(cudaFuncSetAttribute(align_kernel<NT, V>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)(kAlignSmemBudget + 16 * 1024)));
    return MOE_LORA_OK;
  });
  if (st != MOE_LORA_OK) return st;
  return launch_pdl(align_kernel<NT, V>, 1, NT, plan.bytes, stream, pdl, ids, token_adapter, v,
                    al->T, al->k, al->E, al->L, al->bm_base, al->bm_lora, a.S, a.nbuckets,
                    a.key_bits, a.slot_bits, logits, w);
}

bool align_can_route(const AlignLayout& a, int T, int E) {
  return a.ctas == 0 && a.S <= 4096 && T <= kAlignRouteMaxTokens && E <= 64;
}

int launch_route_align(const float* logits, int* ids, float* w, const int* token_adapter,
                       const moe_lora_align_t* al, const AlignLayout& a, cudaStream_t stream,
                       bool pdl) {
  if (!align_can_route(a, al->T, al->E)) return MOE_LORA_ERR_UNSUPPORTED;
  // 1024 threads: two tokens a warp, up to eight lanes a word of the rank sort
  return al->E <= 32 ? launch_align_t<1024, 1>(ids, token_adapter, al, a, stream, pdl, logits, w)
                     : launch_align_t<1024, 2>(ids, token_adapter, al, a, stream, pdl, logits, w);
}

int launch_align(const int* ids, const int* token_adapter, const moe_lora_align_t* al,
                 const AlignLayout& a, cudaStream_t stream, bool pdl) {
  if (a.ctas > 0) {  // many slots: spread the sort over a.ctas CTAs
    AlignView v = align_view(al->buf, a);
    int st = launch_pdl(align_local_kernel<256>, a.ctas, 256, 0, stream, pdl, ids, token_adapter,
                        v, al->k, al->E, al->L, a.S, a.nbuckets, a.key_bits, a.slot_bits, a.ctas);
    if (st != MOE_LORA_OK) return st;
    st = launch_pdl(align_scan_kernel<1024>, 1, 1024, 0, stream, pdl, v, al->T, al->k, al->E,
                    al->L, al->bm_base, al->bm_lora, a.S, a.nbuckets, a.ctas);
    if (st != MOE_LORA_OK) return st;
    return launch_pdl(align_place_kernel<256>, a.ctas, 256, 0, stream, pdl, v, al->L, a.S,
                      a.nbuckets, a.slot_bits, a.ctas);
  }
  // one CTA of 1024 threads (at 1024 and 2048 slots, with the radix sort: 15.3 and 25.7 us
  // against 17.5 and 33.8 us with 256 threads)
  return launch_align_t<1024, 0>(ids, token_adapter, al, a, stream, pdl);
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
