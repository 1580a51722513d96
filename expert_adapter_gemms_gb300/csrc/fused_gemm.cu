// The expert grouped GEMM with the LoRA expand fused in by concatenation along the
// reduction dimension (the tensor-core form of "adding the LoRA result to the base
// output inside the expand kernel", vllm.com.cn, section "Kernel optimizations";
// agentlenshq.com, "Kernel-Level Optimizations"). For the rows of adapter l in a
// token tile of expert e,
//
//   out = x W_e^T + z B_{l,e}^T = [x | z] [W_e | B_{l,e}]^T,
//
// so the expand is a few more K-steps of the same tcgen05 accumulation and the base
// output never makes an fp32 round trip through HBM. Two epilogues:
//
// * gate_up (kGLU): the 128 rows of a CTA's weight block are 64 rows of the gate half
//   of W1 and the matching 64 rows of the up half, so one M = 128 accumulator holds
//   gate (TMEM lanes 0..63) and up (lanes 64..127) of 64 output features for every
//   token of the tile. The four epilogue warps pass their lanes through a small
//   shared-memory tile so that one thread sees the gate and the up value of a feature,
//   and write the SwiGLU output h = silu(gate) * up in bf16.
// * down: 128 rows of W2, fp32 rows out (the weighted top-k combine follows).
//
// The z operand. The shrink writes z for sorted row j of pair (e, l) to row
// j + (e L + l + 1) * gap of a "shifted" z buffer, and zero rows in the `gap` rows
// before and after every pair it writes (gap >= the GEMM's token tile). A tile's rows
// [r0, r0 + BN) all belong to one expert and are ordered by adapter, so the one TMA
// box of BN rows at row r0 + (e L + l + 1) * gap returns z for exactly the tile's
// rows of adapter l and zeros for its other rows: the rows of other pairs map into
// the zero gaps around pair (e, l)'s own rows (a later pair's rows lie at least one
// gap further on, an earlier pair's one gap further back). No masking, no per-tile
// staging. Each z value is stored as two bf16 values (its rounding and the rounding
// of the remainder) that multiply the same bf16 B, which keeps the fp32 z to about
// 2^-16 relative, as the unfused expand does.
//
// Stage ring: STAGES slots of [W block | token rows]; a LoRA stage uses the same slot for
// [B block | z rows], its boxes only as wide as the rank (32-, 64- or 128-byte swizzled
// rows). Per job the producer issues the K/64 base stages, then the stages of every run
// of rows with an adapter in the tile; their MMAs stop at the run's last row. Warp roles
// (a TMA producer, one MMA-issuing thread, four epilogue warps), TMEM double buffering,
// bounded waits and the work decompositions (expert-major, per tile, persistent) follow
// the plain grouped GEMM; token-tile jobs go expert by expert, weight block by weight
// block over groups of the expert's tiles, so a weight block is read from memory about
// once. At 256-row tiles a cluster of two CTAs computes each job as one
// tcgen05.mma.cta_group::2 of M = 256 (kPair).
#include <algorithm>
#include <atomic>

#include "internal.h"

namespace moe_lora {

constexpr int kFBM = 128;  // weight rows per block (MMA M)
constexpr int kFBK = 64;   // K per stage
constexpr int kFusedThreads = 192;
constexpr int kFGroupTiles = 16;  // token tiles that share their weight blocks (<= 24 MB of rows)
constexpr int kFMaxExperts = 1024;
constexpr int kXStride = 17;  // floats per row of the gate/up exchange tile (conflict-free)
enum { kFModeTile = 0, kFModeExpert = 1, kFModePersistent = 2 };

// kPair: a cluster of two CTAs computes each job as one M = 256 tcgen05.mma.cta_group::2
// (CTA c: weight block 2 wbp + c, and half of the tile's token rows).
template <int BN, int STAGES, bool kGLU, bool kPair = false>
struct FusedCfg {
  static constexpr int kRowsPerCta = kPair ? BN / 2 : BN;  // token rows a CTA stages
  static constexpr int kWBytes = kFBM * kFBK * 2;
  static constexpr int kABytes = kRowsPerCta * kFBK * 2;
  static constexpr int kStageBytes = kWBytes + kABytes;
  static constexpr int kBarOff = STAGES * kStageBytes;
  static constexpr int kXOff = kBarOff + 256;  // gate/up exchange tile [128][kXStride] fp32
  static constexpr int kT0Off = kXOff + (kGLU ? kFBM * kXStride * 4 : 0);  // first tile per expert
  // expert-major launches take kSmemBytes (two CTAs an SM at the decode shapes); the token
  // tile modes add the first-tile table
  static constexpr int kSmemBytes = kT0Off + 1024;
  static constexpr int kSmemTiles = kSmemBytes + 4 * (kFMaxExperts + 8);
  static constexpr uint32_t kAccCols = BN < 32 ? 32 : BN;  // one fp32 accumulator
  static constexpr uint32_t kTmemCols = 2 * kAccCols;     // two, used alternately
  static_assert((2 * STAGES + 5) * 8 + 16 <= 256, "barrier area");
  static_assert(kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM allocation");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "token tile");
  static_assert(kABytes % 1024 == 0, "stage alignment");
  static_assert(kSmemTiles <= 227 * 1024, "shared memory");
  static_assert(!kPair || BN == 256, "CTA pairs take 256-row token tiles");
};

struct FusedArgs {
  int* hdr;
  const int4* tiles;
  const int* expert_begin;
  const int* row_adapter;
  void* out;        // kGLU: h [S, n_out] bf16; else [S, n_out] fp32 (sorted rows)
  int n_out;        // output features: I (kGLU) or N
  int up_off;       // kGLU: first row of the up half of W and B (= I)
  int K;            // reduction length of the base part
  int n_wblocks, max_tiles, mode, early;
  int ksplit;       // expert-major, down form: CTAs per (expert, weight block), each a
                    // contiguous share of the k-blocks writing its own partial output
  size_t part_stride;  // elements between the partial outputs
  int E, L, gap;    // z of sorted row j of pair (e, l) sits at row j + (e L + l + 1) gap
  int lora;         // 0: no adapter term (B and z maps unused)
  int zchunks;      // LoRA stages per run of an adapter in a tile
  int zk;           // > 0: one stage, z row = [high (zk K16 steps) | low (zk)]; 0: chunked
  int rp16;         // rank rounded up to a multiple of 16
  // LoRA tiles: columns per box of B and of z, and their shared-memory swizzle (descriptor
  // layout 2/4/6 for 128/64/32-byte rows, stride of 8 rows in bytes)
  int b_cols, z_cols;
  uint32_t b_layout, b_sbo, z_layout, z_sbo;
  unsigned long long wait_ns;
};

// The adapters of a job's rows (sorted by (e, l), so each adapter present is one run),
// loaded into registers when the job starts -- G groups of 32 rows, one value per lane --
// and walked when its LoRA stages come, so no warp waits on these loads at that point.
template <int G>
struct AdapterRows {
  int v[G];
  int rows;
  __device__ __forceinline__ void load(const int* row_adapter, int r0, int n) {
    const int lane = threadIdx.x & 31;
    rows = n;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int i = 32 * g + lane;
      v[g] = i < n ? __ldcg(row_adapter + r0 + i) : -1;
    }
  }
  // f(l, begin, end) for every run of rows [begin, end) with adapter l >= 0, in order.
  // Warp-wide: every lane calls f with the same arguments.
  template <typename F>
  __device__ __forceinline__ void for_each_run(F&& f) const {
    const int lane = threadIdx.x & 31;
    unsigned m[G];
    int carry = -1;  // adapter of the last row of the previous group (-1 before the first)
#pragma unroll
    for (int g = 0; g < G; ++g) {
      int prev = __shfl_up_sync(0xffffffffu, v[g], 1);
      if (lane == 0) prev = carry;
      m[g] = __ballot_sync(0xffffffffu, v[g] >= 0 && v[g] != prev);
      carry = __shfl_sync(0xffffffffu, v[g], 31);
    }
    // a run ends where the next one starts, or at the job's last row (rows without an
    // adapter come first in an expert's order, never after a run)
    int cur = -1, cur_l = -1;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      unsigned mm = m[g];
      while (mm) {
        const int b = __ffs(mm) - 1;
        mm &= mm - 1;
        const int l = __shfl_sync(0xffffffffu, v[g], b);
        if (cur >= 0) f(cur_l, cur, 32 * g + b);
        cur = 32 * g + b;
        cur_l = l;
      }
    }
    if (cur >= 0) f(cur_l, cur, rows);
  }
};

// The CTA's abort flag as lane 0 of the warp reads it: every lane of a warp that loops
// with warp-wide operations takes the same branch.
__device__ __forceinline__ bool warp_aborted(volatile int* flag) {
  const int v = (threadIdx.x & 31) == 0 ? *flag : 0;
  return __shfl_sync(0xffffffffu, v, 0) != 0;
}

// AND of a predicate over the `n` threads that meet at named barrier `id`.
__device__ __forceinline__ bool bar_and(uint32_t id, uint32_t n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void bar_sync(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

template <int BN, int STAGES, bool kGLU, bool kPair>
__global__ void __launch_bounds__(kFusedThreads, 1)
    fused_gemm_kernel(const __grid_constant__ CUtensorMap tm_w,
                      const __grid_constant__ CUtensorMap tm_a,
                      const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_z, const FusedArgs p) {
  using C = FusedCfg<BN, STAGES, kGLU, kPair>;
  // weight rows per output block: 64 gate + 64 up rows (kGLU) or 128 rows
  constexpr int kWR = kGLU ? kFBM / 2 : kFBM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* empty = full + STAGES;
  uint64_t* tmem_full = empty + STAGES;  // [2]: one per accumulator
  uint64_t* tmem_empty = tmem_full + 2;  // [2]
  uint64_t* mma_done = tmem_empty + 2;   // after an abort: every MMA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_job = reinterpret_cast<int*>(tmem_slot + 2);  // expert-major: first row, row count
  float* xt = reinterpret_cast<float*>(smem + C::kXOff);  // [128][kXStride] (kGLU)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool expert_major = p.mode == kFModeExpert;
  const bool persistent = p.mode == kFModePersistent;
  // A CTA pair (persistent mode only) walks its jobs as one unit: CTA c takes weight block
  // 2 wbp + c of job wbp, the leader (c = 0) issues the MMAs of both.
  const uint32_t crank = kPair ? cluster_ctarank() : 0u;
  const bool leader = crank == 0;
  const int unit = kPair ? (int)blockIdx.x / 2 : (int)blockIdx.x;
  const int nunits = kPair ? (int)gridDim.x / 2 : (int)gridDim.x;
  const int n_wblocks = kPair ? (p.n_wblocks + 1) / 2 : p.n_wblocks;  // weight jobs per tile
  // (token tile, weight block) jobs expert by expert, in groups of up to kFGroupTiles of the
  // expert's tiles taken weight block by weight block: the CTAs that share a weight block
  // run together and the group's token rows stay in L2, so each weight block is read from
  // memory about once. s_t0[e] = the first tile of expert e (the align cuts every expert's
  // rows into tiles of BN rows, in expert order); expert e's jobs are [s_t0[e] nwb,
  // s_t0[e + 1] nwb), so tile w / nwb is one of e's own.
  int* s_t0 = reinterpret_cast<int*>(smem + C::kT0Off);
  auto tile_job = [&](int w, int& e, int& wb, int& r0, int& rows) {
    const int ew = __ldcg(p.tiles + w / n_wblocks).x;
    const int t0 = s_t0[ew], nt = s_t0[ew + 1] - t0;
    const int u = w - t0 * n_wblocks;
    const int per_group = kFGroupTiles * n_wblocks;
    const int grp = u / per_group;
    const int first = grp * kFGroupTiles;
    const int gsz = min(kFGroupTiles, nt - first);
    const int within = u - grp * per_group;
    wb = within / gsz;
    if (kPair) wb = 2 * wb + (int)crank;
    const int4 tile = __ldcg(p.tiles + t0 + first + within % gsz);
    e = tile.x;
    r0 = tile.y;
    rows = tile.z;
  };

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 2);  // one arrival for the weight copies, one for the row copy
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tmem_full[a], 1);
      mbar_init(&tmem_empty[a], kPair ? 8 : 4);  // one arrival per epilogue warp (of both)
    }
    mbar_init(mma_done, 1);
    *s_abort = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_a);
    if (p.lora) {
      tma_prefetch_desc(&tm_b);
      tma_prefetch_desc(&tm_z);
    }
  }
  // the pair: each CTA's barriers are initialised before the other arrives on them
  if constexpr (kPair) cluster_sync();
  else __syncthreads();

  // Pair-aware pieces. Copies complete on the leader's full barrier (which the leader arms
  // for the bytes of both CTAs); waits acquire at cluster scope; an abort is mirrored into
  // the other CTA of the pair.
  auto full_bar = [&](int s) -> uint32_t {
    return kPair ? smem_in_cta(&full[s], 0) : smem_u32(&full[s]);
  };
  auto copy2d = [&](void* dst, const CUtensorMap* m, int s, int c0, int c1, uint64_t pol) {
    if constexpr (kPair) tma_load_2d_pair(dst, m, full_bar(s), c0, c1, pol);
    else tma_load_2d(dst, m, &full[s], c0, c1, pol);
  };
  auto copy3d = [&](void* dst, const CUtensorMap* m, int s, int c0, int c1, int c2, uint64_t pol) {
    if constexpr (kPair) tma_load_3d_pair(dst, m, full_bar(s), c0, c1, c2, pol);
    else tma_load_3d(dst, m, &full[s], c0, c1, c2, pol);
  };
  auto arm = [&](int s, uint32_t bytes_per_cta) {  // the leader arms for the whole pair
    if (leader) mbar_arrive_expect_tx(&full[s], kPair ? 2 * bytes_per_cta : bytes_per_cta);
  };
  auto wait_bar = [&](uint64_t* bar, uint32_t parity) -> bool {
    if constexpr (kPair) return mbar_wait_cluster(bar, parity, p.wait_ns);
    else return mbar_wait_bounded(bar, parity, p.wait_ns);
  };
  auto set_abort = [&]() {
    *s_abort = 1;
    if constexpr (kPair) st_cluster_u32(smem_in_cta((const void*)s_abort, crank ^ 1u), 1u);
  };

  // With `early`, everything but z was produced two or more launches back (the
  // predecessor, a shrink, triggers its dependents only after its own wait), so only
  // the first z copy waits for the predecessor; without it, every read waits.
  // Expert-major CTAs know their weights from their index: they stream the first ring of
  // weight stages before waiting in either case.
  int njobs, e0, wb0, r00 = 0, rows0 = 0, n_tiles = 0, ks = 0;
  if (!p.early && !expert_major) pdl_wait();
  if (expert_major) {
    const int jb = blockIdx.x / p.ksplit;
    ks = blockIdx.x - jb * p.ksplit;
    e0 = jb / n_wblocks;
    wb0 = jb - e0 * n_wblocks;
    njobs = -1;  // known once the expert's rows are read
  } else {
    n_tiles = __ldcg(p.hdr + HDR_NTILES);
    if (warp == 0) {  // s_t0: exclusive prefix of the experts' tile counts
      int carry = 0;
      for (int base = 0; base < p.E; base += 32) {
        const int e = base + lane;
        const int c = e < p.E ? (__ldcg(p.expert_begin + e + 1) - __ldcg(p.expert_begin + e) + BN - 1) / BN : 0;
        int v = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, v, off);
          if (lane >= off) v += y;
        }
        if (e < p.E) s_t0[e] = carry + v - c;
        carry += __shfl_sync(0xffffffffu, v, 31);
      }
      if (lane == 0) s_t0[p.E] = carry;
    }
    __syncthreads();
    const int total = n_tiles * n_wblocks;
    if (persistent) {
      njobs = unit < total ? (total - 1 - unit) / nunits + 1 : 0;
      if (njobs > 0) tile_job(unit, e0, wb0, r00, rows0);
    } else {
      njobs = (int)blockIdx.x < total ? 1 : 0;
      if (njobs) tile_job(blockIdx.x, e0, wb0, r00, rows0);
    }
    if (njobs == 0) {
      if (p.early) pdl_wait();  // a CTA leaves only once its predecessor has completed
      return;
    }
  }
  // this CTA's k-blocks: [kb0, kb0 + nk) (all of them unless the K range is split)
  const int nk_all = (p.K + kFBK - 1) / kFBK;
  const int kper = (nk_all + p.ksplit - 1) / p.ksplit;
  const int kb0 = ks * kper;
  const int nk = max(0, min(nk_all, kb0 + kper) - kb0);
  const bool lora = p.lora && ks == 0;  // the adapter term goes with the first K share
  void* const out = static_cast<char*>(p.out) + (size_t)ks * p.part_stride * (kGLU ? 2 : 4);
  const int pre = nk < STAGES ? nk : STAGES;

  if (warp == 1) {
    if constexpr (kPair) {  // one warp of each CTA of the pair
      tmem_alloc_pair(tmem_slot, C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, C::kTmemCols);
      tmem_relinquish();
    }
  }
  // Weight block wb of expert e into stage s: rows [wb kWR, +kWR) of the gate half and,
  // kGLU, of the up half (at up_off) below them -- one 128-row operand.
  auto load_w = [&](uint8_t* sw, int s, int kb, int wb, int e, uint64_t pol) {
    copy3d(sw, &tm_w, s, (kb0 + kb) * kFBK, wb * kWR, e, pol);
    if (kGLU) copy3d(sw + kWR * 128, &tm_w, s, (kb0 + kb) * kFBK, p.up_off + wb * kWR, e, pol);
  };
  // the first ring of weight stages of the first job (a weight never depends on a launch)
  if (threadIdx.x == 0) {
    const uint64_t pol_w = expert_major ? l2_policy_evict_first() : l2_policy_evict_normal();
    for (int kb = 0; kb < pre; ++kb) {
      arm(kb, C::kWBytes);
      load_w(smem + kb * C::kStageBytes, kb, kb, wb0, e0, pol_w);
    }
  }
  if (!p.early && expert_major) pdl_wait();  // every thread, after the weights went out
  if (threadIdx.x == 0) {
    if (!p.early) pdl_trigger();
    if (expert_major) {
      const int eb = __ldcg(p.expert_begin + e0), ee = __ldcg(p.expert_begin + e0 + 1);
      s_job[0] = eb;
      s_job[1] = ee - eb;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (expert_major) njobs = (s_job[1] + BN - 1) / BN;

  auto job = [&](int j, int& e, int& wb, int& r0, int& rows) {
    if (expert_major) {
      e = e0;
      wb = wb0;
      r0 = s_job[0] + j * BN;
      rows = min(BN, s_job[1] - j * BN);
    } else if (persistent && j > 0) {
      tile_job(unit + j * nunits, e, wb, r0, rows);
    } else {
      e = e0; wb = wb0; r0 = r00; rows = rows0;
    }
  };
  // A pair splits a job's token rows at half its MMA width nj (rows rounded up to 32):
  // CTA c stages rows [c nj / 2, c nj / 2 + 128) of the tile, and the MMA reads nj / 2 of
  // them from each CTA. One CTA: the MMA width follows the rows (16-row steps).
  auto job_n = [&](int rows) -> int { return kPair ? (rows + 31) & ~31 : (rows + 15) & ~15; };
  auto row_off = [&](int rows) -> int { return kPair ? (int)crank * (job_n(rows) / 2) : 0; };
  const int cph = p.zk ? 1 : p.zchunks / 2;  // chunked layout: stages per half (high, low)
  // bytes of one B row and of one z row in shared memory (their boxes' widths)
  const int b_row = p.b_cols * 2, z_row = p.z_cols * 2;

  bool waited0 = !p.early;  // thread 0 has passed griddepcontrol.wait
  int issued = 0;           // producer: stages whose row (or z) copy went out
  if (warp == 0) {
    // producer: the whole warp walks the jobs (the adapter runs are found warp-wide);
    // lane 0 issues the copies. Expert-major, a weight block is read by one CTA: it streams
    // through L2 marked to go first; token tiles share each weight block with the other
    // tiles of their group, which read it moments later.
    const uint64_t pol_w = expert_major ? l2_policy_evict_first() : l2_policy_evict_normal();
    const uint64_t pol_a = l2_policy_evict_last();
    int g = 0;
    if (njobs == 0 && lane == 0) {  // expert-major with no row: complete the prefetched stages
      for (int kb = 0; kb < pre; ++kb) mbar_arrive_expect_tx(&full[kb], 0);
      for (int kb = 0; kb < pre; ++kb) mbar_wait_bounded(&full[kb], 0);
    }  // (a pair always has jobs: persistent CTAs without one have left)
    for (int j = 0; j < njobs && !warp_aborted(s_abort); ++j) {
      int e, wb, r0, rows;
      job(j, e, wb, r0, rows);
      AdapterRows<(BN + 31) / 32> ar;
      if (lora) ar.load(p.row_adapter, r0, rows);
      // Every stage, base or adapter, takes the next ring index g: the job's K/64 base
      // stages, then its adapter stages (the accumulator was cleared by the first base
      // stage; placed last, they also give the predecessor that writes z the most time).
      for (int kb = 0; kb < nk; ++kb) {
        const int s = g % STAGES;
        const uint32_t ph = (g / STAGES) & 1;
        if (lane == 0) {
          uint8_t* sw = smem + s * C::kStageBytes;
          bool ok = !*s_abort;
          if (ok && g >= pre) {
            ok = wait_bar(&empty[s], ph ^ 1);
            if (ok) {
              arm(s, C::kWBytes);
              load_w(sw, s, kb, wb, e, pol_w);
            }
          }
          if (ok) {
            arm(s, C::kABytes);
            copy2d(sw + C::kWBytes, &tm_a, s, (kb0 + kb) * kFBK, r0 + row_off(rows), pol_a);
            ++issued;
          } else {
            set_abort();
          }
        }
        ++g;
        __syncwarp();
        if (warp_aborted(s_abort)) break;
      }
      if (!lora || warp_aborted(s_abort)) continue;
      if (!waited0) {  // z comes from the predecessor
        if (lane == 0) {
          pdl_wait();
          pdl_trigger();
        }
        waited0 = true;
      }
      ar.for_each_run([&](int l, int, int) {
        for (int c = 0; c < p.zchunks; ++c) {
          if (warp_aborted(s_abort)) return;
          const int s = g % STAGES;
          const uint32_t ph = (g / STAGES) & 1;
          if (lane == 0) {
            uint8_t* sw = smem + s * C::kStageBytes;
            if (wait_bar(&empty[s], ph ^ 1)) {
              const int bcol = 64 * (c % cph);
              const int pair = l * p.E + e;
              arm(s, (uint32_t)(kFBM * b_row));
              copy3d(sw, &tm_b, s, bcol, wb * kWR, pair, pol_w);
              if (kGLU) copy3d(sw + kWR * b_row, &tm_b, s, bcol, p.up_off + wb * kWR, pair, pol_w);
              arm(s, (uint32_t)(C::kRowsPerCta * z_row));
              copy2d(sw + C::kWBytes, &tm_z, s, 64 * c,
                     r0 + row_off(rows) + (e * p.L + l + 1) * p.gap, pol_a);
              ++issued;
            } else {
              set_abort();
            }
          }
          ++g;
          __syncwarp();
        }
      });
    }
  } else if (warp == 1 && leader) {
    // MMA issuer (lane 0); the warp walks the same jobs and adapter runs as the producer.
    // A pair's MMAs (M = 256 over both CTAs) and commits (to the barriers of both) are
    // issued by the leader alone.
    constexpr uint32_t kM = kPair ? 2 * kFBM : kFBM;
    auto mma = [&](uint32_t d, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t acc_in) {
      if constexpr (kPair) tc_mma_bf16_pair(d, a_desc, b_desc, idesc, acc_in);
      else tc_mma_bf16(d, a_desc, b_desc, idesc, acc_in);
    };
    auto commit = [&](uint64_t* bar) {
      if constexpr (kPair) tc_commit_pair_mc(bar);
      else tc_commit(bar);
    };
    int g = 0;
    for (int j = 0; j < njobs && !warp_aborted(s_abort); ++j) {
      int e, wb, r0, rows;
      job(j, e, wb, r0, rows);
      const int a = j & 1;
      const uint32_t acc = tmem + static_cast<uint32_t>(a * C::kAccCols);
      const uint32_t idesc = idesc_bf16_f32(kM, static_cast<uint32_t>(job_n(rows)));
      AdapterRows<(BN + 31) / 32> ar;
      if (lora) ar.load(p.row_adapter, r0, rows);
      if (lane == 0 && j >= 2) {  // the epilogue must have read this accumulator's last job
        if (!wait_bar(&tmem_empty[a], ((j >> 1) - 1) & 1)) set_abort();
        tc_fence_after();
      }
      __syncwarp();
      if (warp_aborted(s_abort)) break;
      for (int kb = 0; kb < nk; ++kb) {
        const int s = g % STAGES;
        const uint32_t ph = (g / STAGES) & 1;
        if (lane == 0) {
          if (!wait_bar(&full[s], ph)) {
            set_abort();
          } else {
            tc_fence_after();
            const uint8_t* sw = smem + s * C::kStageBytes;
            const uint64_t dw = smem_desc_sw128(smem_u32(sw));
            const uint64_t da = smem_desc_sw128(smem_u32(sw + C::kWBytes));
#pragma unroll
            for (int kk = 0; kk < kFBK / 16; ++kk)
              mma(acc, dw + 2 * kk, da + 2 * kk, idesc, (kb | kk) != 0);
            commit(&empty[s]);
          }
        }
        ++g;
        __syncwarp();
        if (warp_aborted(s_abort)) break;
      }
      if (lora && !warp_aborted(s_abort)) {
        ar.for_each_run([&](int, int, int end) {
          // the run's z rows are zero past its last row: the MMAs stop there (N = the run's
          // end rounded up to 16), the accumulator columns beyond are left as they are (a
          // pair keeps the job's width: its split of the rows between the CTAs follows it)
          const uint32_t idr =
              idesc_bf16_f32(kM, static_cast<uint32_t>(kPair ? job_n(rows) : (end + 15) & ~15));
          for (int c = 0; c < p.zchunks; ++c) {
            if (warp_aborted(s_abort)) return;
            const int s = g % STAGES;
            const uint32_t ph = (g / STAGES) & 1;
            if (lane == 0) {
              if (!wait_bar(&full[s], ph)) {
                set_abort();
              } else {
                tc_fence_after();
                const uint8_t* sw = smem + s * C::kStageBytes;
                const uint64_t db = smem_desc_swz(smem_u32(sw), p.b_layout, p.b_sbo);
                const uint64_t dz = smem_desc_swz(smem_u32(sw + C::kWBytes), p.z_layout, p.z_sbo);
                if (p.zk) {  // [high | low] in one row: both against the same B steps
                  for (int kk = 0; kk < p.zk; ++kk) {
                    mma(acc, db + 2 * kk, dz + 2 * kk, idr, 1);
                    mma(acc, db + 2 * kk, dz + 2 * (p.zk + kk), idr, 1);
                  }
                } else {  // chunk c of the high or the low half
                  const int rem = (p.rp16 - 64 * (c % cph)) / 16;
                  const int nm = rem < 4 ? rem : 4;
                  for (int kk = 0; kk < nm; ++kk) mma(acc, db + 2 * kk, dz + 2 * kk, idr, 1);
                }
                commit(&empty[s]);
              }
            }
            ++g;
            __syncwarp();
          }
        });
      }
      if (warp_aborted(s_abort)) break;
      if (lane == 0) commit(&tmem_full[a]);  // fires when every MMA issued above completes
      __syncwarp();
    }
  } else if (warp >= 2) {
    // epilogue: warp w reads TMEM lanes [32 (w % 4), 32 (w % 4) + 32), i.e. 32 rows of the
    // weight block, for every token of the job
    const int quad = warp & 3;
    bool waited = !p.early;
    for (int j = 0; j < njobs; ++j) {
      int e, wb, r0, rows;
      job(j, e, wb, r0, rows);
      const int a = j & 1;
      bool ok = __all_sync(0xffffffffu, wait_bar(&tmem_full[a], (j >> 1) & 1) ? 1 : 0);
      if (!ok && lane == 0) set_abort();
      ok = ok && !warp_aborted(s_abort);
      if (kGLU) ok = bar_and(1, 128, ok);  // the four warps meet at the exchange below
      if (!ok) break;
      tc_fence_after();
      if (!waited) {  // nothing is written before the predecessor has completed
        pdl_wait();
        waited = true;
      }
      const uint32_t taddr = tmem + static_cast<uint32_t>(a * C::kAccCols) +
                             (static_cast<uint32_t>(quad * 32) << 16);
      const uint32_t nmma = static_cast<uint32_t>((rows + 15) & ~15);
      if (kGLU) {
        // lanes 0..63 hold gate, 64..127 up of features f0 .. f0 + 63: every warp parks its
        // 32 rows x 16 tokens in the exchange tile, then thread t takes feature t % 64 for
        // 8 tokens (a warp stores 32 consecutive features of a token row)
        const int t = (warp - 2) * 32 + lane;  // 0..127 over the epilogue warps
        const int f = t & 63, tq = (t >> 6) * 8;
        const int n = wb * kWR + f;
        __nv_bfloat16* h = static_cast<__nv_bfloat16*>(out);
        for (uint32_t c0 = 0; c0 < nmma; c0 += 16) {
          uint32_t v[16];
          tmem_ld_x16(taddr + c0, v);
          tmem_ld_wait();
          float* xr = xt + (quad * 32 + lane) * kXStride;
#pragma unroll
          for (int q = 0; q < 16; ++q) xr[q] = __uint_as_float(v[q]);
          bar_sync(1, 128);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int tok = static_cast<int>(c0) + tq + q;
            const float gv = xt[f * kXStride + tq + q], uv = xt[(64 + f) * kXStride + tq + q];
            if (tok < rows && n < p.n_out)
              h[(size_t)(r0 + tok) * p.n_out + n] = __float2bfloat16_rn(silu_fast(gv) * uv);
          }
          bar_sync(1, 128);  // the tile is read before the next chunk overwrites it
        }
      } else {
        const int n = wb * kWR + quad * 32 + lane;
        float* o = static_cast<float*>(out);
        for (uint32_t c0 = 0; c0 < nmma; c0 += 16) {
          uint32_t v[16];
          tmem_ld_x16(taddr + c0, v);
          tmem_ld_wait();
          if (n < p.n_out) {
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const int tok = static_cast<int>(c0) + q;
              if (tok < rows) o[(size_t)(r0 + tok) * p.n_out + n] = __uint_as_float(v[q]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (kPair && !leader) mbar_arrive_remote(smem_in_cta(&tmem_empty[a], 0));
        else mbar_arrive(&tmem_empty[a]);
      }
    }
  }
  tc_fence_before();
  if constexpr (kPair) cluster_sync();
  else __syncthreads();
  // Past this barrier every role (of both CTAs of a pair) has stopped issuing and the
  // abort flag is final. After a give-up -- by any warp, possibly after another role had
  // already finished its loop -- copies may still be landing in shared memory and MMAs
  // still writing TMEM: both are drained before the CTA frees its tensor memory and exits
  // (these waits keep the full limit).
  const bool aborted = *s_abort != 0;
  if (!kPair && aborted && threadIdx.x == 0) {
    // prefetched weight stages whose row copy was never issued miss one arrival
    for (int kb = issued; kb < pre; ++kb) mbar_arrive_expect_tx(&full[kb], 0);
    for (int gg = (issued > pre ? issued : pre) - 1; gg >= 0 && gg >= issued - STAGES; --gg)
      mbar_wait_bounded(&full[gg % STAGES], (gg / STAGES) & 1);
  }
  if (kPair && aborted && threadIdx.x == 0) {
    // A pair's copies complete on the leader's barriers, armed for both CTAs' bytes: once
    // the two CTAs stopped at different stages no phase can be awaited exactly. Each
    // copy is at most a 32 KB box; 100 us is far beyond its flight time.
    const unsigned long long t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 100000ull) {
    }
  }
  if (aborted && threadIdx.x == 32 && leader) {
    if constexpr (kPair) tc_commit_pair(mma_done);  // once every MMA issued has completed
    else tc_commit(mma_done);
    mbar_wait_bounded(mma_done, 0);
  }
  if (threadIdx.x == 0) {
    if (aborted) set_dev_error(p.hdr, MOE_LORA_DEVERR_TIMEOUT);
    if (!waited0) pdl_wait();  // a CTA leaves only once its predecessor has completed
  }
  // a pair: the leader's MMAs into this CTA's TMEM and the other CTA's arrivals on this
  // CTA's barriers are over before either frees anything
  if constexpr (kPair) cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (kPair) tmem_dealloc_pair(tmem, C::kTmemCols);
    else tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------
template <int BN, int STAGES, bool kGLU, bool kPair = false>
static int launch_fused_t(const CUtensorMap& tw, const CUtensorMap& ta, const CUtensorMap& tb,
                          const CUtensorMap& tz, const FusedArgs& args, int E,
                          cudaStream_t stream, bool pdl) {
  using C = FusedCfg<BN, STAGES, kGLU, kPair>;
  auto kernel = fused_gemm_kernel<BN, STAGES, kGLU, kPair>;
  static std::atomic<uint64_t> configured[kMaxDevices];
  int st = once_per_context(configured, [] {
    ML_CHECK_CUDA(cudaFuncSetAttribute(fused_gemm_kernel<BN, STAGES, kGLU, kPair>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemTiles));
    return MOE_LORA_OK;
  });
  if (st != MOE_LORA_OK) return st;
  const int smem = args.mode == kFModeExpert ? C::kSmemBytes : C::kSmemTiles;
  if (kPair) {  // persistent CTA pairs: as many as can be resident at once
    if (args.mode != kFModePersistent) return MOE_LORA_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (unsigned)num_sms());
    cfg.blockDim = dim3(kFusedThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    ML_CHECK_CUDA(cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg));
    if (clusters < 1) return MOE_LORA_ERR_UNSUPPORTED;
    int64_t units = (int64_t)args.max_tiles * ((args.n_wblocks + 1) / 2);
    if (units > clusters) units = clusters;
    if (units < 1) units = 1;
    return launch_pdl_cluster(kernel, dim3(2 * (unsigned)units), kFusedThreads, smem,
                              stream, pdl, 2, tw, ta, tb, tz, args);
  }
  int64_t grid = (int64_t)(args.mode == kFModeExpert ? E * args.ksplit : args.max_tiles) *
                 args.n_wblocks;
  if (args.mode == kFModePersistent) {  // one resident CTA per SM slot, each looping over jobs
    int per_sm = 0;
    ML_CHECK_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kFusedThreads,
                                                                smem));
    const int64_t slots = (int64_t)num_sms() * (per_sm > 0 ? per_sm : 1);
    if (grid > slots) grid = slots;
  }
  if (grid > 0x7fffffff) return MOE_LORA_ERR_UNSUPPORTED;
  return launch_pdl(kernel, dim3((unsigned)grid), kFusedThreads, smem, stream, pdl, tw,
                    ta, tb, tz, args);
}

ZPadLayout zpad_layout(int S, int E, int L, int r, int gap) {
  ZPadLayout z = {};
  if (L <= 0 || r <= 0) return z;
  z.rp16 = (r + 15) / 16 * 16;
  if (z.rp16 <= 32) {  // one 64-column row: [high | low | unused]
    z.zw = 64;
    z.zk = z.rp16 / 16;
    z.zchunks = 1;
    z.lo_off = z.rp16;
  } else {  // high and low halves, each a whole number of 64-column chunks
    const int half = (z.rp16 + 63) / 64 * 64;
    z.zw = 2 * half;
    z.zk = 0;
    z.zchunks = 2 * (half / 64);
    z.lo_off = half;
  }
  z.gap = gap;
  z.rows = (int64_t)S + ((int64_t)E * L + 1) * gap;
  return z;
}

int launch_fused_gemm(const void* a_sorted, const void* W, const void* B, const void* zpad,
                      const ZPadLayout& zl, const moe_lora_align_t* al, const AlignLayout& a,
                      int N_w, int K, int r, bool glu, void* out, cudaStream_t stream, bool pdl,
                      bool early, int expert_major_bn, unsigned long long wait_ns, int ksplit,
                      bool pairs) {
  if (a.S == 0) return MOE_LORA_OK;
  // a split of the K range: expert-major down form only, at least two k-blocks a share
  if (ksplit < 1 || (ksplit > 1 && (glu || expert_major_bn == 0 || ceil_div(K, kFBK) < 2 * ksplit)))
    return MOE_LORA_ERR_UNSUPPORTED;
  AlignView v = align_view(al->buf, a);
  // rows per job: the expert-major chunk, else the align's token tile
  const int bn = expert_major_bn > 0 ? expert_major_bn : al->bm_base;
  const int mode = expert_major_bn > 0 ? kFModeExpert : bn >= 128 ? kFModePersistent : kFModeTile;
  const bool lora = al->L > 0 && B != nullptr && zpad != nullptr;
  if (lora && (zl.gap < bn || r % 8 != 0 || zl.rows >= (1ll << 31))) return MOE_LORA_ERR_UNSUPPORTED;
  if (mode != kFModeExpert && al->E > kFMaxExperts) return MOE_LORA_ERR_UNSUPPORTED;
  // 256-row token tiles: CTA pairs, each CTA staging 128 of the tile's rows
  const bool pair = pairs && mode == kFModePersistent && bn == 256;
  const uint32_t rows_per_cta = pair ? (uint32_t)bn / 2 : (uint32_t)bn;
  const int wrows = glu ? kFBM / 2 : kFBM;  // weight rows per box (gate and up halves: 64 each)
  CUtensorMap tw, ta, tb, tz;
  {
    const uint64_t dims[3] = {(uint64_t)K, (uint64_t)N_w, (uint64_t)al->E};
    const uint64_t strides[2] = {(uint64_t)K * 2, (uint64_t)N_w * K * 2};
    const uint32_t box[3] = {kFBK, (uint32_t)wrows, 1};
    int st = make_tmap_bf16(&tw, W, 3, dims, strides, box);
    if (st != MOE_LORA_OK) return st;
  }
  {  // the token rows in sorted order (a CTA of a pair stages half the tile's rows)
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)a.S};
    const uint64_t strides[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {kFBK, rows_per_cta};
    int st = make_tmap_bf16(&ta, a_sorted, 2, dims, strides, box);
    if (st != MOE_LORA_OK) return st;
  }
  // LoRA tiles only as wide as the rank needs: B of rank 16 or 32 in 32- or 64-byte rows,
  // z [high | low] of rank 16 or 32 in 64- or 128-byte rows; larger ranks in 64-column
  // chunks of 128-byte rows. The TMA engine writes every byte of a box (its out-of-range
  // part as zeros), so narrower boxes move less through shared memory.
  const int b_cols = zl.zk ? zl.rp16 : kFBK;
  const int z_cols = zl.zk ? 2 * zl.rp16 : kFBK;
  auto swz = [](int cols) {
    return cols == 16 ? CU_TENSOR_MAP_SWIZZLE_32B : cols == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                              : CU_TENSOR_MAP_SWIZZLE_128B;
  };
  auto layout = [](int cols) { return cols == 16 ? 6u : cols == 32 ? 4u : 2u; };
  if (lora) {
    const uint64_t dims[3] = {(uint64_t)r, (uint64_t)N_w, (uint64_t)al->L * al->E};
    const uint64_t strides[2] = {(uint64_t)r * 2, (uint64_t)N_w * r * 2};
    const uint32_t box[3] = {(uint32_t)b_cols, (uint32_t)wrows, 1};
    int st = make_tmap_bf16(&tb, B, 3, dims, strides, box, swz(b_cols));
    if (st != MOE_LORA_OK) return st;
    const uint64_t zdims[2] = {(uint64_t)zl.zw, (uint64_t)zl.rows};
    const uint64_t zstrides[1] = {(uint64_t)zl.zw * 2};
    const uint32_t zbox[2] = {(uint32_t)z_cols, rows_per_cta};
    st = make_tmap_bf16(&tz, zpad, 2, zdims, zstrides, zbox, swz(z_cols));
    if (st != MOE_LORA_OK) return st;
  } else {
    tb = tw;
    tz = ta;
  }
  FusedArgs args = {};
  args.hdr = v.hdr;
  args.tiles = v.tiles;
  args.expert_begin = v.expert_begin;
  args.row_adapter = v.row_adapter;
  args.out = out;
  args.n_out = glu ? N_w / 2 : N_w;
  args.up_off = glu ? N_w / 2 : 0;
  args.K = K;
  args.n_wblocks = ceil_div(args.n_out, wrows);
  args.max_tiles = a.max_tiles;
  args.mode = mode;
  args.ksplit = ksplit;
  args.part_stride = (size_t)a.S * (size_t)args.n_out;
  args.early = early ? 1 : 0;
  args.E = al->E;
  args.L = al->L;
  args.gap = zl.gap;
  args.lora = lora ? 1 : 0;
  args.zchunks = lora ? zl.zchunks : 0;
  args.zk = zl.zk;
  args.rp16 = zl.rp16;
  args.b_cols = b_cols;
  args.z_cols = z_cols;
  args.b_layout = layout(b_cols);
  args.b_sbo = 8u * (uint32_t)b_cols * 2u;
  args.z_layout = layout(z_cols);
  args.z_sbo = 8u * (uint32_t)z_cols * 2u;
  args.wait_ns = wait_ns;
  // stages: 192-200 KB of ring with one CTA per SM (128 and 256 rows), about 100 KB with
  // two (16 to 64 rows, the decode shapes)
  switch (bn) {
    case 16: return glu ? launch_fused_t<16, 6, true>(tw, ta, tb, tz, args, al->E, stream, pdl)
                        : launch_fused_t<16, 6, false>(tw, ta, tb, tz, args, al->E, stream, pdl);
    case 32: return glu ? launch_fused_t<32, 5, true>(tw, ta, tb, tz, args, al->E, stream, pdl)
                        : launch_fused_t<32, 5, false>(tw, ta, tb, tz, args, al->E, stream, pdl);
    case 64: return glu ? launch_fused_t<64, 4, true>(tw, ta, tb, tz, args, al->E, stream, pdl)
                        : launch_fused_t<64, 4, false>(tw, ta, tb, tz, args, al->E, stream, pdl);
    case 128: return glu ? launch_fused_t<128, 6, true>(tw, ta, tb, tz, args, al->E, stream, pdl)
                         : launch_fused_t<128, 6, false>(tw, ta, tb, tz, args, al->E, stream, pdl);
    case 256:
      if (pair)  // 32 KB stages: six in the ring
        return glu ? launch_fused_t<256, 6, true, true>(tw, ta, tb, tz, args, al->E, stream, pdl)
                   : launch_fused_t<256, 6, false, true>(tw, ta, tb, tz, args, al->E, stream, pdl);
      return glu ? launch_fused_t<256, 4, true>(tw, ta, tb, tz, args, al->E, stream, pdl)
                 : launch_fused_t<256, 4, false>(tw, ta, tb, tz, args, al->E, stream, pdl);
    default: return MOE_LORA_ERR_UNSUPPORTED;
  }
}

}  // namespace moe_lora
