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
// * gate_up (kGLU): a CTA holds a 128-row block of the gate rows of W1 and the
//   matching 128-row block of the up rows in two TMEM accumulators and writes the
//   SwiGLU output h = silu(gate) * up in bf16 directly.
// * down: one accumulator, fp32 rows out (the weighted top-k combine follows).
//
// The z operand. The shrink writes z for sorted row j of pair (e, l) to row
// j + (e L + l + 1) * gap of a "shifted" z buffer, and zero rows in the `gap` rows
// before and after every pair it writes (gap = the GEMM's token tile). A tile's rows
// [r0, r0 + BN) all belong to one expert and are ordered by adapter, so the one TMA
// box of BN rows at row r0 + (e L + l + 1) * gap returns z for exactly the tile's
// rows of adapter l and zeros for its other rows: the rows of other pairs map into
// the zero gaps around pair (e, l)'s own rows (a later pair's rows lie at least one
// gap further on, an earlier pair's one gap further back). No masking, no per-tile
// staging. Each z value is stored as two bf16 values (its rounding and the rounding
// of the remainder) that multiply the same bf16 B, which keeps the fp32 z to about
// 2^-16 relative, as the unfused expand does.
//
// Stage ring: STAGES slots of [W (gate) | W (up, kGLU) | token rows]; a LoRA stage
// uses the same slots for [B (gate) | B (up) | z rows]. Per job the producer issues the
// K/64 base stages, then, for every run of rows with an adapter in the tile, the
// stages of that adapter's B and z. Warp roles, TMEM double buffering, bounded waits
// and the work decompositions (expert-major, per tile, persistent) follow the plain
// grouped GEMM.
#include <atomic>

#include "internal.h"

namespace moe_lora {

constexpr int kFBM = 128;  // weight rows per block (MMA M)
constexpr int kFBK = 64;   // K per stage
constexpr int kFusedThreads = 192;
constexpr int kFGroupTiles = 8;
enum { kFModeTile = 0, kFModeExpert = 1, kFModePersistent = 2 };

template <int BN, int STAGES, bool kGLU>
struct FusedCfg {
  static constexpr int kNW = kGLU ? 2 : 1;  // weight tiles per stage (gate and up)
  static constexpr int kWBytes = kFBM * kFBK * 2;
  static constexpr int kABytes = BN * kFBK * 2;
  static constexpr int kStageBytes = kNW * kWBytes + kABytes;
  static constexpr int kBarOff = STAGES * kStageBytes;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;  // barriers + alignment slack
  static constexpr uint32_t kAccCols = BN < 32 ? 32 : BN;   // one fp32 accumulator
  static constexpr uint32_t kSetCols = kNW * kAccCols;      // gate (+ up) of one job
  static constexpr uint32_t kTmemCols = 2 * kSetCols;       // two sets, used alternately
  static_assert((2 * STAGES + 5) * 8 + 16 <= 256, "barrier area");
  static_assert(kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM allocation");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "token tile");
  static_assert(kABytes % 1024 == 0, "stage alignment");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
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
  int E, L, gap;    // z of sorted row j of pair (e, l) sits at row j + (e L + l + 1) gap
  int lora;         // 0: no adapter term (B and z maps unused)
  int zchunks;      // LoRA stages per run of an adapter in a tile
  int zk;           // > 0: one stage, z row = [high (zk K16 steps) | low (zk)]; 0: chunked
  int rp16;         // rank rounded up to a multiple of 16
  unsigned long long wait_ns;
};

// Calls f(l) for every run of rows with an adapter (l >= 0) among sorted rows
// [r0, r0 + rows), in order. Rows of one expert are ordered by adapter, so each adapter
// present is one run. Warp-wide: every lane calls f with the same l.
template <typename F>
__device__ __forceinline__ void for_each_adapter_run(const int* row_adapter, int r0, int rows,
                                                     F&& f) {
  const int lane = threadIdx.x & 31;
  int carry = -1;  // adapter of the last row of the previous 32-row group (-1 at r0)
  for (int base = 0; base < rows; base += 32) {
    const int i = base + lane;
    const int l = i < rows ? __ldcg(row_adapter + r0 + i) : -1;
    int prev = __shfl_up_sync(0xffffffffu, l, 1);
    if (lane == 0) prev = carry;
    unsigned m = __ballot_sync(0xffffffffu, l >= 0 && l != prev);
    while (m) {
      const int b = __ffs(m) - 1;
      m &= m - 1;
      f(__shfl_sync(0xffffffffu, l, b));
    }
    carry = __shfl_sync(0xffffffffu, l, 31);
  }
}

// The CTA's abort flag as lane 0 of the warp reads it: every lane of a warp that loops
// with warp-wide operations takes the same branch.
__device__ __forceinline__ bool warp_aborted(volatile int* flag) {
  const int v = (threadIdx.x & 31) == 0 ? *flag : 0;
  return __shfl_sync(0xffffffffu, v, 0) != 0;
}

template <int BN, int STAGES, bool kGLU>
__global__ void __launch_bounds__(kFusedThreads, 1)
    fused_gemm_kernel(const __grid_constant__ CUtensorMap tm_w,
                      const __grid_constant__ CUtensorMap tm_a,
                      const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_z, const FusedArgs p) {
  using C = FusedCfg<BN, STAGES, kGLU>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* empty = full + STAGES;
  uint64_t* tmem_full = empty + STAGES;  // [2]: one per accumulator set
  uint64_t* tmem_empty = tmem_full + 2;  // [2]
  uint64_t* mma_done = tmem_empty + 2;   // after an abort: every MMA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_job = reinterpret_cast<int*>(tmem_slot + 2);  // expert-major: first row, row count

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool expert_major = p.mode == kFModeExpert;
  const bool persistent = p.mode == kFModePersistent;
  const int n_wblocks = p.n_wblocks;
  // (tile, weight block) jobs in groups of kFGroupTiles tiles, so that CTAs sharing a
  // weight block run together
  auto tile_job = [&](int w, int n_tiles, int& e, int& wb, int& r0, int& rows) {
    const int per_group = kFGroupTiles * n_wblocks;
    const int grp = w / per_group;
    const int first = grp * kFGroupTiles;
    const int gsz = min(kFGroupTiles, n_tiles - first);
    const int within = w - grp * per_group;
    wb = within / gsz;
    const int4 tile = __ldcg(p.tiles + first + within % gsz);
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
      mbar_init(&tmem_empty[a], 4);  // one arrival per epilogue warp
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
  __syncthreads();

  // With `early`, everything but z was produced two or more launches back (the
  // predecessor, a shrink, triggers its dependents only after its own wait), so only
  // the first z copy waits for the predecessor; without it, every read waits.
  int njobs, e0, wb0, r00 = 0, rows0 = 0, n_tiles = 0;
  if (!p.early) pdl_wait();
  if (expert_major) {
    e0 = blockIdx.x / n_wblocks;
    wb0 = blockIdx.x - e0 * n_wblocks;
    njobs = -1;  // known once the expert's rows are read
  } else {
    n_tiles = __ldcg(p.hdr + HDR_NTILES);
    const int total = n_tiles * n_wblocks;
    if (persistent) {
      njobs = blockIdx.x < total ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
      if (njobs > 0) tile_job(blockIdx.x, n_tiles, e0, wb0, r00, rows0);
    } else {
      const int lin = blockIdx.x;
      const int per_group = kFGroupTiles * n_wblocks;
      const int grp = lin / per_group;
      const int first = grp * kFGroupTiles;
      const int gsz = min(kFGroupTiles, p.max_tiles - first);
      const int within = lin - grp * per_group;
      wb0 = within / gsz;
      const int ti = first + within % gsz;
      njobs = ti < n_tiles ? 1 : 0;
      if (njobs) {
        const int4 tile = __ldcg(p.tiles + ti);
        e0 = tile.x;
        r00 = tile.y;
        rows0 = tile.z;
      }
    }
    if (njobs == 0) {
      if (p.early) pdl_wait();  // a CTA leaves only once its predecessor has completed
      return;
    }
  }
  const int nk = (p.K + kFBK - 1) / kFBK;
  const int pre = nk < STAGES ? nk : STAGES;

  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  // the first ring of weight stages of the first job (a weight never depends on a launch)
  if (threadIdx.x == 0) {
    const uint64_t pol_w = l2_policy_evict_first();
    for (int kb = 0; kb < pre; ++kb) {
      uint8_t* sw = smem + kb * C::kStageBytes;
      mbar_arrive_expect_tx(&full[kb], C::kNW * C::kWBytes);
      tma_load_3d(sw, &tm_w, &full[kb], kb * kFBK, wb0 * kFBM, e0, pol_w);
      if (kGLU) tma_load_3d(sw + C::kWBytes, &tm_w, &full[kb], kb * kFBK, p.up_off + wb0 * kFBM, e0, pol_w);
    }
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
      tile_job(blockIdx.x + j * gridDim.x, n_tiles, e, wb, r0, rows);
    } else {
      e = e0; wb = wb0; r0 = r00; rows = rows0;
    }
  };
  const int cph = p.zk ? 1 : p.zchunks / 2;  // chunked layout: stages per half (high, low)

  bool waited0 = !p.early;  // thread 0 has passed griddepcontrol.wait
  if (warp == 0) {
    // producer: the whole warp walks the jobs (the adapter runs are found warp-wide);
    // lane 0 issues the copies
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_a = l2_policy_evict_last();
    int g = 0, issued = 0;
    if (njobs == 0 && lane == 0) {  // expert-major with no row: complete the prefetched stages
      for (int kb = 0; kb < pre; ++kb) mbar_arrive_expect_tx(&full[kb], 0);
      for (int kb = 0; kb < pre; ++kb) mbar_wait_bounded(&full[kb], 0);
    }
    for (int j = 0; j < njobs && !warp_aborted(s_abort); ++j) {
      int e, wb, r0, rows;
      job(j, e, wb, r0, rows);
      for (int kb = 0; kb < nk; ++kb, ++g) {
        const int s = g % STAGES;
        const uint32_t ph = (g / STAGES) & 1;
        if (lane == 0) {
          uint8_t* sw = smem + s * C::kStageBytes;
          bool ok = !*s_abort;
          if (ok && g >= pre) {
            ok = mbar_wait_bounded(&empty[s], ph ^ 1, p.wait_ns);
            if (ok) {
              mbar_arrive_expect_tx(&full[s], C::kNW * C::kWBytes);
              tma_load_3d(sw, &tm_w, &full[s], kb * kFBK, wb * kFBM, e, pol_w);
              if (kGLU)
                tma_load_3d(sw + C::kWBytes, &tm_w, &full[s], kb * kFBK, p.up_off + wb * kFBM, e, pol_w);
            }
          }
          if (ok) {
            mbar_arrive_expect_tx(&full[s], C::kABytes);
            tma_load_2d(sw + C::kNW * C::kWBytes, &tm_a, &full[s], kb * kFBK, r0, pol_a);
            ++issued;
          } else {
            *s_abort = 1;
          }
        }
        __syncwarp();
        if (warp_aborted(s_abort)) break;
      }
      if (!p.lora || warp_aborted(s_abort)) continue;
      if (!waited0) {  // z comes from the predecessor
        if (lane == 0) {
          pdl_wait();
          pdl_trigger();
        }
        waited0 = true;
      }
      for_each_adapter_run(p.row_adapter, r0, rows, [&](int l) {
        for (int c = 0; c < p.zchunks; ++c, ++g) {
          if (warp_aborted(s_abort)) return;
          const int s = g % STAGES;
          const uint32_t ph = (g / STAGES) & 1;
          if (lane == 0) {
            uint8_t* sw = smem + s * C::kStageBytes;
            if (mbar_wait_bounded(&empty[s], ph ^ 1, p.wait_ns)) {
              const int bcol = 64 * (c % cph);
              const int pair = l * p.E + e;
              mbar_arrive_expect_tx(&full[s], C::kNW * C::kWBytes);
              tma_load_3d(sw, &tm_b, &full[s], bcol, wb * kFBM, pair, pol_w);
              if (kGLU) tma_load_3d(sw + C::kWBytes, &tm_b, &full[s], bcol, p.up_off + wb * kFBM, pair, pol_w);
              mbar_arrive_expect_tx(&full[s], C::kABytes);
              tma_load_2d(sw + C::kNW * C::kWBytes, &tm_z, &full[s], 64 * c,
                          r0 + (e * p.L + l + 1) * p.gap, pol_a);
              ++issued;
            } else {
              *s_abort = 1;
            }
          }
          __syncwarp();
        }
      });
    }
    if (lane == 0 && *s_abort) {  // drain own copies in flight before the CTA may exit
      // prefetched weight stages whose row copy was never issued miss one arrival
      for (int kb = issued; kb < pre; ++kb) mbar_arrive_expect_tx(&full[kb], 0);
      for (int gg = (issued > pre ? issued : pre) - 1; gg >= 0 && gg >= issued - STAGES; --gg)
        mbar_wait_bounded(&full[gg % STAGES], (gg / STAGES) & 1);
    }
  } else if (warp == 1) {
    // MMA issuer (lane 0); the warp walks the same jobs and adapter runs as the producer
    int g = 0;
    for (int j = 0; j < njobs && !warp_aborted(s_abort); ++j) {
      int e, wb, r0, rows;
      job(j, e, wb, r0, rows);
      const int a = j & 1;
      const uint32_t acc = tmem + static_cast<uint32_t>(a * C::kSetCols);
      const uint32_t idesc = idesc_bf16_f32(kFBM, static_cast<uint32_t>((rows + 15) & ~15));
      if (lane == 0 && j >= 2) {  // the epilogue must have read this set's previous job
        if (!mbar_wait_bounded(&tmem_empty[a], ((j >> 1) - 1) & 1, p.wait_ns)) *s_abort = 1;
        tc_fence_after();
      }
      __syncwarp();
      if (warp_aborted(s_abort)) break;
      for (int kb = 0; kb < nk; ++kb, ++g) {
        const int s = g % STAGES;
        const uint32_t ph = (g / STAGES) & 1;
        if (lane == 0) {
          if (!mbar_wait_bounded(&full[s], ph, p.wait_ns)) {
            *s_abort = 1;
          } else {
            tc_fence_after();
            const uint8_t* sw = smem + s * C::kStageBytes;
            const uint64_t dw = smem_desc_sw128(smem_u32(sw));
            const uint64_t da = smem_desc_sw128(smem_u32(sw + C::kNW * C::kWBytes));
#pragma unroll
            for (int kk = 0; kk < kFBK / 16; ++kk) {
              tc_mma_bf16(acc, dw + 2 * kk, da + 2 * kk, idesc, (kb | kk) != 0);
              if (kGLU) {
                const uint64_t du = smem_desc_sw128(smem_u32(sw + C::kWBytes));
                tc_mma_bf16(acc + C::kAccCols, du + 2 * kk, da + 2 * kk, idesc, (kb | kk) != 0);
              }
            }
            tc_commit(&empty[s]);
          }
        }
        __syncwarp();
        if (warp_aborted(s_abort)) break;
      }
      if (warp_aborted(s_abort)) break;
      if (p.lora) {
        for_each_adapter_run(p.row_adapter, r0, rows, [&](int l) {
          (void)l;
          for (int c = 0; c < p.zchunks; ++c, ++g) {
            if (warp_aborted(s_abort)) return;
            const int s = g % STAGES;
            const uint32_t ph = (g / STAGES) & 1;
            if (lane == 0) {
              if (!mbar_wait_bounded(&full[s], ph, p.wait_ns)) {
                *s_abort = 1;
              } else {
                tc_fence_after();
                const uint8_t* sw = smem + s * C::kStageBytes;
                const uint64_t db = smem_desc_sw128(smem_u32(sw));
                const uint64_t du = smem_desc_sw128(smem_u32(sw + C::kWBytes));
                const uint64_t dz = smem_desc_sw128(smem_u32(sw + C::kNW * C::kWBytes));
                if (p.zk) {  // [high | low] in one row: both against the same B steps
                  for (int kk = 0; kk < p.zk; ++kk) {
                    tc_mma_bf16(acc, db + 2 * kk, dz + 2 * kk, idesc, 1);
                    tc_mma_bf16(acc, db + 2 * kk, dz + 2 * (p.zk + kk), idesc, 1);
                    if (kGLU) {
                      tc_mma_bf16(acc + C::kAccCols, du + 2 * kk, dz + 2 * kk, idesc, 1);
                      tc_mma_bf16(acc + C::kAccCols, du + 2 * kk, dz + 2 * (p.zk + kk), idesc, 1);
                    }
                  }
                } else {  // chunk c of the high or the low half
                  const int rem = (p.rp16 - 64 * (c % cph)) / 16;
                  const int nm = rem < 4 ? rem : 4;
                  for (int kk = 0; kk < nm; ++kk) {
                    tc_mma_bf16(acc, db + 2 * kk, dz + 2 * kk, idesc, 1);
                    if (kGLU) tc_mma_bf16(acc + C::kAccCols, du + 2 * kk, dz + 2 * kk, idesc, 1);
                  }
                }
                tc_commit(&empty[s]);
              }
            }
            __syncwarp();
          }
        });
      }
      if (warp_aborted(s_abort)) break;
      if (lane == 0) tc_commit(&tmem_full[a]);  // fires when every MMA issued above completes
      __syncwarp();
    }
    if (lane == 0 && *s_abort) {  // MMAs still in flight read shared memory and write TMEM
      tc_commit(mma_done);
      mbar_wait_bounded(mma_done, 0);
    }
  } else {
    // epilogue: warp w reads TMEM lanes [32 (w % 4), 32 (w % 4) + 32), i.e. 32 output
    // features, for every row of the job
    const int quad = warp & 3;
    bool waited = !p.early;
    for (int j = 0; j < njobs; ++j) {
      int e, wb, r0, rows;
      job(j, e, wb, r0, rows);
      const int a = j & 1;
      const bool ok =
          __all_sync(0xffffffffu, mbar_wait_bounded(&tmem_full[a], (j >> 1) & 1, p.wait_ns) ? 1 : 0);
      if (!ok) *s_abort = 1;
      if (!ok || warp_aborted(s_abort)) break;
      tc_fence_after();
      if (!waited) {  // nothing is written before the predecessor has completed
        pdl_wait();
        waited = true;
      }
      const int n = wb * kFBM + quad * 32 + lane;
      const uint32_t taddr = tmem + static_cast<uint32_t>(a * C::kSetCols) +
                             (static_cast<uint32_t>(quad * 32) << 16);
      const uint32_t nmma = static_cast<uint32_t>((rows + 15) & ~15);
      for (uint32_t c0 = 0; c0 < nmma; c0 += 16) {
        uint32_t v[16];
        tmem_ld_x16(taddr + c0, v);
        if (kGLU) {
          uint32_t u[16];
          tmem_ld_x16(taddr + C::kAccCols + c0, u);
          tmem_ld_wait();
          if (n < p.n_out) {
            __nv_bfloat16* h = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const int tok = static_cast<int>(c0) + q;
              if (tok < rows)
                h[(size_t)(r0 + tok) * p.n_out + n] =
                    __float2bfloat16_rn(silu_fast(__uint_as_float(v[q])) * __uint_as_float(u[q]));
            }
          }
        } else {
          tmem_ld_wait();
          if (n < p.n_out) {
            float* o = static_cast<float*>(p.out);
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
      if (lane == 0) mbar_arrive(&tmem_empty[a]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    if (*s_abort) set_dev_error(p.hdr, MOE_LORA_DEVERR_TIMEOUT);
    if (!waited0) pdl_wait();  // a CTA leaves only once its predecessor has completed
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------
template <int BN, int STAGES, bool kGLU>
static int launch_fused_t(const CUtensorMap& tw, const CUtensorMap& ta, const CUtensorMap& tb,
                          const CUtensorMap& tz, const FusedArgs& args, int E,
                          cudaStream_t stream, bool pdl) {
  using C = FusedCfg<BN, STAGES, kGLU>;
  static std::atomic<uint64_t> configured[kMaxDevices];
  int st = once_per_context(configured, [] {
    ML_CHECK_CUDA(cudaFuncSetAttribute(fused_gemm_kernel<BN, STAGES, kGLU>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes));
    return MOE_LORA_OK;
  });
  if (st != MOE_LORA_OK) return st;
  int64_t grid = (int64_t)(args.mode == kFModeExpert ? E : args.max_tiles) * args.n_wblocks;
  if (args.mode == kFModePersistent) {  // one resident CTA per SM slot, each looping over jobs
    int per_sm = 0;
    ML_CHECK_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, fused_gemm_kernel<BN, STAGES, kGLU>, kFusedThreads, C::kSmemBytes));
    const int64_t slots = (int64_t)num_sms() * (per_sm > 0 ? per_sm : 1);
    if (grid > slots) grid = slots;
  }
  if (grid > 0x7fffffff) return MOE_LORA_ERR_UNSUPPORTED;
  return launch_pdl(fused_gemm_kernel<BN, STAGES, kGLU>, dim3((unsigned)grid), kFusedThreads,
                    C::kSmemBytes, stream, pdl, tw, ta, tb, tz, args);
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
                      bool early, int expert_major_bn, unsigned long long wait_ns) {
  if (a.S == 0) return MOE_LORA_OK;
  AlignView v = align_view(al->buf, a);
  const int bn = expert_major_bn > 0 ? expert_major_bn : al->bm_base;
  const int mode = expert_major_bn > 0 ? kFModeExpert : bn >= 128 ? kFModePersistent : kFModeTile;
  const bool lora = al->L > 0 && B != nullptr && zpad != nullptr;
  if (lora && (zl.gap < bn || r % 8 != 0 || zl.rows >= (1ll << 31))) return MOE_LORA_ERR_UNSUPPORTED;
  CUtensorMap tw, ta, tb, tz;
  {
    const uint64_t dims[3] = {(uint64_t)K, (uint64_t)N_w, (uint64_t)al->E};
    const uint64_t strides[2] = {(uint64_t)K * 2, (uint64_t)N_w * K * 2};
    const uint32_t box[3] = {kFBK, kFBM, 1};
    int st = make_tmap_bf16(&tw, W, 3, dims, strides, box);
    if (st != MOE_LORA_OK) return st;
  }
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)a.S};
    const uint64_t strides[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {kFBK, (uint32_t)bn};
    int st = make_tmap_bf16(&ta, a_sorted, 2, dims, strides, box);
    if (st != MOE_LORA_OK) return st;
  }
  if (lora) {
    const uint64_t dims[3] = {(uint64_t)r, (uint64_t)N_w, (uint64_t)al->L * al->E};
    const uint64_t strides[2] = {(uint64_t)r * 2, (uint64_t)N_w * r * 2};
    const uint32_t box[3] = {kFBK, kFBM, 1};
    int st = make_tmap_bf16(&tb, B, 3, dims, strides, box);
    if (st != MOE_LORA_OK) return st;
    const uint64_t zdims[2] = {(uint64_t)zl.zw, (uint64_t)zl.rows};
    const uint64_t zstrides[1] = {(uint64_t)zl.zw * 2};
    const uint32_t zbox[2] = {kFBK, (uint32_t)bn};
    st = make_tmap_bf16(&tz, zpad, 2, zdims, zstrides, zbox);
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
  args.n_wblocks = ceil_div(args.n_out, kFBM);
  args.max_tiles = a.max_tiles;
  args.mode = mode;
  args.early = early ? 1 : 0;
  args.E = al->E;
  args.L = al->L;
  args.gap = zl.gap;
  args.lora = lora ? 1 : 0;
  args.zchunks = lora ? zl.zchunks : 0;
  args.zk = zl.zk;
  args.rp16 = zl.rp16;
  args.wait_ns = wait_ns;
  if (glu) {
    switch (bn) {
      case 16: return launch_fused_t<16, 5, true>(tw, ta, tb, tz, args, al->E, stream, pdl);
      case 32: return launch_fused_t<32, 5, true>(tw, ta, tb, tz, args, al->E, stream, pdl);
      case 64: return launch_fused_t<64, 4, true>(tw, ta, tb, tz, args, al->E, stream, pdl);
      case 128: return launch_fused_t<128, 4, true>(tw, ta, tb, tz, args, al->E, stream, pdl);
      default: return MOE_LORA_ERR_UNSUPPORTED;
    }
  }
  switch (bn) {
    case 16: return launch_fused_t<16, 6, false>(tw, ta, tb, tz, args, al->E, stream, pdl);
    case 32: return launch_fused_t<32, 5, false>(tw, ta, tb, tz, args, al->E, stream, pdl);
    case 64: return launch_fused_t<64, 4, false>(tw, ta, tb, tz, args, al->E, stream, pdl);
    case 128: return launch_fused_t<128, 6, false>(tw, ta, tb, tz, args, al->E, stream, pdl);
    default: return MOE_LORA_ERR_UNSUPPORTED;
  }
}

}  // namespace moe_lora
