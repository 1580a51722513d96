// Base expert grouped GEMM (vLLM's fused_moe group GEMM: one GEMM per expert over
// the tokens routed to it; vllm.com.cn, section "Implementing multi-LoRA
// inference for MoE models in vLLM") on the sm_103a tensor cores.
//
//   out[row, n] = sum_c a[row, c] * W[e(row), n, c]
//
// Design (GB300-first):
// * The weights take the MMA's M side: a CTA owns 128 consecutive rows of W_e
//   (output features) and one token tile of expert e (at most BN sorted rows) on
//   the N side. At decode an expert sees a handful of tokens, so N shrinks to a
//   multiple of 16 that covers the tile while the weight stream, which bounds
//   the kernel, stays full-width. At prefill the same tile is 128 x 256.
// * Operands are staged in shared memory by TMA (128-byte swizzle, K-major) in a
//   STAGES-deep mbarrier ring; one elected thread issues tcgen05.mma
//   (kind::f16, bf16 in, fp32 accumulate) into a TMEM accumulator of BN columns;
//   four epilogue warps read TMEM with tcgen05.ld and store fp32 rows.
// * The weight tensor map is 3-D [E][N][K], so weight rows past N read zeros;
//   K tails read zeros too (TMA out-of-bounds fill) -- no masks in the main loop.
// * Token tiles are ordered by expert and CTAs are rasterised in groups of
//   tiles so CTAs that share a weight block run together (L2 reuse).
// * Every mbarrier wait is bounded; on timeout the CTA records
//   MOE_LORA_DEVERR_TIMEOUT, drains its own copies and frees TMEM.
#include <atomic>
#include <mutex>

#include "internal.h"

namespace moe_lora {

constexpr int kBM = 128;  // weight rows per CTA (MMA M)
constexpr int kBK = 64;   // K per stage: one 128-byte swizzle row of bf16
constexpr int kGemmThreads = 192;
constexpr int kGroupTiles = 8;
enum { kModeTile = 0, kModeExpert = 1, kModePersistent = 2 };

template <int BN, int STAGES>
struct GemmCfg {
  static constexpr int kWBytes = kBM * kBK * 2;
  static constexpr int kABytes = BN * kBK * 2;
  static constexpr int kStageBytes = kWBytes + kABytes;
  static constexpr int kBarOff = STAGES * kStageBytes;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;  // barriers + alignment slack
  static_assert((2 * STAGES + 5) * 8 + 24 <= 256, "barrier area");
  static constexpr uint32_t kAccCols = BN < 32 ? 32 : BN;  // one fp32 accumulator
  static constexpr uint32_t kTmemCols = 2 * kAccCols;     // two, used alternately
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "token tile");
  static_assert(kABytes % 1024 == 0, "stage alignment");
};

// ----------------------------------------------------------------------------
// gather: xs[row] = x[token of sorted slot row]
// ----------------------------------------------------------------------------
constexpr int kGatherU = 4;  // 16-byte chunks per lane per row segment

template <bool kVec>
__global__ void __launch_bounds__(256) gather_rows_kernel(const __nv_bfloat16* __restrict__ x,
                                                          const int* __restrict__ hdr,
                                                          const int* __restrict__ sorted_slots,
                                                          int k, int H,
                                                          __nv_bfloat16* __restrict__ xs,
                                                          int trigger_first) {
  // trigger_first: the next launch reads nothing of the align step before its own
  // wait (the expert-major GEMM), so it may start streaming weights right away
  if (trigger_first) pdl_trigger();
  pdl_wait();
  const int n_valid = __ldcg(hdr + HDR_NVALID);
  if (!trigger_first) pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (kVec) {
    // A warp copies one segment of a row (32 x kGatherU 16-byte chunks): one slot lookup,
    // then every load of the segment before the first store, so a row costs two round
    // trips rather than one per 512 bytes, and rows x segments spread over the whole GPU.
    const int n8 = H / 8;
    const int segs = (n8 + 32 * kGatherU - 1) / (32 * kGatherU);
    const int64_t items = (int64_t)n_valid * segs;
    for (int64_t item = gw; item < items; item += warps) {
      const int row = (int)(item / segs), seg = (int)(item - (int64_t)row * segs);
      const int t = __ldcg(sorted_slots + row) / k;
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
      uint4* dst = reinterpret_cast<uint4*>(xs + (size_t)row * H);
      const int c0 = seg * 32 * kGatherU + lane;
      uint4 v[kGatherU];
#pragma unroll
      for (int u = 0; u < kGatherU; ++u)
        if (c0 + 32 * u < n8) v[u] = __ldcg(src + c0 + 32 * u);
#pragma unroll
      for (int u = 0; u < kGatherU; ++u)
        if (c0 + 32 * u < n8) dst[c0 + 32 * u] = v[u];
    }
  } else {
    for (int row = gw; row < n_valid; row += warps) {
      const int t = __ldcg(sorted_slots + row) / k;
      for (int c = lane; c < H; c += 32) xs[(size_t)row * H + c] = __ldcg(x + (size_t)t * H + c);
    }
  }
}

int launch_gather(const void* x, const moe_lora_align_t* al, const AlignLayout& a, int H, void* xs,
                  cudaStream_t stream, bool pdl, bool trigger_first) {
  if (a.S == 0) return MOE_LORA_OK;
  AlignView v = align_view(al->buf, a);
  const auto* xp = static_cast<const __nv_bfloat16*>(x);
  auto* xsp = static_cast<__nv_bfloat16*>(xs);
  const bool vec = H % 8 == 0 && aligned16(x) && aligned16(xs);
  // one warp per row segment (vector path) or per row, eight warps per CTA, at most
  // eight CTAs per SM
  const int segs = vec ? ceil_div(H / 8, 32 * kGatherU) : 1;
  const int64_t blocks = std::min<int64_t>(ceil_div64((int64_t)a.S * segs, 8), (int64_t)num_sms() * 8);
  if (vec)
    return launch_pdl(gather_rows_kernel<true>, (unsigned)blocks, 256, 0, stream, pdl, xp, v.hdr,
                      v.sorted_slots, al->k, H, xsp, trigger_first ? 1 : 0);
  return launch_pdl(gather_rows_kernel<false>, (unsigned)blocks, 256, 0, stream, pdl, xp, v.hdr,
                    v.sorted_slots, al->k, H, xsp, trigger_first ? 1 : 0);
}

// ----------------------------------------------------------------------------
// grouped GEMM kernel
// ----------------------------------------------------------------------------
template <int BN, int STAGES>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_w,
                        const __grid_constant__ CUtensorMap tm_a, int* __restrict__ hdr,
                        const int4* __restrict__ tiles, const int* __restrict__ expert_begin,
                        float* __restrict__ out, int N, int K, int n_wblocks, int max_tiles,
                        int mode, int early, unsigned long long wait_ns) {
  using C = GemmCfg<BN, STAGES>;
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
  int* s_issued = s_job + 2;  // the producer's count of stages whose token copy went out

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Work decomposition (see the mode constants): a job is one token chunk of one
  // expert against one 128-row weight block.
  //  kModeTile:       one job, (token tile, weight block) from blockIdx
  //  kModeExpert:     the expert's rows in chunks of BN against one weight block
  //  kModePersistent: jobs w = blockIdx.x, + gridDim.x, ... over every
  //                   (token tile, weight block) in grouped order
  const bool expert_major = mode == kModeExpert;
  const bool persistent = mode == kModePersistent;
  auto tile_job = [&](int w, int n_tiles, int& e, int& wb, int& r0, int& rows) {
    const int per_group = kGroupTiles * n_wblocks;
    const int grp = w / per_group;
    const int first = grp * kGroupTiles;
    const int gsz = min(kGroupTiles, n_tiles - first);
    const int within = w - grp * per_group;
    wb = within / gsz;
    const int4 tile = __ldcg(tiles + first + within % gsz);
    e = tile.x;
    r0 = tile.y;
    rows = tile.z;
  };

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 2);  // one arrival for the weight copy, one for the token copy
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
  }
  __syncthreads();

  // First job's expert and weight block. Tile modes with `early` read the tile table
  // (from the align launch, two or more launches back) before griddepcontrol.wait;
  // expert-major reads nothing of the align step before the wait.
  int njobs, e0, wb0, r00 = 0, rows0 = 0, n_tiles = 0;
  if (expert_major) {
    e0 = blockIdx.x / n_wblocks;
    wb0 = blockIdx.x - e0 * n_wblocks;
    njobs = -1;  // known after the wait
  } else {
    if (!early) pdl_wait();
    n_tiles = __ldcg(hdr + HDR_NTILES);
    const int total = n_tiles * n_wblocks;
    if (persistent) {
      njobs = blockIdx.x < total ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
      if (njobs > 0) tile_job(blockIdx.x, n_tiles, e0, wb0, r00, rows0);
    } else {
      // one job from the grouped mapping over the host's tile bound
      const int lin = blockIdx.x;
      const int per_group = kGroupTiles * n_wblocks;
      const int grp = lin / per_group;
      const int first = grp * kGroupTiles;
      const int gsz = min(kGroupTiles, max_tiles - first);
      const int within = lin - grp * per_group;
      wb0 = within / gsz;
      const int ti = first + within % gsz;
      njobs = ti < n_tiles ? 1 : 0;
      if (njobs) {
        const int4 tile = __ldcg(tiles + ti);
        e0 = tile.x;
        r00 = tile.y;
        rows0 = tile.z;
      }
    }
    if (njobs == 0) {
      if (early) pdl_wait();
      return;
    }
  }
  const int nk = (K + kBK - 1) / kBK;
  const int pre = nk < STAGES ? nk : STAGES;

  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  // the first ring of weight stages of the first job (a weight never depends on a launch)
  if (threadIdx.x == 0) {
    const uint64_t pol_w = l2_policy_evict_first();
    for (int kb = 0; kb < pre; ++kb) {
      mbar_arrive_expect_tx(&full[kb], C::kWBytes);
      tma_load_3d(smem + kb * C::kStageBytes, &tm_w, &full[kb], kb * kBK, wb0 * kBM, e0, pol_w);
    }
  }
  if (expert_major || early) pdl_wait();
  if (threadIdx.x == 0) {
    pdl_trigger();
    if (expert_major) {
      const int eb = __ldcg(expert_begin + e0), ee = __ldcg(expert_begin + e0 + 1);
      s_job[0] = eb;
      s_job[1] = ee - eb;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (expert_major) njobs = (s_job[1] + BN - 1) / BN;

  // job j -> expert, weight block, first row, rows
  auto job = [&](int j, int& e, int& wb, int& r0, int& rows) {
    if (expert_major) {
      e = e0;
      wb = wb0;
      r0 = s_job[0] + j * BN;
      rows = min(BN, s_job[1] - j * BN);
    } else if (persistent) {
      if (j == 0) {
        e = e0; wb = wb0; r0 = r00; rows = rows0;
      } else {
        tile_job(blockIdx.x + j * gridDim.x, n_tiles, e, wb, r0, rows);
      }
    } else {
      e = e0; wb = wb0; r0 = r00; rows = rows0;
    }
  };

  if (warp == 0) {
    if (lane == 0) {
      // producer: TMA ring over every k-block of every job
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_a = l2_policy_evict_last();
      int issued = 0;
      if (njobs == 0) {  // expert-major with no token: complete the prefetched stages, drain
        for (int kb = 0; kb < pre; ++kb) mbar_arrive_expect_tx(&full[kb], 0);
        for (int kb = 0; kb < pre; ++kb) mbar_wait_bounded(&full[kb], 0);
      }
      for (int j = 0; j < njobs && !*s_abort; ++j) {
        int e, wb, r0, rows;
        job(j, e, wb, r0, rows);
        for (int kb = 0; kb < nk; ++kb) {
          const int g = j * nk + kb;
          const int s = g % STAGES;
          const uint32_t ph = (g / STAGES) & 1;
          uint8_t* sw = smem + s * C::kStageBytes;
          if (g >= pre) {
            if (*s_abort || !mbar_wait_bounded(&empty[s], ph ^ 1, wait_ns)) {
              *s_abort = 1;
              break;
            }
            mbar_arrive_expect_tx(&full[s], C::kWBytes);
            tma_load_3d(sw, &tm_w, &full[s], kb * kBK, wb * kBM, e, pol_w);
          }
          mbar_arrive_expect_tx(&full[s], C::kABytes);
          tma_load_2d(sw + C::kWBytes, &tm_a, &full[s], kb * kBK, r0, pol_a);
          ++issued;
        }
      }
      s_issued[0] = issued;  // for the drain after the final barrier
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // MMA issuer: job j accumulates in buffer j % 2
      for (int j = 0; j < njobs && !*s_abort; ++j) {
        int e, wb, r0, rows;
        job(j, e, wb, r0, rows);
        const int a = j & 1;
        const uint32_t acc = tmem + static_cast<uint32_t>(a * C::kAccCols);
        const uint32_t idesc = idesc_bf16_f32(kBM, static_cast<uint32_t>((rows + 15) & ~15));
        if (j >= 2) {  // the epilogue must have read this buffer's previous job
          if (!mbar_wait_bounded(&tmem_empty[a], ((j >> 1) - 1) & 1, wait_ns)) {
            *s_abort = 1;
            break;
          }
          tc_fence_after();
        }
        for (int kb = 0; kb < nk; ++kb) {
          const int g = j * nk + kb;
          const int s = g % STAGES;
          const uint32_t ph = (g / STAGES) & 1;
          if (*s_abort || !mbar_wait_bounded(&full[s], ph, wait_ns)) {
            *s_abort = 1;
            break;
          }
          tc_fence_after();
          const uint8_t* sw = smem + s * C::kStageBytes;
          const uint64_t da = smem_desc_sw128(smem_u32(sw));
          const uint64_t db = smem_desc_sw128(smem_u32(sw + C::kWBytes));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            tc_mma_bf16(acc, da + 2 * kk, db + 2 * kk, idesc, (kb | kk) != 0);
          tc_commit(&empty[s]);
        }
        tc_commit(&tmem_full[a]);  // fires when every MMA issued above has completed
      }
    }
  } else {
    // epilogue: warp w may read TMEM lanes [32 (w % 4), 32 (w % 4) + 32)
    const int quad = warp & 3;
    for (int j = 0; j < njobs; ++j) {
      int e, wb, r0, rows;
      job(j, e, wb, r0, rows);
      const int a = j & 1;
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&tmem_full[a], (j >> 1) & 1, wait_ns) ? 1 : 0);
      if (!ok) *s_abort = 1;
      if (!ok || *s_abort) break;
      tc_fence_after();
      const int n = wb * kBM + quad * 32 + lane;
      const uint32_t taddr = tmem + static_cast<uint32_t>(a * C::kAccCols) +
                             (static_cast<uint32_t>(quad * 32) << 16);
      const uint32_t nmma = static_cast<uint32_t>((rows + 15) & ~15);
      for (uint32_t c0 = 0; c0 < nmma; c0 += 16) {
        uint32_t v[16];
        tmem_ld_x16(taddr + c0, v);
        tmem_ld_wait();
        if (n < N) {
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int tok = static_cast<int>(c0) + q;
            if (tok < rows) out[(size_t)(r0 + tok) * N + n] = __uint_as_float(v[q]);
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
  // Past this barrier every role has stopped issuing and the abort flag is final. After a
  // give-up -- by any warp, possibly after another role had already finished its loop --
  // copies may still be landing in shared memory and MMAs still writing TMEM: both are
  // drained before the CTA frees its tensor memory and exits (these waits keep the full
  // limit).
  const bool aborted = *s_abort != 0;
  if (aborted && threadIdx.x == 0) {
    const int issued = s_issued[0];
    // prefetched weight stages whose token copy was never issued miss one arrival
    for (int kb = issued; kb < pre; ++kb) mbar_arrive_expect_tx(&full[kb], 0);
    for (int g = (issued > pre ? issued : pre) - 1; g >= 0 && g >= issued - STAGES; --g)
      mbar_wait_bounded(&full[g % STAGES], (g / STAGES) & 1);
  }
  if (aborted && threadIdx.x == 32) {
    tc_commit(mma_done);  // arrives once every MMA this thread issued has completed
    mbar_wait_bounded(mma_done, 0);
  }
  if (threadIdx.x == 0 && aborted) set_dev_error(hdr, MOE_LORA_DEVERR_TIMEOUT);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// bf16 tensor map, innermost dimension K (contiguous), 128-byte swizzle, box {64, box_rows[, 1]}.
int make_tmap_bf16(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                   const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return MOE_LORA_ERR_CUDA;
  cuuint64_t gd[3], gs[2];
  cuuint32_t bd[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bd[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), gd, gs, bd,
                   es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_LORA_OK : MOE_LORA_ERR_CUDA;
}

template <int BN, int STAGES>
static int launch_gemm_t(const CUtensorMap& tw, const CUtensorMap& ta, const AlignView& v,
                         int max_tiles, int E, int N, int K, float* out, cudaStream_t stream,
                         bool pdl, int mode, int early, unsigned long long wait_ns) {
  using C = GemmCfg<BN, STAGES>;
  static std::atomic<uint64_t> configured[kMaxDevices];
  int st = once_per_context(configured, [] {
    ML_CHECK_CUDA(cudaFuncSetAttribute(grouped_gemm_kernel<BN, STAGES>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes));
    return MOE_LORA_OK;
  });
  if (st != MOE_LORA_OK) return st;
  const int n_wblocks = ceil_div(N, kBM);
  int64_t grid = (int64_t)(mode == kModeExpert ? E : max_tiles) * n_wblocks;
  if (mode == kModePersistent) {  // one resident CTA per SM slot, each looping over jobs
    int per_sm = 0;
    ML_CHECK_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &per_sm, grouped_gemm_kernel<BN, STAGES>, kGemmThreads, C::kSmemBytes));
    const int64_t slots = (int64_t)num_sms() * (per_sm > 0 ? per_sm : 1);
    if (grid > slots) grid = slots;
  }
  if (grid > 0x7fffffff) return MOE_LORA_ERR_UNSUPPORTED;
  return launch_pdl(grouped_gemm_kernel<BN, STAGES>, dim3((unsigned)grid), kGemmThreads,
                    C::kSmemBytes, stream, pdl, tw, ta, v.hdr, (const int4*)v.tiles,
                    (const int*)v.expert_begin, out, N, K, n_wblocks, max_tiles, mode, early,
                    wait_ns);
}

int launch_grouped_gemm_impl(const void* a_sorted, const void* W, const moe_lora_align_t* al,
                             const AlignLayout& a, int N, int K, float* out, cudaStream_t stream,
                             bool pdl, bool early, int expert_major_bn,
                             unsigned long long wait_ns) {
  if (a.S == 0) return MOE_LORA_OK;
  AlignView v = align_view(al->buf, a);
  // expert-major when asked; else persistent for large token tiles (prefill), whose
  // epilogue then overlaps the next job's main loop; else one job per CTA
  const int bn = expert_major_bn > 0 ? expert_major_bn : al->bm_base;
  const int em = expert_major_bn > 0 ? kModeExpert : bn >= 128 ? kModePersistent : kModeTile;
  const int ea = early ? 1 : 0;
  CUtensorMap tw, ta;
  {
    const uint64_t dims[3] = {(uint64_t)K, (uint64_t)N, (uint64_t)al->E};
    const uint64_t strides[2] = {(uint64_t)K * 2, (uint64_t)N * K * 2};
    const uint32_t box[3] = {kBK, kBM, 1};
    int st = make_tmap_bf16(&tw, W, 3, dims, strides, box);
    if (st != MOE_LORA_OK) return st;
  }
  {
    const uint64_t dims[2] = {(uint64_t)K, (uint64_t)a.S};
    const uint64_t strides[1] = {(uint64_t)K * 2};
    const uint32_t box[2] = {kBK, (uint32_t)bn};
    int st = make_tmap_bf16(&ta, a_sorted, 2, dims, strides, box);
    if (st != MOE_LORA_OK) return st;
  }
  switch (bn) {
    case 16: return launch_gemm_t<16, 6>(tw, ta, v, a.max_tiles, al->E, N, K, out, stream, pdl, em, ea, wait_ns);
    case 32: return launch_gemm_t<32, 5>(tw, ta, v, a.max_tiles, al->E, N, K, out, stream, pdl, em, ea, wait_ns);
    case 64: return launch_gemm_t<64, 4>(tw, ta, v, a.max_tiles, al->E, N, K, out, stream, pdl, em, ea, wait_ns);
    case 128: return launch_gemm_t<128, 6>(tw, ta, v, a.max_tiles, al->E, N, K, out, stream, pdl, em, ea, wait_ns);
    case 256: return launch_gemm_t<256, 4>(tw, ta, v, a.max_tiles, al->E, N, K, out, stream, pdl, em, ea, wait_ns);
    default: return MOE_LORA_ERR_UNSUPPORTED;
  }
}

int launch_grouped_gemm(const void* a_sorted, const void* W, const moe_lora_align_t* al,
                        const AlignLayout& a, int N, int K, float* out, cudaStream_t stream,
                        bool pdl) {
  return launch_grouped_gemm_impl(a_sorted, W, al, a, N, K, out, stream, pdl, false, 0);
}

}  // namespace moe_lora

extern "C" int moe_gather_rows(const void* x, const moe_lora_align_t* al, int H, void* xs,
                               moe_lora_stream_t stream) {
  using namespace moe_lora;
  AlignLayout a;
  int st = check_align(al, &a);
  if (st != MOE_LORA_OK) return st;
  if (H < 1 || (a.S > 0 && (!x || !xs))) return MOE_LORA_ERR_INVALID_ARG;
  if ((st = check_device()) != MOE_LORA_OK) return st;
  return launch_gather(x, al, a, H, xs, reinterpret_cast<cudaStream_t>(stream), true, false);
}

extern "C" int moe_grouped_gemm(const void* a_sorted, const void* W, const moe_lora_align_t* al,
                                int N, int K, float* out, moe_lora_stream_t stream) {
  using namespace moe_lora;
  AlignLayout a;
  int st = check_align(al, &a);
  if (st != MOE_LORA_OK) return st;
  if (N < 1 || K < 1) return MOE_LORA_ERR_INVALID_ARG;
  if (a.S > 0 && (!a_sorted || !W || !out)) return MOE_LORA_ERR_INVALID_ARG;
  if (a.S > 0 && (!aligned16(a_sorted) || !aligned16(W))) return MOE_LORA_ERR_INVALID_ARG;
  if (K % 8 != 0) return MOE_LORA_ERR_UNSUPPORTED;  // TMA row stride must be a multiple of 16 bytes
  if ((st = check_device()) != MOE_LORA_OK) return st;
  return launch_grouped_gemm(a_sorted, W, al, a, N, K, out, reinterpret_cast<cudaStream_t>(stream),
                             true);
}
