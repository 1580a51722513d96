// Shared helpers of the MoE-LoRA kernels: status plumbing, PDL launches, and thin
// inline-PTX wrappers for mbarrier, TMA bulk tensor copies and tcgen05 (5th-gen
// tensor cores with tensor-memory accumulators) on sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "../../include/moe_lora.h"

namespace moe_lora {

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------
#define ML_CHECK_CUDA(expr)                              \
  do {                                                   \
    cudaError_t _e = (expr);                             \
    if (_e != cudaSuccess) return MOE_LORA_ERR_CUDA;     \
  } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
inline int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Checks once per device that it is an sm_103 part (the only target compiled).
int check_device();
int num_sms();

// An id of the CUDA context current on this thread; it changes when the primary
// context is destroyed and re-created (cudaDeviceReset), so state that belongs to a
// context -- function attributes, the device address of a __device__ array -- is
// cached per (device, context id). 0 when no context is current or the id cannot be
// read.
uint64_t current_context_id();

constexpr int kMaxDevices = 64;

// Runs `set` (which returns a status) unless it already succeeded in the current
// context of the current device; `seen` holds, per device, the context id it last
// succeeded in. Concurrent first calls may both run `set`: it must be idempotent.
template <typename F>
inline int once_per_context(std::atomic<uint64_t> (&seen)[kMaxDevices], F&& set) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_LORA_ERR_CUDA;
  const uint64_t id = current_context_id();
  const bool cache = dev >= 0 && dev < kMaxDevices && id != 0;
  if (cache && seen[dev].load(std::memory_order_acquire) == id) return MOE_LORA_OK;
  const int st = set();
  if (st == MOE_LORA_OK && cache) seen[dev].store(id, std::memory_order_release);
  return st;
}

// Launch with programmatic dependent launch (the kernel may start while its
// predecessor on the stream drains; it must call pdl_wait() before touching
// the predecessor's outputs).
template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t stream, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  return e == cudaSuccess ? MOE_LORA_OK : MOE_LORA_ERR_CUDA;
}

// The same launch in clusters of `cluster_x` CTAs along x (grid.x a multiple of it).
template <typename... KArgs, typename... Args>
inline int launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, bool pdl, int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  return e == cudaSuccess ? MOE_LORA_OK : MOE_LORA_ERR_CUDA;
}

// ----------------------------------------------------------------------------
// align buffer layout (host and device agree through this one function)
// ----------------------------------------------------------------------------
struct AlignLayout {
  int64_t off[MOE_LORA_ALIGN_NFIELDS];
  int S, max_tiles, max_blocks, nbuckets, key_bits, slot_bits;
  int64_t off_bucket_count, off_bucket_start, off_sort0, off_sort1, off_counts;
  int ctas;  // CTAs of the multi-CTA align (kAlignChunk slots each); 0: one-CTA align
  bool valid;
};

// Multi-CTA align: from kAlignMultiMin slots on, with at most half as many buckets as
// slots (else the (bucket, CTA) count table, not the sort, is the work) and the table
// within kAlignMaxCounts entries.
constexpr int kAlignChunk = 512;
constexpr int kAlignMultiMin = 2048;
constexpr int64_t kAlignMaxCounts = 1 << 22;

// header word indices
enum { HDR_ERR = 0, HDR_NVALID = 1, HDR_NTILES = 2, HDR_NBLOCKS = 3, HDR_NLORAROWS = 4,
       HDR_T = 5, HDR_K = 6, HDR_E = 7, HDR_L = 8, HDR_BMB = 9, HDR_BML = 10 };
constexpr int kHeaderInts = 64;
constexpr uint32_t kMaxSlots = 1u << 22;

inline int bits_for(uint64_t v) {  // bits needed to represent values 0..v
  int b = 0;
  while ((1ull << b) <= v) ++b;
  return b == 0 ? 1 : b;
}

inline AlignLayout align_layout(int T, int k, int E, int L, int bm_base, int bm_lora) {
  AlignLayout a = {};
  a.valid = false;
  if (T < 0 || k < 1 || E < 1 || L < 0 || bm_base < 16 || bm_base > 256 || bm_base % 16 != 0 ||
      bm_lora < 1 || bm_lora > 16)
    return a;
  int64_t S64 = (int64_t)T * k;
  if (S64 > (int64_t)kMaxSlots) return a;
  int S = (int)S64;
  int64_t nb = (int64_t)E * (L + 1) + 1;  // buckets incl. one for dropped slots
  if (nb >= (1ll << 30)) return a;
  a.slot_bits = bits_for(S > 0 ? S - 1 : 0);
  a.key_bits = bits_for(nb - 1);
  if (a.slot_bits + a.key_bits > 32) return a;
  a.S = S;
  a.nbuckets = (int)nb;
  a.max_tiles = S / bm_base + (E < S ? E : S) + 1;
  int64_t mb = (int64_t)S / bm_lora + ((int64_t)E * L < S ? (int64_t)E * L : S) + 1;
  a.max_blocks = (int)(mb < S + 1 ? mb : S + 1);
  int64_t o = 0;
  auto take = [&](int64_t bytes) { int64_t r = o; o = (int64_t)round_up(o + bytes, 256); return r; };
  a.off[MOE_LORA_AF_HEADER] = take(kHeaderInts * 4);
  a.off[MOE_LORA_AF_SORTED_SLOTS] = take((int64_t)S * 4);
  a.off[MOE_LORA_AF_SLOT_ROW] = take((int64_t)S * 4);
  a.off[MOE_LORA_AF_ROW_EXPERT] = take((int64_t)S * 4);
  a.off[MOE_LORA_AF_ROW_ADAPTER] = take((int64_t)S * 4);
  a.off[MOE_LORA_AF_EXPERT_BEGIN] = take((int64_t)(E + 1) * 4);
  a.off[MOE_LORA_AF_TILES] = take((int64_t)a.max_tiles * 16);
  a.off[MOE_LORA_AF_LORA_BLOCKS] = take((int64_t)a.max_blocks * 16);
  a.off[MOE_LORA_AF_MAX_TILES] = a.max_tiles;
  a.off[MOE_LORA_AF_MAX_LORA_BLOCKS] = a.max_blocks;
  a.off[MOE_LORA_AF_SCRATCH] = o;
  a.off_bucket_count = take(nb * 4);
  a.off_bucket_start = take(nb * 4);
  a.off_sort0 = take((int64_t)S * 4);
  a.off_sort1 = take((int64_t)S * 4);
  const int64_t ctas = ((int64_t)S + kAlignChunk - 1) / kAlignChunk;
  a.ctas = (S >= kAlignMultiMin && 2 * nb <= S && nb * ctas <= kAlignMaxCounts) ? (int)ctas : 0;
  a.off_counts = take(a.ctas ? nb * ctas * 4 : 0);
  a.off[MOE_LORA_AF_TOTAL_BYTES] = o;
  a.valid = true;
  return a;
}

// Device-side view of an align buffer.
struct AlignView {
  int* hdr;
  int* sorted_slots;
  int* slot_row;
  int* row_expert;
  int* row_adapter;
  int* expert_begin;
  int4* tiles;
  int4* blocks;
  int* bucket_count;
  int* bucket_start;
  uint32_t* sort0;
  uint32_t* sort1;
  int* counts;  // [ctas][nbuckets] of the multi-CTA align
};

inline AlignView align_view(void* buf, const AlignLayout& a) {
  char* b = static_cast<char*>(buf);
  AlignView v;
  v.hdr = reinterpret_cast<int*>(b + a.off[MOE_LORA_AF_HEADER]);
  v.sorted_slots = reinterpret_cast<int*>(b + a.off[MOE_LORA_AF_SORTED_SLOTS]);
  v.slot_row = reinterpret_cast<int*>(b + a.off[MOE_LORA_AF_SLOT_ROW]);
  v.row_expert = reinterpret_cast<int*>(b + a.off[MOE_LORA_AF_ROW_EXPERT]);
  v.row_adapter = reinterpret_cast<int*>(b + a.off[MOE_LORA_AF_ROW_ADAPTER]);
  v.expert_begin = reinterpret_cast<int*>(b + a.off[MOE_LORA_AF_EXPERT_BEGIN]);
  v.tiles = reinterpret_cast<int4*>(b + a.off[MOE_LORA_AF_TILES]);
  v.blocks = reinterpret_cast<int4*>(b + a.off[MOE_LORA_AF_LORA_BLOCKS]);
  v.bucket_count = reinterpret_cast<int*>(b + a.off_bucket_count);
  v.bucket_start = reinterpret_cast<int*>(b + a.off_bucket_start);
  v.sort0 = reinterpret_cast<uint32_t*>(b + a.off_sort0);
  v.sort1 = reinterpret_cast<uint32_t*>(b + a.off_sort1);
  v.counts = reinterpret_cast<int*>(b + a.off_counts);
  return v;
}

// Validates a moe_lora_align_t and computes its layout.
inline int check_align(const moe_lora_align_t* al, AlignLayout* out) {
  if (!al || !al->buf) return MOE_LORA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(al->buf) & 255u) != 0) return MOE_LORA_ERR_INVALID_ARG;
  AlignLayout a = align_layout(al->T, al->k, al->E, al->L, al->bm_base, al->bm_lora);
  if (!a.valid) return MOE_LORA_ERR_UNSUPPORTED;
  *out = a;
  return MOE_LORA_OK;
}

// ----------------------------------------------------------------------------
// device side
// ----------------------------------------------------------------------------
// Bounded waits give up after this much wall time and report
// MOE_LORA_DEVERR_TIMEOUT instead of spinning forever.
constexpr unsigned long long kWaitLimitNs = 4000000000ull;

// Under programmatic dependent launch a kernel is already running while earlier
// launches write their results. Everything produced by an earlier launch is
// therefore read with ld.global.cg (__ldcg, coherent at L2) or through TMA, never
// through the read-only path (__ldg / const __restrict__ loads), whose contents
// may be stale; only weights and caller inputs take the read-only path.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void set_dev_error(int* hdr, uint32_t bits) {
  atomicOr(reinterpret_cast<unsigned int*>(hdr + HDR_ERR), bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier ----
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return done;
}
// Waits for the phase of `parity` to complete; false once `limit_ns` of wall time has
// passed. limit_ns == 0 gives up at the first unsuccessful poll (a test of the give-up
// paths uses it; the layer passes the default).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  if (limit_ns == 0) return false;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(a, parity)) return true;
    if ((it & 255u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
  }
}

// Pulls `bytes` (a multiple of 16, 16-byte aligned) of global memory into L2 without
// waiting for it (the bulk-copy engine's prefetch; a hint, nothing to complete).
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)),
               "r"(bytes)
               : "memory");
}

// ---- TMA (bulk tensor copies global -> shared, completion on an mbarrier) ----
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0,
                                            int c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int c0,
                                            int c1, int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---- tcgen05 ----
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives on `bar` once all previously issued tcgen05.mma of this thread complete.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns; lane i of the warp gets TMEM lane (base+i).
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major bf16 tile written by TMA with
// 128-byte swizzling: rows of 128 bytes (64 elements), 8-row atoms 1024 bytes
// apart (stride byte offset), tile base 1024-byte aligned. Layout: start address
// >> 4 in bits [0,14), leading byte offset >> 4 in [16,30) (unused for swizzled
// K-major, set to 1), stride byte offset >> 4 in [32,46), the fixed value 1 in
// [46,48), swizzle mode 2 (128B) in [61,64).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1u << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// The same descriptor for the other swizzle widths of a K-major bf16 tile: layout 2
// (128-byte rows), 4 (64-byte rows) or 6 (32-byte rows); stride byte offset = 8 rows of
// the tile (1024, 512 or 256 bytes); tile base aligned to 8 rows.
__device__ __forceinline__ uint64_t smem_desc_swz(uint32_t saddr, uint32_t layout, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1u << 16;
  d |= (uint64_t)(sbo >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)layout << 61;
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits [4,6) = 1), A and B
// bf16 (bits [7,10) and [10,13) = 1), both K-major (bits 15, 16 = 0),
// N >> 3 in bits [17,23), M >> 4 in bits [24,29).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// ---- CTA pairs (a cluster of two CTAs sharing each tcgen05.mma.cta_group::2) ----
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The shared::cluster address of the same shared-memory location in CTA `rank`.
__device__ __forceinline__ uint32_t smem_in_cta(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// As mbar_wait_bounded, acquiring at cluster scope (for barriers another CTA arrives on).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  const uint32_t a = smem_u32(bar);
  auto poll = [&]() {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    return done != 0;
  };
  if (poll()) return true;
  if (limit_ns == 0) return false;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (poll()) return true;
    if ((it & 255u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
  }
}
// TMA into this CTA's shared memory, completing on an mbarrier of either CTA of the pair
// (`bar` is a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* m, uint32_t bar,
                                                 int c0, int c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".cta_group::2.L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* m, uint32_t bar,
                                                 int c0, int c1, int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".cta_group::2.L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}
// tcgen05 with cta_group::2 (every tcgen05 instruction of a kernel uses one cta_group).
// Allocation, relinquish and free are issued by one warp in each CTA of the pair.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D[256 x N] (+)= A[256 x K16] B[N x K16]^T over the pair: each CTA holds 128 rows of A
// and N/2 rows of B at the same shared-memory offsets, and 128 rows of D in its TMEM.
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives on the mbarrier at `bar`'s offset in both CTAs of the pair once every
// tcgen05.mma this thread issued has completed.
__device__ __forceinline__ void tc_commit_pair_mc(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"((unsigned short)3)
      : "memory");
}
// The same, on this CTA's barrier only.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

}  // namespace moe_lora
