// Floor of a short streaming kernel on this GPU: how long does one launch take to
// read N bytes, whatever the kernel does? Several read patterns over 644 x 46 KB
// (the decode shrink's A stream: 161 (expert, adapter) pairs x 4 rank groups x
// 8 ranks x 2880 bf16) are timed as single launches after a clean L2 flush (a
// read of 512 MB) and back to back over 16 distinct copies (475 MB > L2): register
// loads (12, 6 per thread), a grid-stride loop, bulk asynchronous copies into
// shared memory (one 46 KB copy or 45 x 1 KB), and the same grid-stride read at
// 300 MB for the large-size rate. The difference between the two sizes gives the
// fixed cost of a launch that no kernel design removes; it bounds the fraction of
// HBM bandwidth that a kernel of a few tens of MB can show.
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//        -o /tmp/stream_floor expert_adapter_gemms_gb300/probes/stream_floor.cu && /tmp/stream_floor
#include <cstdio>
#include <cstdint>
#include <vector>
#include <algorithm>
#include <cuda_runtime.h>
#define CK(x) do { cudaError_t e = (x); if (e != cudaSuccess) { printf("CUDA %s at %d\n", cudaGetErrorString(e), __LINE__); return 1; } } while (0)

constexpr int kSlab = 46080;             // bytes per work item
constexpr int kItems = 644;
constexpr int kV = kSlab / 16;           // uint4 per item: 2880

__device__ __forceinline__ uint32_t mix(uint4 v) { return v.x ^ v.y ^ v.z ^ v.w; }

template <int PER>  // uint4 loads per thread, all issued before use
__global__ void __launch_bounds__(256) k_regs(const uint4* __restrict__ a, int item_v, uint32_t* out) {
  const uint4* p = a + (size_t)blockIdx.x * item_v;
  uint4 v[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int i = threadIdx.x + 256 * j;
    v[j] = i < item_v ? __ldg(p + i) : make_uint4(0, 0, 0, 0);
  }
  uint32_t s = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) s ^= mix(v[j]);
  for (int o = 16; o; o >>= 1) s ^= __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) atomicXor(out, s);
}

__global__ void __launch_bounds__(256) k_stride(const uint4* __restrict__ a, size_t n, uint32_t* out) {
  uint32_t s = 0;
  const size_t st = (size_t)gridDim.x * 256;
  size_t i = (size_t)blockIdx.x * 256 + threadIdx.x;
  for (; i + 3 * st < n; i += 4 * st) {
    uint4 v0 = __ldg(a + i), v1 = __ldg(a + i + st), v2 = __ldg(a + i + 2 * st), v3 = __ldg(a + i + 3 * st);
    s ^= mix(v0) ^ mix(v1) ^ mix(v2) ^ mix(v3);
  }
  for (; i < n; i += st) s ^= mix(__ldg(a + i));
  for (int o = 16; o; o >>= 1) s ^= __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) atomicXor(out, s);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// one item per CTA through shared memory: `pieces` bulk copies of kSlab / pieces bytes
__global__ void __launch_bounds__(256) k_bulk(const uint8_t* __restrict__ a, int pieces, uint32_t* out, int* err) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const uint8_t* src = a + (size_t)blockIdx.x * kSlab;
  const uint32_t piece = kSlab / pieces;
  if (threadIdx.x == 0)
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&bar)), "r"((uint32_t)kSlab) : "memory");
  __syncthreads();
  if (threadIdx.x < 32) {
    for (int c = threadIdx.x; c < pieces; c += 32)
      asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                   ::"r"(smem_u32(sm + c * piece)), "l"(src + (size_t)c * piece), "r"(piece), "r"(smem_u32(&bar)) : "memory");
  }
  uint32_t done = 0;
  for (uint32_t it = 0; it < (1u << 26) && !done; ++it)
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"(smem_u32(&bar)) : "memory");
  if (!done) { atomicOr(err, 1); return; }
  uint32_t s = 0;
  const uint4* v = reinterpret_cast<const uint4*>(sm);
  for (int i = threadIdx.x; i < kV; i += 256) s ^= mix(v[i]);
  for (int o = 16; o; o >>= 1) s ^= __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) atomicXor(out, s);
}

__global__ void k_empty(uint32_t* out) { if (threadIdx.x == 0 && blockIdx.x == 1u << 30) *out = 1; }

int main() {
  const size_t bytes = (size_t)kItems * kSlab;
  constexpr int NB = 16;  // distinct copies of the 30 MB input, 475 MB in all (> L2)
  uint8_t* a; uint32_t* out; int* err; uint4* flush;
  const size_t fl = 512u << 20;
  CK(cudaMalloc(&a, bytes * NB)); CK(cudaMalloc(&out, 4)); CK(cudaMalloc(&err, 4));
  CK(cudaMalloc(&flush, fl));
  CK(cudaMemset(a, 1, bytes * NB)); CK(cudaMemset(flush, 2, fl)); CK(cudaMemset(err, 0, 4));
  CK(cudaDeviceSynchronize());
  CK(cudaFuncSetAttribute(k_bulk, cudaFuncAttributeMaxDynamicSharedMemorySize, kSlab));
  int sms; CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  cudaEvent_t e0, e1; CK(cudaEventCreate(&e0)); CK(cudaEventCreate(&e1));
  // single launch after a clean (read) flush, and NB back-to-back launches on distinct inputs
  auto timeit = [&](const char* name, size_t nbytes, auto launch) -> int {
    std::vector<float> t1, tb;
    for (int i = 0; i < 25; ++i) {
      k_stride<<<4 * sms, 256>>>(flush, fl / 16, out);
      cudaEventRecord(e0); launch(0); cudaEventRecord(e1);
      if (cudaEventSynchronize(e1) != cudaSuccess) { printf("%s failed\n", name); return 1; }
      float ms; cudaEventElapsedTime(&ms, e0, e1); if (i >= 5) t1.push_back(ms * 1000.f);
      k_stride<<<4 * sms, 256>>>(flush, fl / 16, out);
      cudaEventRecord(e0); for (int b = 0; b < NB; ++b) launch(b); cudaEventRecord(e1);
      if (cudaEventSynchronize(e1) != cudaSuccess) { printf("%s failed\n", name); return 1; }
      cudaEventElapsedTime(&ms, e0, e1); if (i >= 5) tb.push_back(ms * 1000.f / NB);
    }
    std::sort(t1.begin(), t1.end()); std::sort(tb.begin(), tb.end());
    const float m1 = t1[t1.size() / 2], mb = tb[tb.size() / 2];
    printf("%-28s single %7.2f us (%5.0f GB/s)   back-to-back %7.2f us/launch (%5.0f GB/s)\n", name, m1,
           nbytes / (m1 * 1e3), mb, nbytes / (mb * 1e3));
    return 0;
  };
  auto A4 = [&](int b) { return reinterpret_cast<const uint4*>(a + (size_t)b * bytes); };
  auto A8 = [&](int b) { return a + (size_t)b * bytes; };
  printf("reads of %.1f MB per launch (300 MB in the last line)\n", bytes / 1e6);
  if (timeit("empty 644 CTAs", bytes, [&](int) { k_empty<<<kItems, 256>>>(out); })) return 1;
  if (timeit("regs 644x46KB (12/thr)", bytes, [&](int b) { k_regs<12><<<kItems, 256>>>(A4(b), kV, out); })) return 1;
  if (timeit("regs 1288x23KB (6/thr)", bytes, [&](int b) { k_regs<6><<<2 * kItems, 256>>>(A4(b), kV / 2, out); })) return 1;
  if (timeit("stride 4/SM", bytes, [&](int b) { k_stride<<<4 * sms, 256>>>(A4(b), bytes / 16, out); })) return 1;
  if (timeit("stride 8/SM", bytes, [&](int b) { k_stride<<<8 * sms, 256>>>(A4(b), bytes / 16, out); })) return 1;
  if (timeit("bulk 1 x 46KB", bytes, [&](int b) { k_bulk<<<kItems, 256, kSlab>>>(A8(b), 1, out, err); })) return 1;
  if (timeit("bulk 45 x 1KB", bytes, [&](int b) { k_bulk<<<kItems, 256, kSlab>>>(A8(b), 45, out, err); })) return 1;
  // the same reads at 10x the size, for the asymptote
  if (timeit("stride 4/SM, 300 MB", bytes * 10, [&](int b) { k_stride<<<4 * sms, 256>>>(A4(0), bytes * 10 / 16, out); })) return 1;
  int h = 0; CK(cudaMemcpy(&h, err, 4, cudaMemcpyDeviceToHost));
  printf("bulk wait errors: %d\n", h);
  return 0;
}
