// moe_lora_layer without a caller workspace.
//
// Some callers cannot allocate device memory for our intermediates: a serving
// engine that reserves nearly all HBM up front for weights and KV cache and hands
// out only its own buffers; a plugin interface that passes inputs and outputs but
// offers no allocator; or a latency-critical path where cudaMalloc/cudaFree may
// synchronise the whole device. This entry point serves them: the layer's
// intermediates (align tables, gathered rows, gate_up and down outputs, LoRA
// shrink results) live in one array in device global memory that the library
// itself holds, so the caller passes only inputs and outputs.
//
// Limits and sharing rules:
// * The array holds kNoallocBytes (64 MiB). Shapes whose workspace
//   (moe_lora_workspace_size) exceeds it are rejected with
//   MOE_LORA_ERR_WORKSPACE_TOO_SMALL before anything is launched.
// * Every GPU that loads this part of the library keeps the 64 MiB until the
//   process exits.
// * All calls on a device share the one array and it keeps the previous call's
//   contents. Calls whose work overlaps on the GPU (different streams without
//   ordering between them) race on it; order such calls on one stream.
// * The first call on each device looks up the array's device address (with that
//   device current); make that first call before any stream capture. The address
//   belongs to the device's current context: when that context is replaced (after
//   cudaDeviceReset, say) the next call looks it up again.
#include <mutex>

#include "internal.h"

namespace moe_lora {
namespace {

constexpr size_t kNoallocBytes = 64ull << 20;

// The library-held workspace. In host code this name is only a stand-in for the
// symbol, never a device address: host code uses the address looked up below.
__device__ __align__(256) unsigned char g_noalloc_ws[kNoallocBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {nullptr};
uint64_t g_addr_ctx[kMaxDevices] = {0};  // context id the address was looked up in

// Device address of g_noalloc_ws in the current context of the current device:
// looked up on the first call in each context (a module's __device__ arrays are
// placed anew in every context that loads it) and cached against the context id.
int noalloc_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_LORA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_LORA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  uint64_t id = current_context_id();
  if (!g_addr[dev] || id == 0 || g_addr_ctx[dev] != id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess || !p) return MOE_LORA_ERR_CUDA;
    if (id == 0) id = current_context_id();  // the lookup made the primary context current
    g_addr[dev] = p;
    g_addr_ctx[dev] = id;
  }
  *out = g_addr[dev];
  return MOE_LORA_OK;
}

}  // namespace
}  // namespace moe_lora

extern "C" int moe_lora_layer_noalloc(const void* x, const float* logits,
                                      const int32_t* topk_ids, const float* topk_w,
                                      const int32_t* token_adapter, int T, int H, int I, int E,
                                      int k, const void* W1, const void* W2, const void* A1,
                                      const void* B1, const void* A2, const void* B2, int L,
                                      int r, void* y, int y_fp32, uint32_t* err_out,
                                      moe_lora_stream_t stream) {
  using namespace moe_lora;
  if (T < 0 || H < 1 || I < 1 || E < 1 || k < 1 || L < 0) return MOE_LORA_ERR_INVALID_ARG;
  const size_t need = moe_lora_workspace_size(T, k, E, L, H, I, r);
  if (need == 0) return MOE_LORA_ERR_INVALID_ARG;
  if (need > kNoallocBytes) return MOE_LORA_ERR_WORKSPACE_TOO_SMALL;
  if (T == 0) return MOE_LORA_OK;
  void* ws = nullptr;
  int st = noalloc_workspace(&ws);
  if (st != MOE_LORA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the sticky error word (first bytes of the workspace) must start clear
  ML_CHECK_CUDA(cudaMemsetAsync(ws, 0, 256, s));
  st = moe_lora_layer(x, logits, topk_ids, topk_w, token_adapter, T, H, I, E, k, W1, W2, A1, B1,
                      A2, B2, L, r, y, y_fp32, ws, kNoallocBytes, stream);
  if (st != MOE_LORA_OK) return st;
  if (err_out)
    ML_CHECK_CUDA(cudaMemcpyAsync(err_out, ws, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s));
  return MOE_LORA_OK;
}
