// Router top-k + softmax over the chosen logits: the router picks each token's
// top-k experts (vllm.com.cn, section "Implementing multi-LoRA inference for MoE
// models in vLLM"). One warp per token; HBM-light.
#include "route.cuh"

namespace moe_lora {

template <int V>
__global__ void __launch_bounds__(256) topk_softmax_kernel(const float* __restrict__ logits, int T,
                                                           int E, int k, int* __restrict__ ids,
                                                           float* __restrict__ w) {
  // the next launch (align) waits before reading ids/w, so it may start right away
  pdl_trigger();
  pdl_wait();
  const int warps = blockDim.x >> 5;
  for (int t = blockIdx.x * warps + (threadIdx.x >> 5); t < T; t += gridDim.x * warps)
    topk_softmax_token<V>(logits + (size_t)t * E, E, k, ids + (size_t)t * k, w + (size_t)t * k);
}

int launch_topk_softmax(const float* logits, int T, int E, int k, int* ids, float* w,
                        cudaStream_t stream, bool pdl) {
  if (T == 0) return MOE_LORA_OK;
  const int threads = 256, per_block = threads / 32;
  int blocks = ceil_div(T, per_block);
  const int cap = num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (E <= 32) return launch_pdl(topk_softmax_kernel<1>, blocks, threads, 0, stream, pdl, logits, T, E, k, ids, w);
  if (E <= 64) return launch_pdl(topk_softmax_kernel<2>, blocks, threads, 0, stream, pdl, logits, T, E, k, ids, w);
  if (E <= 128) return launch_pdl(topk_softmax_kernel<4>, blocks, threads, 0, stream, pdl, logits, T, E, k, ids, w);
  if (E <= 256) return launch_pdl(topk_softmax_kernel<8>, blocks, threads, 0, stream, pdl, logits, T, E, k, ids, w);
  if (E <= 512) return launch_pdl(topk_softmax_kernel<16>, blocks, threads, 0, stream, pdl, logits, T, E, k, ids, w);
  return launch_pdl(topk_softmax_kernel<32>, blocks, threads, 0, stream, pdl, logits, T, E, k, ids, w);
}

int check_route_args(const float* logits, int T, int E, int k, const int32_t* ids, const float* w) {
  if (T < 0 || E < 1 || k < 1 || k > E || k > 32) return MOE_LORA_ERR_INVALID_ARG;
  if (E > 1024) return MOE_LORA_ERR_UNSUPPORTED;
  if (T > 0 && (!logits || !ids || !w)) return MOE_LORA_ERR_INVALID_ARG;
  return MOE_LORA_OK;
}

}  // namespace moe_lora

extern "C" int moe_topk_softmax(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                                moe_lora_stream_t stream) {
  using namespace moe_lora;
  int st = check_route_args(logits, T, E, k, ids, w);
  if (st != MOE_LORA_OK) return st;
  if ((st = check_device()) != MOE_LORA_OK) return st;
  return launch_topk_softmax(logits, T, E, k, ids, w, reinterpret_cast<cudaStream_t>(stream), true);
}
