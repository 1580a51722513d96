// The fused MoE-LoRA expert layer as one chain of launches on the caller's
// stream (vllm.com.cn, sections "Implementing multi-LoRA inference for MoE
// models in vLLM" and "Kernel optimizations"; aib.vote, programmatic dependent
// launch removing the idle gaps between kernels):
//
//   route -> align -> gather -> gate_up GEMM -> gate_up shrink ->
//   gate_up expand + SwiGLU -> down GEMM -> down shrink -> down expand + combine
//
// Every launch uses programmatic dependent launch; nothing synchronises with the
// host, no device count is read back, and every size is a runtime argument, so a
// new token count never triggers a compile or a module load. Intermediates live
// in the caller's workspace, carved here.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace moe_lora {

// ---------------------------------------------------------------------------
// device checks
// ---------------------------------------------------------------------------
namespace {
std::atomic<int> g_dev_state[kMaxDevices];  // 0 unknown, 1 ok, 2 unsupported
std::atomic<int> g_dev_sms[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
std::once_flag g_ctx_once;
}  // namespace

uint64_t current_context_id() {
  std::call_once(g_ctx_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!g_ctx_current || !g_ctx_id) return 0;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  unsigned long long id = 0;
  if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return static_cast<uint64_t>(id);
}

int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_LORA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_LORA_ERR_UNSUPPORTED;
  int s = g_dev_state[dev].load(std::memory_order_relaxed);
  if (s == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_LORA_ERR_CUDA;
    g_dev_sms[dev].store(sms);
    s = (major == 10 && minor == 3) ? 1 : 2;
    g_dev_state[dev].store(s);
  }
  return s == 1 ? MOE_LORA_OK : MOE_LORA_ERR_UNSUPPORTED;
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  int n = g_dev_sms[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
    g_dev_sms[dev].store(n);
  }
  return n;
}

// ---------------------------------------------------------------------------
// tiles and workspace
// ---------------------------------------------------------------------------
static void pick_tiles(int T, int k, int E, int L, int32_t* bm_base, int32_t* bm_lora) {
  const int64_t S = (int64_t)T * k;
  const int64_t per_expert = (S + E - 1) / E;
  int64_t b = (2 * per_expert + 15) / 16 * 16;
  if (b < 16) b = 16;
  // the tile sizes with a compiled kernel
  const int allowed[5] = {16, 32, 64, 128, 256};
  int pick = 256;
  for (int i = 0; i < 5; ++i)
    if (allowed[i] >= b) { pick = allowed[i]; break; }
  *bm_base = pick;
  // short (expert, adapter) segments (decode): blocks of at most 8 rows
  *bm_lora = S <= 2 * (int64_t)E * (L > 0 ? L : 1) ? 8 : 16;
}

// Rows per expert-major chunk: with few rows per expert (decode) each grouped-GEMM CTA
// takes one (expert, weight block) and all of the expert's rows, so it can stream its
// weights before routing and alignment have finished; 0: token tiles. An expert with more
// rows than the chunk streams its weights once per chunk, so chunks of 64 rows are taken
// up to 32 rows per expert on average, and up to 64 where the count is exact (one expert:
// a dense layer). At 48 and 64 rows per expert of 32 experts (GPT-OSS dims), 64-row chunks
// ran 0.352 against 0.363 ms and 0.488 against 0.377 ms for token tiles.
static int expert_major_rows(int T, int k, int E) {
  const int64_t per_expert = ((int64_t)T * k + E - 1) / E;
  return per_expert <= 16 ? 32 : per_expert <= 32 || (E == 1 && per_expert <= 64) ? 64 : 0;
}

// The expert-major down GEMM's K shares (partial outputs the combine sums): two where the
// (expert, weight block) CTAs already fill the SMs' slots (2.4 -> 4.8 waves at the GPT-OSS
// decode shape, where one and three shares were slower), else as many as fill about one
// wave of two CTAs per SM (dense, E = 1: 8 shares at H = 4096, 4 at H = 8192 were the best
// measured), at most 8 and at least two k-blocks each. Shape-only (a fixed 304 slots), so
// the workspace layout does not depend on the device.
static int down_ksplit(int E, int H, int I) {
  const int64_t blocks = (int64_t)E * ((H + 127) / 128);
  const int nk = (I + 63) / 64;
  if (nk < 4) return 1;
  int s = blocks >= 304 ? 2 : (int)std::min<int64_t>(8, std::max<int64_t>(2, 304 / blocks));
  s = std::min(s, nk / 2);
  // the kernel gives share i the k-blocks [i q, (i + 1) q), q = ceil(nk / s): every share
  // must hold some (an empty one would publish an accumulator it never wrote)
  while (s > 1 && (s - 1) * ((nk + s - 1) / s) >= nk) --s;
  return s;
}

// The fused expand's token tile (and so the zero gap of its shifted z buffers) that the
// heuristics give a shape: the expert-major chunk, else the align's token tile.
static int fused_gap(int T, int k, int E, int L) {
  const int em = expert_major_rows(T, k, E);
  if (em) return em;
  int32_t hb, hl;
  pick_tiles(T, k, E, L, &hb, &hl);
  return hb;
}

struct LayerPlan {
  AlignLayout al;
  int bm_base, bm_lora, em_bn;
  bool fused;    // expand (and SwiGLU) inside the grouped GEMMs
  ZPadLayout z;  // the shifted z buffers of the fused chain (both the same shape)
  int ksplit;    // fused, expert-major: CTAs per down weight block (partial outputs)
  int64_t off_align, off_ids, off_w, off_xs, off_G, off_Z1, off_h, off_Z2, off_O, off_Z1p,
      off_Z2p, total;
  bool valid;
};

// The workspace layout depends on the shape only; the chain (fused or not) and the tiles
// may also depend on the options. The fp32 gate_up output G of the unfused chain and the
// two shifted z buffers of the fused chain share one region.
static LayerPlan plan_layer(int T, int k, int E, int L, int H, int I, int r,
                            const moe_lora_layer_opts& opt) {
  LayerPlan p = {};
  p.valid = false;
  int32_t hb, hl;
  pick_tiles(T, k, E, L, &hb, &hl);
  const int64_t S = (int64_t)T * k;
  const int64_t rr = L > 0 ? r : 0;
  const bool pdl = !opt.disable_pdl;
  const int slices = opt.gate_up_slices == 0 ? 1 : opt.gate_up_slices;
  // the fused chain: shapes whose shifted z buffers stay small next to G (they grow with
  // E L); adapters of one rank with one gate_up slice and r % 8 == 0 (the B tensor maps)
  const int gap = fused_gap(T, k, E, L);
  p.z = zpad_layout((int)S, E, L, (int)rr, gap);
  const int64_t zbytes = L > 0 ? (int64_t)round_up((size_t)(p.z.rows * p.z.zw * 2), 256) : 0;
  const int64_t g_bytes = S * 2 * (int64_t)I * 4;
  const bool shape_ok = L == 0 || (r % 8 == 0 && 2 * zbytes <= std::max<int64_t>(g_bytes, 64ll << 20));
  // ... where it pays: with adapters at few rows per expert (the grouped GEMMs then stream
  // weights, and the adapter stages add bytes, not time) or where the (expert, adapter) runs
  // are long (each run's stages multiply a whole token tile, so short runs waste tensor
  // work); without adapters where token tiles, not expert-major chunks, are used
  const int em_shape = expert_major_rows(T, k, E);
  const bool long_runs = L > 0 && S >= 16 * std::min<int64_t>((int64_t)E * L, S);
  const bool pays = L == 0 ? em_shape == 0 : (em_shape > 0 || long_runs);
  const bool want = shape_ok && opt.expand_mode != 1 && (pays || opt.expand_mode == 2) &&
                    (L == 0 || (opt.adapter_ranks == nullptr && slices == 1));
  p.em_bn = pdl ? em_shape : 0;
  p.bm_base = opt.bm_base > 0 ? opt.bm_base : hb;
  p.bm_lora = opt.bm_lora > 0 ? opt.bm_lora : hl;
  const int chunk = p.em_bn > 0 ? p.em_bn : p.bm_base;
  p.fused = want && chunk <= gap;
  // few rows per expert: each down weight block's K range is split (down_ksplit) and the
  // combine sums the partial outputs
  p.ksplit = p.fused && p.em_bn > 0 ? down_ksplit(E, H, I) : 1;
  p.al = align_layout(T, k, E, L, p.bm_base, p.bm_lora);
  // the align region is sized for the smallest tiles so any tile choice fits
  AlignLayout worst = align_layout(T, k, E, L, 16, 1);
  if (!p.al.valid || !worst.valid) return p;
  int64_t o = 0;
  auto take = [&](int64_t bytes) { int64_t at = o; o = (int64_t)round_up(o + bytes, 256); return at; };
  p.off_align = take(worst.off[MOE_LORA_AF_TOTAL_BYTES]);
  p.off_ids = take(S * 4);
  p.off_w = take(S * 4);
  p.off_xs = take(S * H * 2);
  p.off_G = take(std::max<int64_t>(g_bytes, shape_ok ? 2 * zbytes : 0));
  p.off_Z1p = p.off_G;
  p.off_Z2p = p.off_G + zbytes;
  p.off_Z1 = take(S * 2 * rr * 4);  // two z slices with separate gate and up adapters
  p.off_h = take(S * (int64_t)I * 2);
  p.off_Z2 = take(S * rr * 4);
  p.off_O = take(S * (int64_t)H * 4 * (em_shape > 0 ? down_ksplit(E, H, I) : 1));  // partial outputs
  p.total = o;
  p.valid = true;
  return p;
}

// ---------------------------------------------------------------------------
// The chain of launches and the reads made before a kernel's wait
// ---------------------------------------------------------------------------
// Under programmatic dependent launch a kernel starts once every CTA of its predecessor
// has triggered its dependents (or exited), and no kernel of the layer completes before
// its own griddepcontrol.wait has returned, i.e. before its predecessor completed. So
// when launch c starts, an earlier launch p has completed if p <= c - 2 and launch c - 1
// triggers only after its own wait. Reads a kernel makes before its wait ("early" reads:
// weights, older activations, the align tables) rely on exactly that. The chain records,
// per step, its launches, whether they trigger only after waiting, and the steps whose
// outputs the step reads early; the layer refuses a chain that breaks the rule, and every
// launch takes its early flag from here.
enum Step { kRoute, kAlign, kGather, kShrink1, kGemm1, kExpand1, kShrink2, kGemm2, kExpand2,
            kCombine, kNumSteps };
struct Chain {
  int first[kNumSteps], last[kNumSteps];  // launch indices of each step (-1: not launched)
  int src[kNumSteps][3];                  // steps read before the wait (-1: none)
  bool after_wait[24];                    // per launch: triggers only after its wait
  int n;                                  // launches
  bool early(Step s) const { return src[s][0] >= 0; }
  int early_reads() const {
    int c = 0;
    for (int s = 0; s < kNumSteps; ++s)
      for (int i = 0; i < 3; ++i) c += src[s][i] >= 0 && last[src[s][i]] >= 0;
    return c;
  }
  // every early read comes from a launch that has completed when the reader starts
  bool ok() const {
    for (int s = 0; s < kNumSteps; ++s) {
      for (int i = 0; i < 3; ++i) {
        const int t = src[s][i];
        if (t < 0 || last[t] < 0) continue;  // a caller input (e.g. routing given by the caller)
        const int c = first[s];
        if (c < 0 || c - last[t] < 2 || !after_wait[c - 1]) return false;
      }
    }
    return true;
  }
};

static Chain layer_chain(const LayerPlan& p, int T, int k, int E, int L, bool have_logits,
                         bool pdl) {
  Chain c;
  for (int s = 0; s < kNumSteps; ++s) {
    c.first[s] = c.last[s] = -1;
    c.src[s][0] = c.src[s][1] = c.src[s][2] = -1;
  }
  c.n = 0;
  auto add = [&](Step s, int kernels, bool after_wait) {
    c.first[s] = c.n;
    for (int i = 0; i < kernels; ++i) c.after_wait[c.n++] = after_wait;
    c.last[s] = c.n - 1;
  };
  auto reads = [&](Step s, int a, int b = -1, int d = -1) {
    if (!pdl) return;  // plain stream order: every read follows its producer's completion
    c.src[s][0] = a;
    c.src[s][1] = b;
    c.src[s][2] = d;
  };
  const bool lora = L > 0;
  // few tokens: the one-CTA align routes them itself (no route launch)
  if (have_logits && !align_can_route(p.al, T, E)) add(kRoute, 1, false);  // triggers at its start
  add(kAlign, p.al.ctas > 0 ? 3 : 1, false);    // each align kernel triggers at its start
  if (p.fused) {
    add(kGather, 1, lora || p.em_bn == 0);  // base only, expert-major: triggers at its start
    if (lora) {
      add(kShrink1, 1, true);
      reads(kShrink1, kAlign);                  // x by token (a caller input), the tables
    }
    add(kGemm1, 1, true);
    if (lora) reads(kGemm1, kGather, kAlign);   // gathered rows, tables; z only after the wait
    if (lora) {                                 // h is its predecessor's: waits for it, but
      add(kShrink2, 1, true);                   // reads its block and prefetches A first
      reads(kShrink2, kAlign);
    }
    add(kGemm2, 1, true);
    if (lora) reads(kGemm2, kGemm1, kAlign);    // h, tables; z only after the wait
    add(kCombine, 1, true);
    reads(kCombine, kAlign, kRoute);            // slot rows, routing weights
    return c;
  }
  const bool em = p.em_bn > 0;
  add(kGather, 1, !em);  // expert-major: the gate_up GEMM reads nothing of it early
  add(kGemm1, 1, true);
  if (!em) reads(kGemm1, kAlign);  // the token tiles
  if (lora) {
    add(kShrink1, 1, true);
    if (p.bm_lora <= 8) reads(kShrink1, kGather, kAlign);  // gathered rows
    else reads(kShrink1, kAlign);                          // x by token
  }
  add(kExpand1, 1, true);
  if (lora) reads(kExpand1, kGemm1, kAlign);  // G, B, tables; z after the wait
  add(kGemm2, 1, true);
  if (!em) reads(kGemm2, kAlign);
  if (lora) {
    add(kShrink2, 1, true);
    reads(kShrink2, kExpand1, kAlign);  // h
  }
  // the down expand: a token walk, or (several rows per pair) an in-place add and a combine
  const bool add_then_combine = lora && (int64_t)T * k >= 2 * (int64_t)E * L;
  add(kExpand2, add_then_combine ? 2 : 1, true);
  if (lora) reads(kExpand2, kGemm2, kAlign, kRoute);  // O, tables, routing weights
  return c;
}

}  // namespace moe_lora

using namespace moe_lora;

extern "C" const char* moe_lora_status_string(int status) {
  switch (status) {
    case MOE_LORA_OK: return "ok";
    case MOE_LORA_ERR_INVALID_ARG: return "invalid argument";
    case MOE_LORA_ERR_UNSUPPORTED: return "unsupported shape or device";
    case MOE_LORA_ERR_CUDA: return "CUDA runtime error";
    case MOE_LORA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_LORA_ERR_TIMEOUT: return "a bounded wait inside a kernel gave up";
    default: return "unknown status";
  }
}

extern "C" int moe_lora_get_error(const void* buf, moe_lora_stream_t stream, uint32_t* err) {
  if (!buf || !err) return MOE_LORA_ERR_INVALID_ARG;
  uint32_t v = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  ML_CHECK_CUDA(cudaMemcpyAsync(&v, buf, sizeof(v), cudaMemcpyDeviceToHost, s));
  ML_CHECK_CUDA(cudaStreamSynchronize(s));
  *err = v;
  return (v & MOE_LORA_DEVERR_TIMEOUT) ? MOE_LORA_ERR_TIMEOUT : MOE_LORA_OK;
}

extern "C" int moe_lora_clear_error(void* buf, moe_lora_stream_t stream) {
  if (!buf) return MOE_LORA_ERR_INVALID_ARG;
  ML_CHECK_CUDA(cudaMemsetAsync(buf, 0, sizeof(uint32_t), reinterpret_cast<cudaStream_t>(stream)));
  return MOE_LORA_OK;
}

extern "C" int moe_lora_layer_tiles(int T, int k, int E, int L, int H, int I, int r,
                                    int32_t* bm_base, int32_t* bm_lora) {
  (void)H; (void)I; (void)r;
  if (!bm_base || !bm_lora || T < 0 || k < 1 || E < 1 || L < 0) return MOE_LORA_ERR_INVALID_ARG;
  pick_tiles(T, k, E, L, bm_base, bm_lora);
  return MOE_LORA_OK;
}

extern "C" size_t moe_lora_workspace_size(int T, int k, int E, int L, int H, int I, int r) {
  if (T < 0 || k < 1 || E < 1 || L < 0 || H < 1 || I < 1 || (L > 0 && r < 1)) return 0;
  const moe_lora_layer_opts o = {};
  LayerPlan p = plan_layer(T, k, E, L, H, I, r, o);
  return p.valid ? (size_t)p.total : 0;
}

extern "C" int moe_lora_layer_plan(int T, int k, int E, int L, int H, int I, int r,
                                   const moe_lora_layer_opts* opts, moe_lora_layer_plan_t* out) {
  if (!out || T < 0 || k < 1 || E < 1 || L < 0 || H < 1 || I < 1 || (L > 0 && r < 1))
    return MOE_LORA_ERR_INVALID_ARG;
  moe_lora_layer_opts o = {};
  if (opts) o = *opts;
  LayerPlan p = plan_layer(T, k, E, L, H, I, r, o);
  if (!p.valid) return MOE_LORA_ERR_UNSUPPORTED;
  const bool pdl = !o.disable_pdl;
  const Chain c = layer_chain(p, T, k, E, L, true, pdl);
  if (!c.ok() || !layer_chain(p, T, k, E, L, false, pdl).ok()) return MOE_LORA_ERR_UNSUPPORTED;
  out->bm_base = p.bm_base;
  out->bm_lora = p.bm_lora;
  out->expert_major_rows = p.em_bn;
  out->fused_expand = p.fused ? 1 : 0;
  out->launches = T > 0 ? c.n : 0;
  out->early_reads = c.early_reads();
  out->route_in_align = T > 0 && align_can_route(p.al, T, E) ? 1 : 0;
  return MOE_LORA_OK;
}

// Host-side checks of a layer call; nothing is launched or copied on error. On success
// *plan holds the layer's workspace plan (T = 0 passes with nothing to do).
static int check_layer_args(const void* x, const float* logits, const int32_t* topk_ids,
                            const float* topk_w, int T, int H, int I, int E, int k,
                            const void* W1, const void* W2, const void* A1, const void* B1,
                            const void* A2, const void* B2, int L, int r, const void* y,
                            const void* workspace, size_t workspace_bytes,
                            const moe_lora_layer_opts& o, LayerPlan* plan) {
  if (T < 0 || H < 1 || I < 1 || E < 1 || k < 1 || k > E || L < 0) return MOE_LORA_ERR_INVALID_ARG;
  if (k > 32 || E > 1024 || L >= 65535) return MOE_LORA_ERR_UNSUPPORTED;
  if (L > 0 && (r < 1 || !A1 || !B1 || !A2 || !B2)) return MOE_LORA_ERR_INVALID_ARG;
  if (L > 0 && r > 256) return MOE_LORA_ERR_UNSUPPORTED;
  if (H % 8 != 0 || I % 8 != 0) return MOE_LORA_ERR_UNSUPPORTED;
  const bool have_logits = logits != nullptr;
  const bool have_ids = topk_ids != nullptr || topk_w != nullptr;
  if (T > 0) {
    if (have_logits == have_ids) return MOE_LORA_ERR_INVALID_ARG;
    if (have_ids && (!topk_ids || !topk_w)) return MOE_LORA_ERR_INVALID_ARG;
    if (!x || !W1 || !W2 || !y || !workspace) return MOE_LORA_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W1) || !aligned16(W2)) return MOE_LORA_ERR_INVALID_ARG;
    if (L > 0 && (!aligned16(A1) || !aligned16(B1) || !aligned16(A2) || !aligned16(B2)))
      return MOE_LORA_ERR_INVALID_ARG;
  }
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return MOE_LORA_ERR_INVALID_ARG;
  if (o.num_events < 0 || (o.num_events > 0 && !o.events)) return MOE_LORA_ERR_INVALID_ARG;
  if (o.gate_up_slices < 0 || o.gate_up_slices > 2) return MOE_LORA_ERR_INVALID_ARG;
  if (o.expand_mode < 0 || o.expand_mode > 2) return MOE_LORA_ERR_INVALID_ARG;
  *plan = plan_layer(T, k, E, L, H, I, r, o);
  if (!plan->valid) return MOE_LORA_ERR_UNSUPPORTED;
  if (T == 0) return MOE_LORA_OK;
  if (workspace_bytes < (size_t)plan->total) return MOE_LORA_ERR_WORKSPACE_TOO_SMALL;
  return check_device();
}

extern "C" int moe_lora_layer_ex(const void* x, const float* logits, const int32_t* topk_ids,
                                 const float* topk_w, const int32_t* token_adapter, int T, int H,
                                 int I, int E, int k, const void* W1, const void* W2,
                                 const void* A1, const void* B1, const void* A2, const void* B2,
                                 int L, int r, void* y, int y_fp32, void* workspace,
                                 size_t workspace_bytes, const moe_lora_layer_opts* opts,
                                 moe_lora_stream_t stream_) {
  // ---- host-side validation: nothing is launched on error ----
  moe_lora_layer_opts o = {};
  if (opts) o = *opts;
  LayerPlan p;
  int st = check_layer_args(x, logits, topk_ids, topk_w, T, H, I, E, k, W1, W2, A1, B1, A2, B2,
                            L, r, y, workspace, workspace_bytes, o, &p);
  if (st != MOE_LORA_OK || T == 0) return st;
  const int slices = o.gate_up_slices == 0 ? 1 : o.gate_up_slices;
  const bool have_logits = logits != nullptr;

  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const bool pdl = !o.disable_pdl;
  const Chain ch = layer_chain(p, T, k, E, L, have_logits, pdl);
  if (!ch.ok()) return MOE_LORA_ERR_UNSUPPORTED;
  char* ws = static_cast<char*>(workspace);
  moe_lora_align_t al;
  al.buf = ws + p.off_align;
  al.T = T;
  al.k = k;
  al.E = E;
  al.L = L;
  al.bm_base = p.bm_base;
  al.bm_lora = p.bm_lora;
  al.adapter_ranks = L > 0 ? o.adapter_ranks : nullptr;
  int32_t* ids = reinterpret_cast<int32_t*>(ws + p.off_ids);
  float* w = reinterpret_cast<float*>(ws + p.off_w);
  void* xs = ws + p.off_xs;
  float* G = reinterpret_cast<float*>(ws + p.off_G);
  float* Z1 = reinterpret_cast<float*>(ws + p.off_Z1);
  void* h = ws + p.off_h;
  float* Z2 = reinterpret_cast<float*>(ws + p.off_Z2);
  float* O = reinterpret_cast<float*>(ws + p.off_O);
  const int rr = L > 0 ? r : 0;
  const unsigned long long wait_ns = o.wait_limit_ns == 0 ? kWaitLimitNs
                                     : o.wait_limit_ns < 0 ? 0ull
                                                           : (unsigned long long)o.wait_limit_ns;

  auto mark = [&](int i) -> int {
    if (i < o.num_events && o.events[i])
      if (cudaEventRecord(static_cast<cudaEvent_t>(o.events[i]), stream) != cudaSuccess)
        return MOE_LORA_ERR_CUDA;
    return MOE_LORA_OK;
  };
#define ML_STEP(expr)                       \
  do {                                      \
    int _s = (expr);                        \
    if (_s != MOE_LORA_OK) return _s;       \
  } while (0)

  ML_STEP(mark(0));
  const bool route_in_align = have_logits && align_can_route(p.al, T, E);
  if (have_logits && !route_in_align) {
    ML_STEP(launch_topk_softmax(logits, T, E, k, ids, w, stream, pdl));
  } else if (!have_logits) {
    ids = const_cast<int32_t*>(topk_ids);
    w = const_cast<float*>(topk_w);
  }
  ML_STEP(mark(1));
  if (route_in_align)  // few tokens: the align's one CTA routes them first
    ML_STEP(launch_route_align(logits, ids, w, L > 0 ? token_adapter : nullptr, &al, p.al, stream,
                               pdl));
  else
    ML_STEP(launch_align(ids, L > 0 ? token_adapter : nullptr, &al, p.al, stream, pdl));
  ML_STEP(mark(2));
  const int em_bn = p.em_bn;
  if (p.fused) {
    // route -> align -> gather -> gate_up shrink -> gate_up GEMM with the expand and
    // SwiGLU -> down shrink -> down GEMM with the expand -> combine. Each shrink writes
    // z into its shifted buffer; each GEMM reads everything but z before its wait (its
    // predecessor, the shrink, triggers only after its own wait).
    __nv_bfloat16* Z1p = reinterpret_cast<__nv_bfloat16*>(ws + p.off_Z1p);
    __nv_bfloat16* Z2p = reinterpret_cast<__nv_bfloat16*>(ws + p.off_Z2p);
    ZPadOut zo = {};
    zo.zw = p.z.zw;
    zo.lo_off = p.z.lo_off;
    zo.rp16 = p.z.rp16;
    zo.gap = p.z.gap;
    zo.L = L;
    AlignView av = align_view(al.buf, p.al);
    zo.row_expert = av.row_expert;
    zo.row_adapter = av.row_adapter;
    const bool lora = L > 0;
    // without adapters the gate_up GEMM follows the gather and reads nothing of it early:
    // the gather then triggers at its start so that the (expert-major) GEMM streams weights
    ML_STEP(launch_gather(x, &al, p.al, H, xs, stream, pdl, !lora && em_bn > 0));
    ML_STEP(mark(3));
    if (lora) {  // by token: x is a caller input, the align tables two launches back
      zo.p = Z1p;
      ML_STEP(launch_shrink_impl(x, 0, A1, &al, p.al, H, r, r, nullptr, stream, pdl,
                                 ch.early(kShrink1), wait_ns, &zo, kShrinkOneWave));
    }
    ML_STEP(mark(4));
    ML_STEP(launch_fused_gemm(xs, W1, lora ? B1 : nullptr, Z1p, p.z, &al, p.al, 2 * I, H, r, true, h,
                              stream, pdl, ch.early(kGemm1), em_bn, wait_ns, 1,
                              o.mma_pairs >= 0));
    ML_STEP(mark(5));
    ML_STEP(mark(6));
    if (lora) {  // h comes from the predecessor: the shrink waits for it, A streams first
      zo.p = Z2p;
      ML_STEP(launch_shrink_impl(h, 1, A2, &al, p.al, I, r, r, nullptr, stream, pdl, false, wait_ns,
                                 &zo, kShrinkOneWave | (ch.early(kShrink2) ? kShrinkPrefetchA : 0)));
    }
    ML_STEP(mark(7));
    ML_STEP(launch_fused_gemm(h, W2, lora ? B2 : nullptr, Z2p, p.z, &al, p.al, H, I, r, false, O,
                              stream, pdl, ch.early(kGemm2), em_bn, wait_ns, p.ksplit,
                              o.mma_pairs >= 0));
    ML_STEP(mark(8));
    ML_STEP(launch_combine(O, w, &al, p.al, H, y, y_fp32, stream, pdl, p.ksplit,
                           (size_t)T * k * H, ch.early(kCombine)));
    ML_STEP(mark(9));
    return MOE_LORA_OK;
  }
  // Few rows per expert (decode): the gate_up GEMM runs expert-major, so its weights
  // stream from the start of the layer while routing, align and gather finish.
  ML_STEP(launch_gather(x, &al, p.al, H, xs, stream, pdl, em_bn > 0));
  ML_STEP(mark(3));
  ML_STEP(launch_grouped_gemm_impl(xs, W1, &al, p.al, 2 * I, H, G, stream, pdl, ch.early(kGemm1),
                                   em_bn, wait_ns));
  ML_STEP(mark(4));
  // Short LoRA blocks (decode-like) read the gathered rows: addressed by sorted row, they
  // need no slot lookup before the load (and are recent in L2).
  if (L > 0) {
    // with separate gate and up adapters the gate_up shrink is one of rank 2r
    if (p.bm_lora <= 8)
      ML_STEP(launch_shrink_impl(xs, 1, A1, &al, p.al, H, slices * r, r, Z1, stream, pdl,
                                 ch.early(kShrink1), wait_ns));
    else
      ML_STEP(launch_shrink_impl(x, 0, A1, &al, p.al, H, slices * r, r, Z1, stream, pdl,
                                 ch.early(kShrink1), wait_ns));
  }
  ML_STEP(mark(5));
  ML_STEP(launch_expand_impl(Z1, L > 0 ? B1 : nullptr, &al, p.al, 2 * I, rr, L > 0 && slices == 2 ? 3 : 1, G, h, 0,
                             nullptr, stream, pdl, ch.early(kExpand1)));
  ML_STEP(mark(6));
  // the down GEMM likewise runs expert-major when experts hold few rows: its weights stream
  // while the SwiGLU expand drains
  ML_STEP(launch_grouped_gemm_impl(h, W2, &al, p.al, H, I, O, stream, pdl, ch.early(kGemm2), em_bn,
                                   wait_ns));
  ML_STEP(mark(7));
  if (L > 0)
    ML_STEP(launch_shrink_impl(h, 1, A2, &al, p.al, I, r, r, Z2, stream, pdl, ch.early(kShrink2),
                               wait_ns));
  ML_STEP(mark(8));
  ML_STEP(launch_expand_impl(Z2, L > 0 ? B2 : nullptr, &al, p.al, H, rr, 2, O, y, y_fp32, w,
                             stream, pdl, ch.early(kExpand2)));
  ML_STEP(mark(9));
#undef ML_STEP
  return MOE_LORA_OK;
}

extern "C" int moe_lora_layer(const void* x, const float* logits, const int32_t* topk_ids,
                              const float* topk_w, const int32_t* token_adapter, int T, int H,
                              int I, int E, int k, const void* W1, const void* W2, const void* A1,
                              const void* B1, const void* A2, const void* B2, int L, int r,
                              void* y, int y_fp32, void* workspace, size_t workspace_bytes,
                              moe_lora_stream_t stream) {
  return moe_lora_layer_ex(x, logits, topk_ids, topk_w, token_adapter, T, H, I, E, k, W1, W2, A1,
                           B1, A2, B2, L, r, y, y_fp32, workspace, workspace_bytes, nullptr,
                           stream);
}

extern "C" int moe_lora_host_io_layout(int T, int H, int E, int with_adapter, int y_fp32,
                                       int64_t* offsets, size_t* in_bytes, size_t* staging_bytes) {
  if (T < 0 || H < 1 || E < 1 || !offsets) return MOE_LORA_ERR_INVALID_ARG;
  if ((with_adapter != 0 && with_adapter != 1) || (y_fp32 != 0 && y_fp32 != 1))
    return MOE_LORA_ERR_INVALID_ARG;
  int64_t o = 0, end = 0;
  auto take = [&](int64_t bytes) {
    const int64_t at = (int64_t)round_up((size_t)o, 256);
    o = end = at + bytes;
    return at;
  };
  offsets[0] = take((int64_t)T * H * 2);
  offsets[1] = take((int64_t)T * E * 4);
  offsets[2] = with_adapter ? take((int64_t)T * 4) : -1;
  const int64_t in_end = end;
  offsets[3] = take((int64_t)T * H * (y_fp32 ? 4 : 2));
  if (in_bytes) *in_bytes = (size_t)in_end;
  if (staging_bytes) *staging_bytes = (size_t)end;
  return MOE_LORA_OK;
}

extern "C" int moe_lora_layer_host(const void* in_host, void* y_host, void* staging,
                                   size_t staging_bytes, int with_adapter, int T, int H, int I,
                                   int E, int k, const void* W1, const void* W2, const void* A1,
                                   const void* B1, const void* A2, const void* B2, int L, int r,
                                   int y_fp32, void* workspace, size_t workspace_bytes,
                                   const moe_lora_layer_opts* opts, moe_lora_stream_t stream_) {
  int64_t off[4];
  size_t in_bytes = 0, need = 0;
  int st = moe_lora_host_io_layout(T, H, E, with_adapter, y_fp32, off, &in_bytes, &need);
  if (st != MOE_LORA_OK) return st;
  if (T > 0 && (!in_host || !y_host || !staging)) return MOE_LORA_ERR_INVALID_ARG;
  if (staging && (reinterpret_cast<uintptr_t>(staging) & 255u) != 0) return MOE_LORA_ERR_INVALID_ARG;
  if (T > 0 && staging_bytes < need) return MOE_LORA_ERR_WORKSPACE_TOO_SMALL;
  char* sg = static_cast<char*>(staging);
  const void* x = sg ? sg + off[0] : nullptr;
  const float* logits = sg ? reinterpret_cast<const float*>(sg + off[1]) : nullptr;
  const int32_t* ta = sg && with_adapter ? reinterpret_cast<const int32_t*>(sg + off[2]) : nullptr;
  void* y = sg ? sg + off[3] : nullptr;
  moe_lora_layer_opts o = {};
  if (opts) o = *opts;
  LayerPlan p;
  st = check_layer_args(x, logits, nullptr, nullptr, T, H, I, E, k, W1, W2, A1, B1, A2, B2, L, r,
                        y, workspace, workspace_bytes, o, &p);
  if (st != MOE_LORA_OK || T == 0) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (cudaMemcpyAsync(sg, in_host, in_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return MOE_LORA_ERR_CUDA;
  st = moe_lora_layer_ex(x, logits, nullptr, nullptr, ta, T, H, I, E, k, W1, W2, A1, B1, A2, B2,
                         L, r, y, y_fp32, workspace, workspace_bytes, opts, stream_);
  if (st != MOE_LORA_OK) return st;
  const size_t y_bytes = (size_t)T * H * (y_fp32 ? 4 : 2);
  if (cudaMemcpyAsync(y_host, y, y_bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return MOE_LORA_ERR_CUDA;
  return MOE_LORA_OK;
}
