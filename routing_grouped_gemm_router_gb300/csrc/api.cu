// api.cu — the C ABI (include/moe.h): argument checks, workspace layout and the order in
// which the kernels of the layer are enqueued. No entry point allocates, frees,
// synchronises or reads device memory on the host (moe_device_status excepted).
#include <mutex>

#include "common.cuh"

namespace moe {

int num_sms() {
  static int cache[64];
  static std::once_flag once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  std::call_once(once[dev], [dev] {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = v > 0 ? v : 148;
  });
  return cache[dev];
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

static constexpr int kMaxE = 512;
static constexpr int kFewTokens = 128;  // router on CUDA cores up to this many tokens

static moe_status_t check_cfg(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 1 || c->H < 8 || c->I < 8 || c->E < 1 || c->k < 1 || c->k > c->E || c->k > 32)
    return MOE_ERR_INVALID_ARG;
  if (c->H % 8 || c->I % 8) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->mode != MOE_ROUTE_SOFTMAX && c->mode != MOE_ROUTE_SIGMOID_GROUPED)
    return MOE_ERR_INVALID_ARG;
  if (c->mode == MOE_ROUTE_SIGMOID_GROUPED) {
    if (c->n_group < 1 || c->n_group > 32 || c->E % c->n_group) return MOE_ERR_INVALID_ARG;
    if (c->topk_group < 1 || c->topk_group > c->n_group) return MOE_ERR_INVALID_ARG;
    if ((int64_t)c->topk_group * (c->E / c->n_group) < c->k) return MOE_ERR_INVALID_ARG;
  }
  if (c->n_shared < 0 || c->n_shared > 8 || c->k + c->n_shared > 32) return MOE_ERR_INVALID_ARG;
  if (c->weight_format != MOE_WEIGHTS_NATIVE && c->weight_format != MOE_WEIGHTS_FP8_E4M3_B128)
    return MOE_ERR_INVALID_ARG;
  if (c->weight_format == MOE_WEIGHTS_FP8_E4M3_B128) {
    // FP8 codes feed the bf16 tensor-core path; byte rows must be 16-byte multiples.
    if (c->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (c->H % 16 || c->I % 16) return MOE_ERR_INVALID_ARG;
    if (!c->w13_scale || !c->w2_scale || ((uintptr_t)c->w13_scale & 3u) ||
        ((uintptr_t)c->w2_scale & 3u))
      return MOE_ERR_INVALID_ARG;
  }
  if (c->E + c->n_shared > kMaxE) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)c->T * (c->k + c->n_shared) > (int64_t)1 << 30) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// The configuration the align step, the grouped GEMMs and the combine see: shared experts
// are ordinary experts E..E+n_shared-1 present in slots k..k+n_shared-1 of every token.
static moe_config_t effective(const moe_config_t* c) {
  moe_config_t e = *c;
  e.k = c->k + c->n_shared;
  e.E = c->E + c->n_shared;
  e.n_shared = 0;
  return e;
}

static int block_m_for(moe_dtype_t d) { return d == MOE_BF16 ? 128 : 16; }

static bool block_m_ok(const moe_config_t* c, int block_m) {
  return block_m >= 1 && block_m % block_m_for(c->dtype) == 0 && block_m <= 4096;
}

// Bytes of the gathered routed rows in padded order (bf16 path only).
static size_t gather_bytes(const moe_config_t* c, int block_m) {
  if (c->dtype != MOE_BF16) return 0;
  return align_up(moe_max_padded_rows(c->T, c->k, c->E, block_m) * (size_t)c->H * 2, 256);
}
// Bytes of GEMM1's scratch: the gathered rows (bf16).
static size_t gemm1_scratch_bytes(const moe_config_t* c, int block_m) {
  return gather_bytes(c, block_m);
}

// FP8 weights at batches the CTA-pair kernels take with at least kDequantRows routed rows per
// expert on average: moe_forward turns each grouped GEMM's weights into bf16 in its workspace
// first and runs the bf16 kernel, instead of converting inside the GEMM (see dequant.cu).
// The pass costs 3 bytes a weight; it pays where the GEMMs are compute-bound. Measured on
// GB300 (layer, CUDA graph): Mixtral shape (1024 rows an expert) 4.48 -> 2.46 ms, Qwen3
// shape (512 on average) 4.79 -> 3.28 ms, DeepSeek-V3 shape (128) 9.18 -> 11.07 ms.
constexpr int64_t kDequantRows = 256;
static bool fp8_dequant_applies(const moe_config_t& e, int max_padded) {
  return e.weight_format == MOE_WEIGHTS_FP8_E4M3_B128 && e.dtype == MOE_BF16 &&
         !gemv_applies(e, max_padded) && !dec_gemm_applies(e, max_padded) &&
         (int64_t)e.T * e.k >= kDequantRows * e.E;
}
static size_t dequant_bytes(const moe_config_t& e, int max_padded) {
  return fp8_dequant_applies(e, max_padded)
             ? align_up((size_t)e.E * 2 * (size_t)e.I * (size_t)e.H * 2, 256)
             : 0;
}

// Argument checks of the align entry points (moe_align, moe_align_noalloc) and the padded
// table length they write.
moe_status_t align_check_args(const int32_t* topk_ids, int T, int k, int E, int block_m,
                              const int32_t* sorted_ids, const int32_t* expert_ids,
                              const int32_t* num_post_padded, int* max_padded) {
  if (!topk_ids || !sorted_ids || !expert_ids || !num_post_padded) return MOE_ERR_INVALID_ARG;
  if (T < 1 || k < 1 || E < 1 || k > E || block_m < 1 || block_m > 4096)
    return MOE_ERR_INVALID_ARG;
  if (E > kMaxE) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)T * k > (int64_t)1 << 30) return MOE_ERR_UNSUPPORTED;
  *max_padded = (int)moe_max_padded_rows(T, k, E, block_m);
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_abi_version(void) { return MOE_ABI_VERSION; }

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

int moe_block_m(const moe_config_t* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return block_m_for(cfg->dtype);
}

int moe_small_batch(const moe_config_t* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  const moe_config_t e = effective(cfg);
  const int B = block_m_for(e.dtype);
  return gemv_applies(e, (int)moe_max_padded_rows(e.T, e.k, e.E, B)) ? 1 : 0;
}

moe_status_t moe_dequant_fp8_weights(const moe_config_t* cfg, int matrix, const void* codes,
                                     const int32_t* counts, void* out, cudaStream_t stream) {
  moe_status_t st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (cfg->weight_format != MOE_WEIGHTS_FP8_E4M3_B128 || (matrix != 1 && matrix != 2))
    return MOE_ERR_INVALID_ARG;
  if (!codes || !out || !aligned16(codes) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  const moe_config_t e = effective(cfg);
  if (matrix == 1)
    return launch_dequant_fp8(codes, cfg->w13_scale, e.E, 2 * e.I, e.I, e.H,
                              (int)ceil_div(e.I, 128), (int)ceil_div(e.H, 128), counts, out,
                              stream);
  return launch_dequant_fp8(codes, cfg->w2_scale, e.E, e.H, e.H, e.I, (int)ceil_div(e.H, 128),
                            (int)ceil_div(e.I, 128), counts, out, stream);
}

moe_gemm_kernel_t moe_gemm_kernel(const moe_config_t* cfg) {
  if (check_cfg(cfg) != MOE_OK) return MOE_GEMM_INVALID;
  const moe_config_t e = effective(cfg);
  if (e.dtype != MOE_BF16) return MOE_GEMM_SIMT;
  const int mp = (int)moe_max_padded_rows(e.T, e.k, e.E, block_m_for(e.dtype));
  if (gemv_applies(e, mp)) return MOE_GEMM_SMALL_BATCH;
  if (dec_gemm_applies(e, mp)) return MOE_GEMM_DECODE_TC;
  return MOE_GEMM_PAIR_TC;
}

size_t moe_max_padded_rows(int T, int k, int E, int block_m) {
  if (T < 1 || k < 1 || E < 1 || block_m < 1) return 0;
  // total = sum_e ceil(n_e / B) * B <= T*k + min(E, T*k) * (B - 1), and total is a
  // multiple of B, so it also fits the bound rounded down to whole tiles.
  const int64_t n = (int64_t)T * k;
  const int64_t bound = n + std::min<int64_t>(E, n) * (block_m - 1);
  return (size_t)(bound / block_m * block_m);
}

moe_status_t moe_align_workspace_size(int T, int k, int E, int block_m, size_t* bytes) {
  if (!bytes || T < 1 || k < 1 || k > E || E < 1 || block_m < 1) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE) return MOE_ERR_UNSUPPORTED;
  *bytes = align_scratch_bytes(T, k, E, block_m);
  return MOE_OK;
}

moe_status_t moe_workspace_layout(const moe_config_t* cfg, moe_ws_layout_t* L) {
  moe_status_t st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (!L) return MOE_ERR_INVALID_ARG;
  const moe_config_t eff = effective(cfg);
  const moe_config_t* c = &eff;
  const int B = block_m_for(c->dtype);
  const size_t mp = moe_max_padded_rows(c->T, c->k, c->E, B);
  const size_t es = dtype_size(c->dtype);
  const size_t n = (size_t)c->T * c->k;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L->logits = take((size_t)c->T * cfg->E * 4);
  L->topk_ids = take(n * 4);
  L->topk_w = take(n * 4);
  L->sorted_ids = take(mp * 4);
  L->expert_ids = take(mp / B * 4);
  L->num_post_padded = take(4);
  L->counts = take((size_t)c->E * 4);
  L->align_scratch = take(align_scratch_bytes(c->T, c->k, c->E, B));
  L->act = take(mp * c->I * es);
  L->xs = take(gather_bytes(c, B));
  L->y = take(n * c->H * es);
  L->gemm_scratch = take(dequant_bytes(*c, (int)mp));  // bf16 copy of FP8 weights, or empty
  L->total = off;
  L->block_m = B;
  L->max_padded = (int)mp;
  return MOE_OK;
}

moe_status_t moe_workspace_size(const moe_config_t* c, size_t* bytes) {
  moe_ws_layout_t L;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  moe_status_t st = moe_workspace_layout(c, &L);
  if (st == MOE_OK) *bytes = L.total;
  return st;
}

// The router GEMM of moe_route (logits only). Few tokens (decode): CUDA cores, router rows
// spread over many SMs. Otherwise bf16 runs on the tensor cores (E <= 256 fits one MMA N),
// fp32 on FFMA tiles.
static moe_status_t router_logits(const moe_config_t* c, const void* x, const void* Wg,
                                  float* logits, cudaStream_t stream) {
  if (c->dtype == MOE_BF16 && (!aligned16(x) || !aligned16(Wg))) return MOE_ERR_INVALID_ARG;
  if (c->T <= kFewTokens && aligned16(x) && aligned16(Wg))
    return launch_router_few_tokens(*c, x, Wg, logits, stream);
  if (c->dtype == MOE_BF16 && c->E <= 256) return launch_router_tc(*c, x, Wg, logits, stream);
  return launch_router_simt(*c, x, Wg, logits, stream);
}

moe_status_t moe_route_logits(const moe_config_t* c, const void* x, const void* Wg,
                              float* logits, cudaStream_t stream) {
  moe_status_t st = check_cfg(c);
  if (st != MOE_OK) return st;
  if (!x || !Wg || !logits) return MOE_ERR_INVALID_ARG;
  return router_logits(c, x, Wg, logits, stream);
}

moe_status_t moe_route(const moe_config_t* c, const void* x, const void* Wg, float* logits,
                       int32_t* topk_ids, float* topk_w, cudaStream_t stream) {
  moe_status_t st = check_cfg(c);
  if (st != MOE_OK) return st;
  if (!x || !Wg || !logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if ((st = router_logits(c, x, Wg, logits, stream)) != MOE_OK) return st;
  return launch_topk(*c, logits, topk_ids, topk_w, stream);
}

moe_status_t moe_align(const int32_t* topk_ids, int T, int k, int E, int block_m,
                       int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_post_padded,
                       int32_t* counts, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int mp = 0;
  const moe_status_t st = align_check_args(topk_ids, T, k, E, block_m, sorted_ids, expert_ids,
                                           num_post_padded, &mp);
  if (st != MOE_OK) return st;
  const size_t need = align_scratch_bytes(T, k, E, block_m);
  if (need && (!ws || ws_bytes < need)) return MOE_ERR_WORKSPACE;
  return launch_align(topk_ids, T, k, E, block_m, mp, sorted_ids, expert_ids, num_post_padded,
                      counts, ws, stream);
}

static moe_status_t check_gemm_args(const moe_config_t* c, int block_m) {
  moe_status_t st = check_cfg(c);
  if (st != MOE_OK) return st;
  if (!block_m_ok(c, block_m)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status_t moe_expert_gemm1_workspace_size(const moe_config_t* cfg, int block_m,
                                             size_t* bytes) {
  moe_status_t st = check_gemm_args(cfg, block_m);
  const moe_config_t eff = effective(cfg);
  const moe_config_t* c = &eff;
  if (st != MOE_OK) return st;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = gemm1_scratch_bytes(c, block_m);
  return MOE_OK;
}

moe_status_t moe_gather_rows(const void* x, const int32_t* sorted_ids,
                             const int32_t* num_post_padded, int T, int k, int H,
                             moe_dtype_t dtype, void* xs, cudaStream_t stream) {
  if (!x || !sorted_ids || !num_post_padded || !xs || T < 1 || k < 1 || H < 8 || H % 8)
    return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_F32 && dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(xs)) return MOE_ERR_INVALID_ARG;
  return launch_gather_rows(x, sorted_ids, num_post_padded, T * k, k,
                            H * (int)dtype_size(dtype), xs, stream);
}

moe_status_t moe_expert_gemm1_gathered_workspace_size(const moe_config_t* cfg, int block_m,
                                                      size_t* bytes) {
  moe_status_t st = check_gemm_args(cfg, block_m);
  if (st != MOE_OK) return st;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = 0;  // the kernels need no scratch
  return MOE_OK;
}

moe_status_t moe_expert_gemm1_gathered(const moe_config_t* cfg, const void* xs,
                                       const void* W13, const int32_t* sorted_ids,
                                       const int32_t* expert_ids, const int32_t* npp,
                                       int block_m, void* act, void* ws, size_t ws_bytes,
                                       cudaStream_t stream) {
  moe_status_t st = check_gemm_args(cfg, block_m);
  const moe_config_t eff = effective(cfg);
  const moe_config_t* c = &eff;
  if (st != MOE_OK) return st;
  if (c->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (!xs || !W13 || !sorted_ids || !expert_ids || !npp || !act) return MOE_ERR_INVALID_ARG;
  if (!aligned16(xs) || !aligned16(W13) || !aligned16(act)) return MOE_ERR_INVALID_ARG;
  (void)ws;
  (void)ws_bytes;
  const int mp = (int)moe_max_padded_rows(c->T, c->k, c->E, block_m);
  if (gemv_applies(*c, mp))
    return launch_gemv1(*c, xs, true, W13, sorted_ids, expert_ids, npp, block_m, act, stream);
  if (dec_gemm_applies(*c, mp))
    return launch_gemm1_dec(*c, xs, W13, sorted_ids, expert_ids, npp, block_m, mp, act, stream);
  return launch_gemm1_tc(*c, xs, W13, sorted_ids, expert_ids, npp, block_m, mp, act, stream);
}

moe_status_t moe_expert_gemm1(const moe_config_t* cfg, const void* x, const void* W13,
                              const int32_t* sorted_ids, const int32_t* expert_ids,
                              const int32_t* npp, int block_m, void* act, void* ws,
                              size_t ws_bytes, cudaStream_t stream) {
  moe_status_t st = check_gemm_args(cfg, block_m);
  const moe_config_t eff = effective(cfg);
  const moe_config_t* c = &eff;
  if (st != MOE_OK) return st;
  if (!x || !W13 || !sorted_ids || !expert_ids || !npp || !act) return MOE_ERR_INVALID_ARG;
  const int mp = (int)moe_max_padded_rows(c->T, c->k, c->E, block_m);
  if (c->dtype == MOE_BF16) {
    if (gemv_applies(*c, mp)) {  // small batch: the token rows are read in place
      if (!aligned16(x) || !aligned16(W13) || !aligned16(act)) return MOE_ERR_INVALID_ARG;
      return launch_gemv1(*c, x, false, W13, sorted_ids, expert_ids, npp, block_m, act, stream);
    }
    const size_t need = gemm1_scratch_bytes(c, block_m);
    if (!ws || ws_bytes < need || ((uintptr_t)ws & 255u)) return MOE_ERR_WORKSPACE;
    st = moe_gather_rows(x, sorted_ids, npp, c->T, c->k, c->H, c->dtype, ws, stream);
    if (st != MOE_OK) return st;
    const size_t gb = gather_bytes(c, block_m);
    return moe_expert_gemm1_gathered(cfg, ws, W13, sorted_ids, expert_ids, npp, block_m, act,
                                     (uint8_t*)ws + gb, ws_bytes - gb, stream);
  }
  return launch_gemm1_simt(*c, (const float*)x, (const float*)W13, sorted_ids, expert_ids, npp,
                           block_m, mp, (float*)act, stream);
}

moe_status_t moe_expert_gemm2_workspace_size(const moe_config_t* cfg, int block_m,
                                             size_t* bytes) {
  moe_status_t st = check_gemm_args(cfg, block_m);
  if (st != MOE_OK) return st;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = 0;  // the kernels need no scratch
  return MOE_OK;
}

moe_status_t moe_expert_gemm2(const moe_config_t* cfg, const void* act, const void* W2,
                              const int32_t* sorted_ids, const int32_t* expert_ids,
                              const int32_t* npp, int block_m, const float* topk_w, void* y,
                              void* ws, size_t ws_bytes, cudaStream_t stream) {
  moe_status_t st = check_gemm_args(cfg, block_m);
  const moe_config_t eff = effective(cfg);
  const moe_config_t* c = &eff;
  if (st != MOE_OK) return st;
  if (!act || !W2 || !sorted_ids || !expert_ids || !npp || !topk_w || !y)
    return MOE_ERR_INVALID_ARG;
  const int mp = (int)moe_max_padded_rows(c->T, c->k, c->E, block_m);
  if (c->dtype == MOE_BF16) {
    if (!aligned16(act) || !aligned16(W2) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
    (void)ws;
    (void)ws_bytes;
    if (gemv_applies(*c, mp))
      return launch_gemv2(*c, act, W2, sorted_ids, expert_ids, npp, block_m, topk_w, y, stream);
    if (dec_gemm_applies(*c, mp))
      return launch_gemm2_dec(*c, act, W2, sorted_ids, expert_ids, npp, block_m, mp, topk_w, y,
                              stream);
    return launch_gemm2_tc(*c, act, W2, sorted_ids, expert_ids, npp, block_m, mp, topk_w, y,
                           stream);
  }
  return launch_gemm2_simt(*c, (const float*)act, (const float*)W2, sorted_ids, expert_ids, npp,
                           block_m, mp, topk_w, (float*)y, stream);
}

moe_status_t moe_grouped_swiglu_workspace_size(const moe_config_t* cfg, int block_m,
                                               size_t* bytes) {
  moe_status_t st = check_gemm_args(cfg, block_m);
  const moe_config_t eff = effective(cfg);
  const moe_config_t* c = &eff;
  if (st != MOE_OK) return st;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  const size_t mp = moe_max_padded_rows(c->T, c->k, c->E, block_m);
  *bytes = align_up(mp * c->I * dtype_size(c->dtype), 256) + gemm1_scratch_bytes(c, block_m);
  return MOE_OK;
}

moe_status_t moe_grouped_swiglu(const moe_config_t* c, const void* x, const void* W13,
                                const void* W2, const int32_t* sorted_ids,
                                const int32_t* expert_ids, const int32_t* npp, int block_m,
                                const float* topk_w, void* y, void* ws, size_t ws_bytes,
                                cudaStream_t stream) {
  size_t need = 0;
  moe_status_t st = moe_grouped_swiglu_workspace_size(c, block_m, &need);
  if (st != MOE_OK) return st;
  if (!ws || ws_bytes < need || ((uintptr_t)ws & 255u)) return MOE_ERR_WORKSPACE;
  const moe_config_t eff = effective(c);
  const size_t mp = moe_max_padded_rows(eff.T, eff.k, eff.E, block_m);
  const size_t act_bytes = align_up(mp * eff.I * dtype_size(eff.dtype), 256);
  uint8_t* act = (uint8_t*)ws;
  st = moe_expert_gemm1(c, x, W13, sorted_ids, expert_ids, npp, block_m, act, act + act_bytes,
                        ws_bytes - act_bytes, stream);
  if (st != MOE_OK) return st;
  return moe_expert_gemm2(c, act, W2, sorted_ids, expert_ids, npp, block_m, topk_w, y,
                          act + act_bytes, ws_bytes - act_bytes, stream);
}

moe_status_t moe_combine(const void* y, int T, int k, int H, moe_dtype_t dtype, void* out,
                         cudaStream_t stream) {
  if (!y || !out || T < 1 || k < 1 || H < 8 || H % 8) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_F32 && dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  return launch_combine(y, T, k, H, dtype, out, stream);
}

moe_status_t moe_apply_expert_map(int32_t* expert_ids, int num_tiles, const int32_t* expert_map,
                                  int E, cudaStream_t stream) {
  if (!expert_ids || !expert_map || num_tiles < 0 || E < 1) return MOE_ERR_INVALID_ARG;
  if (num_tiles == 0) return MOE_OK;
  return launch_apply_expert_map(expert_ids, num_tiles, expert_map, E, stream);
}

moe_status_t moe_combine_local(const void* y, const int32_t* topk_ids, const int32_t* expert_map,
                               int E, int T, int k, int H, moe_dtype_t dtype, void* out,
                               cudaStream_t stream) {
  if (!y || !topk_ids || !expert_map || !out || E < 1 || T < 1 || k < 1 || H < 8 || H % 8)
    return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_F32 && dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  return launch_combine_local(y, topk_ids, expert_map, E, T, k, H, dtype, out, stream);
}

// ---- fixed-capacity (masked) layout ---------------------------------------------------
// The masked layout is the grouped GEMMs' padded order with the identity as the table: an
// internal configuration with T = E*C rows, one slot each.
static moe_status_t masked_cfg(const moe_config_t* cfg, int capacity, moe_config_t* m) {
  if (!cfg) return MOE_ERR_INVALID_ARG;
  moe_config_t c = *cfg;
  c.T = 1;
  c.k = 1;
  c.mode = MOE_ROUTE_SOFTMAX;
  c.n_group = c.topk_group = 1;
  c.n_shared = 0;
  c.expert_map = nullptr;
  moe_status_t st = check_cfg(&c);
  if (st != MOE_OK) return st;
  const int B = block_m_for(c.dtype);
  if (capacity < B || capacity % B || (int64_t)capacity * c.E > (int64_t)1 << 29)
    return MOE_ERR_INVALID_ARG;
  c.T = capacity * c.E;
  *m = c;
  return MOE_OK;
}

moe_status_t moe_masked_table(const int32_t* counts, int E, int capacity, int block_m,
                              int32_t* sorted_ids, int32_t* expert_ids,
                              int32_t* num_post_padded, cudaStream_t stream) {
  if (!counts || !sorted_ids || !expert_ids || !num_post_padded || E < 1 || block_m < 1 ||
      capacity < block_m || capacity % block_m)
    return MOE_ERR_INVALID_ARG;
  return launch_masked_table(counts, E, capacity, block_m, sorted_ids, expert_ids,
                             num_post_padded, nullptr, stream);
}

moe_status_t moe_masked_workspace_size(const moe_config_t* cfg, int capacity, size_t* bytes) {
  moe_config_t m;
  moe_status_t st = masked_cfg(cfg, capacity, &m);
  if (st != MOE_OK) return st;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  const size_t n = (size_t)m.T, B = block_m_for(m.dtype);
  *bytes = align_up(n * 4, 256) + align_up(n / B * 4, 256) + 256 + align_up(n * 4, 256) +
           align_up(n * m.I * dtype_size(m.dtype), 256);
  return MOE_OK;
}

moe_status_t moe_masked_forward(const moe_config_t* cfg, const void* x_masked,
                                const int32_t* counts, int capacity, const float* row_w,
                                const void* W13, const void* W2, void* y_masked, void* ws,
                                size_t ws_bytes, cudaStream_t stream) {
  moe_config_t m;
  moe_status_t st = masked_cfg(cfg, capacity, &m);
  if (st != MOE_OK) return st;
  if (!x_masked || !counts || !W13 || !W2 || !y_masked) return MOE_ERR_INVALID_ARG;
  size_t need = 0;
  moe_masked_workspace_size(cfg, capacity, &need);
  if (!ws || ws_bytes < need || ((uintptr_t)ws & 255u)) return MOE_ERR_WORKSPACE;
  const size_t n = (size_t)m.T;
  const int B = block_m_for(m.dtype);
  uint8_t* b = (uint8_t*)ws;
  int32_t* sid = (int32_t*)b;
  b += align_up(n * 4, 256);
  int32_t* eid = (int32_t*)b;
  b += align_up(n / B * 4, 256);
  int32_t* npp = (int32_t*)b;
  b += 256;
  float* ones = (float*)b;
  b += align_up(n * 4, 256);
  void* act = b;
  st = launch_masked_table(counts, m.E, capacity, B, sid, eid, npp, row_w ? nullptr : ones,
                           stream);
  if (st != MOE_OK) return st;
  // The masked rows are already in padded order: GEMM1 reads them directly (bf16) or gathers
  // them with one slot per row (fp32). The row extent handed to the kernels is E*C, the size
  // of the caller's buffers, so tile rows past it read as zeros.
  const int rows = (int)n;
  const float* w = row_w ? row_w : ones;
  if (m.dtype == MOE_BF16) {
    if (!aligned16(x_masked) || !aligned16(W13) || !aligned16(W2) || !aligned16(y_masked))
      return MOE_ERR_INVALID_ARG;
    if (dec_masked_applies(m, capacity)) {
      // capacity 128: at most one tile per expert, holding its few tokens (decode); the
      // decode kernels stream each active expert's weights once
      st = launch_gemm1_dec(m, x_masked, W13, sid, eid, npp, B, rows, act, stream);
      if (st != MOE_OK) return st;
      return launch_gemm2_dec(m, act, W2, sid, eid, npp, B, rows, w, y_masked, stream);
    }
    st = launch_gemm1_tc(m, x_masked, W13, sid, eid, npp, B, rows, act, stream);
    if (st != MOE_OK) return st;
    return launch_gemm2_tc(m, act, W2, sid, eid, npp, B, rows, w, y_masked, stream);
  }
  st = launch_gemm1_simt(m, (const float*)x_masked, (const float*)W13, sid, eid, npp, B, rows,
                         (float*)act, stream);
  if (st != MOE_OK) return st;
  return launch_gemm2_simt(m, (const float*)act, (const float*)W2, sid, eid, npp, B, rows, w,
                           (float*)y_masked, stream);
}

moe_status_t moe_forward(const moe_config_t* c, const void* x, const void* Wg, const void* W13,
                         const void* W2, void* out, void* ws, size_t ws_bytes,
                         cudaStream_t stream) {
  moe_ws_layout_t L;
  moe_status_t st = moe_workspace_layout(c, &L);
  if (st != MOE_OK) return st;
  if (!x || !Wg || !W13 || !W2 || !out) return MOE_ERR_INVALID_ARG;
  if (!ws || ws_bytes < L.total || ((uintptr_t)ws & 255u)) return MOE_ERR_WORKSPACE;
  uint8_t* b = (uint8_t*)ws;
  float* logits = (float*)(b + L.logits);
  int32_t* ids = (int32_t*)(b + L.topk_ids);
  float* w = (float*)(b + L.topk_w);
  int32_t* sid = (int32_t*)(b + L.sorted_ids);
  int32_t* eid = (int32_t*)(b + L.expert_ids);
  int32_t* npp = (int32_t*)(b + L.num_post_padded);
  int32_t* counts = (int32_t*)(b + L.counts);
  const moe_config_t e = effective(c);  // shared experts as ordinary slots / experts
  const bool tiny = topk_table_tiny_fits(*c);
  if (tiny && route_table_tiny_fits(*c) && aligned16(x) && aligned16(Wg)) {
    // at most 32 routed slots, bf16: the router GEMM, then top-k and the table (expert map
    // applied), in one launch
    if ((st = launch_route_table_tiny(*c, x, Wg, logits, ids, w, L.block_m, L.max_padded, sid,
                                      eid, npp, counts, stream)) != MOE_OK)
      return st;
  } else if (tiny) {
    // at most 32 routed slots: router GEMM, then top-k and the table (expert map applied) in
    // one small CTA
    if ((st = router_logits(c, x, Wg, logits, stream)) != MOE_OK) return st;
    if ((st = launch_topk_table_tiny(*c, logits, ids, w, L.block_m, L.max_padded, sid, eid, npp,
                                     counts, stream)) != MOE_OK)
      return st;
  } else if (topk_align_fits(*c)) {
    // decode-sized batch: router GEMM, then top-k and the align table in one CTA (the same
    // device code as moe_route's top-k and moe_align's one-CTA table)
    if ((st = router_logits(c, x, Wg, logits, stream)) != MOE_OK) return st;
    if ((st = launch_topk_align_small(*c, logits, ids, w, L.block_m, L.max_padded, sid, eid,
                                      npp, counts, stream)) != MOE_OK)
      return st;
  } else {
    if ((st = moe_route(c, x, Wg, logits, ids, w, stream)) != MOE_OK) return st;
    if ((st = moe_align(ids, e.T, e.k, e.E, L.block_m, sid, eid, npp, counts,
                        b + L.align_scratch, L.act - L.align_scratch, stream)) != MOE_OK)
      return st;
  }
  if (c->expert_map && !tiny &&
      (st = moe_apply_expert_map(eid, L.max_padded / L.block_m, c->expert_map, e.E, stream)) !=
          MOE_OK)
    return st;
  const bool small = e.dtype == MOE_BF16 && gemv_applies(e, (int)L.max_padded);
  // FP8 weights of a large batch: the grouped GEMMs run on bf16 copies in the workspace
  // (cb: the same layer with those weights); experts no row reached are not converted
  // unless an expert map relabels the tiles
  const bool dq = fp8_dequant_applies(e, (int)L.max_padded);
  moe_config_t cb = *c;
  cb.weight_format = MOE_WEIGHTS_NATIVE;
  cb.w13_scale = cb.w2_scale = nullptr;
  const int32_t* dq_counts = c->expert_map ? nullptr : counts;
  if (small) {
    // a small batch: GEMM1 reads the token rows in place, no gather pass; GEMM2 directly
    // follows it, so its first weight loads may start before its dependency wait
    if (!aligned16(x) || !aligned16(W13) || !aligned16(W2)) return MOE_ERR_INVALID_ARG;
    if ((st = launch_gemv1(e, x, false, W13, sid, eid, npp, L.block_m, b + L.act, stream)) !=
        MOE_OK)
      return st;
    if ((st = launch_gemv2(e, b + L.act, W2, sid, eid, npp, L.block_m, w, b + L.y, stream,
                           true)) != MOE_OK)
      return st;
  } else if (e.dtype == MOE_BF16) {  // gather pass, then the tensor-core GEMM1
    if ((st = moe_gather_rows(x, sid, npp, e.T, e.k, e.H, e.dtype, b + L.xs, stream)) != MOE_OK)
      return st;
    const void* w13 = W13;
    if (dq) {  // FP8 weights of a large batch: bf16 gate/up weights first
      if ((st = moe_dequant_fp8_weights(c, 1, W13, dq_counts, b + L.gemm_scratch, stream)) !=
          MOE_OK)
        return st;
      w13 = b + L.gemm_scratch;
    }
    if ((st = moe_expert_gemm1_gathered(dq ? &cb : c, b + L.xs, w13, sid, eid, npp, L.block_m,
                                        b + L.act, nullptr, 0, stream)) != MOE_OK)
      return st;
  } else if ((st = moe_expert_gemm1(c, x, W13, sid, eid, npp, L.block_m, b + L.act, nullptr, 0,
                                    stream)) != MOE_OK) {
    return st;
  }
  if (dq &&  // and bf16 down-projection weights, over the gate/up copy GEMM1 is done with
      (st = moe_dequant_fp8_weights(c, 2, W2, dq_counts, b + L.gemm_scratch, stream)) != MOE_OK)
    return st;
  if (!small && (st = moe_expert_gemm2(dq ? &cb : c, b + L.act, dq ? b + L.gemm_scratch : W2, sid,
                                       eid, npp, L.block_m, w, b + L.y, nullptr, 0, stream)) !=
                    MOE_OK)
    return st;
  if (c->expert_map)
    return moe_combine_local(b + L.y, ids, c->expert_map, e.E, e.T, e.k, e.H, e.dtype, out,
                             stream);
  return moe_combine(b + L.y, e.T, e.k, e.H, e.dtype, out, stream);
}

moe_status_t moe_selftest_wait_timeout(cudaStream_t stream) {
  return launch_selftest_wait(stream);
}

int moe_device_status(int reset) {
  const int a = align_status_read(reset);
  const int r = router_status_read(reset);
  const int g = grouped_status_read(reset);
  const int c = combine_status_read(reset);
  const int t = tiny_status_read(reset);
  const int d = dec_status_read(reset);
  return g ? g : (d ? d : (r ? r : (a ? a : (t ? t : c))));
}

}  // extern "C"
