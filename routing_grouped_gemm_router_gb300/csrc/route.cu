// route.cu — router logits on CUDA cores (fp32 configs) and the warp-per-token top-k.
//
// Router semantics follow "Mixture-of-Experts Kernels: Routing, Permutation, and Grouped
// GEMM": §3 route() (softmax over E, top-k, renormalise) and §4 route_grouped() (sigmoid
// scores, selection-only bias, groups scored by the sum of their two best biased scores,
// top-k inside the kept groups, weights from the unbiased scores, renormalise, scale).
#include "route_dev.cuh"

namespace moe {

// ------------------------------------------------------------------------------------
// Router GEMM on CUDA cores: logits[T,E] = x[T,H] . Wg[E,H]^T, fp32 FMA accumulation.
// 64x64 output tile per 256-thread block, 4x4 outputs per thread, K staged through shared
// memory 32 at a time. Used for fp32 layers (bf16 layers use the tensor-core GEMM).
// ------------------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__global__ void __launch_bounds__(256) router_simt_kernel(const T* __restrict__ x,
                                                          const T* __restrict__ Wg,
                                                          float* __restrict__ logits, int Tn,
                                                          int H, int E) {
  pdl_wait();
  pdl_trigger();
  __shared__ float xs[32][64 + 1];
  __shared__ float ws[32][64 + 1];
  const int t0 = blockIdx.x * 64, e0 = blockIdx.y * 64;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  for (int h0 = 0; h0 < H; h0 += 32) {
    for (int i = threadIdx.x; i < 64 * 32; i += 256) {
      int r = i / 32, kk = i % 32;
      int t = t0 + r, e = e0 + r, h = h0 + kk;
      xs[kk][r] = (t < Tn && h < H) ? to_f32(x[(size_t)t * H + h]) : 0.f;
      ws[kk][r] = (e < E && h < H) ? to_f32(Wg[(size_t)e * H + h]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int t = t0 + ty * 4 + i;
    if (t >= Tn) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int e = e0 + tx * 4 + j;
      if (e < E) logits[(size_t)t * E + e] = acc[i][j];
    }
  }
}

// ------------------------------------------------------------------------------------
// Router GEMM for few tokens (decode): a warp owns one expert and a block of TB tokens,
// streams that expert's router row in 16-byte pieces and keeps one fp32 sum per token; lane
// partial sums are reduced with shuffles. E/8 x ceil(T/TB) CTAs of 8 warps spread the
// router matrix over many SMs instead of one tensor-core tile.
// ------------------------------------------------------------------------------------
template <typename T, int TB>
__global__ void __launch_bounds__(256) router_few_tokens_kernel(const T* __restrict__ x,
                                                                const T* __restrict__ Wg,
                                                                float* __restrict__ logits,
                                                                int Tn, int H, int E) {
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x / 32;
  const int e = blockIdx.x * 8 + warp;
  const int t0 = blockIdx.y * TB;
  if (e >= E) return;
  router_warp_logits<T, TB>(x, Wg, logits, t0, Tn, H, E, e);
}

template <int TB>
static moe_status_t launch_few(const moe_config_t& c, const void* x, const void* Wg,
                               float* logits, cudaStream_t s) {
  dim3 grid(ceil_div(c.E, 8), ceil_div(c.T, TB));
  if (c.dtype == MOE_F32)
    return launch_k(router_few_tokens_kernel<float, TB>, grid, dim3(256), 0, s, (const float*)x,
                    (const float*)Wg, logits, c.T, c.H, c.E);
  return launch_k(router_few_tokens_kernel<__nv_bfloat16, TB>, grid, dim3(256), 0, s,
                  (const __nv_bfloat16*)x, (const __nv_bfloat16*)Wg, logits, c.T, c.H, c.E);
}

moe_status_t launch_router_few_tokens(const moe_config_t& c, const void* x, const void* Wg,
                                      float* logits, cudaStream_t s) {
  if (c.T <= 1) return launch_few<1>(c, x, Wg, logits, s);
  if (c.T <= 8) return launch_few<8>(c, x, Wg, logits, s);
  return launch_few<16>(c, x, Wg, logits, s);
}

moe_status_t launch_router_simt(const moe_config_t& c, const void* x, const void* Wg,
                                float* logits, cudaStream_t s) {
  dim3 grid(ceil_div(c.T, 64), ceil_div(c.E, 64));
  if (c.dtype == MOE_F32)
    return launch_k(router_simt_kernel<float>, grid, dim3(256), 0, s, (const float*)x,
                    (const float*)Wg, logits, c.T, c.H, c.E);
  return launch_k(router_simt_kernel<__nv_bfloat16>, grid, dim3(256), 0, s, (const __nv_bfloat16*)x,
                  (const __nv_bfloat16*)Wg, logits, c.T, c.H, c.E);
}

// ------------------------------------------------------------------------------------
// Top-k: one warp per token. Lane l holds experts e = l + 32*i. Each of the k rounds is a
// warp-wide argmax (larger key wins, equal keys go to the lower id) over the experts not
// taken yet, so slot j holds the j-th largest key.
// ------------------------------------------------------------------------------------
template <int MPL>
__global__ void __launch_bounds__(kTopkWarps * 32) topk_kernel(
    const float* __restrict__ logits, int Tn, int E, int k, int mode, int renorm, float scale,
    int n_group, int topk_group, const float* __restrict__ logit_bias,
    const float* __restrict__ select_bias, int n_shared, int32_t* __restrict__ ids,
    float* __restrict__ w) {
  pdl_wait();
  pdl_trigger();
  __shared__ float skey[kTopkWarps][512];
  const int warp = threadIdx.x / 32;
  const int t = blockIdx.x * kTopkWarps + warp;
  if (t >= Tn) return;
  topk_token<MPL>(logits, t, E, k, mode, renorm, scale, n_group, topk_group, logit_bias, select_bias,
             n_shared, ids, w, skey[warp]);
}

template <int MPL>
static moe_status_t launch_topk_mpl(const moe_config_t& c, const float* logits, int32_t* ids,
                                    float* w, cudaStream_t s) {
  int grid = ceil_div(c.T, kTopkWarps);
  return launch_k(topk_kernel<MPL>, dim3(grid), dim3(kTopkWarps * 32), 0, s, logits, c.T, c.E,
                  c.k, (int)c.mode, c.renormalize, c.scale, c.n_group, c.topk_group,
                  c.logit_bias, c.select_bias, c.n_shared, ids, w);
}

moe_status_t launch_topk(const moe_config_t& c, const float* logits, int32_t* ids, float* w,
                         cudaStream_t s) {
  switch (topk_per_lane(c.E)) {
    case 4: return launch_topk_mpl<4>(c, logits, ids, w, s);
    case 8: return launch_topk_mpl<8>(c, logits, ids, w, s);
    default: return launch_topk_mpl<kMaxPerLane>(c, logits, ids, w, s);
  }
}

}  // namespace moe
