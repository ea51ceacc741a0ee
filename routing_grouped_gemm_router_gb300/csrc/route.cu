// route.cu — router logits on CUDA cores (fp32 configs) and the warp-per-token top-k.
//
// Router semantics follow "Mixture-of-Experts Kernels: Routing, Permutation, and Grouped
// GEMM": §3 route() (softmax over E, top-k, renormalise) and §4 route_grouped() (sigmoid
// scores, selection-only bias, groups scored by the sum of their two best biased scores,
// top-k inside the kept groups, weights from the unbiased scores, renormalise, scale).
#include "common.cuh"

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
template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&v)[8]);
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 q = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename T, int TB>
__global__ void __launch_bounds__(256) router_few_tokens_kernel(const T* __restrict__ x,
                                                                const T* __restrict__ Wg,
                                                                float* __restrict__ logits,
                                                                int Tn, int H, int E) {
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int e = blockIdx.x * 8 + warp;
  const int t0 = blockIdx.y * TB;
  if (e >= E) return;
  // Token rows past the end are clamped to the last row (loaded, never stored), so every
  // load below is unconditional and the loads of a group can all be in flight together.
  const T* xr[TB];
#pragma unroll
  for (int t = 0; t < TB; ++t) xr[t] = x + (size_t)min(t0 + t, Tn - 1) * H;
  float acc[TB];
#pragma unroll
  for (int t = 0; t < TB; ++t) acc[t] = 0.f;
  const T* w = Wg + (size_t)e * H;
#pragma unroll 2
  for (int h = lane * 8; h < H; h += 256) {
    float wv[8];
    load8(w + h, wv);
#pragma unroll
    for (int tg = 0; tg < TB; tg += 8) {
      constexpr int G = TB < 8 ? TB : 8;
      float xv[G][8];
#pragma unroll
      for (int j = 0; j < G; ++j) load8(xr[tg + j] + h, xv[j]);
#pragma unroll
      for (int j = 0; j < G; ++j)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[tg + j] = fmaf(xv[j][q], wv[q], acc[tg + j]);
    }
  }
#pragma unroll
  for (int t = 0; t < TB; ++t) {
    float v = acc[t];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == (t & 31) && t0 + t < Tn) logits[(size_t)(t0 + t) * E + e] = v;
  }
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
struct KeyId {
  float v;
  int e;
};

__device__ __forceinline__ bool better(float v, int e, float v2, int e2) {
  return v > v2 || (v == v2 && e < e2);
}

__device__ __forceinline__ KeyId warp_argmax(float v, int e) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float v2 = __shfl_xor_sync(0xffffffffu, v, off);
    int e2 = __shfl_xor_sync(0xffffffffu, e, off);
    if (better(v2, e2, v, e)) { v = v2; e = e2; }
  }
  return {v, e};
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

constexpr int kTopkWarps = 8;
constexpr int kMaxPerLane = 16;  // E <= 512

__global__ void __launch_bounds__(kTopkWarps * 32) topk_kernel(
    const float* __restrict__ logits, int Tn, int E, int k, int mode, int renorm, float scale,
    int n_group, int topk_group, const float* __restrict__ logit_bias,
    const float* __restrict__ select_bias, int n_shared, int32_t* __restrict__ ids,
    float* __restrict__ w) {
  pdl_wait();
  pdl_trigger();
  __shared__ float skey[kTopkWarps][512];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int t = blockIdx.x * kTopkWarps + warp;
  if (t >= Tn) return;
  const float* lrow = logits + (size_t)t * E;
  const float NEG = -INFINITY;

  float key[kMaxPerLane], val[kMaxPerLane];
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) {
    int e = lane + 32 * i;
    key[i] = NEG;
    val[i] = 0.f;
    if (e < E) {
      float l = lrow[e];
      if (mode == MOE_ROUTE_SOFTMAX) {
        if (logit_bias) l += logit_bias[e];
        key[i] = l;
        val[i] = l;
      } else {
        float sg = 1.f / (1.f + expf(-l));
        val[i] = sg;
        key[i] = select_bias ? sg + select_bias[e] : sg;
      }
    }
  }

  if (mode == MOE_ROUTE_SIGMOID_GROUPED && n_group > 1) {
    // Group score = sum of the two largest biased keys of E/n_group consecutive experts.
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      int e = lane + 32 * i;
      if (e < E) skey[warp][e] = key[i];
    }
    __syncwarp();
    const int per = E / n_group;
    float gscore = NEG;
    if (lane < n_group) {
      float b1 = NEG, b2 = NEG;
      for (int q = 0; q < per; ++q) {
        float v = skey[warp][lane * per + q];
        if (v > b1) { b2 = b1; b1 = v; } else if (v > b2) { b2 = v; }
      }
      gscore = per >= 2 ? b1 + b2 : b1;
    }
    uint32_t kept = 0;
    for (int g = 0; g < topk_group; ++g) {
      KeyId best = warp_argmax(lane < n_group ? gscore : NEG, lane < n_group ? lane : 1 << 30);
      kept |= 1u << best.e;
      if (lane == best.e) gscore = NEG;
    }
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      int e = lane + 32 * i;
      if (e < E && !((kept >> (e / per)) & 1u)) key[i] = NEG;
    }
  }

  // k rounds of warp argmax. Taken entries drop to a key below every real one.
  float my_sel_val = 0.f;   // lane j keeps the value of slot j
  int my_sel_id = 0;
  bool taken[kMaxPerLane];
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) taken[i] = false;
  for (int j = 0; j < k; ++j) {
    float bv = NEG;
    int be = 1 << 30;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      int e = lane + 32 * i;
      if (e < E && !taken[i] && (be == (1 << 30) || better(key[i], e, bv, be))) {
        bv = key[i];
        be = e;
      }
    }
    KeyId best = warp_argmax(bv, be);
    float sel_val = 0.f;
    if ((best.e & 31) == lane) {
      int i = best.e >> 5;
#pragma unroll
      for (int q = 0; q < kMaxPerLane; ++q)
        if (q == i) { taken[q] = true; sel_val = val[q]; }
    }
    sel_val = __shfl_sync(0xffffffffu, sel_val, best.e & 31);
    if (lane == j) { my_sel_val = sel_val; my_sel_id = best.e; }
  }

  float wj;
  if (mode == MOE_ROUTE_SOFTMAX) {
    float top = __shfl_sync(0xffffffffu, my_sel_val, 0);  // slot 0 holds the largest logit
    if (renorm) {
      float ex = lane < k ? expf(my_sel_val - top) : 0.f;
      wj = ex / warp_sum(ex);
    } else {
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i) {
        int e = lane + 32 * i;
        if (e < E) part += expf(val[i] - top);
      }
      wj = expf(my_sel_val - top) / warp_sum(part);
    }
  } else {
    float sv = lane < k ? my_sel_val : 0.f;
    wj = renorm ? sv / warp_sum(sv) : sv;
  }
  const int kk = k + n_shared;  // row stride: routed slots, then the shared experts
  if (lane < k) {
    ids[(size_t)t * kk + lane] = my_sel_id;
    w[(size_t)t * kk + lane] = scale * wj;
  } else if (lane < kk) {
    ids[(size_t)t * kk + lane] = E + (lane - k);
    w[(size_t)t * kk + lane] = 1.f;
  }
}

moe_status_t launch_topk(const moe_config_t& c, const float* logits, int32_t* ids, float* w,
                         cudaStream_t s) {
  int grid = ceil_div(c.T, kTopkWarps);
  return launch_k(topk_kernel, dim3(grid), dim3(kTopkWarps * 32), 0, s, logits, c.T, c.E, c.k,
                  (int)c.mode, c.renormalize, c.scale, c.n_group, c.topk_group, c.logit_bias,
                  c.select_bias, c.n_shared, ids, w);
}

}  // namespace moe
