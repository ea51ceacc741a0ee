// route_dev.cuh — device building blocks of the router shared by the router kernels, the
// top-k kernel and the small-batch top-k + align kernel (internal header). The arithmetic
// lives only here, so the combined and the separate paths produce identical ids and weights.
#pragma once

#include "common.cuh"

namespace moe {

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

// One warp computes the router logits of expert e for tokens t0 .. t0+TB-1 (rows past Tn
// are clamped to the last token, loaded and never stored, so every load is unconditional):
// the expert's router row streams in 16-byte pieces, one fp32 sum per token, lane partial
// sums reduced with shuffles.
template <typename T, int TB>
__device__ __forceinline__ void router_warp_logits(const T* __restrict__ x,
                                                   const T* __restrict__ Wg,
                                                   float* __restrict__ logits, int t0, int Tn,
                                                   int H, int E, int e) {
  const int lane = threadIdx.x % 32;
  const T* xr[TB];
#pragma unroll
  for (int t = 0; t < TB; ++t) xr[t] = x + (size_t)min(t0 + t, Tn - 1) * H;
  float acc[TB];
#pragma unroll
  for (int t = 0; t < TB; ++t) acc[t] = 0.f;
  const T* w = Wg + (size_t)e * H;
  if constexpr (TB == 1 && sizeof(T) == 2) {
    // one bf16 token: eight 16-byte pieces of the router row (and of x) in flight a lane, all
    // loaded before any is used, so a 2880-wide row takes two round trips
    constexpr int kPieces = 8;
    for (int h0 = lane * 8; h0 < H; h0 += 256 * kPieces) {
      uint4 wq[kPieces], xq[kPieces];
#pragma unroll
      for (int j = 0; j < kPieces; ++j) {
        const int h = h0 + j * 256;
        if (h < H) {
          wq[j] = *reinterpret_cast<const uint4*>(w + h);
          xq[j] = *reinterpret_cast<const uint4*>(xr[0] + h);
        }
      }
#pragma unroll
      for (int j = 0; j < kPieces; ++j) {
        if (h0 + j * 256 >= H) break;
        const __nv_bfloat162* wp = reinterpret_cast<const __nv_bfloat162*>(&wq[j]);
        const __nv_bfloat162* xp = reinterpret_cast<const __nv_bfloat162*>(&xq[j]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 wf = __bfloat1622float2(wp[i]), xf = __bfloat1622float2(xp[i]);
          acc[0] = fmaf(xf.x, wf.x, acc[0]);
          acc[0] = fmaf(xf.y, wf.y, acc[0]);
        }
      }
    }
  } else {
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
  }
#pragma unroll
  for (int t = 0; t < TB; ++t) {
    float v = acc[t];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == (t & 31) && t0 + t < Tn) logits[(size_t)(t0 + t) * E + e] = v;
  }
}

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

// The K best (key, expert, value) entries of a warp, sorted (larger key first, equal keys to
// the lower expert id), in every lane. Lane l holds the candidates of experts l + 32*i
// (i < MPL); each lane first keeps its own K best by insertion, then five butterfly steps
// merge each lane's list with its xor partner's: the element-wise better of one list and
// the other list reversed is a bitonic sequence holding the K best of both, which a bitonic
// merge network puts back in order. Both lanes of a pair end with the same list, and after
// the fifth step every lane holds the warp's K best. The order is a total order, so the
// result is the one k rounds of warp argmax give, in a few dependent shuffle steps instead of
// k times five.
template <int MPL, int K>
__device__ __forceinline__ void warp_topk_sorted(const float (&key)[MPL], const float (&val)[MPL],
                                                 int E, float (&lk)[K], int (&li)[K],
                                                 float (&lv)[K]) {
  const int lane = threadIdx.x % 32;
#pragma unroll
  for (int s = 0; s < K; ++s) {
    lk[s] = -INFINITY;
    li[s] = 0x7fffffff;  // an empty slot sorts after every expert
    lv[s] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < MPL; ++i) {
    const int e = lane + 32 * i;
    if (e >= E) continue;
    float ck = key[i], cv = val[i];
    int ci = e;
#pragma unroll
    for (int s = 0; s < K; ++s) {
      if (better(ck, ci, lk[s], li[s])) {
        const float tk = lk[s], tv = lv[s];
        const int ti = li[s];
        lk[s] = ck; li[s] = ci; lv[s] = cv;
        ck = tk; ci = ti; cv = tv;
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float pk[K], pv[K];
    int pi[K];
#pragma unroll
    for (int s = 0; s < K; ++s) {
      pk[s] = __shfl_xor_sync(0xffffffffu, lk[s], off);
      pi[s] = __shfl_xor_sync(0xffffffffu, li[s], off);
      pv[s] = __shfl_xor_sync(0xffffffffu, lv[s], off);
    }
#pragma unroll
    for (int s = 0; s < K; ++s) {
      if (!better(lk[s], li[s], pk[K - 1 - s], pi[K - 1 - s])) {
        lk[s] = pk[K - 1 - s];
        li[s] = pi[K - 1 - s];
        lv[s] = pv[K - 1 - s];
      }
    }
#pragma unroll
    for (int d = K / 2; d >= 1; d >>= 1) {
#pragma unroll
      for (int s = 0; s < K; ++s) {
        if ((s & d) == 0 && !better(lk[s], li[s], lk[s + d], li[s + d])) {
          const float tk = lk[s], tv = lv[s];
          const int ti = li[s];
          lk[s] = lk[s + d]; li[s] = li[s + d]; lv[s] = lv[s + d];
          lk[s + d] = tk; li[s + d] = ti; lv[s + d] = tv;
        }
      }
    }
  }
}

constexpr int kTopkWarps = 8;
constexpr int kMaxPerLane = 16;  // E <= 512

// Experts a lane holds for E router experts (4, 8 or 16): top-k loops run over that many.
inline int topk_per_lane(int E) { return E <= 128 ? 4 : (E <= 256 ? 8 : kMaxPerLane); }

// Top-k of one token, one warp (lane l holds experts l + 32*i, i < MPL, 32*MPL >= E): the k
// largest keys (equal keys to the lower id), slot j holding the j-th, from the butterfly
// merge when k <= KMAX (KMAX 4 or 8: the registers of the sorted lists; kernels of 1024
// threads keep 4) and otherwise from k rounds of a warp-wide argmax over the experts not
// taken yet; then the weights of the mode (softmax over E or over the k kept logits; sigmoid
// scores renormalised and scaled), written to row t of ids / w, after which the shared
// experts' slots follow. skey_w: this warp's 512 floats of shared memory (used by the group
// scores of mode 1). Logits in global memory (written by an earlier kernel) are read from L2
// (ld.global.cg); with LSH they are in shared memory and read with plain loads (a global-only
// load of a shared address faults).
template <int MPL, int KMAX = 8, bool LSH = false>
__device__ __forceinline__ void topk_token(const float* __restrict__ logits, int t, int E, int k,
                                           int mode, int renorm, float scale, int n_group,
                                           int topk_group, const float* __restrict__ logit_bias,
                                           const float* __restrict__ select_bias, int n_shared,
                                           int32_t* __restrict__ ids, float* __restrict__ w,
                                           float* skey_w) {
  const int lane = threadIdx.x % 32;
  const float* lrow = logits + (size_t)t * E;
  const float NEG = -INFINITY;

  float key[MPL], val[MPL];
#pragma unroll
  for (int i = 0; i < MPL; ++i) {
    int e = lane + 32 * i;
    key[i] = NEG;
    val[i] = 0.f;
    if (e < E) {
      float l = LSH ? lrow[e] : __ldcg(lrow + e);
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
    for (int i = 0; i < MPL; ++i) {
      int e = lane + 32 * i;
      if (e < E) skey_w[e] = key[i];
    }
    __syncwarp();
    const int per = E / n_group;
    float gscore = NEG;
    if (lane < n_group) {
      float b1 = NEG, b2 = NEG;
      for (int q = 0; q < per; ++q) {
        float v = skey_w[lane * per + q];
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
    for (int i = 0; i < MPL; ++i) {
      int e = lane + 32 * i;
      if (e < E && !((kept >> (e / per)) & 1u)) key[i] = NEG;
    }
  }

  float my_sel_val = 0.f;   // lane j keeps the value of slot j
  int my_sel_id = 0;
  if (k <= KMAX) {
    // the k best from the warp's sorted 4 or 8 best (butterfly merge)
    auto take = [&](auto& lk, auto& li, auto& lv) {
#pragma unroll
      for (int s = 0; s < (int)(sizeof(lk) / sizeof(lk[0])); ++s)
        if (lane == s) {
          my_sel_val = lv[s];
          my_sel_id = li[s];
        }
    };
    if (k <= 4) {
      float lk[4], lv[4];
      int li[4];
      warp_topk_sorted<MPL, 4>(key, val, E, lk, li, lv);
      take(lk, li, lv);
    } else if (KMAX >= 8) {
      float lk[8], lv[8];
      int li[8];
      warp_topk_sorted<MPL, 8>(key, val, E, lk, li, lv);
      take(lk, li, lv);
    }
  }
  // larger k: k rounds of warp argmax. Taken entries drop to a key below every real one.
  bool taken[MPL];
#pragma unroll
  for (int i = 0; i < MPL; ++i) taken[i] = false;
  for (int j = 0; k > KMAX && j < k; ++j) {
    float bv = NEG;
    int be = 1 << 30;
#pragma unroll
    for (int i = 0; i < MPL; ++i) {
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
      for (int q = 0; q < MPL; ++q)
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
      for (int i = 0; i < MPL; ++i) {
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

}  // namespace moe
