// gemv_dev.cuh — device code of the small-batch grouped GEMMs on CUDA cores (internal
// header of gemv.cu).
//
// One warp owns two weight rows of one expert at a time (an item; GEMM1: the gate and up
// rows of output column n; GEMM2: the rows of columns n and n+1): the 32 lanes stream them
// in 16-byte pieces (512 contiguous bytes of a row per step, several steps in flight) and
// multiply every piece against the tile's real rows in fp32 registers; the lane sums meet
// in a shuffle reduction. FP8 E4M3 weights with 128x128 block scales: each lane's 16 codes
// of a step lie in one 128-wide k-block, so the codes (converted exactly through f16) are
// multiplied against the activations in fp32 and the 16-term partial sum is scaled once by
// its block scale.
#pragma once

#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {
namespace gv {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kTile = 128;  // rows of one tile of the padded order

struct Params {
  const uint8_t* a;  // bf16 activation rows: row p (gathered) or token sorted_ids[p] / k
  int a_gathered;
  const uint8_t* w;    // GEMM1: W13 [E, 2N, K]; GEMM2: W2 [E, N, K]; bf16 or E4M3 codes
  const float* scale;  // FP8: [E, grids, ceil(N/128), ceil(K/128)]; else null
  int sc_rb, sc_kb;
  const int32_t* sid;
  const int32_t* eid;
  const int32_t* npp;
  int block_m, n_rows, k, K, N, n_slots;
  const float* topk_w;  // GEMM2
  void* out;            // GEMM1: act [padded, N]; GEMM2: y [T*k, N] (bf16)
  // GEMM2 inside the fused layer: each warp loads the first pieces of its first item's
  // weight rows before the dependency wait (see gemv_kernel)
  int early;
};

// Weights are read once: no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const uint8_t* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Eight bf16 (one 16-byte piece) to fp32, exactly.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& q, float* f) {
  const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf_lo(u[i]);
    f[2 * i + 1] = bf_hi(u[i]);
  }
}

// Sixteen E4M3 codes (one 16-byte piece, lowest byte first) to fp32, exactly: every E4M3
// value is an f16 value, and every f16 value an fp32 value.
__device__ __forceinline__ void e4m3x16_to_f32(const uint4& q, float* f) {
  const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((u[i] >> (16 * h)) & 0xffffu);
      const float2 fv = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3)));
      f[4 * i + 2 * h] = fv.x;
      f[4 * i + 2 * h + 1] = fv.y;
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Real rows of tile t: their count, and their (p, r) in padded order into rl. CG: the table
// is read past L1 (before the dependency wait).
template <bool CG = false>
__device__ __forceinline__ int tile_rows(const Params& P, int t, int2* rl) {
  const int lane = threadIdx.x % 32;
  int n = 0;
#pragma unroll
  for (int i = 0; i < kTile / 32; ++i) {
    const int p = t * kTile + i * 32 + lane;
    const int r = CG ? __ldcg(P.sid + p) : P.sid[p];
    const bool v = r >= 0 && r < P.n_rows;
    const unsigned m = __ballot_sync(0xffffffffu, v);
    if (v) rl[n + __popc(m & ((1u << lane) - 1u))] = make_int2(p, r);
    n += __popc(m);
  }
  return n;
}

// One pass of an item: weight rows w0, w1 (K elements each) against the real rows rl[0..rv)
// (R >= rv), then the epilogue of the item's output column(s) n for those rows. S: 16-byte
// pieces of each weight row in flight.
// Pieces in flight per row and CTAs per SM, measured at one and two tokens on GB300: bf16
// passes of 1-2 rows run 3 CTAs an SM (80 registers; 6 or 4 pieces in flight), 5-6 % faster
// than 2 CTAs with 8 pieces; FP8 codes (half the bytes a piece) keep 2 CTAs and 8 pieces.
template <int MODE, bool FP8, int RMAX>
constexpr int kMinCtas = (!FP8 && RMAX <= 2) ? 3 : 2;
template <int MODE, bool FP8, int RMAX>
constexpr int kPieces = RMAX == 1 ? (FP8 ? 8 : 6) : 4;

// Activation rows: read-only inputs of the launch, through the non-coherent path (L1-cached;
// every warp of a tile reads them).
__device__ __forceinline__ uint4 ld_act(const uint8_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// PRE: the first S pieces of both rows are already in pre0 / pre1 (loaded by the caller).
template <int MODE, bool FP8, int R, int S, bool PRE = false>
__device__ __forceinline__ void item_pass(const Params& P, const uint8_t* w0, const uint8_t* w1,
                                          const float* s0, const float* s1, const int2* rl,
                                          int rv, int n, const uint4 (&pre0)[S] = {},
                                          const uint4 (&pre1)[S] = {}) {
  constexpr int EPL = FP8 ? 16 : 8;  // elements of a 16-byte weight piece
  constexpr int ES = FP8 ? 1 : 2;    // weight element bytes
  constexpr int kStride = 32 * EPL;  // elements per warp step
  // Rows past rv are skipped (warp-uniform branches) where their multiply-adds would cost
  // issue slots: FP8 codes and passes of four rows (a decode tile mostly holds one real row).
  // Measured on GB300 (gpt-oss-shaped layer, FP8 weights): 23-25 % less time a layer at 4 to
  // 16 tokens. bf16 passes of two rows stream well below the issue rate, and the branches
  // would cost them registers.
  constexpr bool kSkip = R > 1 && (FP8 || R > 2);
  const int lane = threadIdx.x % 32;
  const int K = P.K;
  const uint8_t* ar[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int2 q = rl[min(r, rv - 1)];
    ar[r] = P.a + (size_t)(P.a_gathered ? q.x : q.y / P.k) * K * 2;
  }
  float a0[R], a1[R];
#pragma unroll
  for (int r = 0; r < R; ++r) a0[r] = a1[r] = 0.f;
  // one step of S pieces of both rows at k0 into the row sums
  auto step = [&](const uint4 (&q0)[S], const uint4 (&q1)[S], int k0) {
#pragma unroll
    for (int j = 0; j < S; ++j) {
      const int kk = k0 + j * kStride;
      if (kk >= K) break;
      if constexpr (FP8) {
        float f0[16], f1[16];
        e4m3x16_to_f32(q0[j], f0);
        e4m3x16_to_f32(q1[j], f1);
        const float sc0 = __ldg(s0 + kk / 128), sc1 = __ldg(s1 + kk / 128);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          if (kSkip && r >= rv) break;
          float xf[16];
          bf16x8_to_f32(ld_act(ar[r] + (size_t)kk * 2), xf);
          bf16x8_to_f32(ld_act(ar[r] + (size_t)kk * 2 + 16), xf + 8);
          float p0 = 0.f, p1 = 0.f;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            p0 = fmaf(f0[i], xf[i], p0);
            p1 = fmaf(f1[i], xf[i], p1);
          }
          a0[r] = fmaf(sc0, p0, a0[r]);
          a1[r] = fmaf(sc1, p1, a1[r]);
        }
      } else {
        float f0[8], f1[8];
        bf16x8_to_f32(q0[j], f0);
        bf16x8_to_f32(q1[j], f1);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          if (kSkip && r >= rv) break;
          float xf[8];
          bf16x8_to_f32(ld_act(ar[r] + (size_t)kk * 2), xf);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            a0[r] = fmaf(f0[i], xf[i], a0[r]);
            a1[r] = fmaf(f1[i], xf[i], a1[r]);
          }
        }
      }
    }
  };
  int k0 = lane * EPL;
  if constexpr (PRE) {  // the first step from the pieces already loaded
    step(pre0, pre1, k0);
    k0 += kStride * S;
  }
  for (; k0 < K; k0 += kStride * S) {
    uint4 q0[S], q1[S];
#pragma unroll
    for (int j = 0; j < S; ++j) {
      const int kk = k0 + j * kStride;
      if (kk < K) {
        q0[j] = ld_stream(w0 + (size_t)kk * ES);
        q1[j] = ld_stream(w1 + (size_t)kk * ES);
      }
    }
    step(q0, q1, k0);
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (kSkip && r >= rv) break;
    const float d0 = warp_sum(a0[r]), d1 = warp_sum(a1[r]);
    if (r < rv && lane == r) {
      const int2 q = rl[r];
      if (MODE == 0) {
        const float v = d0 / (1.f + __expf(-d0)) * d1;
        reinterpret_cast<__nv_bfloat16*>(P.out)[(size_t)q.x * P.N + n] = __float2bfloat16(v);
      } else {
        const float wr = P.topk_w[q.y];
        *reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(P.out) +
                                     (size_t)q.y * P.N + n) = pack_bf16x2(wr * d0, wr * d1);
      }
    }
  }
}

}  // namespace gv
}  // namespace moe
