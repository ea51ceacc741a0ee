// dequant.cu — FP8 E4M3 expert weights with 128 x 128 block scales turned into bf16 weights
// in device memory: out[e, r, k] = bf16(code[e, r, k] * scale of its block), the value the
// grouped GEMMs' converter warps put into the MMA operand (the same device function, so the
// same bits).
//
// The fused layer runs it before each grouped GEMM of a large batch ("Mixture-of-Experts
// Kernels: Routing, Permutation, and Grouped GEMM", §8: at prefill an expert's rows make its
// GEMMs compute-bound, so the weights' bytes matter less than the tensor rate): the bf16
// CTA-pair kernel then runs at its full rate, where converting inside the GEMM costs the
// tensor pipe most of its time. A bandwidth-bound pass: 1 byte read and 2 bytes written per
// weight.
//
// A weight matrix is [E, R, K] codes, its scales [E, grids, ceil(Rg / 128), K / 128] with
// R = grids * Rg (GEMM1: W13, grid 0 the gate rows and grid 1 the up rows, Rg = I; GEMM2: W2,
// one grid, Rg = H). K is a multiple of 16, so a thread's 16 codes lie in one scale block.
#include "tc_ptx.cuh"

namespace moe {

// 32 bytes to global memory in one instruction (needs a 32-byte aligned address): a warp's
// store covers 1 KB with no gaps, where two 16-byte stores a lane each leave every other
// 16 bytes of a sector to the other instruction.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&v)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

template <bool V8>
__global__ void __launch_bounds__(256) dequant_fp8_kernel(const uint4* __restrict__ codes,
                                                          const float* __restrict__ scale,
                                                          int E, int R, int Rg, int K,
                                                          int sc_rb, int sc_kb,
                                                          const int32_t* __restrict__ counts,
                                                          uint4* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int units_row = K / 16;
  const int64_t units_e = (int64_t)R * units_row;
  const int64_t total = (int64_t)E * units_e;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  constexpr int kU = 4;  // units a thread has in flight
  for (int64_t u0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u0 < total;
       u0 += kU * stride) {
    uint4 q[kU];
    bool live[kU];
#pragma unroll
    for (int i = 0; i < kU; ++i) {
      const int64_t u = u0 + i * stride;
      // no row reached expert e: no tile of it runs, its weights are not needed
      live[i] = u < total && (!counts || counts[(int)(u / units_e)] != 0);
      if (live[i]) q[i] = codes[u];
    }
#pragma unroll
    for (int i = 0; i < kU; ++i) {
      if (!live[i]) continue;
      const int64_t u = u0 + i * stride;
      const int e = (int)(u / units_e);
      const int64_t in_e = u - (int64_t)e * units_e;
      const int r = (int)(in_e / units_row);
      const int kc = (int)(in_e - (int64_t)r * units_row) * 16;
      const int grid = r / Rg, rr = r - grid * Rg;
      const float sc =
          __ldg(scale + (((int64_t)e * (R / Rg) + grid) * sc_rb + rr / 128) * sc_kb + kc / 128);
      uint32_t v[8];
      ptx::e4m3x16_scaled_bf16(q[i], sc, v);
      if constexpr (V8) {
        st_global_v8(out + 2 * u, v);
      } else {
        out[2 * u] = make_uint4(v[0], v[1], v[2], v[3]);
        out[2 * u + 1] = make_uint4(v[4], v[5], v[6], v[7]);
      }
    }
  }
}

moe_status_t launch_dequant_fp8(const void* codes, const float* scale, int E, int R, int Rg,
                                int K, int sc_rb, int sc_kb, const int32_t* counts, void* out,
                                cudaStream_t s) {
  if (K % 16 || R % Rg) return MOE_ERR_INVALID_ARG;
  const int64_t units = (int64_t)E * R * (K / 16);
  const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((units + 255) / 256,
                                                                  (int64_t)num_sms() * 8));
  auto kern = ((uintptr_t)out & 31u) == 0 ? dequant_fp8_kernel<true> : dequant_fp8_kernel<false>;
  return launch_k(kern, dim3(blocks), dim3(256), 0, s, (const uint4*)codes, scale, E, R, Rg, K,
                  sc_rb, sc_kb, counts, (uint4*)out);
}

}  // namespace moe
