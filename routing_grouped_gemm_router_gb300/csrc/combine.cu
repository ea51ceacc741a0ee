// combine.cu — out[t, :] = sum_{j<k} y[t*k + j, :] ("Mixture-of-Experts Kernels: Routing,
// Permutation, and Grouped GEMM", §6: the router weight is already folded into y by
// GEMM2, so the combine is a plain sum over the k slots of each token).
//
// HBM-bound: every y element is read once and every out element written once. Each thread
// handles 16 bytes of a row (8 bf16 or 4 fp32), accumulates the k slots in fp32 in slot
// order j = 0..k-1, and the grid is a multiple of the SM count with a grid-stride loop.
#include "common.cuh"

namespace moe {

__device__ int g_combine_status;

int combine_status_read(int reset) {
  int v = 0;
  cudaMemcpyFromSymbol(&v, g_combine_status, sizeof(int));
  if (reset) {
    int z = 0;
    cudaMemcpyToSymbol(g_combine_status, &z, sizeof(int));
  }
  return v;
}

__global__ void __launch_bounds__(256) combine_bf16_kernel(const uint4* __restrict__ y,
                                                           uint4* __restrict__ out, int T,
                                                           int k, int vec_per_row) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = (int64_t)T * vec_per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / vec_per_row, v = i % vec_per_row;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const uint4* src = y + (t * k) * vec_per_row + v;
    for (int j = 0; j < k; ++j) {
      uint4 q = __ldcs(src + (int64_t)j * vec_per_row);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float2 f = __bfloat1622float2(h[c]);
        acc[2 * c] += f.x;
        acc[2 * c + 1] += f.y;
      }
    }
    uint4 o;
    __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int c = 0; c < 4; ++c) oh[c] = __floats2bfloat162_rn(acc[2 * c], acc[2 * c + 1]);
    out[i] = o;
  }
}

__global__ void __launch_bounds__(256) combine_f32_kernel(const float4* __restrict__ y,
                                                          float4* __restrict__ out, int T,
                                                          int k, int vec_per_row) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = (int64_t)T * vec_per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / vec_per_row, v = i % vec_per_row;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4* src = y + (t * k) * vec_per_row + v;
    for (int j = 0; j < k; ++j) {
      float4 q = __ldcs(src + (int64_t)j * vec_per_row);
      acc.x += q.x; acc.y += q.y; acc.z += q.z; acc.w += q.w;
    }
    out[i] = acc;
  }
}

// Expert parallelism: slots whose expert is on another device (map < 0) are skipped, and so
// are slots with an id outside [0, E) (never aligned, so never computed; status 1).
template <bool BF16>
__global__ void __launch_bounds__(256) combine_local_kernel(const void* __restrict__ y,
                                                            const int32_t* __restrict__ ids,
                                                            const int32_t* __restrict__ map,
                                                            void* __restrict__ out, int E, int T,
                                                            int k, int vec_per_row) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = (int64_t)T * vec_per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / vec_per_row, v = i % vec_per_row;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < k; ++j) {
      const int e = ids[t * k + j];
      if (e < 0 || e >= E) {
        if (v == 0) atomicExch(&g_combine_status, kStatusBadExpert);
        continue;
      }
      if (map[e] < 0) continue;
      if (BF16) {
        const uint4 q = __ldcs((const uint4*)y + (t * k + j) * vec_per_row + v);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float2 f = __bfloat1622float2(h[c]);
          acc[2 * c] += f.x;
          acc[2 * c + 1] += f.y;
        }
      } else {
        const float4 q = __ldcs((const float4*)y + (t * k + j) * vec_per_row + v);
        acc[0] += q.x; acc[1] += q.y; acc[2] += q.z; acc[3] += q.w;
      }
    }
    if (BF16) {
      uint4 o;
      __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int c = 0; c < 4; ++c) oh[c] = __floats2bfloat162_rn(acc[2 * c], acc[2 * c + 1]);
      ((uint4*)out)[i] = o;
    } else {
      ((float4*)out)[i] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    }
  }
}

moe_status_t launch_combine_local(const void* y, const int32_t* ids, const int32_t* map, int E,
                                  int T, int k, int H, moe_dtype_t dt, void* out, cudaStream_t s) {
  const int vec = dt == MOE_BF16 ? H / 8 : H / 4;
  const int64_t total = (int64_t)T * vec;
  int blocks = (int)std::min<int64_t>(ceil_div64(total, 256), (int64_t)num_sms() * 8);
  if (blocks < 1) blocks = 1;
  if (dt == MOE_BF16)
    return launch_k(combine_local_kernel<true>, dim3(blocks), dim3(256), 0, s, y, ids, map, out, E,
                    T, k, vec);
  return launch_k(combine_local_kernel<false>, dim3(blocks), dim3(256), 0, s, y, ids, map, out, E,
                  T, k, vec);
}

moe_status_t launch_combine(const void* y, int T, int k, int H, moe_dtype_t dt, void* out,
                            cudaStream_t s) {
  const int vec = dt == MOE_BF16 ? H / 8 : H / 4;
  const int64_t total = (int64_t)T * vec;
  int blocks = (int)std::min<int64_t>(ceil_div64(total, 256), (int64_t)num_sms() * 8);
  if (blocks < 1) blocks = 1;
  if (dt == MOE_BF16)
    return launch_k(combine_bf16_kernel, dim3(blocks), dim3(256), 0, s, (const uint4*)y,
                    (uint4*)out, T, k, vec);
  return launch_k(combine_f32_kernel, dim3(blocks), dim3(256), 0, s, (const float4*)y,
                  (float4*)out, T, k, vec);
}

}  // namespace moe
