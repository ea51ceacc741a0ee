// gather.cu — the token rows of GEMM1 in padded order: xs[p, :] = x[sorted_ids[p] / k, :]
// for every padded position p < num_post_padded whose flat row r = sorted_ids[p] is real
// (r < T*k); padding positions are left untouched (GEMM1 never stores their results).
//
// This is the gather of "Mixture-of-Experts Kernels: Routing, Permutation, and Grouped GEMM"
// §6 (rows r // TOP_K of x through the sorted_ids table) done as its own bandwidth-bound
// pass, so the tensor-core GEMM can then stream A with plain TMA tiles like its weights.
// One warp copies one row with 16-byte vectors (four independent loads in flight per lane);
// the number of rows comes from num_post_padded on the device.
#include "common.cuh"

namespace moe {

__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x,
                                                          const int32_t* __restrict__ sid,
                                                          const int32_t* __restrict__ npp,
                                                          int n_rows, int k, int vec,
                                                          uint4* __restrict__ xs) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int total = *npp;
  for (int p = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); p < total; p += warps) {
    const int r = sid[p];
    if (r >= n_rows) continue;
    const uint4* src = x + (int64_t)(r / k) * vec;
    uint4* dst = xs + (int64_t)p * vec;
    int v = lane;
    for (; v + 96 < vec; v += 128) {
      const uint4 a = src[v], b = src[v + 32], c = src[v + 64], d = src[v + 96];
      dst[v] = a;
      dst[v + 32] = b;
      dst[v + 64] = c;
      dst[v + 96] = d;
    }
    for (; v < vec; v += 32) dst[v] = src[v];
  }
}

moe_status_t launch_gather_rows(const void* x, const int32_t* sid, const int32_t* npp,
                                int n_rows, int k, int row_bytes, void* xs, cudaStream_t s) {
  const int blocks = num_sms() * 4;
  return launch_k(gather_rows_kernel, dim3(blocks), dim3(256), 0, s, (const uint4*)x, sid, npp,
                  n_rows, k, row_bytes / 16, (uint4*)xs);
}

}  // namespace moe
