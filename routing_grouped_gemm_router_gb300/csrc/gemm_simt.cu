// gemm_simt.cu — grouped expert GEMMs on CUDA cores for fp32 layers.
//
// fp32 layers must match a float64 reference to 1e-5 relative, which the tensor cores'
// tf32 mode cannot, so these kernels use fp32 FFMA. Semantics are those of the fused
// grouped GEMM in "Mixture-of-Experts Kernels: Routing, Permutation, and Grouped GEMM",
// §6: a 16-row tile belongs to one expert (expert_ids[p / block_m]); GEMM1 gathers token
// rows x[sorted_ids[p] / k] and computes the gate and up halves as two accumulators so
// silu(gate) * up is applied before anything is stored; GEMM2 multiplies by topk_w[r] and
// scatters to row r. Tiles past num_post_padded exit at once; padding rows are not stored.
#include "common.cuh"

namespace moe {

constexpr int kSimtBM = 16, kSimtBN = 64, kSimtBK = 32;

__global__ void __launch_bounds__(256) gemm1_simt_kernel(
    const float* __restrict__ x, const float* __restrict__ W13, const int32_t* __restrict__ sid,
    const int32_t* __restrict__ eid, const int32_t* __restrict__ npp, int block_m, int n_rows,
    int k, int H, int I, float* __restrict__ act) {
  pdl_wait();
  pdl_trigger();
  __shared__ float As[kSimtBK][kSimtBM];
  __shared__ float Bg[kSimtBK][kSimtBN + 1];
  __shared__ float Bu[kSimtBK][kSimtBN + 1];
  __shared__ int tok[kSimtBM];
  const int p0 = blockIdx.x * kSimtBM;
  if (p0 >= *npp) return;
  const int e = eid[p0 / block_m];
  if (e < 0) return;
  const int n0 = blockIdx.y * kSimtBN;
  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
  if (tid < kSimtBM) {
    int r = sid[p0 + tid];
    tok[tid] = r < n_rows ? r / k : 0;
  }
  __syncthreads();
  const float* Wgate = W13 + (size_t)e * 2 * I * H;
  const float* Wup = Wgate + (size_t)I * H;
  float ag[4] = {}, au[4] = {};
  for (int h0 = 0; h0 < H; h0 += kSimtBK) {
    for (int i = tid; i < kSimtBM * kSimtBK; i += 256) {
      int m = i / kSimtBK, kk = i % kSimtBK, h = h0 + kk;
      As[kk][m] = h < H ? x[(size_t)tok[m] * H + h] : 0.f;
    }
    for (int i = tid; i < kSimtBN * kSimtBK; i += 256) {
      int nn = i / kSimtBK, kk = i % kSimtBK, h = h0 + kk, n = n0 + nn;
      bool ok = h < H && n < I;
      Bg[kk][nn] = ok ? Wgate[(size_t)n * H + h] : 0.f;
      Bu[kk][nn] = ok ? Wup[(size_t)n * H + h] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kSimtBK; ++kk) {
      float a = As[kk][ty];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        ag[j] = fmaf(a, Bg[kk][tx * 4 + j], ag[j]);
        au[j] = fmaf(a, Bu[kk][tx * 4 + j], au[j]);
      }
    }
    __syncthreads();
  }
  const int p = p0 + ty;
  if (sid[p] >= n_rows) return;  // padding row: never stored
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int n = n0 + tx * 4 + j;
    if (n < I) {
      float g = ag[j];
      act[(size_t)p * I + n] = g / (1.f + expf(-g)) * au[j];
    }
  }
}

__global__ void __launch_bounds__(256) gemm2_simt_kernel(
    const float* __restrict__ act, const float* __restrict__ W2, const int32_t* __restrict__ sid,
    const int32_t* __restrict__ eid, const int32_t* __restrict__ npp, int block_m, int n_rows,
    int H, int I, const float* __restrict__ topk_w, float* __restrict__ y) {
  pdl_wait();
  pdl_trigger();
  __shared__ float As[kSimtBK][kSimtBM];
  __shared__ float Bs[kSimtBK][kSimtBN + 1];
  const int p0 = blockIdx.x * kSimtBM;
  if (p0 >= *npp) return;
  const int e = eid[p0 / block_m];
  if (e < 0) return;
  const int n0 = blockIdx.y * kSimtBN;
  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
  const float* We = W2 + (size_t)e * H * I;
  float acc[4] = {};
  for (int i0 = 0; i0 < I; i0 += kSimtBK) {
    for (int i = tid; i < kSimtBM * kSimtBK; i += 256) {
      int m = i / kSimtBK, kk = i % kSimtBK, c = i0 + kk;
      bool ok = c < I && sid[p0 + m] < n_rows;  // padding rows of act were never written
      As[kk][m] = ok ? act[(size_t)(p0 + m) * I + c] : 0.f;
    }
    for (int i = tid; i < kSimtBN * kSimtBK; i += 256) {
      int nn = i / kSimtBK, kk = i % kSimtBK, c = i0 + kk, n = n0 + nn;
      Bs[kk][nn] = (c < I && n < H) ? We[(size_t)n * I + c] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kSimtBK; ++kk) {
      float a = As[kk][ty];
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[j] = fmaf(a, Bs[kk][tx * 4 + j], acc[j]);
    }
    __syncthreads();
  }
  const int r = sid[p0 + ty];
  if (r >= n_rows) return;
  const float wr = topk_w[r];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int n = n0 + tx * 4 + j;
    if (n < H) y[(size_t)r * H + n] = wr * acc[j];
  }
}

moe_status_t launch_gemm1_simt(const moe_config_t& c, const float* x, const float* W13,
                               const int32_t* sid, const int32_t* eid, const int32_t* npp,
                               int block_m, int max_padded, float* act, cudaStream_t s) {
  dim3 grid(max_padded / kSimtBM, ceil_div(c.I, kSimtBN));
  return launch_k(gemm1_simt_kernel, grid, dim3(256), 0, s, x, W13, sid, eid, npp, block_m,
                  c.T * c.k, c.k, c.H, c.I, act);
}

moe_status_t launch_gemm2_simt(const moe_config_t& c, const float* act, const float* W2,
                               const int32_t* sid, const int32_t* eid, const int32_t* npp,
                               int block_m, int max_padded, const float* topk_w, float* y,
                               cudaStream_t s) {
  dim3 grid(max_padded / kSimtBM, ceil_div(c.H, kSimtBN));
  return launch_k(gemm2_simt_kernel, grid, dim3(256), 0, s, act, W2, sid, eid, npp, block_m,
                  c.T * c.k, c.H, c.I, topk_w, y);
}

}  // namespace moe
