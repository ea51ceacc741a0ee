// common.cuh — shared host/device helpers of the MoE library (internal header).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <utility>

#include "moe.h"

namespace moe {

// Device status codes (moe_device_status).
enum : int { kStatusOk = 0, kStatusBadExpert = 1, kStatusTimeout = 2, kStatusPairTmem = 3 };

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ inline int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Number of SMs of the current device (cached per device).
int num_sms();

// Launch-error check shared by all entry points.
inline moe_status_t last_launch_status() {
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

inline size_t dtype_size(moe_dtype_t d) { return d == MOE_BF16 ? 2 : 4; }

// ---------------------------------------------------------------- programmatic dependent launch
// Every kernel of the library is launched with programmatic stream serialisation and starts
// with pdl_wait() (before any global-memory access, before any early return): its launch and
// prologue overlap the previous kernel's tail, while its memory operations still begin only
// after the previous grid has completed and its writes are visible. pdl_trigger() lets the
// next kernel launch as soon as every CTA of this grid has started.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline moe_status_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...) == cudaSuccess ? MOE_OK
                                                                                    : MOE_ERR_CUDA;
}

// ---------------------------------------------------------------- kernel entry wrappers
// Implemented in the .cu files; all enqueue on `stream` and return MOE_OK/MOE_ERR_CUDA.

moe_status_t launch_router_simt(const moe_config_t& c, const void* x, const void* Wg,
                                float* logits, cudaStream_t s);
moe_status_t launch_router_few_tokens(const moe_config_t& c, const void* x, const void* Wg,
                                      float* logits, cudaStream_t s);
moe_status_t launch_router_tc(const moe_config_t& c, const void* x, const void* Wg,
                              float* logits, cudaStream_t s);
moe_status_t launch_topk(const moe_config_t& c, const float* logits, int32_t* ids, float* w,
                         cudaStream_t s);
size_t align_scratch_bytes(int T, int k, int E, int block_m);
// Argument checks shared by the align entry points; sets the padded table length.
moe_status_t align_check_args(const int32_t* topk_ids, int T, int k, int E, int block_m,
                              const int32_t* sorted_ids, const int32_t* expert_ids,
                              const int32_t* num_post_padded, int* max_padded);
moe_status_t launch_align(const int32_t* ids, int T, int k, int E, int block_m, int max_padded,
                          int32_t* sorted_ids, int32_t* expert_ids, int32_t* npp,
                          int32_t* counts, void* scratch, cudaStream_t s);
// Top-k of a batch of at most 8 tokens and its align table in one single-CTA launch (the
// routing tail of moe_forward for decode); topk_align_fits says whether cfg qualifies.
bool topk_align_fits(const moe_config_t& c);
moe_status_t launch_topk_align_small(const moe_config_t& c, const float* logits, int32_t* ids,
                                     float* w, int B, int max_padded, int32_t* sorted_ids,
                                     int32_t* expert_ids, int32_t* npp, int32_t* counts,
                                     cudaStream_t s);
// Decode batches of at most 32 routed slots: top-k and the table from one warp per token and
// one lane per slot, with cfg.expert_map applied to the tile labels, in one small CTA
// (align.cu).
bool topk_table_tiny_fits(const moe_config_t& c);
moe_status_t launch_topk_table_tiny(const moe_config_t& c, const float* logits, int32_t* ids,
                                    float* w, int B, int max_padded, int32_t* sorted_ids,
                                    int32_t* expert_ids, int32_t* npp, int32_t* counts,
                                    cudaStream_t s);
// The same for one token with the router GEMM fused in front (bf16 x and Wg, 16-byte
// aligned): one cluster launch writes the logits too (align.cu).
bool route_table_tiny_fits(const moe_config_t& c);
moe_status_t launch_route_table_tiny(const moe_config_t& c, const void* x, const void* Wg,
                                     float* logits, int32_t* ids, float* w, int B,
                                     int max_padded, int32_t* sorted_ids, int32_t* expert_ids,
                                     int32_t* npp, int32_t* counts, cudaStream_t s);
moe_status_t launch_gemm1_simt(const moe_config_t& c, const float* x, const float* W13,
                               const int32_t* sid, const int32_t* eid, const int32_t* npp,
                               int block_m, int max_padded, float* act, cudaStream_t s);
moe_status_t launch_gemm2_simt(const moe_config_t& c, const float* act, const float* W2,
                               const int32_t* sid, const int32_t* eid, const int32_t* npp,
                               int block_m, int max_padded, const float* topk_w, float* y,
                               cudaStream_t s);
moe_status_t launch_gemm1_tc(const moe_config_t& c, const void* xs, const void* W13,
                             const int32_t* sid, const int32_t* eid, const int32_t* npp,
                             int block_m, int max_padded, void* act, cudaStream_t s);
moe_status_t launch_gemm2_tc(const moe_config_t& c, const void* act, const void* W2,
                             const int32_t* sid, const int32_t* eid, const int32_t* npp,
                             int block_m, int max_padded, const float* topk_w, void* y,
                             cudaStream_t s);
// Grouped GEMMs of small bf16 batches on CUDA cores (gemv.cu): whether they apply to a
// layer, and the two GEMMs with the tensor-core kernels' inputs and outputs (GEMM1 reads
// the routed rows gathered in padded order, or the token rows through sorted_ids).
bool gemv_applies(const moe_config_t& c, int max_padded);
moe_status_t launch_gemv1(const moe_config_t& c, const void* a, bool gathered, const void* W13,
                          const int32_t* sid, const int32_t* eid, const int32_t* npp,
                          int block_m, void* act, cudaStream_t s);
// FP8 E4M3 weights [E, R, K] with block scales [E, R / Rg grids, ceil(Rg / 128), K / 128]
// into bf16 weights (code times block scale, as the converter warps round it); experts whose
// counts entry is 0 are skipped when counts is given (dequant.cu).
moe_status_t launch_dequant_fp8(const void* codes, const float* scale, int E, int R, int Rg,
                                int K, int sc_rb, int sc_kb, const int32_t* counts, void* out,
                                cudaStream_t s);
// early: the launch directly follows launch_gemv1 on the same table (the fused layer), so the
// kernel may read the table and the weights before its dependency wait.
moe_status_t launch_gemv2(const moe_config_t& c, const void* act, const void* W2,
                          const int32_t* sid, const int32_t* eid, const int32_t* npp,
                          int block_m, const float* topk_w, void* y, cudaStream_t s,
                          bool early = false);
// Grouped GEMMs of decode-sized batches on the tensor cores with the weights as the 128-row
// MMA operand (gemm_dec.cu): whether they apply, and the two GEMMs with the pair kernels'
// inputs and outputs (GEMM1 reads the routed rows gathered in padded order).
bool dec_gemm_applies(const moe_config_t& c, int max_padded);
bool dec_masked_applies(const moe_config_t& m, int capacity);
moe_status_t launch_gemm1_dec(const moe_config_t& c, const void* xs, const void* W13,
                              const int32_t* sid, const int32_t* eid, const int32_t* npp,
                              int block_m, int max_padded, void* act, cudaStream_t s);
moe_status_t launch_gemm2_dec(const moe_config_t& c, const void* act, const void* W2,
                              const int32_t* sid, const int32_t* eid, const int32_t* npp,
                              int block_m, int max_padded, const float* topk_w, void* y,
                              cudaStream_t s);
int dec_status_read(int reset);
moe_status_t launch_gather_rows(const void* x, const int32_t* sid, const int32_t* npp,
                                int n_rows, int k, int row_bytes, void* xs, cudaStream_t s);
moe_status_t launch_masked_table(const int32_t* counts, int E, int C, int B, int32_t* sid,
                                 int32_t* eid, int32_t* npp, float* ones, cudaStream_t s);
moe_status_t launch_apply_expert_map(int32_t* eid, int tiles, const int32_t* map, int E,
                                     cudaStream_t s);
moe_status_t launch_combine_local(const void* y, const int32_t* ids, const int32_t* map, int E,
                                  int T, int k, int H, moe_dtype_t dt, void* out, cudaStream_t s);
moe_status_t launch_combine(const void* y, int T, int k, int H, moe_dtype_t dt, void* out,
                            cudaStream_t s);

moe_status_t launch_selftest_wait(cudaStream_t s);

int align_status_read(int reset);
int router_status_read(int reset);
int grouped_status_read(int reset);
int combine_status_read(int reset);
int tiny_status_read(int reset);

}  // namespace moe
