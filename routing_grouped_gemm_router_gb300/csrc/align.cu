// align.cu — the block-aligned indirection table (sorted_ids / expert_ids / padded total).
//
// "Mixture-of-Experts Kernels: Routing, Permutation, and Grouped GEMM", §5: histogram of
// the flat rows r = t*k + j over experts, round each count up to BLOCK_M, exclusive scan
// for each expert's run start, scatter r to start[e] + rank. The rank is the number of
// earlier rows (smaller r) routed to the same expert, so each run is in ascending r and
// the table is deterministic. Nothing is sorted: the rank comes from a warp match
// (__match_any_sync) inside a warp plus per-warp counts in shared memory across warps.
//
// Small problems (T*k <= kSmallRows) run all steps in one CTA. Larger ones split the rows
// into chunks of kChunk: a per-chunk histogram kernel, a single-CTA scan kernel that turns
// the chunk histograms into absolute write offsets, and a per-chunk scatter kernel. Inside
// the layer, a batch of at most kTopkWarps tokens also takes its top-k in that one CTA
// (topk_align_small_kernel): the routing tail of a decode step is then a single launch.
#include <mutex>

#include <cooperative_groups.h>

#include "route_dev.cuh"

namespace moe {

constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr int kSmallRows = 4096;
constexpr int kChunk = 1024;  // rows per CTA in the multi-CTA path (one round)

__device__ int g_align_status;

int align_status_read(int reset) {
  int v = 0;
  cudaMemcpyFromSymbol(&v, g_align_status, sizeof(int));
  if (reset) {
    int z = 0;
    cudaMemcpyToSymbol(g_align_status, &z, sizeof(int));
  }
  return v;
}

size_t align_scratch_bytes(int T, int k, int E, int /*block_m*/) {
  int64_t n = (int64_t)T * k;
  if (n <= kSmallRows) return 0;
  int64_t chunks = ceil_div64(n, kChunk);
  return (size_t)(chunks * E) * sizeof(int32_t);
}

__device__ __forceinline__ int load_expert(const int32_t* ids, int r, int E) {
  int e = ids[r];
  if (e < 0 || e >= E) {
    atomicExch(&g_align_status, kStatusBadExpert);
    return -1;
  }
  return e;
}

// Block-wide exclusive scan over E <= kAlignThreads values (one per thread).
__device__ int block_exclusive_scan(int v, int* warp_tot, int* total_out) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  int inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int wv = lane < kAlignWarps ? warp_tot[lane] : 0;
    int wi = wv;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int o = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += o;
    }
    if (lane < kAlignWarps) warp_tot[lane] = wi - wv;  // exclusive warp offsets
    if (lane == 31) *total_out = wi;
  }
  __syncthreads();
  return warp_tot[warp] + inc - v;
}

// Pads, scans and writes the per-expert metadata from cnt[E] (in shared memory).
// Leaves start[e] in shared memory. Also writes expert_ids, the padding sentinels, the
// sentinel tail of sorted_ids, num_post_padded and counts.
__device__ void scan_and_fill(const int* cnt, int* start, int* warp_tot, int* total_sh, int n,
                              int E, int B, int max_padded, int32_t* sorted_ids,
                              int32_t* expert_ids, int32_t* npp, int32_t* counts) {
  const int tid = threadIdx.x;
  int c = tid < E ? cnt[tid] : 0;
  int p = (c + B - 1) / B * B;
  int st = block_exclusive_scan(p, warp_tot, total_sh);
  if (tid < E) start[tid] = st;
  __syncthreads();
  const int total = *total_sh;
  if (tid == 0) *npp = total;
  if (counts && tid < E) counts[tid] = c;
  // Sentinels: the padding slots of each run, then the tail [total, max_padded).
  if (tid < E)
    for (int q = st + c; q < st + p; ++q) sorted_ids[q] = n;
  for (int q = total + tid; q < max_padded; q += blockDim.x) sorted_ids[q] = n;
  // expert_ids: tile -> the expert whose run covers it (largest e with start[e] <= pos).
  const int tiles = max_padded / B;
  for (int tile = tid; tile < tiles; tile += blockDim.x) {
    int pos = tile * B, e = -1;
    if (pos < total) {
      int lo = 0, hi = E - 1;
      while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (start[mid] <= pos) lo = mid; else hi = mid - 1;
      }
      e = lo;
    }
    expert_ids[tile] = e;
  }
}

// Stable scatter of rows [r0, r1) given each expert's next free slot run_base[e] (shared).
// wcnt[kAlignWarps][E] (shared) must be zero on entry and is zero on exit.
__device__ void stable_scatter(const int32_t* ids, int r0, int r1, int E, int* run_base,
                               int* wcnt, int32_t* sorted_ids) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = r0; base < r1; base += blockDim.x) {
    int r = base + threadIdx.x;
    int e = r < r1 ? load_expert(ids, r, E) : -1;
    unsigned peers = __match_any_sync(0xffffffffu, e);
    int rank = __popc(peers & lt_mask);
    if (e >= 0 && rank == 0) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int off = run_base[e] + rank;
      for (int w = 0; w < warp; ++w) off += wcnt[w * E + e];
      sorted_ids[off] = r;
    }
    __syncthreads();
    for (int q = threadIdx.x; q < E; q += blockDim.x) {
      int s = 0;
      for (int w = 0; w < kAlignWarps; ++w) {
        s += wcnt[w * E + q];
        wcnt[w * E + q] = 0;
      }
      run_base[q] += s;
    }
    __syncthreads();
  }
}

// ---- single CTA: histogram, scan, fill, scatter --------------------------------------
__device__ __forceinline__ void align_small_body(const int32_t* __restrict__ ids, int n, int E,
                                                 int B, int max_padded,
                                                 int32_t* __restrict__ sorted_ids,
                                                 int32_t* __restrict__ expert_ids, int32_t* npp,
                                                 int32_t* counts, int* sm) {
  int* cnt = sm;                   // [E]
  int* start = cnt + E;            // [E]
  int* wcnt = start + E;           // [kAlignWarps * E]
  int* warp_tot = wcnt + kAlignWarps * E;  // [32]
  int* total_sh = warp_tot + 32;
  for (int q = threadIdx.x; q < E * (2 + kAlignWarps); q += blockDim.x) sm[q] = 0;
  __syncthreads();
  for (int r = threadIdx.x; r < n; r += blockDim.x) {
    int e = load_expert(ids, r, E);
    if (e >= 0) atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  scan_and_fill(cnt, start, warp_tot, total_sh, n, E, B, max_padded, sorted_ids, expert_ids,
                npp, counts);
  __syncthreads();
  stable_scatter(ids, 0, n, E, start, wcnt, sorted_ids);
}

__global__ void __launch_bounds__(kAlignThreads) align_small_kernel(
    const int32_t* __restrict__ ids, int n, int E, int B, int max_padded,
    int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids, int32_t* npp,
    int32_t* counts) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int sm[];
  align_small_body(ids, n, E, B, max_padded, sorted_ids, expert_ids, npp, counts, sm);
}

// ---- single CTA: top-k of at most kTopkWarps tokens, then the table ---------------------
// Warp t routes token t with the same top-k as the separate top-k kernel (writing its ids
// and weights), the CTA synchronises (its global writes are then visible to all of its
// threads) and builds the table from those ids. Router experts: c.E; table experts and
// slots: the effective E_eff, kk (shared experts included).
struct TopkArgs {
  const float* logits;
  int Tn, E, k, mode, renorm;
  float scale;
  int n_group, topk_group;
  const float* logit_bias;
  const float* select_bias;
  int n_shared;
};

template <int MPL>
__global__ void __launch_bounds__(kAlignThreads) topk_align_small_kernel(
    const TopkArgs a, int32_t* __restrict__ ids, float* __restrict__ w, int n, int E_eff, int B,
    int max_padded, int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
    int32_t* npp, int32_t* counts) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int sm[];
  const int warp = threadIdx.x / 32;
  if (warp < a.Tn)
    topk_token<MPL, 4>(a.logits, warp, a.E, a.k, a.mode, a.renorm, a.scale, a.n_group,
                       a.topk_group, a.logit_bias, a.select_bias, a.n_shared, ids, w,
                       reinterpret_cast<float*>(sm) + warp * 512);
  __syncthreads();
  align_small_body(ids, n, E_eff, B, max_padded, sorted_ids, expert_ids, npp, counts, sm);
}

// ---- multi CTA: per-chunk histogram ---------------------------------------------------
__global__ void __launch_bounds__(256) align_hist_kernel(const int32_t* __restrict__ ids,
                                                         int n, int E,
                                                         int32_t* __restrict__ chunk_cnt) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int hist[];
  for (int q = threadIdx.x; q < E; q += blockDim.x) hist[q] = 0;
  __syncthreads();
  const int r0 = blockIdx.x * kChunk, r1 = min(n, r0 + kChunk);
  for (int r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
    int e = load_expert(ids, r, E);
    if (e >= 0) atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int q = threadIdx.x; q < E; q += blockDim.x) chunk_cnt[(size_t)blockIdx.x * E + q] = hist[q];
}

// ---- multi CTA: totals, scan, fill, absolute chunk offsets ----------------------------
__global__ void __launch_bounds__(kAlignThreads) align_scan_kernel(
    int32_t* __restrict__ chunk_cnt, int chunks, int n, int E, int B, int max_padded,
    int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids, int32_t* npp,
    int32_t* counts) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int sm[];
  int* cnt = sm;
  int* start = cnt + E;
  int* warp_tot = start + E;
  int* total_sh = warp_tot + 32;
  // Per expert: running prefix over chunks (chunk-relative base) and the total count.
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int c = 0; c < chunks; ++c) {
      int v = chunk_cnt[(size_t)c * E + e];
      chunk_cnt[(size_t)c * E + e] = run;
      run += v;
    }
    cnt[e] = run;
  }
  __syncthreads();
  scan_and_fill(cnt, start, warp_tot, total_sh, n, E, B, max_padded, sorted_ids, expert_ids,
                npp, counts);
  __syncthreads();
  for (int i = threadIdx.x; i < chunks * E; i += blockDim.x) chunk_cnt[i] += start[i % E];
}

// ---- multi CTA: stable scatter of one chunk --------------------------------------------
__global__ void __launch_bounds__(kAlignThreads) align_scatter_kernel(
    const int32_t* __restrict__ ids, const int32_t* __restrict__ chunk_base, int n, int E,
    int32_t* __restrict__ sorted_ids) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int sm[];
  int* run_base = sm;        // [E]
  int* wcnt = run_base + E;  // [kAlignWarps * E]
  for (int q = threadIdx.x; q < E; q += blockDim.x) run_base[q] = chunk_base[(size_t)blockIdx.x * E + q];
  for (int q = threadIdx.x; q < kAlignWarps * E; q += blockDim.x) wcnt[q] = 0;
  __syncthreads();
  const int r0 = blockIdx.x * kChunk, r1 = min(n, r0 + kChunk);
  stable_scatter(ids, r0, r1, E, run_base, wcnt, sorted_ids);
}

// ---- variant without caller-provided scratch ------------------------------------------
// Some callers cannot hand this library any device memory beyond their own inputs and
// outputs: code running inside a host application or inference server whose device memory
// is wholly owned by someone else's pool, or latency-critical paths where cudaMalloc (which
// may synchronise the device) is not allowed. For them the per-chunk histograms live in a
// fixed array of this file, which every GPU that loads the library keeps until exit.
constexpr int kNoAllocScratchInts = 1 << 16;  // 256 KiB per GPU: chunks * E <= 65536
static __device__ __align__(256) int32_t g_align_noalloc_scratch[kNoAllocScratchInts];

// Device address of the array for the current device, looked up once per device with that
// device current (in host code the array's name is not a device address).
static int32_t* noalloc_scratch(moe_status_t* st) {
  static std::mutex mu;
  static int32_t* ptr[64] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *st = MOE_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_align_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      *st = MOE_ERR_CUDA;
      return nullptr;
    }
    ptr[dev] = (int32_t*)p;
  }
  return ptr[dev];
}

}  // namespace moe

extern "C" moe_status_t moe_align_noalloc(const int32_t* topk_ids, int T, int k, int E,
                                          int block_m, int32_t* sorted_ids,
                                          int32_t* expert_ids, int32_t* num_post_padded,
                                          int32_t* counts, cudaStream_t stream) {
  using namespace moe;
  int mp = 0;
  moe_status_t st = align_check_args(topk_ids, T, k, E, block_m, sorted_ids, expert_ids,
                                     num_post_padded, &mp);
  if (st != MOE_OK) return st;
  // Histograms beyond the fixed array: refuse rather than write past it.
  if (align_scratch_bytes(T, k, E, block_m) > sizeof(int32_t) * (size_t)kNoAllocScratchInts)
    return MOE_ERR_UNSUPPORTED;
  int32_t* scratch = noalloc_scratch(&st);
  if (!scratch) return st;
  return launch_align(topk_ids, T, k, E, block_m, mp, sorted_ids, expert_ids, num_post_padded,
                      counts, scratch, stream);
}

namespace moe {

// ---- expert parallelism: relabel tiles with local weight slots ------------------------
__global__ void __launch_bounds__(256) apply_expert_map_kernel(int32_t* __restrict__ eid,
                                                               int tiles,
                                                               const int32_t* __restrict__ map,
                                                               int E) {
  pdl_wait();
  pdl_trigger();
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < tiles; t += gridDim.x * blockDim.x) {
    const int e = eid[t];
    if (e < 0) continue;
    int slot = e < E ? map[e] : -1;
    if (slot < -1 || slot >= E) {
      atomicExch(&g_align_status, kStatusBadExpert);
      slot = -1;
    }
    eid[t] = slot;
  }
}

moe_status_t launch_apply_expert_map(int32_t* eid, int tiles, const int32_t* map, int E,
                                     cudaStream_t s) {
  const int blocks = std::max(1, std::min(ceil_div(tiles, 256), 64));
  return launch_k(apply_expert_map_kernel, dim3(blocks), dim3(256), 0, s, eid, tiles, map, E);
}

// ---- fixed-capacity (masked) layout: the table is the identity on valid rows ----------
// Position p = e*C + i holds row p itself when i < counts[e], else the sentinel E*C; a tile
// is labelled e when its first row is valid, else -1 (skipped). Optionally fills ones[].
__global__ void __launch_bounds__(256) masked_table_kernel(const int32_t* __restrict__ counts,
                                                           int E, int C, int B,
                                                           int32_t* __restrict__ sid,
                                                           int32_t* __restrict__ eid,
                                                           int32_t* __restrict__ npp,
                                                           float* __restrict__ ones) {
  pdl_wait();
  pdl_trigger();
  const int n = E * C;
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < n; p += gridDim.x * blockDim.x) {
    const int e = p / C, i = p - e * C;
    int c = counts[e];
    if (c < 0 || c > C) {
      atomicExch(&g_align_status, kStatusBadExpert);
      c = c < 0 ? 0 : C;
    }
    sid[p] = i < c ? p : n;
    if (ones) ones[p] = 1.f;
    if (i % B == 0) eid[p / B] = i < c ? e : -1;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *npp = n;
}

moe_status_t launch_masked_table(const int32_t* counts, int E, int C, int B, int32_t* sid,
                                 int32_t* eid, int32_t* npp, float* ones, cudaStream_t s) {
  const int blocks = std::max(1, std::min(ceil_div(E * C, 256), num_sms() * 4));
  return launch_k(masked_table_kernel, dim3(blocks), dim3(256), 0, s, counts, E, C, B, sid, eid,
                  npp, ones);
}

static bool set_smem(const void* fn, size_t bytes) {
  if (bytes <= 48 * 1024) return true;
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) ==
         cudaSuccess;
}

moe_status_t launch_align(const int32_t* ids, int T, int k, int E, int B, int max_padded,
                          int32_t* sorted_ids, int32_t* expert_ids, int32_t* npp,
                          int32_t* counts, void* scratch, cudaStream_t s) {
  const int n = T * k;
  if (n <= kSmallRows) {
    size_t smem = (size_t)(E * (2 + kAlignWarps) + 33) * sizeof(int);
    if (!set_smem((const void*)align_small_kernel, smem)) return MOE_ERR_CUDA;
    return launch_k(align_small_kernel, dim3(1), dim3(kAlignThreads), smem, s, ids, n, E, B,
                    max_padded, sorted_ids, expert_ids, npp, counts);
  }
  const int chunks = ceil_div(n, kChunk);
  int32_t* cc = (int32_t*)scratch;
  if (launch_k(align_hist_kernel, dim3(chunks), dim3(256), E * sizeof(int), s, ids, n, E, cc) !=
      MOE_OK)
    return MOE_ERR_CUDA;
  size_t smem_scan = (size_t)(2 * E + 33) * sizeof(int);
  if (launch_k(align_scan_kernel, dim3(1), dim3(kAlignThreads), smem_scan, s, cc, chunks, n, E, B,
               max_padded, sorted_ids, expert_ids, npp, counts) != MOE_OK)
    return MOE_ERR_CUDA;
  size_t smem_sc = (size_t)(E * (1 + kAlignWarps)) * sizeof(int);
  if (!set_smem((const void*)align_scatter_kernel, smem_sc)) return MOE_ERR_CUDA;
  return launch_k(align_scatter_kernel, dim3(chunks), dim3(kAlignThreads), smem_sc, s, ids, cc, n,
                  E, sorted_ids);
}

bool topk_align_fits(const moe_config_t& c) {
  const int64_t kk = c.k + c.n_shared;
  return c.T <= kTopkWarps && c.T * kk <= kSmallRows;
}

moe_status_t launch_topk_align_small(const moe_config_t& c, const float* logits, int32_t* ids,
                                     float* w, int B, int max_padded, int32_t* sorted_ids,
                                     int32_t* expert_ids, int32_t* npp, int32_t* counts,
                                     cudaStream_t s) {
  if (!topk_align_fits(c)) return MOE_ERR_UNSUPPORTED;
  const int kk = c.k + c.n_shared, E_eff = c.E + c.n_shared;
  const size_t smem = std::max((size_t)(E_eff * (2 + kAlignWarps) + 33) * sizeof(int),
                               (size_t)kTopkWarps * 512 * sizeof(float));
  const TopkArgs a{logits, c.T, c.E, c.k, (int)c.mode, c.renormalize, c.scale, c.n_group,
                   c.topk_group, c.logit_bias, c.select_bias, c.n_shared};
  auto run = [&](auto kern) {
    if (!set_smem((const void*)kern, smem)) return MOE_ERR_CUDA;
    return launch_k(kern, dim3(1), dim3(kAlignThreads), smem, s, a, ids, w, c.T * kk, E_eff, B,
                    max_padded, sorted_ids, expert_ids, npp, counts);
  };
  switch (topk_per_lane(c.E)) {
    case 4: return run(topk_align_small_kernel<4>);
    case 8: return run(topk_align_small_kernel<8>);
    default: return run(topk_align_small_kernel<kMaxPerLane>);
  }
}

}  // namespace moe

namespace moe {

// ---- decode batches: top-k and the table in one small CTA ---------------------------------
// For at most kTinyRows routed slots the table needs no histogram pass: warp t routes token t
// (the top-k device code of the top-k kernel) into shared memory, then warp 0 gives each flat
// row r a lane: a warp match finds the rows of its expert (its rank among them keeps them in
// ascending r), and counting, over the other lanes, the first rows of lower experts gives its
// tile of the table (experts ascending, one tile each). The result is the table moe_align
// writes (and, with an expert map, moe_apply_expert_map after it): rows first in each tile,
// then sentinels, tail tiles -1.
constexpr int kTinyRows = 32;
constexpr int kTinyThreads = 256;

__device__ int g_tiny_status;

int tiny_status_read(int reset) {
  int v = 0;
  cudaMemcpyFromSymbol(&v, g_tiny_status, sizeof(int));
  if (reset) {
    int z = 0;
    cudaMemcpyToSymbol(g_tiny_status, &z, sizeof(int));
  }
  return v;
}

// The router GEMM of a one-token batch fused in front (bf16): a cluster of up to 8 CTAs of 16
// warps, a warp per expert (the few-token router's device code), writes the logits into the
// shared memory of the cluster's first CTA; after a cluster barrier (release / acquire) that CTA
// stores them to the workspace and runs the top-k and the table on them, as the kernel above
// does on the logits in global memory. One launch, and one dependency wait, fewer on the
// decode step's critical path.
constexpr int kRouteTinyWarps = 16;
constexpr int kRouteTinyMaxCtas = 8;
constexpr int kRouteTinyLogits = 512;  // the token's E logits, held by the first CTA

template <int MPL, int TB, bool FUSED>
__global__ void __launch_bounds__(FUSED ? kRouteTinyWarps * 32 : kTinyThreads)
    topk_table_tiny_kernel(const TopkArgs a, int32_t* __restrict__ ids, float* __restrict__ w,
                           int n, int E_eff, int B, int max_padded,
                           int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
                           int32_t* npp, int32_t* counts, const int32_t* __restrict__ map,
                           const __nv_bfloat16* __restrict__ x,
                           const __nv_bfloat16* __restrict__ Wg, int H, float* logits_out) {
  __shared__ float skey[kTopkWarps][512];
  __shared__ int32_t ids_s[kTinyRows];
  __shared__ float w_s[kTinyRows];
  __shared__ int gt_cnt[kTinyRows], gt_label[kTinyRows];
  __shared__ int n_tiles_s;
  __shared__ float lg_sh[FUSED ? kRouteTinyLogits : 1];
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const float* logits = a.logits;
  if constexpr (FUSED) {
    namespace cg = cooperative_groups;
    cg::cluster_group cl = cg::this_cluster();
    float* lg0 = cl.map_shared_rank(&lg_sh[0], 0);  // the first CTA's logits, from any CTA
    const int rank = (int)cl.block_rank(), nw = (int)cl.num_blocks() * kRouteTinyWarps;
    for (int e = rank * kRouteTinyWarps + warp; e < a.E; e += nw)
      router_warp_logits<__nv_bfloat16, TB>(x, Wg, lg0, 0, a.Tn, H, a.E, e);
    cl.sync();  // every CTA's logits are in the first CTA's shared memory
    if (rank != 0) return;
    for (int i = threadIdx.x; i < a.Tn * a.E; i += blockDim.x) logits_out[i] = lg_sh[i];
    logits = lg_sh;
  }
  if (warp < a.Tn)
    topk_token<MPL, 8, FUSED>(logits, warp, a.E, a.k, a.mode, a.renorm, a.scale, a.n_group,
                              a.topk_group, a.logit_bias, a.select_bias, a.n_shared, ids_s, w_s,
                              skey[warp]);
  __syncthreads();
  if (warp == 0) {
    const int e = lane < n ? ids_s[lane] : 0x7fffffff;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const bool first = lane < n && rank == 0;
    int g = 0;
#pragma unroll 8
    for (int j = 0; j < kTinyRows; ++j) {
      const int ej = __shfl_sync(0xffffffffu, e, j);
      const int fj = __shfl_sync(0xffffffffu, (int)first, j);
      g += (fj && ej < e);
    }
    if (first) {
      int label = e;
      if (map) {
        label = map[e];
        if (label < -1 || label >= E_eff) {  // as moe_apply_expert_map: flagged, skipped
          atomicExch(&g_tiny_status, kStatusBadExpert);
          label = -1;
        }
      }
      gt_cnt[g] = __popc(peers);
      gt_label[g] = label;
    }
    if (lane < n) {
      ids[lane] = e;
      w[lane] = w_s[lane];
      sorted_ids[g * B + rank] = lane;
    }
    const int nt = __popc(__ballot_sync(0xffffffffu, first));
    if (lane == 0) n_tiles_s = nt;
  }
  __syncthreads();
  const int nt = n_tiles_s;
  for (int q = threadIdx.x; q < max_padded; q += blockDim.x) {
    const int t = q / B, i = q - t * B;
    if (!(t < nt && i < gt_cnt[t])) sorted_ids[q] = n;
  }
  for (int t = threadIdx.x; t < max_padded / B; t += blockDim.x)
    expert_ids[t] = t < nt ? gt_label[t] : -1;
  for (int e = threadIdx.x; e < E_eff; e += blockDim.x) {
    int c = 0;
    for (int r = 0; r < n; ++r) c += ids_s[r] == e;
    counts[e] = c;
  }
  if (threadIdx.x == 0) *npp = nt * B;
}

bool topk_table_tiny_fits(const moe_config_t& c) {
  return c.T <= kTopkWarps && c.T * (c.k + c.n_shared) <= kTinyRows;
}

moe_status_t launch_topk_table_tiny(const moe_config_t& c, const float* logits, int32_t* ids,
                                    float* w, int B, int max_padded, int32_t* sorted_ids,
                                    int32_t* expert_ids, int32_t* npp, int32_t* counts,
                                    cudaStream_t s) {
  if (!topk_table_tiny_fits(c) || !counts) return MOE_ERR_UNSUPPORTED;
  const int kk = c.k + c.n_shared, E_eff = c.E + c.n_shared;
  const TopkArgs a{logits, c.T, c.E, c.k, (int)c.mode, c.renormalize, c.scale, c.n_group,
                   c.topk_group, c.logit_bias, c.select_bias, c.n_shared};
  auto run = [&](auto kern) {
    return launch_k(kern, dim3(1), dim3(kTinyThreads), 0, s, a, ids, w, c.T * kk, E_eff, B,
                    max_padded, sorted_ids, expert_ids, npp, counts, c.expert_map,
                    (const __nv_bfloat16*)nullptr, (const __nv_bfloat16*)nullptr, 0,
                    (float*)nullptr);
  };
  switch (topk_per_lane(c.E)) {
    case 4: return run(topk_table_tiny_kernel<4, 1, false>);
    case 8: return run(topk_table_tiny_kernel<8, 1, false>);
    default: return run(topk_table_tiny_kernel<kMaxPerLane, 1, false>);
  }
}

// One token only. Measured on GB300 (gpt-oss-shaped layer, CUDA graph): 1 token 49.4 -> 48.7
// us (FP8 weights 41.0 -> 40.0); at 2-8 tokens the router's 8-token path, on the cluster's 8
// SMs instead of 16, is slower than the launch it saves (2 tokens 87.0 -> 88.5 us).
bool route_table_tiny_fits(const moe_config_t& c) {
  return topk_table_tiny_fits(c) && c.dtype == MOE_BF16 && c.T == 1 &&
         c.E <= kRouteTinyLogits;
}

moe_status_t launch_route_table_tiny(const moe_config_t& c, const void* x, const void* Wg,
                                     float* logits, int32_t* ids, float* w, int B,
                                     int max_padded, int32_t* sorted_ids, int32_t* expert_ids,
                                     int32_t* npp, int32_t* counts, cudaStream_t s) {
  if (!route_table_tiny_fits(c) || !counts) return MOE_ERR_UNSUPPORTED;
  const int kk = c.k + c.n_shared, E_eff = c.E + c.n_shared;
  const TopkArgs a{logits, c.T, c.E, c.k, (int)c.mode, c.renormalize, c.scale, c.n_group,
                   c.topk_group, c.logit_bias, c.select_bias, c.n_shared};
  const int ctas = std::max(1, std::min(kRouteTinyMaxCtas, ceil_div(c.E, kRouteTinyWarps)));
  auto run = [&](auto kern) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kRouteTinyWarps * 32);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = ctas;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, a, ids, w, c.T * kk, E_eff, B, max_padded,
                              sorted_ids, expert_ids, npp, counts, c.expert_map,
                              (const __nv_bfloat16*)x, (const __nv_bfloat16*)Wg, c.H,
                              logits) == cudaSuccess
               ? MOE_OK
               : MOE_ERR_CUDA;
  };
  switch (topk_per_lane(c.E)) {
    case 4: return run(topk_table_tiny_kernel<4, 1, true>);
    case 8: return run(topk_table_tiny_kernel<8, 1, true>);
    default: return run(topk_table_tiny_kernel<kMaxPerLane, 1, true>);
  }
}

}  // namespace moe
