// gemv.cu — the grouped expert GEMMs for small batches (decode), on CUDA cores.
//
// Semantics are those of the grouped GEMMs of "Mixture-of-Experts Kernels: Routing,
// Permutation, and Grouped GEMM", §6, on the same inputs and outputs as the tensor-core
// kernels: the rows of a 128-row tile of the padded order belong to expert
// expert_ids[p / block_m]; GEMM1 writes act[p] = silu(x_r W1[e]^T) * (x_r W3[e]^T) for every
// real row p (sorted_ids[p] < T*k), GEMM2 writes y[r] = topk_w[r] * act[p] W2[e]^T at row
// r = sorted_ids[p]; padding rows are neither read nor written.
//
// With a handful of tokens a tile holds one to a few real rows, so the layer is a stream of
// the active experts' weights with about one multiply-add per weight and row; the
// tensor-core kernels pay for 128-row tiles that such a stream does not need. The item
// arithmetic (a warp per pair of weight rows, fp32 sums, shuffle reduction) is in
// gemv_dev.cuh. The activations (a few rows, read by every warp of the tile) come through L1;
// the weights bypass it. Each warp takes a contiguous range of items, adjacent columns of
// one tile, so its tile's row list (kept in the warp's shared memory) and expert change
// rarely; a pass takes up to one, two or four rows (from the batch size) and skips the rows
// a tile does not have. Inside the fused layer GEMM2's first weight loads are issued before
// its dependency wait (see gemv_kernel).
#include "gemv_dev.cuh"

namespace moe {
namespace gv {

// MODE 0: GEMM1 (item = output column n of act: gate row n, up row N + n).
// MODE 1: GEMM2 (item = output columns n, n + 1 of y: W2 rows n, n + 1).
// RMAX: real rows a pass takes (a tile holds at most T of them); one pass shape per kernel.

// The weight rows of item (expert e, output column n) and, with FP8 codes, their block scales.
template <int MODE, bool FP8>
__device__ __forceinline__ void item_rows(const Params& P, int e, int n, const uint8_t*& w0,
                                          const uint8_t*& w1, const float*& s0,
                                          const float*& s1) {
  const size_t row_bytes = (size_t)P.K * (FP8 ? 1 : 2);
  s0 = s1 = nullptr;
  if (MODE == 0) {
    w0 = P.w + ((size_t)e * 2 * P.N + n) * row_bytes;
    w1 = P.w + ((size_t)e * 2 * P.N + P.N + n) * row_bytes;
    if (FP8) {
      s0 = P.scale + (((size_t)e * 2 + 0) * P.sc_rb + n / 128) * P.sc_kb;
      s1 = P.scale + (((size_t)e * 2 + 1) * P.sc_rb + n / 128) * P.sc_kb;
    }
  } else {
    w0 = P.w + ((size_t)e * P.N + n) * row_bytes;
    w1 = w0 + row_bytes;
    if (FP8) s0 = s1 = P.scale + ((size_t)e * P.sc_rb + n / 128) * P.sc_kb;  // n, n+1: one block
  }
}

// Item w (tile w / cols, column c = w % cols) of one warp: the tile's real rows (kept in rl
// while the warp stays on the tile), then one pass over the item's weight rows per RMAX real
// rows.
template <int MODE, bool FP8, int RMAX>
__device__ __forceinline__ void run_item(const Params& P, int w, int cols, int& cur_t,
                                         int& nvalid, int& e, int2* rl) {
  const int t = w / cols, c = w - t * cols;
  if (t != cur_t) {
    __syncwarp();
    cur_t = t;
    e = P.eid[(t * kTile) / P.block_m];
    nvalid = tile_rows(P, t, rl);
    __syncwarp();
  }
  if (e < 0 || e >= P.n_slots || nvalid == 0) return;
  const int n = MODE == 0 ? c : 2 * c;
  const uint8_t *w0, *w1;
  const float *s0, *s1;
  item_rows<MODE, FP8>(P, e, n, w0, w1, s0, s1);
  for (int rc = 0; rc < nvalid; rc += RMAX)
    item_pass<MODE, FP8, RMAX, kPieces<MODE, FP8, RMAX>>(P, w0, w1, s0, s1, rl + rc,
                                                         min(RMAX, nvalid - rc), n);
}

// First item of warp gw's contiguous range of items. BAL: ranges of floor or ceil(total /
// nwarps) items, every warp busy once total >= nwarps; else ranges of ceil(total / nwarps)
// items, which leave the last warps idle (at one token 768 of 3648). Measured on GB300
// (gpt-oss-shaped layer in a CUDA graph, same box): balanced ranges FP8 T = 8 234 vs 242 µs;
// ceil-sized ranges bf16 T = 1 48.7 vs 49.7 µs, T = 2 87.7 vs 88.6. So the passes of up to
// four rows take balanced ranges.
template <bool BAL>
__device__ __forceinline__ int range_begin(int gw, int total, int nwarps) {
  if (BAL) return (int)((int64_t)gw * total / nwarps);
  const int per = (total + nwarps - 1) / nwarps;
  return min(total, gw * per);
}

template <int MODE, bool FP8, int RMAX>
__global__ void __launch_bounds__(kThreads, (kMinCtas<MODE, FP8, RMAX>)) gemv_kernel(const Params P) {
  constexpr int S = kPieces<MODE, FP8, RMAX>;
  constexpr bool kBal = RMAX > 2;
  constexpr int ES = FP8 ? 1 : 2;
  constexpr int EPL = FP8 ? 16 : 8;  // elements of a 16-byte weight piece
  __shared__ int2 rows_sh[kWarps][kTile];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  int2* rl = rows_sh[warp];
  const int cols = MODE == 0 ? P.N : P.N / 2;
  const int nwarps = gridDim.x * kWarps;
  const int gw = blockIdx.x * kWarps + warp;
  int cur_t = -1, nvalid = 0, e = -1;
  // GEMM2 inside the fused layer (P.early): the kernel before this one is GEMM1, which writes
  // only act. The weights are the layer's inputs and the table was written by the routing
  // kernel, which completed before GEMM1 started (and so before this grid was launched), so
  // this warp's first item is set up (table read past L1) and the first pieces of its weight
  // rows are loaded before the dependency wait, during GEMM1's tail; act and y wait.
  uint4 pre0[S], pre1[S];
  bool pre = false;
  int pre_n = 0;
  const uint8_t *pw0 = nullptr, *pw1 = nullptr;
  const float *ps0 = nullptr, *ps1 = nullptr;
  if (MODE == 1 && P.early) {
    const int total0 = __ldcg(P.npp) / kTile * cols;
    const int wb = range_begin<kBal>(gw, total0, nwarps);  // as w_begin below
    if (wb < range_begin<kBal>(gw + 1, total0, nwarps)) {
      const int t = wb / cols, c = wb - t * cols;
      cur_t = t;
      e = __ldcg(P.eid + (t * kTile) / P.block_m);
      nvalid = tile_rows<true>(P, t, rl);
      __syncwarp();
      if (e >= 0 && e < P.n_slots && nvalid > 0) {
        pre_n = 2 * c;
        item_rows<MODE, FP8>(P, e, pre_n, pw0, pw1, ps0, ps1);
#pragma unroll
        for (int j = 0; j < S; ++j) {
          const int kk = lane * EPL + j * 32 * EPL;
          if (kk < P.K) {
            pre0[j] = ld_stream(pw0 + (size_t)kk * ES);
            pre1[j] = ld_stream(pw1 + (size_t)kk * ES);
          }
        }
        pre = true;
      }
    }
  }
  pdl_wait();
  pdl_trigger();
  const int num_m = *P.npp / kTile;
  const int total = num_m * cols;  // bounded on the host
  const int w_begin = range_begin<kBal>(gw, total, nwarps);
  const int w_end = range_begin<kBal>(gw + 1, total, nwarps);
  int w = w_begin;
  if (MODE == 1 && pre) {  // the first item: its first pass from the loaded pieces
    item_pass<MODE, FP8, RMAX, S, true>(P, pw0, pw1, ps0, ps1, rl, min(RMAX, nvalid), pre_n, pre0,
                                        pre1);
    for (int rc = RMAX; rc < nvalid; rc += RMAX)
      item_pass<MODE, FP8, RMAX, S>(P, pw0, pw1, ps0, ps1, rl + rc, min(RMAX, nvalid - rc), pre_n);
    ++w;
  }
  for (; w < w_end; ++w) run_item<MODE, FP8, RMAX>(P, w, cols, cur_t, nvalid, e, rl);
}

template <int MODE, bool FP8, int RMAX>
static moe_status_t launch_r(const Params& P, cudaStream_t s) {
  static int per_sm[64];
  int dev = 0;
  cudaGetDevice(&dev);
  int& occ = per_sm[dev & 63];
  if (occ == 0) {
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, gemv_kernel<MODE, FP8, RMAX>, kThreads,
                                                      0) != cudaSuccess ||
        v < 1)
      v = 1;
    occ = v;
  }
  return launch_k(gemv_kernel<MODE, FP8, RMAX>, dim3(num_sms() * occ), dim3(kThreads), 0, s, P);
}

template <int MODE, bool FP8>
static moe_status_t launch_fmt(const Params& P, int T, cudaStream_t s) {
  // A tile holds at most T real rows (a token takes an expert at most once); rows past RMAX
  // take further passes over the same weights.
  if (T <= 1) return launch_r<MODE, FP8, 1>(P, s);
  if (T <= 2) return launch_r<MODE, FP8, 2>(P, s);
  return launch_r<MODE, FP8, 4>(P, s);
}

static Params base_params(const moe_config_t& c, const int32_t* sid, const int32_t* eid,
                          const int32_t* npp, int block_m) {
  Params P{};
  P.sid = sid;
  P.eid = eid;
  P.npp = npp;
  P.block_m = block_m;
  P.n_rows = c.T * c.k;
  P.k = c.k;
  P.n_slots = c.E;
  return P;
}

}  // namespace gv

// Up to this many tokens the grouped GEMMs of a layer run here. Measured on GB300 against
// the decode tensor-core kernel (gemm_dec.cu; gpt-oss-shaped decode layer, one step in a CUDA
// graph): bf16 weights 49.5 vs 62.6 us at 1 token, 88 vs 117 at 2, behind at 3 (134 vs 124)
// and from 6 tokens (236 vs 220); FP8 weights 41 vs 87 us at 1 token, 242 vs 340 at 8, 411 vs
// 532 at 16, 559 vs 658 at 24, behind at 32 (993 vs 770).
constexpr int kGemvMaxTokens = 2;
constexpr int kGemvMaxTokensFp8 = 24;

bool gemv_applies(const moe_config_t& c, int max_padded) {
  const bool fp8 = c.weight_format == MOE_WEIGHTS_FP8_E4M3_B128;
  if (c.dtype != MOE_BF16 || c.T > (fp8 ? kGemvMaxTokensFp8 : kGemvMaxTokens)) return false;
  const int64_t tiles = max_padded / gv::kTile;
  return tiles * std::max(c.I, c.H) < ((int64_t)1 << 31) - ((int64_t)1 << 24);
}

moe_status_t launch_gemv1(const moe_config_t& c, const void* a, bool gathered, const void* W13,
                          const int32_t* sid, const int32_t* eid, const int32_t* npp,
                          int block_m, void* act, cudaStream_t s) {
  gv::Params P = gv::base_params(c, sid, eid, npp, block_m);
  const bool fp8 = c.weight_format == MOE_WEIGHTS_FP8_E4M3_B128;
  P.a = (const uint8_t*)a;
  P.a_gathered = gathered ? 1 : 0;
  P.w = (const uint8_t*)W13;
  P.scale = fp8 ? c.w13_scale : nullptr;
  P.sc_rb = ceil_div(c.I, 128);
  P.sc_kb = ceil_div(c.H, 128);
  P.K = c.H;
  P.N = c.I;
  P.out = act;
  return fp8 ? gv::launch_fmt<0, true>(P, c.T, s) : gv::launch_fmt<0, false>(P, c.T, s);
}

moe_status_t launch_gemv2(const moe_config_t& c, const void* act, const void* W2,
                          const int32_t* sid, const int32_t* eid, const int32_t* npp,
                          int block_m, const float* topk_w, void* y, cudaStream_t s, bool early) {
  gv::Params P = gv::base_params(c, sid, eid, npp, block_m);
  P.early = early ? 1 : 0;
  const bool fp8 = c.weight_format == MOE_WEIGHTS_FP8_E4M3_B128;
  P.a = (const uint8_t*)act;
  P.a_gathered = 1;
  P.w = (const uint8_t*)W2;
  P.scale = fp8 ? c.w2_scale : nullptr;
  P.sc_rb = ceil_div(c.H, 128);
  P.sc_kb = ceil_div(c.I, 128);
  P.K = c.I;
  P.N = c.H;
  P.topk_w = topk_w;
  P.out = y;
  return fp8 ? gv::launch_fmt<1, true>(P, c.T, s) : gv::launch_fmt<1, false>(P, c.T, s);
}

}  // namespace moe
