// decode.cu — a decode-sized layer after its router GEMM in one launch: top-k, the align
// table, GEMM1 + SwiGLU, GEMM2 with the router weight and the top-k combine.
//
// Semantics: "Mixture-of-Experts Kernels: Routing, Permutation, and Grouped GEMM", §3 route()
// and §4 route_grouped() (top-k), §5 (the sorted_ids / expert_ids table), §6 (GEMM1 with the
// gather, silu(gate) * up, GEMM2 times topk_w, the sum over k); §7 notes that decode needs
// its own small-batch kernels, and §10 that at decode the router, align and combine cost as
// much as the GEMMs and the layer should approach HBM bandwidth.
//
// With a few tokens (bf16 weights: one or two; FP8 E4M3 weights: up to eight, at most 32
// routed slots) the layer streams the few active experts' weights (gpt-oss-shaped, one token:
// 4 experts, 199 MB) and every separate launch costs a ramp and a tail of several
// microseconds. Here one persistent cooperative launch (every CTA resident) does the rest
// of the layer after the router GEMM:
//   1. every CTA routes the batch itself (warp t: top-k of token t, the same device code as
//      the top-k kernel) and builds the tile list in shared memory (a lane per flat row:
//      warp match, ballots); CTA 0 also writes topk_ids / topk_w and the align table
//      (sorted_ids, expert_ids with the expert map applied, num_post_padded, counts) to
//      the workspace, exactly as the separate route, align and expert-map kernels would;
//   2. GEMM1 items (tile, column) spread evenly over all warps in contiguous ranges (the
//      weight-streaming device code of the small-batch GEMV kernels), act in padded order;
//   3. one grid barrier (bounded: after the pipeline time limit it records kStatusTimeout
//      and the CTA returns);
//   4. GEMM2 items (tile, column pair); after its items a warp makes its y columns visible
//      once and arrives on each item's column pair; the arrival that completes a pair (an
//      arrival counter per pair) adds the k slots of every token in slot order and writes
//      those two columns of out: no second barrier, no separate combine launch.
// Results are bit-identical to the separate entry points (same products, same summation
// orders). The barrier word and the per-pair counters must be zero at launch: the router
// GEMM of moe_forward zeroes them, moe_expert_decode clears them with a memset, and each
// launch leaves them zero again.
#include "gemv_dev.cuh"
#include "route_dev.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace dec {

__device__ int g_decode_status;

constexpr int kMaxRows = 32;  // flat rows T*kk of one launch: a lane each
constexpr int kMaxTokens = 8;  // tokens: a warp each for the top-k
constexpr int kWarps = gv::kWarps;
constexpr int kThreads = gv::kThreads;

struct Params {
  // router output and the top-k rule
  const float* logits;
  int T, E, k, mode, renorm;
  float scale;
  int n_group, topk_group;
  const float* logit_bias;
  const float* select_bias;
  int n_shared;
  int kk, E_eff, B, max_padded;  // slots per token and experts incl. shared ones; table shape
  const int32_t* expert_map;     // [E_eff] or null
  // intermediates (moe_forward workspace layout)
  int32_t* ids;
  float* w;
  int32_t* sid;
  int32_t* eid;
  int32_t* npp;
  int32_t* counts;
  // expert GEMMs: bf16 tokens; bf16 weights, or FP8 E4M3 codes with fp32 128 x 128 block
  // scales (W13: [E', 2, ceil(I/128), ceil(H/128)], W2: [E', ceil(H/128), ceil(I/128)])
  const uint8_t* x;
  const uint8_t* W13;
  const uint8_t* W2;
  const float* s13;
  const float* s2;
  int H, I;
  uint8_t* act;
  uint8_t* y;
  uint8_t* out;
  unsigned* bar;  // [0] arrivals, [1] generation (arrivals 0 at launch)
  int* cnt;       // [H / 2] arrivals per output column pair (0 at launch)
};

struct Smem {
  float skey[kMaxTokens][512];  // top-k scratch (group scores of the grouped router)
  int32_t ids[kMaxRows];
  float w[kMaxRows];
  int2 rows[kMaxRows];          // (padded position p, flat row r) of local tiles, by tile
  int tile_slot[kMaxRows];      // local tile -> weight slot
  int tile_c0[kMaxRows];        // local tile -> first entry of rows[]
  int tile_n[kMaxRows];         // local tile -> real rows
  int gt_cnt[kMaxRows];         // tile of the table (all experts) -> real rows
  int gt_label[kMaxRows];       // tile of the table -> expert_ids label
  int local_row[kMaxRows];      // flat row r is computed on this device
  int n_local, n_tiles, ok;
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Sense-reversing grid barrier over n_ctas CTAs (arrival count bar[0], generation bar[1]).
// The last arrival resets the count and advances the generation; the others poll the
// generation. A wait that outlasts the pipeline time limit records kStatusTimeout and
// returns false (the CTA then leaves the kernel): a barrier that cannot complete ends with a
// status, not a hang.
__device__ bool grid_barrier(unsigned* bar, unsigned n_ctas, int* ok_sh) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned g = ld_acquire(bar + 1);
    __threadfence();
    int ok = 1;
    if (atomicAdd(bar, 1u) == n_ctas - 1) {
      atomicExch(bar, 0u);
      __threadfence();
      st_release(bar + 1, g + 1);
    } else {
      const uint64_t t0 = ptx::gtimer();
      while (ld_acquire(bar + 1) == g) {
        if (ptx::gtimer() - t0 > ptx::kTimeoutNs) {
          atomicExch(&g_decode_status, kStatusTimeout);
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
    *ok_sh = ok;
  }
  __syncthreads();
  return *ok_sh != 0;
}

// Steps 1 (routing and the table) of the kernel; returns with the table in shared memory.
template <int MPL>
__device__ __forceinline__ void route_and_table(const Params& P, Smem& S) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n = P.T * P.kk;
  if (warp < P.T)
    topk_token<MPL>(P.logits, warp, P.E, P.k, P.mode, P.renorm, P.scale, P.n_group,
                    P.topk_group, P.logit_bias, P.select_bias, P.n_shared, S.ids, S.w,
                    S.skey[warp]);
  __syncthreads();
  if (warp == 0) {
    // lane r holds flat row r: its expert, its rank among the rows of that expert (rows of an
    // expert stay in ascending r), the table tile of the expert (experts ascending) and its
    // place among the local rows
    const int e = lane < n ? S.ids[lane] : 0x7fffffff;
    const unsigned below = (1u << lane) - 1u;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & below);
    const bool first = lane < n && rank == 0;
    int slot = e;
    if (lane < n && P.expert_map) {
      slot = P.expert_map[e];
      if (slot < -1 || slot >= P.E_eff) {  // as the expert-map kernel: flagged, not computed
        if (blockIdx.x == 0) atomicExch(&g_decode_status, kStatusBadExpert);
        slot = -1;
      }
    }
    const bool local = lane < n && slot >= 0;
    int g = 0, lt = 0, lcs = 0;
#pragma unroll 4
    for (int j = 0; j < kMaxRows; ++j) {
      const int ej = __shfl_sync(0xffffffffu, e, j);
      const int fj = __shfl_sync(0xffffffffu, (int)first, j);
      const int lj = __shfl_sync(0xffffffffu, (int)local, j);
      g += (fj && ej < e);
      lt += (fj && lj && ej < e);
      lcs += (lj && ej < e);
    }
    if (local) S.rows[lcs + rank] = make_int2(g * P.B + rank, lane);
    if (first && local) {
      S.tile_slot[lt] = slot;
      S.tile_c0[lt] = lcs;
      S.tile_n[lt] = __popc(peers);
    }
    if (first) {
      S.gt_cnt[g] = __popc(peers);
      S.gt_label[g] = P.expert_map ? slot : e;
    }
    S.local_row[lane] = local ? 1 : 0;
    const int n_local = __popc(__ballot_sync(0xffffffffu, first && local));
    const int n_tiles = __popc(__ballot_sync(0xffffffffu, first));
    if (lane == 0) {
      S.n_local = n_local;
      S.n_tiles = n_tiles;
    }
    if (blockIdx.x == 0 && lane < n) {
      P.ids[lane] = e;
      P.w[lane] = S.w[lane];
      P.sid[g * P.B + rank] = lane;
    }
  }
  __syncthreads();
  if (blockIdx.x == 0) {  // the rest of the table: sentinels, tile labels, total, counts
    const int nt = S.n_tiles;
    for (int q = threadIdx.x; q < P.max_padded; q += blockDim.x) {
      const int t = q / P.B, i = q - t * P.B;
      if (!(t < nt && i < S.gt_cnt[t])) P.sid[q] = n;
    }
    for (int t = threadIdx.x; t < P.max_padded / P.B; t += blockDim.x)
      P.eid[t] = t < nt ? S.gt_label[t] : -1;
    for (int e = threadIdx.x; e < P.E_eff; e += blockDim.x) {
      int c = 0;
      for (int r = 0; r < n; ++r) c += S.ids[r] == e;
      if (P.counts) P.counts[e] = c;
    }
    if (threadIdx.x == 0) *P.npp = nt * P.B;
  }
}

template <int RMAX, int MPL, bool FP8>
__global__ void __launch_bounds__(kThreads, (gv::kMinCtas<0, FP8, RMAX>))
    decode_kernel(const Params P) {
  __shared__ Smem S;
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  route_and_table<MPL>(P, S);

  const int A = S.n_local;
  const int gw = blockIdx.x * kWarps + warp, nwarps = gridDim.x * kWarps;
  if (A == 0) {  // no expert of the batch on this device: out is zero
    uint32_t* o = reinterpret_cast<uint32_t*>(P.out);
    for (int i = blockIdx.x * kThreads + threadIdx.x; i < P.T * P.H / 2; i += gridDim.x * kThreads)
      o[i] = 0u;
    return;
  }

  // ---- GEMM1 + SwiGLU: item (local tile t, column c) -> act[p][c] for the tile's rows
  {
    gv::Params G{};
    G.a = P.x;
    G.a_gathered = 0;
    G.k = P.kk;
    G.K = P.H;
    G.N = P.I;
    G.out = P.act;
    const size_t row_bytes = (size_t)P.H * (FP8 ? 1 : 2);
    const int rb = (P.I + 127) / 128, kb = (P.H + 127) / 128;
    // every warp takes total / nwarps items, rounded down or up, so every SM carries the
    // same share of the stream
    const int total = A * P.I;
    const int w0i = (int)((int64_t)gw * total / nwarps);
    const int w1i = (int)((int64_t)(gw + 1) * total / nwarps);
    for (int w = w0i; w < w1i; ++w) {
      const int t = w / P.I, c = w - t * P.I;
      const int slot = S.tile_slot[t];
      const uint8_t* wg = P.W13 + ((size_t)slot * 2 * P.I + c) * row_bytes;
      const uint8_t* wu = wg + (size_t)P.I * row_bytes;
      const float* sg = nullptr;
      const float* su = nullptr;
      if (FP8) {
        sg = P.s13 + (((size_t)slot * 2 + 0) * rb + c / 128) * kb;
        su = P.s13 + (((size_t)slot * 2 + 1) * rb + c / 128) * kb;
      }
      const int2* rl = S.rows + S.tile_c0[t];
      const int nv = S.tile_n[t];
      for (int rc = 0; rc < nv; rc += RMAX)
        gv::item_pass<0, FP8, RMAX, gv::kPieces<0, FP8, RMAX>>(G, wg, wu, sg, su, rl + rc,
                                                               min(RMAX, nv - rc), c);
    }
  }

  if (!grid_barrier(P.bar, gridDim.x, &S.ok)) return;

  // ---- GEMM2 * topk_w: item (local tile t, column pair c) -> y[r][2c, 2c+1]; the last
  // item of a column pair adds the slots of every token into out
  {
    gv::Params G{};
    G.a = P.act;
    G.a_gathered = 1;
    G.k = 1;
    G.K = P.I;
    G.N = P.H;
    G.topk_w = S.w;
    G.out = P.y;
    const size_t row_bytes = (size_t)P.I * (FP8 ? 1 : 2);
    const int rb = (P.H + 127) / 128, kb = (P.I + 127) / 128;
    const int pairs = P.H / 2;
    const int total = A * pairs;
    const int w0i = (int)((int64_t)gw * total / nwarps);
    const int w1i = (int)((int64_t)(gw + 1) * total / nwarps);
    for (int w = w0i; w < w1i; ++w) {
      const int t = w / pairs, c = w - t * pairs, n0 = 2 * c;
      const int slot = S.tile_slot[t];
      const uint8_t* wa = P.W2 + ((size_t)slot * P.H + n0) * row_bytes;
      // columns n0 and n0 + 1 lie in one 128-row block (n0 is even)
      const float* sa = FP8 ? P.s2 + ((size_t)slot * rb + n0 / 128) * kb : nullptr;
      const int2* rl = S.rows + S.tile_c0[t];
      const int nv = S.tile_n[t];
      for (int rc = 0; rc < nv; rc += RMAX)
        gv::item_pass<1, FP8, RMAX, gv::kPieces<1, FP8, RMAX>, true>(
            G, wa, wa + row_bytes, sa, sa, rl + rc, min(RMAX, nv - rc), n0);
    }
    // one fence for all of this warp's y columns, then one arrival per item on its column
    // pair; the arrival that completes a pair adds the slots of every token into out
    if (w0i < w1i) {
      __threadfence();
      __syncwarp();
    }
    for (int w = w0i; w < w1i; ++w) {
      const int c = w % pairs, n0 = 2 * c;
      int prev = 0;
      if (lane == 0) prev = atomicAdd(&P.cnt[c], 1);
      prev = __shfl_sync(0xffffffffu, prev, 0);
      if (prev == A - 1) {
        __threadfence();
        for (int tok = lane; tok < P.T; tok += 32) {
          float a0 = 0.f, a1 = 0.f;
          for (int j = 0; j < P.kk; ++j) {
            const int r = tok * P.kk + j;
            if (!S.local_row[r]) continue;
            const uint32_t v = __ldcg(reinterpret_cast<const unsigned*>(
                P.y + ((size_t)r * P.H + n0) * 2));
            a0 += gv::bf_lo(v);
            a1 += gv::bf_hi(v);
          }
          *reinterpret_cast<uint32_t*>(P.out + ((size_t)tok * P.H + n0) * 2) =
              gv::pack_bf16x2(a0, a1);
        }
        __syncwarp();
        if (lane == 0) P.cnt[c] = 0;  // zero again for the next launch
      }
    }
  }
}

// Failure-path self-test of the grid barrier: one CTA enters a barrier of two, which
// nothing completes; after the time limit the wait gives up and records kStatusTimeout.
__device__ unsigned g_selftest_bar[2];

__global__ void __launch_bounds__(64) selftest_barrier_kernel() {
  __shared__ int ok;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) {
    g_selftest_bar[0] = 0u;
    g_selftest_bar[1] = 0u;
    __threadfence();
  }
  grid_barrier(g_selftest_bar, 2u, &ok);
}

// Launch: cooperative (the grid barrier needs every CTA resident) with programmatic stream
// serialisation when the runtime accepts both; the grid is every CTA that fits at once.
template <int RMAX, int MPL, bool FP8>
static moe_status_t launch_rm(const Params& P, cudaStream_t s) {
  auto kern = decode_kernel<RMAX, MPL, FP8>;
  static int per_sm[64];
  static int pdl_state[64];  // 0: untried, 1: cooperative + PDL accepted, 2: cooperative only
  int dev = 0;
  cudaGetDevice(&dev);
  dev &= 63;
  if (per_sm[dev] == 0) {
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, kThreads, 0) != cudaSuccess ||
        v < 1)
      return MOE_ERR_CUDA;
    per_sm[dev] = v;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms() * per_sm[dev]);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  if (pdl_state[dev] != 2) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(s, &cs);
    // the first try of both attributes happens outside stream capture
    if (pdl_state[dev] == 1 || cs == cudaStreamCaptureStatusNone) {
      cfg.numAttrs = 2;
      if (cudaLaunchKernelEx(&cfg, kern, P) == cudaSuccess) {
        pdl_state[dev] = 1;
        return MOE_OK;
      }
      if (pdl_state[dev] == 1) return MOE_ERR_CUDA;
      cudaGetLastError();
      pdl_state[dev] = 2;
    }
  }
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, P) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

template <int RMAX, bool FP8>
static moe_status_t launch_r(const Params& P, cudaStream_t s) {
  switch (topk_per_lane(P.E)) {
    case 4: return launch_rm<RMAX, 4, FP8>(P, s);
    case 8: return launch_rm<RMAX, 8, FP8>(P, s);
    default: return launch_rm<RMAX, kMaxPerLane, FP8>(P, s);
  }
}

// Rows a pass takes: a tile holds at most T real rows (a token takes an expert once).
template <bool FP8>
static moe_status_t launch_fmt(const Params& P, cudaStream_t s) {
  if (P.T <= 1) return launch_r<1, FP8>(P, s);
  if (P.T <= 2) return launch_r<2, FP8>(P, s);
  return launch_r<4, FP8>(P, s);
}

}  // namespace dec

bool decode_applies(const moe_config_t& c) {
  const int kk = c.k + c.n_shared;
  moe_config_t e = c;
  e.k = kk;
  e.E = c.E + c.n_shared;
  e.n_shared = 0;
  const int mp = (int)moe_max_padded_rows(e.T, e.k, e.E, 128);
  // the small-batch GEMMs' range (bf16: up to 2 tokens; FP8 weights: up to 32), a warp per
  // token for the top-k and a lane per routed slot for the table
  return c.dtype == MOE_BF16 && c.T <= dec::kMaxTokens && c.T * kk <= dec::kMaxRows &&
         gemv_applies(e, mp);
}

size_t decode_sync_bytes(const moe_config_t& c) {
  return align_up((size_t)(2 + c.H / 2) * sizeof(int), 256);
}

moe_status_t launch_decode(const moe_config_t& c, const float* logits, const void* x,
                           const void* W13, const void* W2, void* out, const DecodeWs& w,
                           cudaStream_t s) {
  if (!decode_applies(c)) return MOE_ERR_UNSUPPORTED;
  dec::Params P{};
  P.logits = logits;
  P.T = c.T;
  P.E = c.E;
  P.k = c.k;
  P.mode = (int)c.mode;
  P.renorm = c.renormalize;
  P.scale = c.scale;
  P.n_group = c.n_group;
  P.topk_group = c.topk_group;
  P.logit_bias = c.logit_bias;
  P.select_bias = c.select_bias;
  P.n_shared = c.n_shared;
  P.kk = c.k + c.n_shared;
  P.E_eff = c.E + c.n_shared;
  P.B = 128;
  P.max_padded = (int)moe_max_padded_rows(c.T, P.kk, P.E_eff, 128);
  P.expert_map = c.expert_map;
  P.ids = w.ids;
  P.w = w.w;
  P.sid = w.sid;
  P.eid = w.eid;
  P.npp = w.npp;
  P.counts = w.counts;
  P.x = (const uint8_t*)x;
  P.W13 = (const uint8_t*)W13;
  P.W2 = (const uint8_t*)W2;
  const bool fp8 = c.weight_format == MOE_WEIGHTS_FP8_E4M3_B128;
  P.s13 = fp8 ? c.w13_scale : nullptr;
  P.s2 = fp8 ? c.w2_scale : nullptr;
  P.H = c.H;
  P.I = c.I;
  P.act = (uint8_t*)w.act;
  P.y = (uint8_t*)w.y;
  P.out = (uint8_t*)out;
  P.bar = (unsigned*)w.sync;
  P.cnt = (int*)w.sync + 2;
  return fp8 ? dec::launch_fmt<true>(P, s) : dec::launch_fmt<false>(P, s);
}

moe_status_t launch_selftest_decode_wait(cudaStream_t s) {
  return launch_k(dec::selftest_barrier_kernel, dim3(1), dim3(64), 0, s);
}

int decode_status_read(int reset) {
  int v = 0;
  cudaMemcpyFromSymbol(&v, dec::g_decode_status, sizeof(int));
  if (reset) {
    int z = 0;
    cudaMemcpyToSymbol(dec::g_decode_status, &z, sizeof(int));
  }
  return v;
}

}  // namespace moe
