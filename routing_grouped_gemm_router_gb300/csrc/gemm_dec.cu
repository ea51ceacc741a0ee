// gemm_dec.cu — the grouped expert GEMMs for decode-sized batches on the tensor cores, with
// the expert weights as the MMA's 128-row operand.
//
// Semantics are those of the grouped GEMMs of "Mixture-of-Experts Kernels: Routing,
// Permutation, and Grouped GEMM", §6, on the same inputs and outputs as the CTA-pair kernels
// (gemm_tc2.cu): a 128-row tile of the padded order belongs to expert expert_ids[tile];
// GEMM1 writes act[p] = silu(x_r W1[e]^T) * (x_r W3[e]^T) for every real row p
// (sorted_ids[p] < T*k), GEMM2 writes y[r] = topk_w[r] * act[p] W2[e]^T at r = sorted_ids[p].
// Page §7: decode needs kernels of its own; with a handful of rows per expert the layer is a
// stream of the active experts' weights.
//
// Design. A work item is (tile, 128-row block of the expert's weight matrix). The MMA is
// swapped relative to the pair kernels: D[128 weight rows, 128 tile rows] = W[128, K] .
// X[128, K]^T (tcgen05 cta_group::1, M = N = 128), so the weights stream through the
// 128-row operand and the tile's token rows (gathered rows for GEMM1, act for GEMM2) are the
// N operand, read from L2. At decode the tensor work is far below the weight stream, so one
// CTA per SM moves the weights with deep TMA rings and no cross-CTA synchronisation. GEMM1
// runs the gate block and the up block of the same output columns as two MMAs into two
// accumulators, so the thread of TMEM lane m holds gate and up of column m for every tile row.
// The epilogue reads the tile's sorted_ids and stores only the real rows.
//
// FP8 E4M3 weights (128 x 128 block scales): the producer streams raw codes into a ring of
// their own, several k-blocks deep; four converter warps turn each k-block into the bf16
// operand (code * scale, exact for power-of-two scales) in a shallower operand ring, all
// with CTA-local barriers.
//
// Warp roles: 0 TMA producer, 1 MMA issuer (one lane), 2-5 epilogue, 6-9 converters (FP8).
// Every mbarrier wait is bounded (time-out: status kStatusTimeout, abort, copies in flight
// drained, TMEM freed).
#include "tc_ptx.cuh"

namespace moe {
namespace dec {

using namespace ptx;

__device__ int g_dec_status;

enum Mode { kGemm1 = 0, kGemm2 = 1 };
constexpr int kMaxTokens = 128;       // batches this kernel takes (see dec_gemm_applies)
constexpr int kMaxTiles = 1024;       // 128-row tiles of the table a launch may hold
constexpr int A_BYTES = 128 * 128;    // 128 weight rows x 64 bf16 (one swizzled k-block)
constexpr int X_BYTES = 128 * 128;    // 128 tile rows x 64 bf16
constexpr int RAW_BYTES = 128 * BK;   // 128 weight rows x 64 E4M3 codes

struct Params {
  int n_rows;      // T*k: sorted_ids >= n_rows are padding
  int N;           // output columns: I (GEMM1), H (GEMM2)
  int K;           // reduction length: H (GEMM1), I (GEMM2)
  int m_blocks;    // ceil(N / 128)
  int block_m;
  const int32_t* sid;
  const int32_t* eid;
  const int32_t* npp;
  const float* topk_w;
  void* out;       // GEMM1: act [padded, I]; GEMM2: y [T*k, H]
  const float* scale;  // FP8: [slots][grids][row blocks][k blocks]
  int sc_rb, sc_kb;
  int n_slots;
  int max_tiles;   // tiles of the table's buffers (max_padded / 128)
};

template <int MODE, bool FP8>
struct Cfg {
  static constexpr int NA = MODE == kGemm1 ? 2 : 1;  // weight blocks per k-block (gate, up)
  static constexpr int OP_BYTES = NA * A_BYTES + X_BYTES;
  static constexpr int RAWS_BYTES = NA * RAW_BYTES;
  static constexpr int kOpStages = FP8 ? (MODE == kGemm1 ? 3 : 4) : (MODE == kGemm1 ? 4 : 6);
  static constexpr int kRawStages = FP8 ? (MODE == kGemm1 ? 4 : 10) : 0;
  static constexpr int kCvtWarps = 4;
  static constexpr int kThreads = (6 + (FP8 ? kCvtWarps : 0)) * 32;
  static constexpr uint32_t kTmemCols = 2u * NA * 128u;  // two accumulators of NA x 128 columns
  // shared memory (offsets from a 1024-aligned base)
  static constexpr size_t op = 0;
  static constexpr size_t raw = op + (size_t)kOpStages * OP_BYTES;
  static constexpr size_t bars = raw + (size_t)kRawStages * RAWS_BYTES;
  static constexpr size_t n_bars = 2 * kOpStages + 2 * kRawStages + 5;
  static constexpr size_t misc = bars + n_bars * 8;  // tmem slot, abort flag, tile count
  static constexpr size_t tiles = misc + 16;
  static constexpr size_t end = tiles + kMaxTiles * 4;
  static constexpr size_t bytes = 1024 + end;
  // the op-stage barrier completes on: bf16, the producer's expect_tx arrival (weights and
  // tile rows); FP8, converter warp 0's expect_tx arrival (tile rows) plus one arrival of
  // each converter warp once its rows of the weights are written
  static constexpr int kOpArrivals = FP8 ? 1 + kCvtWarps : 1;
};
static_assert(Cfg<kGemm1, false>::bytes <= 232448, "shared memory");
static_assert(Cfg<kGemm1, true>::bytes <= 232448, "shared memory");
static_assert(Cfg<kGemm2, false>::bytes <= 232448, "shared memory");
static_assert(Cfg<kGemm2, true>::bytes <= 232448, "shared memory");

template <int MODE, bool FP8>
__global__ void __launch_bounds__(Cfg<MODE, FP8>::kThreads, 1)
    dec_kernel(const __grid_constant__ CUtensorMap tmW0, const __grid_constant__ CUtensorMap tmW1,
               const __grid_constant__ CUtensorMap tmX, const Params P) {
  using C = Cfg<MODE, FP8>;
  constexpr int NA = C::NA;
  constexpr int S = C::kOpStages;
  constexpr int R = C::kRawStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + C::bars);
  uint64_t* opfull = bars;
  uint64_t* opempty = bars + S;
  uint64_t* rawfull = bars + 2 * S;
  uint64_t* rawempty = rawfull + R;
  uint64_t* tfull = rawempty + R;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = (uint32_t*)(smem + C::misc);
  volatile int* abort_flag = (volatile int*)(smem + C::misc + 4);
  int* ntiles_sh = (int*)(smem + C::misc + 8);
  int* tl = (int*)(smem + C::tiles);  // valid tiles of the table, ascending
  int* status = &g_dec_status;

  pdl_trigger();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&opfull[s], C::kOpArrivals);
      mbar_init(&opempty[s], 1);
    }
    for (int r = 0; r < R; ++r) {
      mbar_init(&rawfull[r], 1);
      mbar_init(&rawempty[r], C::kCvtWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_init_fence();
    prefetch_tmap(&tmW0);
    if (MODE == kGemm1) prefetch_tmap(&tmW1);
    prefetch_tmap(&tmX);
  }
  if (warp == 1) {
    tmem_alloc<1>(tmem_slot, C::kTmemCols);
    tmem_relinquish<1>();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  pdl_wait();  // global memory is touched only past this point
  // ---- the tiles whose expert is on this device, in order
  if (warp == 0) {
    const int num_t = min(*P.npp / 128, min(P.max_tiles, kMaxTiles));
    int n = 0;
    for (int base = 0; base < num_t; base += 32) {
      const int t = base + lane;
      const int e = t < num_t ? P.eid[(t * 128) / P.block_m] : -1;
      const bool ok = e >= 0 && e < P.n_slots;
      const unsigned m = __ballot_sync(0xffffffffu, ok);
      if (ok) tl[n + __popc(m & ((1u << lane) - 1u))] = t;
      n += __popc(m);
    }
    if (lane == 0) *ntiles_sh = n;
  }
  __syncthreads();
  const int total = *ntiles_sh * P.m_blocks;
  const int num_kb = (P.K + BK - 1) / BK;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
        const int t = tl[w / P.m_blocks], j = w % P.m_blocks;
        const int e = P.eid[(t * 128) / P.block_m];
        for (int kb = 0; kb < num_kb; ++kb, ++g) {
          if constexpr (FP8) {  // raw codes of the weight blocks into the raw ring
            const int r = g % R;
            if (!wait_bounded(&rawempty[r], ((uint32_t)(g / R) & 1u) ^ 1u, abort_flag, status)) {
              ok = false;
              break;
            }
            uint8_t* dst = smem + C::raw + (size_t)r * C::RAWS_BYTES;
            mbar_expect_tx(&rawfull[r], C::RAWS_BYTES);
            tma_3d(dst, &tmW0, &rawfull[r], kb * BK, j * 128, e);
            if (MODE == kGemm1) tma_3d(dst + RAW_BYTES, &tmW1, &rawfull[r], kb * BK, j * 128, e);
          } else {  // bf16 weight blocks and the tile rows into the operand ring
            const int s = g % S;
            if (!wait_bounded(&opempty[s], ((uint32_t)(g / S) & 1u) ^ 1u, abort_flag, status)) {
              ok = false;
              break;
            }
            uint8_t* dst = smem + C::op + (size_t)s * C::OP_BYTES;
            mbar_expect_tx(&opfull[s], C::OP_BYTES);
            tma_3d(dst, &tmW0, &opfull[s], kb * BK, j * 128, e);
            if (MODE == kGemm1) tma_3d(dst + A_BYTES, &tmW1, &opfull[s], kb * BK, j * 128, e);
            tma_2d(dst + NA * A_BYTES, &tmX, &opfull[s], kb * BK, t * 128);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (one lane)
    // The MMA's N covers the tile's rows up to its last real one (rounded up to 16): at decode
    // a tile holds a few real rows, and the columns past them would only cost tensor time.
    int g = 0, acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true, issued = false;
    for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const int t = tl[w / P.m_blocks];
      int last = -1;  // the tile's last real row (sorted_ids needs only 4-byte alignment)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (P.sid[t * 128 + i * 32 + lane] < P.n_rows) last = i * 32 + lane;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, off));
      const int n_cols = last < 16 ? 16 : (last + 16) / 16 * 16;
      const uint32_t idesc = idesc_bf16(128, n_cols);
      if (lane == 0) {
        if (!wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, status)) ok = false;
      }
      if (!__shfl_sync(0xffffffffu, (int)ok, 0)) break;
      if (lane == 0) {
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * NA * 128);
        for (int kb = 0; kb < num_kb; ++kb, ++g) {
          const int s = g % S;
          if (!wait_bounded(&opfull[s], (uint32_t)(g / S) & 1u, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t base = su32(smem + C::op + (size_t)s * C::OP_BYTES);
          const uint32_t xb = base + NA * A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk)
#pragma unroll
            for (int a = 0; a < NA; ++a)
              umma_bf16<1>(d + a * 128, sw128_desc(base + a * A_BYTES + kk * 32),
                           sw128_desc(xb + kk * 32), idesc, (kb | kk) != 0 ? 1u : 0u);
          umma_commit<1>(&opempty[s]);
          issued = true;
        }
        if (ok) umma_commit<1>(&tfull[acc]);
      }
      if (!__shfl_sync(0xffffffffu, (int)ok, 0)) break;
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (lane == 0 && issued) {  // every MMA of this thread finished before TMEM is freed
      umma_commit<1>(drain);
      wait_bounded(drain, 0, abort_flag, status);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter: weight rows q*32 .. q*32+31 of the block
    const int m = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int w = blockIdx.x; w < total; w += gridDim.x) {
      const int t = tl[w / P.m_blocks], j = w % P.m_blocks;
      const int col = j * 128 + m;  // output column of this thread
      int sid4[4];                  // flat rows of tile rows c*32 + lane
#pragma unroll
      for (int c = 0; c < 4; ++c) sid4[c] = P.sid[t * 128 + c * 32 + lane];
      int ok = 1;
      if (lane == 0) ok = wait_bounded(&tfull[acc], acc_phase, abort_flag, status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (uint32_t)(acc * NA * 128) + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        const unsigned real = __ballot_sync(0xffffffffu, sid4[c] < P.n_rows);
        if (!real) continue;  // 32 padding rows: nothing to store
        if (MODE == kGemm1) {
          uint32_t gv[32], uv[32];
          tmem_ld32(tb + c * 32, gv);
          tmem_ld32(tb + 128 + c * 32, uv);
          tmem_ld_wait();
          __nv_bfloat16* dst = (__nv_bfloat16*)P.out + (int64_t)(t * 128 + c * 32) * P.N + col;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (!((real >> i) & 1u) || col >= P.N) continue;
            const float g0 = __uint_as_float(gv[i]);
            dst[(int64_t)i * P.N] = __float2bfloat16(g0 / (1.f + __expf(-g0)) * __uint_as_float(uv[i]));
          }
        } else {
          uint32_t dv[32];
          tmem_ld32(tb + c * 32, dv);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int r = __shfl_sync(0xffffffffu, sid4[c], i);
            if (r >= P.n_rows || col >= P.N) continue;
            ((__nv_bfloat16*)P.out)[(int64_t)r * P.N + col] =
                __float2bfloat16(P.topk_w[r] * __uint_as_float(dv[i]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
  } else if constexpr (FP8) {
    // ------------------------------------------------------------ FP8 converters (4 warps)
    // Warp cw turns rows cw*32 .. cw*32+31 of each raw 128 x 64 code block into the
    // 128-byte-swizzled bf16 K-major layout the MMA descriptor expects (16-byte chunk c of
    // row r at r*128 + ((c ^ (r & 7)) << 4)), scaled by the block's scale. Converter warp 0
    // also loads the tile rows into the operand slot once it is free.
    const int cw = warp - 6;
    int g = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const int t = tl[w / P.m_blocks], j = w % P.m_blocks;
      const int e = P.eid[(t * 128) / P.block_m];
      const bool sc_ok = e >= 0 && e < P.n_slots && j < P.sc_rb;
      // block scales of this item in windows of 32 k-block pairs: lane i holds the scale of
      // 128-wide k-block win + i of each weight block, so a k-block's scale is a shuffle, not
      // a global load on the critical path (the raw codes are usually waiting already)
      float scw[NA];
      int win = -32;
      for (int kb = 0; kb < num_kb; ++kb, ++g) {
        const int r = g % R, s = g % S;
        const int sb = kb >> 1;
        if (sb - win >= 32) {
          win = sb & ~31;
#pragma unroll
          for (int a = 0; a < NA; ++a)
            scw[a] = sc_ok && win + lane < P.sc_kb
                         ? __ldg(P.scale + (((int64_t)e * NA + a) * P.sc_rb + j) * P.sc_kb +
                                 win + lane)
                         : 0.f;
        }
        float sc[NA];
#pragma unroll
        for (int a = 0; a < NA; ++a) sc[a] = __shfl_sync(0xffffffffu, scw[a], sb - win);
        int okw = 1;
        if (lane == 0) {
          okw = wait_bounded(&opempty[s], ((uint32_t)(g / S) & 1u) ^ 1u, abort_flag, status) &&
                wait_bounded(&rawfull[r], (uint32_t)(g / R) & 1u, abort_flag, status);
          if (okw && cw == 0) {
            uint8_t* xdst = smem + C::op + (size_t)s * C::OP_BYTES + NA * A_BYTES;
            mbar_expect_tx(&opfull[s], X_BYTES);
            tma_2d(xdst, &tmX, &opfull[s], kb * BK, t * 128);
          }
        }
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) {
          ok = false;
          break;
        }
        const uint8_t* src = smem + C::raw + (size_t)r * C::RAWS_BYTES;
        uint8_t* dst = smem + C::op + (size_t)s * C::OP_BYTES;
#pragma unroll
        for (int a = 0; a < NA; ++a) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            // 16-code unit u of this warp's 32 rows: row u / 4, codes (u % 4) * 16 .. +15
            const int u = i * 32 + lane;
            const int row = cw * 32 + (u >> 2), h = u & 3;
            const uint4 qv = *reinterpret_cast<const uint4*>(src + a * RAW_BYTES + row * BK + h * 16);
            uint32_t v[8];
            e4m3x16_scaled_bf16(qv, sc[a], v);
            uint8_t* drow = dst + a * A_BYTES + row * 128;
            *reinterpret_cast<uint4*>(drow + (((2 * h) ^ (row & 7)) << 4)) =
                make_uint4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<uint4*>(drow + (((2 * h + 1) ^ (row & 7)) << 4)) =
                make_uint4(v[4], v[5], v[6], v[7]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&rawempty[r]);
          mbar_arrive(&opfull[s]);
        }
      }
    }
  }

  __syncthreads();
  if (*abort_flag) {  // let copies already in flight land before shared memory is released
    const uint64_t t0 = gtimer();
    while (gtimer() - t0 < 200000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<1>(tmem_base, C::kTmemCols);
  }
}

template <int MODE, bool FP8>
static moe_status_t launch(const CUtensorMap& w0, const CUtensorMap& w1, const CUtensorMap& x,
                           const Params& P, int max_items, cudaStream_t s) {
  auto kern = dec_kernel<MODE, FP8>;
  constexpr size_t smem = Cfg<MODE, FP8>::bytes;
  static int configured[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (!configured[dev & 63]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    configured[dev & 63] = 1;
  }
  const int grid = std::max(1, std::min(num_sms(), max_items));
  return launch_k(kern, dim3(grid), dim3(Cfg<MODE, FP8>::kThreads), smem, s, w0, w1, x, P);
}

}  // namespace dec

int dec_status_read(int reset) {
  int v = 0;
  cudaMemcpyFromSymbol(&v, dec::g_dec_status, sizeof(int));
  if (reset) {
    int z = 0;
    cudaMemcpyToSymbol(dec::g_dec_status, &z, sizeof(int));
  }
  return v;
}

bool dec_gemm_applies(const moe_config_t& c, int max_padded) {
  return c.dtype == MOE_BF16 && c.T <= dec::kMaxTokens && max_padded / 128 <= dec::kMaxTiles;
}

moe_status_t launch_gemm1_dec(const moe_config_t& c, const void* xs, const void* W13,
                              const int32_t* sid, const int32_t* eid, const int32_t* npp,
                              int block_m, int max_padded, void* act, cudaStream_t s) {
  using namespace dec;
  if (max_padded / 128 > kMaxTiles) return MOE_ERR_UNSUPPORTED;
  const bool fp8 = c.weight_format == MOE_WEIGHTS_FP8_E4M3_B128;
  CUtensorMap mG, mU, mX;
  const uint64_t H = c.H, I = c.I, E = c.E;
  {
    uint64_t d[3] = {H, I, E}, st[2] = {H, 2 * I * H};
    uint32_t box[3] = {BK, 128, 1};
    const uint8_t* up = (const uint8_t*)W13 + I * H * (fp8 ? 1 : 2);
    if (!make_map(&mG, W13, 3, d, st, box, true, fp8)) return MOE_ERR_CUDA;
    if (!make_map(&mU, up, 3, d, st, box, true, fp8)) return MOE_ERR_CUDA;
  }
  {
    uint64_t d[2] = {H, (uint64_t)max_padded}, st[1] = {H};
    uint32_t box[2] = {BK, 128};
    if (!make_map(&mX, xs, 2, d, st, box, false)) return MOE_ERR_CUDA;
  }
  Params P{};
  P.n_rows = c.T * c.k;
  P.N = c.I;
  P.K = c.H;
  P.m_blocks = ceil_div(c.I, 128);
  P.block_m = block_m;
  P.sid = sid;
  P.eid = eid;
  P.npp = npp;
  P.out = act;
  P.scale = c.w13_scale;
  P.sc_rb = ceil_div(c.I, 128);
  P.sc_kb = ceil_div(c.H, 128);
  P.n_slots = c.E;
  P.max_tiles = max_padded / 128;
  const int items = P.max_tiles * P.m_blocks;
  return fp8 ? launch<kGemm1, true>(mG, mU, mX, P, items, s)
             : launch<kGemm1, false>(mG, mU, mX, P, items, s);
}

moe_status_t launch_gemm2_dec(const moe_config_t& c, const void* act, const void* W2,
                              const int32_t* sid, const int32_t* eid, const int32_t* npp,
                              int block_m, int max_padded, const float* topk_w, void* y,
                              cudaStream_t s) {
  using namespace dec;
  if (max_padded / 128 > kMaxTiles) return MOE_ERR_UNSUPPORTED;
  const bool fp8 = c.weight_format == MOE_WEIGHTS_FP8_E4M3_B128;
  CUtensorMap mW, mX;
  const uint64_t H = c.H, I = c.I, E = c.E;
  {
    uint64_t d[3] = {I, H, E}, st[2] = {I, H * I};
    uint32_t box[3] = {BK, 128, 1};
    if (!make_map(&mW, W2, 3, d, st, box, true, fp8)) return MOE_ERR_CUDA;
  }
  {
    uint64_t d[2] = {I, (uint64_t)max_padded}, st[1] = {I};
    uint32_t box[2] = {BK, 128};
    if (!make_map(&mX, act, 2, d, st, box, false)) return MOE_ERR_CUDA;
  }
  Params P{};
  P.n_rows = c.T * c.k;
  P.N = c.H;
  P.K = c.I;
  P.m_blocks = ceil_div(c.H, 128);
  P.block_m = block_m;
  P.sid = sid;
  P.eid = eid;
  P.npp = npp;
  P.topk_w = topk_w;
  P.out = y;
  P.scale = c.w2_scale;
  P.sc_rb = ceil_div(c.H, 128);
  P.sc_kb = ceil_div(c.I, 128);
  P.n_slots = c.E;
  P.max_tiles = max_padded / 128;
  const int items = P.max_tiles * P.m_blocks;
  return fp8 ? launch<kGemm2, true>(mW, mW, mX, P, items, s)
             : launch<kGemm2, false>(mW, mW, mX, P, items, s);
}

}  // namespace moe
