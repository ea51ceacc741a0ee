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
// The tile rows are loaded only up to the tile's last real row (16-row boxes): at decode a
// tile holds a few tokens, and the MMA's N is cut to the same width.
//
// FP8 E4M3 weights (128 x 128 block scales): the producer streams raw codes into a ring of
// their own, several k-blocks deep; eight converter warps turn each k-block into the bf16
// operand (code * scale, exact for power-of-two scales) in a shallower operand ring, and a
// warp of its own streams the tile rows into a third ring (slots sized to the item's rows),
// all with CTA-local barriers, so that no copy waits for an operand slot. Each converter lane
// loads all of its codes of a k-block before it stores any converted operand (the stores
// could otherwise alias the next loads, which serialises them). Measured per k-block
// (timestamps in the kernel): the codes wait in their ring long before they are needed; the
// converters' integer work (~0.5 us a k-block) and the MMA thread (~0.26 us fixed per
// k-block plus ~32 ns per N = 16 MMA) set the pace.
//
// Warp roles: 0 TMA producer (weights; bf16 also the tile rows), 1 MMA issuer (one lane),
// 2-5 epilogue; FP8 adds 8 converters on warps 6-15 and the tile-row producer on warp 16.
// Every mbarrier wait is bounded (time-out: status kStatusTimeout, abort, copies in flight
// drained, TMEM freed). All roles but the MMA issuer wait with a suspend hint, so that
// waiting warps do not take issue slots from the converters.
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
constexpr int X_BOX = 16;             // tile rows per TMA box (2 KB, 1024-byte aligned)
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
  static constexpr int OP_BYTES = NA * A_BYTES + (FP8 ? 0 : X_BYTES);
  static constexpr int RAWS_BYTES = NA * RAW_BYTES;
  static constexpr int kOpStages = FP8 ? (MODE == kGemm1 ? 3 : 4) : (MODE == kGemm1 ? 4 : 6);
  static constexpr int kRawStages = FP8 ? (MODE == kGemm1 ? 6 : 12) : 0;
  // FP8 tile-row ring: XR_BYTES split into slots of one k-block of the item's n_cols rows
  // (n_cols * 128 bytes), at most kMaxXSlots of them (GEMM1: 8 k-blocks ahead at decode, one
  // for a full tile; GEMM2: 24 and 3)
  static constexpr int XR_BYTES = FP8 ? (MODE == kGemm1 ? 16 : 48) * 1024 : 0;
  static constexpr int kMaxXSlots = FP8 ? 32 : 0;
  // FP8 converters: 8 warps of 16 rows each, on warps 6-8, 10-12, 14-15, so that none shares
  // the MMA issuer's scheduler (warp 1; a warp runs on scheduler warp % 4); warps 9 and 13
  // have no role. Warp 16 streams the tile rows.
  static constexpr int kCvtWarps = 8;
  static constexpr int kXWarp = 16;
  static constexpr int kThreads = (FP8 ? 17 : 6) * 32;
  static constexpr uint32_t kTmemCols = 2u * NA * 128u;  // two accumulators of NA x 128 columns
  // shared memory (offsets from a 1024-aligned base)
  static constexpr size_t op = 0;
  static constexpr size_t raw = op + (size_t)kOpStages * OP_BYTES;
  static constexpr size_t xr = raw + (size_t)kRawStages * RAWS_BYTES;
  static constexpr size_t bars = xr + (size_t)XR_BYTES;
  static constexpr size_t n_bars = 2 * kOpStages + 2 * kRawStages + 2 * kMaxXSlots + 5;
  static constexpr size_t misc = bars + n_bars * 8;  // tmem slot, abort flag, tile count
  static constexpr size_t tiles = misc + 16;
  static constexpr size_t end = tiles + kMaxTiles * 4;
  static constexpr size_t bytes = 1024 + end;
  // the op-stage barrier completes on: bf16, the producer's expect_tx arrival (weights and
  // tile rows); FP8, one arrival of each converter warp once its rows are written
  static constexpr int kOpArrivals = FP8 ? kCvtWarps : 1;
};
static_assert(Cfg<kGemm1, false>::bytes <= 232448, "shared memory");
static_assert(Cfg<kGemm1, true>::bytes <= 232448, "shared memory");
static_assert(Cfg<kGemm2, false>::bytes <= 232448, "shared memory");
static_assert(Cfg<kGemm2, true>::bytes <= 232448, "shared memory");

// Tile rows the MMA covers for tile t: up to its last real row (sorted_ids < T*k), rounded up
// to 16. Warp-collective; sorted_ids needs only 4-byte alignment, so four scalar loads a lane.
__device__ __forceinline__ int tile_cols(const Params& P, int t, int lane) {
  int last = -1;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (P.sid[t * 128 + i * 32 + lane] < P.n_rows) last = i * 32 + lane;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, off));
  return last < 16 ? 16 : (last + 16) / 16 * 16;
}

// Bytes of one slot of the FP8 tile-row ring for an item of n_cols tile rows (n_cols rounded
// up to a power of two, so that the slot size changes rarely between items), and the slots.
__device__ __forceinline__ int x_slot_bytes(int n_cols) {
  int r = 16;
  while (r < n_cols) r *= 2;
  return r * 128;
}
template <class C>
__device__ __forceinline__ int x_slots(int slot_bytes) {
  return min(C::kMaxXSlots, C::XR_BYTES / slot_bytes);
}

// The tile rows [t*128, t*128 + n_cols) of k-block kb as n_cols / 16 boxes of 16 rows, laid
// out as the first n_cols rows of a 128-row swizzled block.
__device__ __forceinline__ void load_tile_rows(uint8_t* dst, const CUtensorMap* tm, uint64_t* bar,
                                               int kb, int t, int n_cols) {
  for (int c = 0; c < n_cols / X_BOX; ++c)
    tma_2d(dst + c * X_BOX * 128, tm, bar, kb * BK, t * 128 + c * X_BOX);
}

template <int MODE, bool FP8>
__global__ void __launch_bounds__(Cfg<MODE, FP8>::kThreads, 1)
    dec_kernel(const __grid_constant__ CUtensorMap tmW0, const __grid_constant__ CUtensorMap tmW1,
               const __grid_constant__ CUtensorMap tmX, const Params P) {
  using C = Cfg<MODE, FP8>;
  constexpr int NA = C::NA;
  constexpr int S = C::kOpStages;
  constexpr int R = C::kRawStages;
  constexpr int SX = C::kMaxXSlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = (uint64_t*)(smem + C::bars);
  uint64_t* opfull = bars;
  uint64_t* opempty = bars + S;
  uint64_t* rawfull = bars + 2 * S;
  uint64_t* rawempty = rawfull + R;
  uint64_t* xfull = rawempty + R;
  uint64_t* xempty = xfull + SX;
  uint64_t* tfull = xempty + SX;
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
    for (int x = 0; x < SX; ++x) {  // slots of the tile-row ring
      mbar_init(&xfull[x], 1);
      mbar_init(&xempty[x], 1);
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
  // Items go to the first `active` CTAs, each taking the same count (the last possibly fewer):
  // the weight stream bounds these GEMMs, so the bandwidth of CTAs left without an item goes
  // to the others instead of a last round in which most SMs idle (GEMM1 at 8 tokens: 644
  // items on 152 CTAs took 5 rounds, the last with 36 CTAs; now 129 CTAs take 5 each).
  const int per_cta = (total + gridDim.x - 1) / gridDim.x;
  const int active = per_cta > 0 ? (total + per_cta - 1) / per_cta : 0;
  const int first = (int)blockIdx.x < active ? (int)blockIdx.x : total;
  const int num_kb = (P.K + BK - 1) / BK;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int g = 0;
    bool ok = true;
    for (int w = first; w < total && ok; w += active) {
      const int t = tl[w / P.m_blocks], j = w % P.m_blocks;
      const int n_cols = FP8 ? 0 : tile_cols(P, t, lane);
      if (lane == 0) {
        const int e = P.eid[(t * 128) / P.block_m];
        for (int kb = 0; kb < num_kb; ++kb, ++g) {
          if constexpr (FP8) {  // raw codes of the weight blocks into the raw ring
            const int r = g % R;
            if (!wait_bounded_sleep(&rawempty[r], ((uint32_t)(g / R) & 1u) ^ 1u, abort_flag, status)) {
              ok = false;
              break;
            }
            uint8_t* dst = smem + C::raw + (size_t)r * C::RAWS_BYTES;
            mbar_expect_tx(&rawfull[r], C::RAWS_BYTES);
            tma_3d(dst, &tmW0, &rawfull[r], kb * BK, j * 128, e);
            if (MODE == kGemm1) tma_3d(dst + RAW_BYTES, &tmW1, &rawfull[r], kb * BK, j * 128, e);
          } else {  // bf16 weight blocks and the tile rows into the operand ring
            const int s = g % S;
            if (!wait_bounded_sleep(&opempty[s], ((uint32_t)(g / S) & 1u) ^ 1u, abort_flag, status)) {
              ok = false;
              break;
            }
            uint8_t* dst = smem + C::op + (size_t)s * C::OP_BYTES;
            mbar_expect_tx(&opfull[s], NA * A_BYTES + n_cols * 128);
            tma_3d(dst, &tmW0, &opfull[s], kb * BK, j * 128, e);
            if (MODE == kGemm1) tma_3d(dst + A_BYTES, &tmW1, &opfull[s], kb * BK, j * 128, e);
            load_tile_rows(dst + NA * A_BYTES, &tmX, &opfull[s], kb, t, n_cols);
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, (int)ok, 0);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (one lane)
    // The MMA's N covers the tile's rows up to its last real one (rounded up to 16): at decode
    // a tile holds a few real rows, and the columns past them would only cost tensor time.
    // One thread issues every MMA of the CTA, so its instructions per k-block set the pace at
    // decode (measured: about 10 cycles an instruction with all barriers already complete):
    // descriptors are low words plus constants, ring positions are counters, not divisions.
    int acc = 0, s = 0, x = 0, prev_xsb = 0;
    uint32_t acc_phase = 0, sph = 0, xph = 0;  // xph: phase bit of each tile-row slot
    bool ok = true, issued = false;
    const uint32_t op_lo = sw128_desc_lo(su32(smem + C::op));
    const uint32_t xr_lo = sw128_desc_lo(su32(smem + C::xr));
    for (int w = first; w < total && ok; w += active) {
      const int n_cols = tile_cols(P, tl[w / P.m_blocks], lane);
      const int xsb = x_slot_bytes(n_cols), nxs = FP8 ? x_slots<C>(xsb) : 1;
      if (xsb != prev_xsb) x = 0;  // the tile-row producer restarts the same way
      prev_xsb = xsb;
      const uint32_t idesc = idesc_bf16(128, n_cols);
      if (lane == 0) {
        if (!wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, status)) ok = false;
      }
      if (!__shfl_sync(0xffffffffu, (int)ok, 0)) break;
      if (lane == 0) {
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * NA * 128);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded(&opfull[s], sph, abort_flag, status) ||
              (FP8 && !wait_bounded(&xfull[x], (xph >> x) & 1u, abort_flag, status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t alo = op_lo + (uint32_t)s * (C::OP_BYTES >> 4);
          const uint32_t blo = FP8 ? xr_lo + (uint32_t)x * ((uint32_t)xsb >> 4)
                                   : alo + ((NA * A_BYTES) >> 4);
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk)
#pragma unroll
            for (int a = 0; a < NA; ++a)
              umma_bf16_lo(d + a * 128, alo + ((a * A_BYTES + kk * 32) >> 4), blo + kk * 2, idesc,
                           (kb | kk) != 0 ? 1u : 0u);
          umma_commit<1>(&opempty[s]);
          if (++s == S) {
            s = 0;
            sph ^= 1u;
          }
          if (FP8) {
            umma_commit<1>(&xempty[x]);
            xph ^= 1u << x;
            if (++x == nxs) x = 0;
          }
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
    for (int w = first; w < total; w += active) {
      const int t = tl[w / P.m_blocks], j = w % P.m_blocks;
      const int col = j * 128 + m;  // output column of this thread
      int sid4[4];                  // flat rows of tile rows c*32 + lane
#pragma unroll
      for (int c = 0; c < 4; ++c) sid4[c] = P.sid[t * 128 + c * 32 + lane];
      int ok = 1;
      if (lane == 0) ok = wait_bounded_sleep(&tfull[acc], acc_phase, abort_flag, status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (uint32_t)(acc * NA * 128) + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        const unsigned real = __ballot_sync(0xffffffffu, sid4[c] < P.n_rows);
        if (!real) continue;  // 32 padding rows: nothing to store
        if (MODE == kGemm1) {
#pragma unroll 1
          for (int hf = 0; hf < 2; ++hf) {  // 16 tile rows at a time (gate and up in registers)
            if (!((real >> (hf * 16)) & 0xFFFFu)) continue;
            uint32_t gv[16], uv[16];
            tmem_ld16(tb + c * 32 + hf * 16, gv);
            tmem_ld16(tb + 128 + c * 32 + hf * 16, uv);
            tmem_ld_wait();
            __nv_bfloat16* dst =
                (__nv_bfloat16*)P.out + (int64_t)(t * 128 + c * 32 + hf * 16) * P.N + col;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              if (!((real >> (hf * 16 + i)) & 1u) || col >= P.N) continue;
              const float g0 = __uint_as_float(gv[i]);
              dst[(int64_t)i * P.N] =
                  __float2bfloat16(g0 / (1.f + __expf(-g0)) * __uint_as_float(uv[i]));
            }
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
    if (warp == C::kXWarp) {
      // ---------------------------------------------------------- tile-row producer (FP8)
      // The tile rows of each k-block into the tile-row ring, as many k-blocks ahead of the
      // MMA as the item's slots allow; the MMA frees a slot with its commit. Both sides walk
      // the slots in the same order (the slot index wraps at the item's slot count and
      // restarts at 0 when the slot size changes) and keep one phase bit per slot. When the
      // slot size changes, every slot of the old layout is first released (the new slots
      // overlap the old ones).
      int x = 0, prev_nxs = 0, prev_xsb = 0;
      uint32_t xph = 0;
      bool ok = true;
      for (int w = first; w < total && ok; w += active) {
        const int t = tl[w / P.m_blocks];
        const int n_cols = tile_cols(P, t, lane);
        const int xsb = x_slot_bytes(n_cols), nxs = x_slots<C>(xsb);
        if (lane == 0) {
          if (xsb != prev_xsb) {
            for (int y = 0; y < prev_nxs && ok; ++y)
              ok = wait_bounded_sleep(&xempty[y], ((xph >> y) & 1u) ^ 1u, abort_flag, status);
            x = 0;
          }
          prev_xsb = xsb;
          prev_nxs = nxs;
          for (int kb = 0; kb < num_kb && ok; ++kb) {
            if (!wait_bounded_sleep(&xempty[x], ((xph >> x) & 1u) ^ 1u, abort_flag, status)) {
              ok = false;
              break;
            }
            xph ^= 1u << x;
            mbar_expect_tx(&xfull[x], n_cols * 128);
            load_tile_rows(smem + C::xr + (size_t)x * xsb, &tmX, &xfull[x], kb, t, n_cols);
            if (++x == nxs) x = 0;
          }
        }
        ok = __shfl_sync(0xffffffffu, (int)ok, 0);
      }
      __syncwarp();
    } else if ((warp - 6) % 4 != 3) {
      // ---------------------------------------------------------- FP8 converters
      // Converter cw turns rows cw*16 .. cw*16+15 of each raw 128 x 64 code block into the
      // 128-byte-swizzled bf16 K-major layout the MMA descriptor expects (16-byte chunk c of
      // row r at r*128 + ((c ^ (r & 7)) << 4)), scaled by the block's scale.
      const int cw = (warp - 6) - (warp - 6) / 4;
      constexpr int kRows = 128 / C::kCvtWarps;  // rows of each block this warp converts
      constexpr int kUnits = kRows * 4 / 32;     // 16-code units per lane and block
      static_assert(kRows * 4 % 32 == 0, "each lane converts whole units");
      int g = 0;
      bool ok = true;
      for (int w = first; w < total && ok; w += active) {
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
            okw = wait_bounded_sleep(&opempty[s], ((uint32_t)(g / S) & 1u) ^ 1u, abort_flag, status) &&
                  wait_bounded_sleep(&rawfull[r], (uint32_t)(g / R) & 1u, abort_flag, status);
          }
          okw = __shfl_sync(0xffffffffu, okw, 0);
          if (!okw) {
            ok = false;
            break;
          }
          const uint8_t* src = smem + C::raw + (size_t)r * C::RAWS_BYTES;
          uint8_t* dst = smem + C::op + (size_t)s * C::OP_BYTES;
          // all of this lane's 16-code units first (row u / 4, codes (u % 4) * 16 .. +15 of the
          // warp's rows), then the conversions and stores
          uint4 qv[NA][kUnits];
  #pragma unroll
          for (int a = 0; a < NA; ++a)
  #pragma unroll
            for (int i = 0; i < kUnits; ++i) {
              const int u = i * 32 + lane;
              const int row = cw * kRows + (u >> 2), h = u & 3;
              qv[a][i] = *reinterpret_cast<const uint4*>(src + a * RAW_BYTES + row * BK + h * 16);
            }
  #pragma unroll
          for (int a = 0; a < NA; ++a)
  #pragma unroll
            for (int i = 0; i < kUnits; ++i) {
              const int u = i * 32 + lane;
              const int row = cw * kRows + (u >> 2), h = u & 3;
              uint32_t v[8];
              e4m3x16_scaled_bf16(qv[a][i], sc[a], v);
              uint8_t* drow = dst + a * A_BYTES + row * 128;
              *reinterpret_cast<uint4*>(drow + (((2 * h) ^ (row & 7)) << 4)) =
                  make_uint4(v[0], v[1], v[2], v[3]);
              *reinterpret_cast<uint4*>(drow + (((2 * h + 1) ^ (row & 7)) << 4)) =
                  make_uint4(v[4], v[5], v[6], v[7]);
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

// The fixed-capacity layout with at most one 128-row tile per expert (capacity 128, the
// decode case: each tile holds an expert's few tokens, empty tiles are labelled -1).
bool dec_masked_applies(const moe_config_t& m, int capacity) {
  return m.dtype == MOE_BF16 && capacity == 128 && m.T / 128 <= dec::kMaxTiles;
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
    uint32_t box[2] = {BK, X_BOX};
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
    uint32_t box[2] = {BK, X_BOX};
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
