// gemm_tc.cu — the router GEMM on the tensor cores: logits[T, E] = x[T, H] . Wg[E, H]^T,
// bf16 inputs, fp32 accumulation in TMEM ("Mixture-of-Experts Kernels: Routing,
// Permutation, and Grouped GEMM", §3: logits = x @ w_gate.T, the scores every router starts
// from). E <= 256 fits one MMA N; with few 128-token tiles, E is split into BN-wide tiles so
// every SM gets one.
//
// One persistent CTA per SM (up to ceil(T/128) CTAs) with three warp roles: warp 0 issues
// TMA copies of x and Wg k-blocks into a shared-memory ring (4 to 10 stages, see stages_for),
// warp 1 (one lane) issues tcgen05.mma, warps 2-5 read the fp32 accumulator back
// (tcgen05.ld) and store the logits; two TMEM accumulators let the epilogue of one tile
// overlap the next tile's MMAs.
// Every mbarrier wait is bounded: on time-out the kernel records kStatusTimeout, stops
// issuing work, lets copies in flight land and frees its TMEM before returning.
#include "tc_ptx.cuh"

namespace moe {
namespace tc {

using namespace ptx;

__device__ int g_router_status;

constexpr int kThreads = 192;
// A ring stage holds kKbStage k-blocks of x and Wg (one full-barrier wait and one commit of
// the MMA thread per stage: with a narrow N the MMA thread's round trip per stage, not the
// bytes in flight, sets a tile's time), and the ring is as deep as about 200 KB of shared
// memory holds (2 stages at BN = 256, 5 at BN = 32).
constexpr int kKbStage = 2;
__host__ __device__ constexpr int stages_for(int bn) {
  const int s = (200 * 1024) / (kKbStage * (BM * 128 + bn * 128));
  return s < 2 ? 2 : (s > 8 ? 8 : s);
}

struct RouterParams {
  int T, E, H;
  int m_tiles, n_tiles;  // 128-token tiles x BN-expert tiles
  float* logits;
};

__host__ __device__ constexpr int tmem_cols_for(int bn) {
  return 2 * bn <= 32 ? 32 : 2 * bn <= 64 ? 64 : 2 * bn <= 128 ? 128 : 2 * bn <= 256 ? 256 : 512;
}
__host__ __device__ constexpr size_t router_smem_bytes(int bn) {
  return 1024 + (size_t)stages_for(bn) * kKbStage * (BM * 128 + (size_t)bn * 128) + 256;
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmW, const RouterParams P) {
  constexpr int A_BYTES = kKbStage * BM * 128;  // x: kKbStage k-blocks of 128 rows
  constexpr int B_BYTES = kKbStage * BN * 128;  // Wg: kKbStage k-blocks of BN rows
  constexpr int kStages = stages_for(BN);
  constexpr uint32_t TMEM_COLS = tmem_cols_for(BN);
  constexpr uint32_t IDESC = idesc_bf16(BM, BN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * A_BYTES;
  uint64_t* bars = (uint64_t*)(sB + kStages * B_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = (uint32_t*)(drain + 1);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  int* status = &g_router_status;

  pdl_trigger();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_init_fence();
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
  }
  if (warp == 1) {
    tmem_alloc<1>(tmem_slot, TMEM_COLS);
    tmem_relinquish<1>();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_kb = (P.H + kKbStage * BK - 1) / (kKbStage * BK);  // ring stages per tile
  pdl_wait();  // x, Wg and logits are touched only past this point

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    for (int w = blockIdx.x; w < P.m_tiles * P.n_tiles; w += gridDim.x) {
      const int m = w / P.n_tiles, n = w - m * P.n_tiles;
      for (int kb = 0; kb < num_kb; ++kb) {
        int ok = 1;
        if (lane == 0) ok = wait_bounded(&empty[stage], phase ^ 1u, abort_flag, status);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) goto producer_done;
        if (lane == 0) {  // a k-block past H reads zeros (TMA fill) and adds nothing
          mbar_expect_tx(&full[stage], A_BYTES + B_BYTES);
#pragma unroll
          for (int h = 0; h < kKbStage; ++h) {
            const int kx = (kb * kKbStage + h) * BK;
            tma_2d(sA + stage * A_BYTES + h * (BM * 128), &tmX, &full[stage], kx, m * BM);
            tma_2d(sB + stage * B_BYTES + h * (BN * 128), &tmW, &full[stage], kx, n * BN);
          }
        }
        __syncwarp();
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
  producer_done:;
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (one lane)
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true, issued = false;
      for (int w = blockIdx.x; w < P.m_tiles * P.n_tiles && ok; w += gridDim.x) {
        if (!wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, status)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded(&full[stage], phase, abort_flag, status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a = su32(sA + stage * A_BYTES);
          const uint32_t b = su32(sB + stage * B_BYTES);
#pragma unroll
          for (int h = 0; h < kKbStage; ++h)
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk)
              umma_bf16<1>(d, sw128_desc(a + h * (BM * 128) + kk * 32),
                           sw128_desc(b + h * (BN * 128) + kk * 32), IDESC,
                           (kb | h | kk) != 0 ? 1u : 0u);
          umma_commit<1>(&empty[stage]);
          issued = true;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit<1>(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (issued) {  // every MMA of this thread finished before TMEM is freed
        umma_commit<1>(drain);
        wait_bounded(drain, 0, abort_flag, status);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int w = blockIdx.x; w < P.m_tiles * P.n_tiles; w += gridDim.x) {
      const int m = w / P.n_tiles, n = w - m * P.n_tiles;
      int ok = 1;
      if (lane == 0) ok = wait_bounded(&tfull[acc], acc_phase, abort_flag, status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
      const int t = m * BM + q * 32 + lane;
      float* dst = P.logits + (int64_t)t * P.E + n * BN;
      const int ncols = P.E - n * BN;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t v32[32];
        tmem_ld32(tbase + c * 32, v32);
        tmem_ld_wait();
        if (t < P.T) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c * 32 + j < ncols) dst[c * 32 + j] = __uint_as_float(v32[j]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
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
    tmem_dealloc<1>(tmem_base, TMEM_COLS);
  }
}

template <int BN>
static moe_status_t launch_router(const CUtensorMap& mx, const CUtensorMap& mw,
                                  const RouterParams& P, cudaStream_t s) {
  auto kern = router_tc_kernel<BN>;
  const size_t smem = router_smem_bytes(BN);
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    configured_dev = dev;
  }
  const int grid = std::min(num_sms(), P.m_tiles * P.n_tiles);
  return launch_k(kern, dim3(grid), dim3(kThreads), smem, s, mx, mw, P);
}

}  // namespace tc

int router_status_read(int reset) {
  int v = 0;
  cudaMemcpyFromSymbol(&v, tc::g_router_status, sizeof(int));
  if (reset) {
    int z = 0;
    cudaMemcpyToSymbol(tc::g_router_status, &z, sizeof(int));
  }
  return v;
}

moe_status_t launch_router_tc(const moe_config_t& c, const void* x, const void* Wg,
                              float* logits, cudaStream_t s) {
  using namespace tc;
  // Expert tile BN (multiple of 32, <= 256): split E into narrower tiles while all tiles
  // still run in one wave. A tile's time is set by its K loop, not by BN, so a second wave
  // of narrower tiles costs a whole tile time more.
  const int m_tiles = ceil_div(c.T, BM);
  int bn = (c.E + 31) / 32 * 32;
  while (bn > 32) {
    const int half = (bn / 2 + 31) / 32 * 32;
    if (m_tiles * ceil_div(c.E, half) > num_sms()) break;
    bn = half;
  }
  if (bn > 256) return MOE_ERR_UNSUPPORTED;
  CUtensorMap mx, mw;
  const uint64_t H = c.H, E = c.E, T = c.T;
  {
    uint64_t d[2] = {H, T}, st[1] = {H};
    uint32_t box[2] = {BK, BM};
    if (!make_map(&mx, x, 2, d, st, box, false)) return MOE_ERR_CUDA;
  }
  {
    uint64_t d[2] = {H, E}, st[1] = {H};
    uint32_t box[2] = {BK, (uint32_t)bn};
    if (!make_map(&mw, Wg, 2, d, st, box, true)) return MOE_ERR_CUDA;
  }
  RouterParams P{c.T, c.E, c.H, m_tiles, ceil_div(c.E, bn), logits};
  switch (bn) {
    case 32: return launch_router<32>(mx, mw, P, s);
    case 64: return launch_router<64>(mx, mw, P, s);
    case 96: return launch_router<96>(mx, mw, P, s);
    case 128: return launch_router<128>(mx, mw, P, s);
    case 160: return launch_router<160>(mx, mw, P, s);
    case 192: return launch_router<192>(mx, mw, P, s);
    case 224: return launch_router<224>(mx, mw, P, s);
    case 256: return launch_router<256>(mx, mw, P, s);
    default: return MOE_ERR_UNSUPPORTED;
  }
}

}  // namespace moe
