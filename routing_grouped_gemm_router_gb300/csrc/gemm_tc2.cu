// gemm_tc2.cu — the grouped expert GEMMs on CTA pairs (tcgen05.mma.cta_group::2, M=256).
//
// Functional contract ("Mixture-of-Experts Kernels: Routing, Permutation, and Grouped
// GEMM", §6, and the "fused-moe-kernel" skill card, Grouped GEMM Structure):
//   * every 128-row m-tile belongs to ONE expert, expert_ids[p / block_m];
//   * tiles at or past num_post_padded (read on the device) are never started;
//   * GEMM1 multiplies the token rows x[sorted_ids[p] / k], gathered into padded order by a
//     bandwidth-bound pass just before (gather.cu), and computes gate and up as the two
//     halves of one N=256 MMA, so the epilogue applies silu(gate) * up (§6 fused into the
//     GEMM1 epilogue, as the page's exercise suggests);
//   * GEMM2 reads act in padded order, multiplies by topk_w[r] and scatters each row to
//     y[r], r = sorted_ids[p]; padding rows are never stored.
//
// Design. A cluster of two CTAs on two SMs runs M=256 MMAs: each CTA holds 128 rows of A,
// half of the weight panel (B) and its own 128 rows of the fp32 accumulator in TMEM. The
// weight panel per SM is therefore half of a one-CTA tile's, which halves the shared-memory
// traffic per MMA and leaves room for 6 pipeline stages. The two m-tiles of a pair come from
// the SAME expert: an expert with an odd number of m-tiles ends with a pair whose second
// half is masked (its rows are loaded but never stored).
//
// Warp roles in each CTA: one producer warp issues the TMA copies of A and of the CTA's half
// of B into a 6-slot ring of 32 KB stages; both CTAs' copies complete on the LEADER's stage
// barrier (pair form of the copy), whose expect_tx counts the bytes of both. The leader's MMA
// warp (one lane) issues the pair's MMAs and commits with a multicast to both CTAs (stage
// free / accumulator ready); four epilogue warps per CTA drain their TMEM rows
// (double-buffered accumulators, 2 x 256 columns) and release the accumulator on the
// leader's barrier.
//
// An earlier version gathered A inside this kernel (TMA gather4, then cp.async producer
// warps); on GB300 the gather kept the MMA pipe half idle, while the separate gather pass
// costs one extra write and read of the routed rows (about 2.5 % of the Mixtral-shaped
// layer's bytes).
//
// Work order: expert by expert, each weight panel with all of that expert's m-tile pairs
// back to back (the skill card's L2 grouping at expert granularity), so the pairs running at
// the same time share a few panels. Each CTA builds the (expert run -> pair) table in shared
// memory from expert_ids at start-up. Every mbarrier wait is bounded (time-out: status
// kStatusTimeout, abort, copies in flight drained, TMEM freed).
#include "tc_ptx.cuh"

namespace moe {
namespace tc2 {

using namespace ptx;

__device__ int g_grouped_status;

enum Mode { kGemm1 = 0, kGemm2 = 1 };
constexpr int kStages = 6;
constexpr int kMaxTiles = 4096;  // 128-row m-tiles per launch (max_padded <= 524288)
constexpr int kMaxRuns = 1024;   // run boundaries in the m-tile sequence (<= 2E)
constexpr int kAccs = 2;                 // 256-column accumulators in TMEM
constexpr int kTmemCols = 256 * kAccs;
constexpr int A_BYTES = BM * 128;
constexpr int B_BYTES = 128 * 128;  // this CTA's half of an N=256 weight panel

struct Params {
  int n_rows;     // valid flat rows T*k; sorted_ids >= n_rows are padding
  int k;          // GEMM1: experts per token (row r reads token r / k)
  int N;          // output columns: I (GEMM1), H (GEMM2)
  int K;          // reduction length: H (GEMM1), I (GEMM2)
  int n_tiles;    // GEMM1: ceil(I / 128); GEMM2: ceil(H / 256)
  int block_m;
  const int32_t* sid;
  const int32_t* eid;
  const int32_t* npp;
  const float* topk_w;
  void* out;
  int64_t ld_out;
};

template <int MODE>
struct Roles {
  static constexpr int kProdWarps = 1;
  static constexpr int kMmaWarp = 1;
  static constexpr int kEpiWarp0 = 2;
  static constexpr int kThreads = 6 * 32;
  // The leader's full barrier of a stage completes on the leader's expect_tx arrival, which
  // counts the TMA bytes of BOTH CTAs: their copies all complete on this one barrier.
  static constexpr int kFullArrivals = 1;
  static constexpr uint32_t kPairTmaBytes = 2u * (A_BYTES + B_BYTES);
};

struct Layout {
  static constexpr size_t a = 0;
  static constexpr size_t b = a + (size_t)kStages * A_BYTES;
  static constexpr size_t bars = b + (size_t)kStages * B_BYTES;
  static constexpr size_t n_bars = 2 * kStages + 5;
  static constexpr size_t misc = bars + n_bars * 8;  // tmem slot, abort flag, run count
  static constexpr size_t bnd = misc + 16;
  static constexpr size_t run_first = bnd + kMaxRuns * 4;
  static constexpr size_t run_len = run_first + kMaxRuns * 4;
  static constexpr size_t run_e = run_len + kMaxRuns * 4;
  static constexpr size_t run_pref = run_e + kMaxRuns * 4;
  static constexpr size_t flags = run_pref + (kMaxRuns + 1) * 4;
  static constexpr size_t end = flags + kMaxTiles;
  static constexpr size_t bytes = 1024 + end;  // + alignment slack
};
static_assert(Layout::bytes <= 232448, "shared memory");

struct Table {
  const int* run_first;
  const int* run_len;
  const int* run_e;
  const int* run_pref;
  int nruns;
};

// Work item w -> (first m-tile of the pair, weight panel, expert, second half live).
__device__ __forceinline__ void item_of(int w, int n_tiles, const Table& tb, int& m0, int& n,
                                        int& e, bool& live1) {
  int lo = 0, hi = tb.nruns - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tb.run_pref[mid] * n_tiles <= w) lo = mid; else hi = mid - 1;
  }
  const int c = tb.run_pref[lo + 1] - tb.run_pref[lo];
  const int local = w - tb.run_pref[lo] * n_tiles;
  n = local / c;
  const int i = local - n * c;
  m0 = tb.run_first[lo] + 2 * i;
  live1 = 2 * i + 1 < tb.run_len[lo];
  e = tb.run_e[lo];
}

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Roles<MODE>::kThreads, 1)
    grouped_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB0,
                        const __grid_constant__ CUtensorMap tmB1, const Params P) {
  using R = Roles<MODE>;
  constexpr uint32_t IDESC = idesc_bf16(256, 256);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem + Layout::a;
  uint8_t* sB = smem + Layout::b;
  uint64_t* bars = (uint64_t*)(smem + Layout::bars);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = (uint32_t*)(smem + Layout::misc);
  volatile int* abort_flag = (volatile int*)(smem + Layout::misc + 4);
  int* nruns_sh = (int*)(smem + Layout::misc + 8);
  int* bnd = (int*)(smem + Layout::bnd);
  int* run_first = (int*)(smem + Layout::run_first);
  int* run_len = (int*)(smem + Layout::run_len);
  int* run_e = (int*)(smem + Layout::run_e);
  int* run_pref = (int*)(smem + Layout::run_pref);
  uint8_t* flags = smem + Layout::flags;
  int* status = &g_grouped_status;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], R::kFullArrivals);  // only the leader's are used
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 8);  // 4 epilogue warps of each CTA (used in the leader)
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_init_fence();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB0);
    if (MODE == kGemm1) prefetch_tmap(&tmB1);
  }
  if (warp == R::kMmaWarp) {
    tmem_alloc<2>(tmem_slot, kTmemCols);
    tmem_relinquish<2>();
    tc_fence_before();
  }

  // ---- run table: expert runs of the m-tile sequence, pairs per run, prefix of pairs
  const int num_m = min((*P.npp) / BM, kMaxTiles);
  for (int t = threadIdx.x; t < num_m; t += blockDim.x) {
    const int e = P.eid[(t * BM) / P.block_m];
    const int pe = t ? P.eid[((t - 1) * BM) / P.block_m] : -1;
    flags[t] = (t == 0 || e != pe) ? 1 : 0;
  }
  __syncthreads();
  if (warp == 0) {
    const unsigned lt = (1u << lane) - 1u;
    int nb = 0;
    for (int base = 0; base < num_m; base += 32) {
      const int t = base + lane;
      const bool f = t < num_m && flags[t];
      const unsigned msk = __ballot_sync(0xffffffffu, f);
      if (f && nb + __popc(msk & lt) < kMaxRuns) bnd[nb + __popc(msk & lt)] = t;
      nb += __popc(msk);
    }
    nb = min(nb, kMaxRuns);
    __syncwarp();
    int nr = 0, pairs = 0;
    for (int base = 0; base < nb; base += 32) {
      const int i = base + lane;
      int start = 0, len = 0, e = -1;
      if (i < nb) {
        start = bnd[i];
        len = (i + 1 < nb ? bnd[i + 1] : num_m) - start;
        e = P.eid[(start * BM) / P.block_m];
      }
      const bool ok = i < nb && e >= 0;
      const int c = ok ? (len + 1) / 2 : 0;
      int inc = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += o;
      }
      const unsigned msk = __ballot_sync(0xffffffffu, ok);
      if (ok) {
        const int idx = nr + __popc(msk & lt);
        run_first[idx] = start;
        run_len[idx] = len;
        run_e[idx] = e;
        run_pref[idx] = pairs + inc - c;
      }
      nr += __popc(msk);
      pairs += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) {
      run_pref[nr] = pairs;
      *nruns_sh = nr;
    }
  }
  __syncthreads();
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (threadIdx.x == 0) {
    // Both CTAs of the pair must see the same TMEM columns: the leader's MMAs write the
    // peer's rows at the leader's address. A mismatch stops the kernel with a status code.
    uint32_t peer_slot, other;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(peer_slot) : "r"(su32(tmem_slot)), "r"(rank ^ 1u));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(other) : "r"(peer_slot) : "memory");
    if (other != tmem_base) {
      *abort_flag = 1;
      atomicExch(status, kStatusPairTmem);
    }
  }
  __syncthreads();
  const Table tb{run_first, run_len, run_e, run_pref, *nruns_sh};
  const int total = tb.nruns > 0 ? tb.run_pref[tb.nruns] * P.n_tiles : 0;
  const int pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;
  const int num_kb = (P.K + BK - 1) / BK;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int g = 0;
      for (int w = pair; w < total; w += num_pairs) {
        int m0, n, e;
        bool live1;
        item_of(w, P.n_tiles, tb, m0, n, e, live1);
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb, ++g) {
          const int s = g % kStages;
          if (!wait_bounded(&empty[s], ((uint32_t)(g / kStages) & 1u) ^ 1u, abort_flag, status)) {
            ok = false;
            break;
          }
          const uint32_t fl = cluster_addr(&full[s], 0);
          if (leader) mbar_expect_tx(&full[s], R::kPairTmaBytes);
          tma_2d_pair(sA + s * A_BYTES, &tmA, fl, kb * BK, (m0 + (int)rank) * BM);
          if (MODE == kGemm1)  // leader: gate rows of panel n, peer: up rows
            tma_3d_pair(sB + s * B_BYTES, rank ? &tmB1 : &tmB0, fl, kb * BK, n * 128, e);
          else                 // leader: rows n*256 .. +127 of W2[e], peer: the next 128
            tma_3d_pair(sB + s * B_BYTES, &tmB0, fl, kb * BK, n * 256 + (int)rank * 128, e);
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp == R::kMmaWarp) {
    // ------------------------------------------------------------ leader: MMA issuer
    if (leader && lane == 0) {
      int g = 0, acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued = false;
      for (int w = pair; w < total && ok; w += num_pairs) {
        if (!wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, status)) break;
        tc_fence_after();
        if (*abort_flag) break;
        const uint32_t d = tmem_base + (uint32_t)(acc * 256);
        for (int kb = 0; kb < num_kb; ++kb, ++g) {
          const int s = g % kStages;
          if (!wait_bounded(&full[s], (uint32_t)(g / kStages) & 1u, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = su32(sA + s * A_BYTES);
          const uint32_t b = su32(sB + s * B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk)
            umma_bf16<2>(d, sw128_desc(a + kk * 32), sw128_desc(b + kk * 32), IDESC,
                         (kb | kk) != 0 ? 1u : 0u);
          umma_commit_pair(&empty[s], 0x3);
          issued = true;
        }
        if (!ok) break;
        umma_commit_pair(&tfull[acc], 0x3);
        if (++acc == kAccs) { acc = 0; acc_phase ^= 1u; }
      }
      if (issued) {  // every MMA of this thread finished before TMEM is freed
        umma_commit<2>(drain);
        wait_bounded(drain, 0, abort_flag, status);
      }
    }
    __syncwarp();
  } else if (warp >= R::kEpiWarp0) {
    // ------------------------------------------------------------ epilogue (4 warps)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int w = pair; w < total; w += num_pairs) {
      int m0, n, e;
      bool live1;
      item_of(w, P.n_tiles, tb, m0, n, e, live1);
      const bool live = leader || live1;
      int ok = 1;
      if (lane == 0) ok = wait_bounded(&tfull[acc], acc_phase, abort_flag, status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (uint32_t)(acc * 256) + ((uint32_t)(q * 32) << 16);
      const int p = (m0 + (int)rank) * BM + row;
      const int r = live ? P.sid[p] : P.n_rows;
      const bool valid = r < P.n_rows;
      if (MODE == kGemm1) {
        __nv_bfloat16* dst = (__nv_bfloat16*)P.out + (int64_t)p * P.ld_out + n * 128;
        const int col0 = n * 128;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t gv[32], uv[32];
          tmem_ld32(tbase + c * 32, gv);
          tmem_ld32(tbase + 128 + c * 32, uv);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              if (col0 + c * 32 + v * 8 < P.N) {
                uint32_t pk[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                  const float g0 = __uint_as_float(gv[v * 8 + 2 * h]);
                  const float g1 = __uint_as_float(gv[v * 8 + 2 * h + 1]);
                  const float a0 = g0 / (1.f + __expf(-g0)) * __uint_as_float(uv[v * 8 + 2 * h]);
                  const float a1 =
                      g1 / (1.f + __expf(-g1)) * __uint_as_float(uv[v * 8 + 2 * h + 1]);
                  pk[h] = pack_bf16(a0, a1);
                }
                *reinterpret_cast<uint4*>(dst + c * 32 + v * 8) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
              }
            }
          }
        }
      } else {
        const float wr = valid ? P.topk_w[r] : 0.f;
        __nv_bfloat16* dst = (__nv_bfloat16*)P.out + (int64_t)(valid ? r : 0) * P.ld_out + n * 256;
        const int col0 = n * 256;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t v32[32];
          tmem_ld32(tbase + c * 32, v32);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              if (col0 + c * 32 + v * 8 < P.N) {
                uint32_t pk[4];
#pragma unroll
                for (int h = 0; h < 4; ++h)
                  pk[h] = pack_bf16(wr * __uint_as_float(v32[v * 8 + 2 * h]),
                                    wr * __uint_as_float(v32[v * 8 + 2 * h + 1]));
                *reinterpret_cast<uint4*>(dst + c * 32 + v * 8) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(&tempty[acc]);
        else mbar_arrive_cta(&tempty[acc], 0);
      }
      if (++acc == kAccs) { acc = 0; acc_phase ^= 1u; }
    }
  }

  __syncthreads();
  if (*abort_flag) {  // let copies already in flight land before shared memory is released
    const uint64_t t0 = gtimer();
    while (gtimer() - t0 < 200000ull) {
    }
  }
  cluster_sync();  // no remote arrival still targets this CTA; both CTAs are done with TMEM
  if (warp == R::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc<2>(tmem_base, kTmemCols);
  }
}

template <int MODE>
static moe_status_t launch(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                           const Params& P, int max_items, cudaStream_t s) {
  auto kern = grouped_pair_kernel<MODE>;
  constexpr size_t smem = Layout::bytes;
  // Persistent grid: as many CTA pairs as can be resident at once (SMs that cannot be
  // paired inside a GPC stay idle rather than forming a second wave).
  static thread_local int configured_dev = -1, resident_pairs = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms() / 2));
    cfg.blockDim = dim3(Roles<MODE>::kThreads);
    cfg.dynamicSmemBytes = smem;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, (void*)kern, &cfg) != cudaSuccess ||
        clusters < 1) {
      cudaGetLastError();
      clusters = num_sms() / 2;
    }
    resident_pairs = std::min(clusters, num_sms() / 2);
    configured_dev = dev;
  }
  const int pairs = std::min(resident_pairs, max_items);
  if (pairs < 1) return MOE_OK;
  kern<<<2 * pairs, Roles<MODE>::kThreads, smem, s>>>(a, b0, b1, P);
  return last_launch_status();
}

// Upper bound on work items: pairs <= (m-tiles + experts that can own a run) / 2.
static int max_items_for(int max_padded, int n_rows, int E, int n_tiles) {
  const int tiles = max_padded / BM;
  return ((tiles + std::min(E, n_rows)) / 2 + 1) * n_tiles;
}

}  // namespace tc2

int grouped_status_read(int reset) {
  int v = 0;
  cudaMemcpyFromSymbol(&v, tc2::g_grouped_status, sizeof(int));
  if (reset) {
    int z = 0;
    cudaMemcpyToSymbol(tc2::g_grouped_status, &z, sizeof(int));
  }
  return v;
}

moe_status_t launch_gemm1_tc(const moe_config_t& c, const void* xs, const void* W13,
                             const int32_t* sid, const int32_t* eid, const int32_t* npp,
                             int block_m, int max_padded, void* act, cudaStream_t s) {
  using namespace tc2;
  if (max_padded / BM > kMaxTiles) return MOE_ERR_UNSUPPORTED;
  CUtensorMap mA, mG, mU;
  const uint64_t H = c.H, I = c.I, E = c.E;
  {
    uint64_t d[2] = {H, (uint64_t)max_padded}, st[1] = {H};
    uint32_t box[2] = {BK, BM};
    if (!make_map(&mA, xs, 2, d, st, box, false)) return MOE_ERR_CUDA;
  }
  {
    uint64_t d[3] = {H, I, E}, st[2] = {H, 2 * I * H};
    uint32_t box[3] = {BK, 128, 1};
    if (!make_map(&mG, W13, 3, d, st, box, true)) return MOE_ERR_CUDA;
    const __nv_bfloat16* up = (const __nv_bfloat16*)W13 + I * H;
    if (!make_map(&mU, up, 3, d, st, box, true)) return MOE_ERR_CUDA;
  }
  Params P{};
  P.n_rows = c.T * c.k;
  P.k = c.k;
  P.N = c.I;
  P.K = c.H;
  P.n_tiles = ceil_div(c.I, 128);
  P.block_m = block_m;
  P.sid = sid;
  P.eid = eid;
  P.npp = npp;
  P.out = act;
  P.ld_out = c.I;
  return launch<kGemm1>(mA, mG, mU, P, max_items_for(max_padded, P.n_rows, c.E, P.n_tiles), s);
}

moe_status_t launch_gemm2_tc(const moe_config_t& c, const void* act, const void* W2,
                             const int32_t* sid, const int32_t* eid, const int32_t* npp,
                             int block_m, int max_padded, const float* topk_w, void* y,
                             cudaStream_t s) {
  using namespace tc2;
  if (max_padded / BM > kMaxTiles) return MOE_ERR_UNSUPPORTED;
  CUtensorMap mA, mB;
  const uint64_t H = c.H, I = c.I, E = c.E;
  {
    uint64_t d[2] = {I, (uint64_t)max_padded}, st[1] = {I};
    uint32_t box[2] = {BK, BM};
    if (!make_map(&mA, act, 2, d, st, box, false)) return MOE_ERR_CUDA;
  }
  {
    uint64_t d[3] = {I, H, E}, st[2] = {I, H * I};
    uint32_t box[3] = {BK, 128, 1};
    if (!make_map(&mB, W2, 3, d, st, box, true)) return MOE_ERR_CUDA;
  }
  Params P{};
  P.n_rows = c.T * c.k;
  P.k = 1;
  P.N = c.H;
  P.K = c.I;
  P.n_tiles = ceil_div(c.H, 256);
  P.block_m = block_m;
  P.sid = sid;
  P.eid = eid;
  P.npp = npp;
  P.topk_w = topk_w;
  P.out = y;
  P.ld_out = c.H;
  return launch<kGemm2>(mA, mB, mB, P, max_items_for(max_padded, P.n_rows, c.E, P.n_tiles), s);
}

}  // namespace moe
