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
// memory from expert_ids at start-up, after the programmatic-launch dependency wait; barrier
// set-up, TMEM allocation and the pair check come before it and overlap the previous
// kernel. Every mbarrier wait is bounded (time-out: status kStatusTimeout, abort, copies in
// flight drained, TMEM freed).
//
// A variant of the same kernel takes FP8 E4M3 weights with 128 x 128 block scales, turned
// into the bf16 operand by converter warps (see Roles below). Batches of at most 128 tokens
// run the decode kernel (gemm_dec.cu) instead.
#include "tc_ptx.cuh"

namespace moe {
namespace tc2 {

using namespace ptx;

__device__ int g_grouped_status;

enum Mode { kGemm1 = 0, kGemm2 = 1 };
constexpr int kMaxTiles = 4096;  // 128-row m-tiles per launch (max_padded <= 524288)
constexpr int kMaxRuns = 1024;   // run boundaries in the m-tile sequence (<= 2E)
constexpr int kAccs = 2;                 // 256-column accumulators in TMEM
constexpr int kTmemCols = 256 * kAccs;
constexpr int A_BYTES = BM * 128;
constexpr int B_BYTES = 128 * 128;  // this CTA's half of an N=256 weight panel
constexpr int RAW_BYTES = 128 * BK;  // the same half panel as FP8 codes (no swizzle)

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
  // FP8 weights: fp32 scale of each 128 x 128 block, [slots][grids][row blocks][k blocks]
  // (GEMM1: grid 0 = gate rows, grid 1 = up rows; GEMM2: one grid).
  const float* scale;
  int sc_rb, sc_kb;  // row blocks and k blocks of one grid
  int n_slots;       // expert slots the weights hold
};

// FP8 weights add kCvtGroups groups of kCvtWarps converter warps (6..) and a ring of raw
// FP8 tiles; the shared memory they take costs two pipeline stages. Group i owns the ring
// slots s with s % kCvtGroups == i (the slot count is a multiple of the group count), so
// every raw-tile barrier is waited on by one group, phase after phase: a parity wait must
// never start while the phase before the awaited one is still open, or it would pass at
// once. Each group then has several stage-times for a stage, and each converter warp
// arrives once on the leader's stage barrier (from the peer a cluster-scope release).
template <bool FP8>
struct Roles {
  static constexpr int kProdWarps = 1;
  static constexpr int kMmaWarp = 1;
  static constexpr int kEpiWarp0 = 2;
  static constexpr int kCvtWarp0 = 6;
  static constexpr int kCvtGroups = 2;
  static constexpr int kCvtWarps = 4;  // warps per group; each converts 128 / kCvtWarps rows
  static constexpr int kThreads = (FP8 ? 6 + kCvtWarps * kCvtGroups : 6) * 32;
  // The leader's full barrier of a stage completes on the leader's expect_tx arrival, which
  // counts the TMA bytes of BOTH CTAs: their copies all complete on this one barrier. With
  // FP8 weights the B halves are written by the converter warps of both CTAs instead: the
  // four converter warps of each CTA arrive once.
  static constexpr int kFullArrivals = FP8 ? 1 + 2 * kCvtWarps : 1;
  static constexpr uint32_t kPairTmaBytes = FP8 ? 2u * A_BYTES : 2u * (A_BYTES + B_BYTES);
};

template <bool FP8>
struct Layout {
  static constexpr int kStages = FP8 ? 4 : 6;
  static constexpr size_t a = 0;
  static constexpr size_t b = a + (size_t)kStages * A_BYTES;
  static constexpr size_t raw = b + (size_t)kStages * B_BYTES;
  static constexpr size_t bars = raw + (FP8 ? (size_t)kStages * RAW_BYTES : 0);
  static constexpr size_t n_bars = 3 * kStages + 5;  // full, empty, raw full; tfull, tempty, drain
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
static_assert(Layout<false>::bytes <= 232448, "shared memory");
static_assert(Layout<true>::bytes <= 232448, "shared memory");
static_assert(Layout<true>::kStages % Roles<true>::kCvtGroups == 0,
              "each converter group must own whole ring slots");

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

template <int MODE, bool FP8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Roles<FP8>::kThreads, 1)
    grouped_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB0,
                        const __grid_constant__ CUtensorMap tmB1, const Params P) {
  using R = Roles<FP8>;
  using L = Layout<FP8>;
  constexpr int kStages = L::kStages;
  constexpr uint32_t IDESC = idesc_bf16(256, 256);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem + L::a;
  uint8_t* sB = smem + L::b;
  uint8_t* sRaw = smem + L::raw;
  uint64_t* bars = (uint64_t*)(smem + L::bars);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* rawfull = bars + 2 * kStages;
  uint64_t* tfull = bars + 3 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = (uint32_t*)(smem + L::misc);
  volatile int* abort_flag = (volatile int*)(smem + L::misc + 4);
  int* nruns_sh = (int*)(smem + L::misc + 8);
  int* bnd = (int*)(smem + L::bnd);
  int* run_first = (int*)(smem + L::run_first);
  int* run_len = (int*)(smem + L::run_len);
  int* run_e = (int*)(smem + L::run_e);
  int* run_pref = (int*)(smem + L::run_pref);
  uint8_t* flags = smem + L::flags;
  int* status = &g_grouped_status;

  pdl_trigger();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], R::kFullArrivals);  // only the leader's are used
      mbar_init(&empty[s], 1);
      mbar_init(&rawfull[s], 1);              // FP8: this CTA's raw weight tile landed
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

  // Everything up to griddepcontrol.wait touches shared and tensor memory only, so it
  // overlaps the previous kernel's tail.
  cluster_sync();  // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  bool pair_tmem_mismatch = false;
  if (threadIdx.x == 0) {
    // Both CTAs of the pair must see the same TMEM columns: the leader's MMAs write the
    // peer's rows at the leader's address. A mismatch stops the kernel with a status code.
    uint32_t peer_slot, other;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(peer_slot) : "r"(su32(tmem_slot)), "r"(rank ^ 1u));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(other) : "r"(peer_slot) : "memory");
    if (other != tmem_base) {
      *abort_flag = 1;
      pair_tmem_mismatch = true;
    }
  }

  pdl_wait();  // global memory is touched only past this point
  if (pair_tmem_mismatch) atomicExch(status, kStatusPairTmem);
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
          // An expert's odd last m-tile runs in a pair whose peer half is masked (its rows are
          // never stored): the peer copies no A tile then, and its MMA rows read whatever the
          // slot held. That is one 16 KB tile a stage less through L2 on every such item
          // (all of them when experts hold one tile, as in DeepSeek-V3-shaped layers).
          if (leader)
            mbar_expect_tx(&full[s], live1 ? R::kPairTmaBytes : R::kPairTmaBytes - A_BYTES);
          if (leader || live1)
            tma_2d_pair(sA + s * A_BYTES, &tmA, fl, kb * BK, (m0 + (int)rank) * BM);
          // leader: gate rows of panel n (GEMM1) / rows n*256 .. +127 of W2[e] (GEMM2);
          // peer: the up rows / the next 128 rows
          const CUtensorMap* tb_map = (MODE == kGemm1 && rank) ? &tmB1 : &tmB0;
          const int brow = MODE == kGemm1 ? n * 128 : n * 256 + (int)rank * 128;
          if (FP8) {  // raw codes to this CTA's ring; the converter warps write sB
            mbar_expect_tx(&rawfull[s], RAW_BYTES);
            tma_3d(sRaw + s * RAW_BYTES, tb_map, &rawfull[s], kb * BK, brow, e);
          } else {
            tma_3d_pair(sB + s * B_BYTES, tb_map, fl, kb * BK, brow, e);
          }
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
  } else if (warp >= R::kEpiWarp0 && warp < R::kEpiWarp0 + 4) {
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
  } else if (FP8 && warp >= R::kCvtWarp0) {
    // ------------------------------------------------------------ FP8 converters (4 warps)
    // Warp cw turns rows cw*32 .. cw*32+31 of this CTA's raw 128 x 64 code tile into the
    // 128-byte-swizzled bf16 K-major layout the MMA descriptor expects (16-byte chunk c of
    // row r at r*128 + ((c ^ (r & 7)) << 4)), scaled by the tile's block scale; then makes
    // the writes visible to the tensor cores and arrives on the leader's stage barrier.
    const int cw = (warp - R::kCvtWarp0) % R::kCvtWarps;
    const int grp = (warp - R::kCvtWarp0) / R::kCvtWarps;
    const int grid = MODE == kGemm1 ? (int)rank : 0;
    int g = 0;
    for (int w = pair; w < total; w += num_pairs) {
      int m0, n, e;
      bool live1;
      item_of(w, P.n_tiles, tb, m0, n, e, live1);
      const int rb = MODE == kGemm1 ? n : 2 * n + (int)rank;
      const bool sc_ok = e >= 0 && e < P.n_slots && rb < P.sc_rb;
      const float* srow =
          P.scale + (((int64_t)e * (MODE == kGemm1 ? 2 : 1) + grid) * P.sc_rb + rb) * P.sc_kb;
      bool ok = true;
      for (int kb = 0; kb < num_kb; ++kb, ++g) {
        if ((g % kStages) % R::kCvtGroups != grp) continue;  // the group's own slots
        const int s = g % kStages;
        const float sc = sc_ok ? __ldg(srow + (kb >> 1)) : 0.f;  // in flight during the wait
        int okw = 1;
        if (lane == 0) okw = wait_bounded(&rawfull[s], (uint32_t)(g / kStages) & 1u, abort_flag, status);
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) {
          ok = false;
          break;
        }
        // A power-of-two scale below 2^8 (or 0) times 2^120 is an exact bf16: one packed
        // bf16 multiply per two weights, exact. Any other scale: fp32 products.
        const float scb = sc * 0x1p120f;
        const bool fast = (__float_as_uint(sc) & 0x807FFFFFu) == 0 && sc < 0x1p8f;
        const uint32_t sc2 = (__float_as_uint(scb) >> 16) * 0x10001u;
        const uint8_t* src = sRaw + s * RAW_BYTES;
        uint8_t* dst = sB + s * B_BYTES;
#pragma unroll
        for (int j = 0; j < 16 / R::kCvtWarps; ++j) {
          // 16-code unit u: row u/4, codes (u%4)*16 .. +15; 512 units per stage
          const int u = cw * (512 / R::kCvtWarps) + j * 32 + lane;
          const int r = u >> 2, h = u & 3;
          const uint4 q = *reinterpret_cast<const uint4*>(src + u * 16);
          uint32_t v[8];
          e4m3x4_to_bf16x4_lowexp(q.x, v[0], v[1]);
          e4m3x4_to_bf16x4_lowexp(q.y, v[2], v[3]);
          e4m3x4_to_bf16x4_lowexp(q.z, v[4], v[5]);
          e4m3x4_to_bf16x4_lowexp(q.w, v[6], v[7]);
          if (fast) {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = bf16x2_mul(v[i], sc2);
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = bf16x2_lowexp_scale_f32(v[i], sc);
          }
          uint8_t* drow = dst + r * 128;
          *reinterpret_cast<uint4*>(drow + (((2 * h) ^ (r & 7)) << 4)) = make_uint4(v[0], v[1], v[2], v[3]);
          *reinterpret_cast<uint4*>(drow + (((2 * h + 1) ^ (r & 7)) << 4)) = make_uint4(v[4], v[5], v[6], v[7]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(&full[s]);
          else mbar_arrive_cta(&full[s], 0);
        }
      }
      if (!ok) break;
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

template <int MODE, bool FP8>
static moe_status_t launch(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                           const Params& P, int max_items, cudaStream_t s) {
  auto kern = grouped_pair_kernel<MODE, FP8>;
  constexpr size_t smem = Layout<FP8>::bytes;
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
    cfg.blockDim = dim3(Roles<FP8>::kThreads);
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
  return launch_k(kern, dim3(2 * pairs), dim3(Roles<FP8>::kThreads), smem, s, a, b0, b1, P);
}

// Upper bound on work items: pairs <= (m-tiles + experts that can own a run) / 2.
static int max_items_for(int max_padded, int n_rows, int E, int n_tiles) {
  const int tiles = max_padded / BM;
  return ((tiles + std::min(E, n_rows)) / 2 + 1) * n_tiles;
}

// Failure-path self-test: one CTA allocates tensor memory, then two warps wait, through the
// same bounded wait as the GEMM pipelines, on mbarriers that nothing ever arrives on. The
// first wait gives up after the pipeline time limit, raises the CTA's abort flag and records
// kStatusTimeout; the second sees the flag and gives up too; the CTA frees its tensor
// memory and returns.
__global__ void __launch_bounds__(64, 1) selftest_wait_kernel() {
  pdl_wait();
  pdl_trigger();
  __shared__ uint64_t bars[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_sh;
  volatile int* abort_flag = &abort_sh;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 1) {
    tmem_alloc<1>(&tmem_slot, 32);
    tmem_relinquish<1>();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  if (lane == 0) wait_bounded(&bars[warp], 0, abort_flag, &g_grouped_status);
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<1>(tmem_slot, 32);
  }
}

}  // namespace tc2

moe_status_t launch_selftest_wait(cudaStream_t s) {
  return launch_k(tc2::selftest_wait_kernel, dim3(1), dim3(64), 0, s);
}

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
  const bool fp8 = c.weight_format == MOE_WEIGHTS_FP8_E4M3_B128;
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
    const uint8_t* up = (const uint8_t*)W13 + I * H * (fp8 ? 1 : 2);
    if (!make_map(&mG, W13, 3, d, st, box, true, fp8)) return MOE_ERR_CUDA;
    if (!make_map(&mU, up, 3, d, st, box, true, fp8)) return MOE_ERR_CUDA;
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
  P.scale = c.w13_scale;
  P.sc_rb = ceil_div(c.I, 128);
  P.sc_kb = ceil_div(c.H, 128);
  P.n_slots = c.E;
  const int items = max_items_for(max_padded, P.n_rows, c.E, P.n_tiles);
  return fp8 ? launch<kGemm1, true>(mA, mG, mU, P, items, s)
             : launch<kGemm1, false>(mA, mG, mU, P, items, s);
}

moe_status_t launch_gemm2_tc(const moe_config_t& c, const void* act, const void* W2,
                             const int32_t* sid, const int32_t* eid, const int32_t* npp,
                             int block_m, int max_padded, const float* topk_w, void* y,
                             cudaStream_t s) {
  using namespace tc2;
  if (max_padded / BM > kMaxTiles) return MOE_ERR_UNSUPPORTED;
  const bool fp8 = c.weight_format == MOE_WEIGHTS_FP8_E4M3_B128;
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
    if (!make_map(&mB, W2, 3, d, st, box, true, fp8)) return MOE_ERR_CUDA;
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
  P.scale = c.w2_scale;
  P.sc_rb = ceil_div(c.H, 128);
  P.sc_kb = ceil_div(c.I, 128);
  P.n_slots = c.E;
  const int items = max_items_for(max_padded, P.n_rows, c.E, P.n_tiles);
  return fp8 ? launch<kGemm2, true>(mA, mB, mB, P, items, s)
             : launch<kGemm2, false>(mA, mB, mB, P, items, s);
}

}  // namespace moe
