// gemm_tc.cu — grouped expert GEMMs and the router GEMM on the 5th-generation tensor cores
// (tcgen05, sm_103a): TMA copies into 128-byte-swizzled shared memory, MMAs issued by one
// thread into fp32 accumulators in tensor memory (TMEM), epilogues read back with
// tcgen05.ld.
//
// Functional contract ("Mixture-of-Experts Kernels: Routing, Permutation, and Grouped
// GEMM", §6, and the "fused-moe-kernel" skill card, Grouped GEMM Structure):
//   * every 128-row M tile belongs to ONE expert, expert_ids[p / block_m];
//   * tiles at or past num_post_padded (read on the device) are never started;
//   * GEMM1 gathers the token rows x[sorted_ids[p] / k] itself (no permuted copy of x) and
//     computes gate and up as the two halves of one N=256 MMA, so the epilogue applies
//     silu(gate) * up (§6 fused into the GEMM1 epilogue, as the page's exercise suggests);
//   * GEMM2 reads act in padded order with plain 2-D TMA, multiplies by topk_w[r] and
//     scatters each row to y[r], r = sorted_ids[p]; padding rows are never stored.
//
// Design (GB300-first, not the page's Triton kernel): one persistent CTA per SM walks a
// static tile sequence (expert-major: every m-tile of an expert per weight panel, the skill
// card's L2 grouping taken to expert granularity) with three warp roles: producer warps fill a ring of STAGES shared-memory
// stages, one MMA warp (one lane) issues tcgen05.mma into one of two TMEM accumulators, and
// four epilogue warps drain the other accumulator while the next tile accumulates.
// Producers: GEMM2 and the router use one warp issuing 2-D/3-D TMA tiles. GEMM1 uses eight
// warps (two per ring slot) that gather A with 16-byte cp.async (each warp instruction moves
// four whole 128-byte token rows, written straight into the swizzled layout the MMA reads)
// while one lane per slot moves the weight panels by TMA. (A TMA gather4 producer moves only four rows per instruction;
// on GB300 it capped GEMM1 near 470 TFLOP/s, against ~1300 TFLOP/s with contiguous tiles.)
// Every mbarrier wait is bounded: on time-out the kernel records kStatusTimeout, stops
// issuing work, lets copies in flight land and frees its TMEM before returning.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128;          // MMA M (TMEM lanes)
constexpr int BK = 64;           // 64 bf16 = 128 bytes = one swizzle row
constexpr int UMMA_K = 16;       // K of one kind::f16 MMA
constexpr int kGroupM = 8;       // m-tiles that share one weight panel in the raster
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait

enum Mode { kGemm1 = 0, kGemm2 = 1, kRouter = 2 };

__device__ int g_tc_status;

// --------------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t su32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of parity `parity`. Returns false (and raises the CTA's
// abort flag and the device status) when it runs out of time or another role aborted.
__device__ __noinline__ bool wait_slow(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  const uint64_t t0 = gtimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(b, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (gtimer() - t0 > kTimeoutNs) {
        *abort_flag = 1;
        atomicExch(&g_tc_status, kStatusTimeout);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool wait_bounded(uint64_t* b, uint32_t parity,
                                             volatile int* abort_flag) {
  if (mbar_try_wait(b, parity)) return true;
  return wait_slow(b, parity, abort_flag);
}

__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* tm, uint64_t* bar, int c0,
                                       int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(su32(dst)),
      "l"((uint64_t)tm), "r"(c0), "r"(c1), "r"(su32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* tm, uint64_t* bar, int c0,
                                       int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(su32(dst)),
      "l"((uint64_t)tm), "r"(c0), "r"(c1), "r"(c2), "r"(su32(bar))
      : "memory");
}
// 16-byte global -> shared copy that bypasses L1; src_bytes = 0 fills the 16 bytes with zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global.L2::128B [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Orders this thread's generic-proxy shared-memory writes before later async-proxy reads
// (the tensor core reads its operands through the async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)tm) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   su32(slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The mbarrier completes one arrival when every MMA issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          su32(bar))
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of 128 bytes,
// 8-row swizzle atoms 1024 bytes apart (stride byte offset). Tile bases are 1024-aligned;
// stepping K by 16 elements inside the atom advances the start address by 32 bytes.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);      // bits 0-13: start address / 16
  d |= (uint64_t)1 << 16;                        // bits 16-29: leading byte offset (unused)
  d |= (uint64_t)(1024 >> 4) << 32;              // bits 32-45: stride byte offset / 16
  d |= (uint64_t)1 << 46;                        // bits 46-47: descriptor version 1
  d |= (uint64_t)2 << 61;                        // bits 61-63: 128-byte swizzle
  return d;
}
// Instruction descriptor for kind::f16: fp32 accumulator, bf16 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// --------------------------------------------------------------------- parameters
struct Params {
  int n_rows;      // GEMM1/GEMM2: T*k (valid flat rows); router: T
  int k;           // GEMM1: experts per token (row r reads token r / k)
  int N;           // output columns: I (GEMM1), H (GEMM2), E (router)
  int K;           // reduction length: H (GEMM1, router), I (GEMM2)
  int n_tiles;     // output column tiles
  int m_tiles;     // router: ceil(T / 128); GEMM1/GEMM2: 0 = read num_post_padded
  int block_m;
  const int32_t* sid;
  const int32_t* eid;
  const int32_t* npp;
  const float* topk_w;
  void* out;
  int64_t ld_out;  // elements per output row
  const void* x;   // GEMM1: token rows [T, K] bf16, gathered with cp.async
};

// Warp roles: producers, then one MMA warp, then four epilogue warps.
template <int MODE>
struct Roles {
  static constexpr int kProdWarps = MODE == kGemm1 ? 8 : 1;   // GEMM1: two per ring slot
  static constexpr int kMmaWarp = kProdWarps;
  static constexpr int kThreads = (kProdWarps + 5) * 32;
  // GEMM1: the weight TMA's expect_tx arrival plus one arrival per producer warp of the slot
  static constexpr int kFullArrivals = MODE == kGemm1 ? 3 : 1;
};

template <int MODE>
struct Cfg;
template <>
struct Cfg<kGemm1> {  // N=256: gate cols 0..127, up cols 128..255 -> 128 output columns
  static constexpr int BN = 256, OUT_COLS = 128, STAGES = 4;
};
template <>
struct Cfg<kGemm2> {
  static constexpr int BN = 256, OUT_COLS = 256, STAGES = 4;
};

__host__ __device__ constexpr int tmem_cols_for(int bn) {
  return 2 * bn <= 32 ? 32 : 2 * bn <= 64 ? 64 : 2 * bn <= 128 ? 128 : 2 * bn <= 256 ? 256 : 512;
}
__host__ __device__ constexpr size_t smem_bytes_for(int bn, int stages) {
  return 1024 + (size_t)stages * (BM * 128 + (size_t)bn * 128) + 256;
}

// Expert-major raster for the grouped GEMMs: work item w visits, expert by expert, each
// weight panel n with ALL of that expert's m-tiles back to back, so the CTAs running at the
// same time share a few weight panels (one HBM read each) and the expert's token rows stay
// in L2 across its panels. w / n_tiles always lands inside the owning expert's run of
// m-tiles, so its expert id is expert_ids[w / n_tiles]; the run [lo, hi) is found by binary
// search (each expert's tiles are contiguous). Returns the expert (-1: skip the tile).
__device__ __forceinline__ int expert_tile_of(int w, int num_m, int n_tiles, const int32_t* eid,
                                              int block_m, int& m, int& n) {
  const int v = w / n_tiles;
  const int e = eid[(v * BM) / block_m];
  if (e < 0) {
    m = v;
    n = w - v * n_tiles;
    return e;
  }
  int lo = 0, hi = v;  // first tile of the run: smallest t <= v with eid == e
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (eid[(mid * BM) / block_m] == e) hi = mid; else lo = mid + 1;
  }
  const int first = lo;
  lo = v + 1;
  hi = num_m;  // one past the last tile of the run
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (eid[(mid * BM) / block_m] == e) lo = mid + 1; else hi = mid;
  }
  const int mt = lo - first;
  const int local = w - first * n_tiles;
  m = first + local % mt;
  n = local / mt;
  return e;
}

// Router raster: GROUP_M m-tiles per panel (only one panel, n_tiles = 1, in practice).
__device__ __forceinline__ void tile_of(int w, int num_m, int n_tiles, int& m, int& n) {
  const int per_group = kGroupM * n_tiles;
  const int g = w / per_group;
  const int first_m = g * kGroupM;
  const int gm = min(num_m - first_m, kGroupM);
  const int r = w - g * per_group;
  m = first_m + r % gm;
  n = r / gm;
}

// --------------------------------------------------------------------- the kernel
template <int MODE, int BN, int STAGES>
__global__ void __launch_bounds__(Roles<MODE>::kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmB2, const Params P) {
  constexpr int A_BYTES = BM * 128;
  constexpr int B_BYTES = BN * 128;
  constexpr uint32_t TMEM_COLS = tmem_cols_for(BN);
  constexpr uint32_t IDESC = idesc_bf16(BM, BN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint64_t* bars = (uint64_t*)(sB + STAGES * B_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = (uint32_t*)(drain + 1);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);

  constexpr int kProdWarps = Roles<MODE>::kProdWarps;
  constexpr int kMmaWarp = Roles<MODE>::kMmaWarp;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], Roles<MODE>::kFullArrivals);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (MODE != kGemm1) prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (MODE == kGemm1) prefetch_tmap(&tmB2);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int num_m = MODE == kRouter ? P.m_tiles : (*P.npp) / BM;
  const int total = num_m * P.n_tiles;
  const int num_kb = (P.K + BK - 1) / BK;

  if (MODE == kGemm1 && warp < kProdWarps) {
    // ------------------------------------------------------------ GEMM1 producers
    // Producer warps 2s and 2s+1 own ring slot s and fill every STAGES-th k-block of this
    // CTA's tile sequence. Warp 2s's lane 0 issues the weight TMA (expect_tx arrival). Each
    // warp copies 64 of the tile's 128 token rows: lane l moves 16-byte chunk l%8 of rows
    // base + 4*i + l/8 (i = 0..15), so every warp instruction moves four whole 128-byte
    // rows. Padding rows (sentinel ids) are zero-filled without reading memory. The warp
    // waits for its own copies, fences the async proxy, and lane 0 arrives. Each slot's
    // stage loads independently of the others, so STAGES stages are in flight.
    static_assert(MODE != kGemm1 || kProdWarps == 2 * STAGES, "two producer warps per slot");
    const int slot = warp >> 1;
    const int rbase = (warp & 1) * 64;
    const int sub = lane & 7, rsub = lane >> 3;
    const char* xb = (const char*)P.x;
    const uint32_t a = su32(sA + slot * A_BYTES);
    uint8_t* b = sB + slot * B_BYTES;
    int g = 0;  // k-blocks of this CTA's tile sequence before the current tile
    bool ok = true;
    for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
      int m, n;
      const int e = expert_tile_of(w, num_m, P.n_tiles, P.eid, P.block_m, m, n);
      if (e < 0) continue;
      const int kb0 = ((slot - g) % STAGES + STAGES) % STAGES;
      if (kb0 < num_kb) {
        int tok[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = P.sid[m * BM + rbase + 4 * i + rsub];
          tok[i] = r < P.n_rows ? r / P.k : -1;
        }
        for (int kb = kb0; kb < num_kb; kb += STAGES) {
          const uint32_t use = (uint32_t)((g + kb) / STAGES);
          int okw = 1;
          if (lane == 0) okw = wait_bounded(&empty[slot], (use & 1u) ^ 1u, abort_flag);
          okw = __shfl_sync(0xffffffffu, okw, 0);
          if (!okw) { ok = false; break; }
          if (lane == 0 && rbase == 0) {
            mbar_expect_tx(&full[slot], B_BYTES);
            tma_3d(b, &tmB, &full[slot], kb * BK, n * 128, e);
            tma_3d(b + 128 * 128, &tmB2, &full[slot], kb * BK, n * 128, e);
          }
          const int col = kb * BK + sub * 8;
          const bool col_ok = col < P.K;
          const int64_t coff = (int64_t)(col_ok ? col : 0) * 2;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int row = rbase + 4 * i + rsub;
            const bool live = col_ok && tok[i] >= 0;
            cp_async16(a + row * 128 + ((sub ^ (row & 7)) << 4),
                       xb + (int64_t)(tok[i] >= 0 ? tok[i] : 0) * P.K * 2 + coff,
                       live ? 16u : 0u);
          }
          cp_async_commit();
          cp_async_wait<0>();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[slot]);
        }
      }
      g += num_kb;
    }
    cp_async_wait<0>();
  } else if (MODE != kGemm1 && warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    for (int w = blockIdx.x; w < total; w += gridDim.x) {
      int m, n, e = 0;
      if (MODE == kRouter) tile_of(w, num_m, P.n_tiles, m, n);
      else e = expert_tile_of(w, num_m, P.n_tiles, P.eid, P.block_m, m, n);
      if (e < 0) continue;
      for (int kb = 0; kb < num_kb; ++kb) {
        int ok = 1;
        if (lane == 0) ok = wait_bounded(&empty[stage], phase ^ 1u, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) goto producer_done;
        if (lane == 0) {
          uint8_t* a = sA + stage * A_BYTES;
          uint8_t* b = sB + stage * B_BYTES;
          mbar_expect_tx(&full[stage], A_BYTES + B_BYTES);
          tma_2d(a, &tmA, &full[stage], kb * BK, m * BM);
          if (MODE == kGemm2)
            tma_3d(b, &tmB, &full[stage], kb * BK, n * BN, e);
          else
            tma_2d(b, &tmB, &full[stage], kb * BK, 0);
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
  producer_done:;
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer (one lane)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, issued = false;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
        int m, n, e = 0;
        if (MODE == kRouter) tile_of(w, num_m, P.n_tiles, m, n);
        else e = expert_tile_of(w, num_m, P.n_tiles, P.eid, P.block_m, m, n);
        if (e < 0) continue;
        if (!wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded(&full[stage], phase, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a = su32(sA + stage * A_BYTES);
          const uint32_t b = su32(sB + stage * B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk)
            umma_bf16(d, sw128_desc(a + kk * 32), sw128_desc(b + kk * 32), IDESC,
                      (kb | kk) != 0 ? 1u : 0u);
          umma_commit(&empty[stage]);
          issued = true;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // Wait until every MMA issued by this thread has finished before TMEM is freed.
      if (issued) {
        umma_commit(drain);
        wait_bounded(drain, 0, abort_flag);
      }
    }
    __syncwarp();
  } else if (warp > kMmaWarp) {
    // ------------------------------------------------------------ epilogue (4 warps)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int w = blockIdx.x; w < total; w += gridDim.x) {
      int m, n, e = 0;
      if (MODE == kRouter) tile_of(w, num_m, P.n_tiles, m, n);
      else e = expert_tile_of(w, num_m, P.n_tiles, P.eid, P.block_m, m, n);
      if (e < 0) continue;
      int ok = 1;
      if (lane == 0) ok = wait_bounded(&tfull[acc], acc_phase, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
      const int p = m * BM + row;
      if (MODE == kGemm1) {
        const int r = P.sid[p];
        const bool valid = r < P.n_rows;
        __nv_bfloat16* dst = (__nv_bfloat16*)P.out + (int64_t)p * P.ld_out + n * 128;
        const int col0 = n * 128;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(tbase + c * 32, g);
          tmem_ld32(tbase + 128 + c * 32, u);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              if (col0 + c * 32 + v * 8 < P.N) {
                uint32_t pk[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                  float g0 = __uint_as_float(g[v * 8 + 2 * h]);
                  float g1 = __uint_as_float(g[v * 8 + 2 * h + 1]);
                  float a0 = g0 / (1.f + __expf(-g0)) * __uint_as_float(u[v * 8 + 2 * h]);
                  float a1 = g1 / (1.f + __expf(-g1)) * __uint_as_float(u[v * 8 + 2 * h + 1]);
                  pk[h] = pack_bf16(a0, a1);
                }
                *reinterpret_cast<uint4*>(dst + c * 32 + v * 8) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
              }
            }
          }
        }
      } else if (MODE == kGemm2) {
        const int r = P.sid[p];
        const bool valid = r < P.n_rows;
        const float wr = valid ? P.topk_w[r] : 0.f;
        __nv_bfloat16* dst =
            (__nv_bfloat16*)P.out + (int64_t)(valid ? r : 0) * P.ld_out + n * BN;
        const int col0 = n * BN;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
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
      } else {
        const bool valid = p < P.n_rows;
        float* dst = (float*)P.out + (int64_t)p * P.ld_out;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v32[32];
          tmem_ld32(tbase + c * 32, v32);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c * 32 + j < P.N) dst[c * 32 + j] = __uint_as_float(v32[j]);
          }
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
  if (*abort_flag) {
    // Let copies already in flight land before the shared memory is released.
    const uint64_t t0 = gtimer();
    while (gtimer() - t0 < 200000ull) {
    }
  }
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// Router: BN = E rounded up to 32 (N <= 256), 4 stages.
template <int BN>
struct RouterCfg {
  static constexpr int STAGES = 4;
};

// --------------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  });
  return fn;
}

// bf16 tensor map, 128-byte swizzle. dims/strides in elements (dim 0 innermost).
static bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides_elems, const uint32_t* box, bool weights) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[3], gstr[2];
  cuuint32_t bdim[3], estr[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) gstr[i] = strides_elems[i] * 2;
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), gdim, gstr,
                  bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  weights ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int MODE, int BN, int STAGES>
static moe_status_t launch(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b2,
                           const Params& P, int max_tiles, cudaStream_t s) {
  auto kern = gemm_tc_kernel<MODE, BN, STAGES>;
  const size_t smem = smem_bytes_for(BN, STAGES);
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    configured_dev = dev;
  }
  int grid = std::min(num_sms(), max_tiles);
  if (grid < 1) return MOE_OK;
  kern<<<grid, Roles<MODE>::kThreads, smem, s>>>(a, b, b2, P);
  return last_launch_status();
}

}  // namespace tc

int tc_status_read(int reset) {
  int v = 0;
  cudaMemcpyFromSymbol(&v, tc::g_tc_status, sizeof(int));
  if (reset) {
    int z = 0;
    cudaMemcpyToSymbol(tc::g_tc_status, &z, sizeof(int));
  }
  return v;
}

moe_status_t launch_gemm1_tc(const moe_config_t& c, const void* x, const void* W13,
                             const int32_t* sid, const int32_t* eid, const int32_t* npp,
                             int block_m, int max_padded, void* act, cudaStream_t s) {
  using namespace tc;
  CUtensorMap mG, mU;
  const uint64_t H = c.H, I = c.I, E = c.E;
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
  P.n_tiles = ceil_div(c.I, Cfg<kGemm1>::OUT_COLS);
  P.m_tiles = 0;
  P.block_m = block_m;
  P.sid = sid;
  P.eid = eid;
  P.npp = npp;
  P.out = act;
  P.ld_out = c.I;
  P.x = x;
  const int max_tiles = (max_padded / BM) * P.n_tiles;
  return launch<kGemm1, Cfg<kGemm1>::BN, Cfg<kGemm1>::STAGES>(mG, mG, mU, P, max_tiles, s);
}

moe_status_t launch_gemm2_tc(const moe_config_t& c, const void* act, const void* W2,
                             const int32_t* sid, const int32_t* eid, const int32_t* npp,
                             int block_m, int max_padded, const float* topk_w, void* y,
                             cudaStream_t s) {
  using namespace tc;
  constexpr int BN = Cfg<kGemm2>::BN;
  CUtensorMap mA, mB;
  const uint64_t H = c.H, I = c.I, E = c.E;
  {
    uint64_t d[2] = {I, (uint64_t)max_padded}, st[1] = {I};
    uint32_t box[2] = {BK, BM};
    if (!make_map(&mA, act, 2, d, st, box, false)) return MOE_ERR_CUDA;
  }
  {
    uint64_t d[3] = {I, H, E}, st[2] = {I, H * I};
    uint32_t box[3] = {BK, BN, 1};
    if (!make_map(&mB, W2, 3, d, st, box, true)) return MOE_ERR_CUDA;
  }
  Params P{};
  P.n_rows = c.T * c.k;
  P.k = 1;
  P.N = c.H;
  P.K = c.I;
  P.n_tiles = ceil_div(c.H, BN);
  P.m_tiles = 0;
  P.block_m = block_m;
  P.sid = sid;
  P.eid = eid;
  P.npp = npp;
  P.topk_w = topk_w;
  P.out = y;
  P.ld_out = c.H;
  const int max_tiles = (max_padded / BM) * P.n_tiles;
  return launch<kGemm2, BN, Cfg<kGemm2>::STAGES>(mA, mB, mB, P, max_tiles, s);
}

moe_status_t launch_router_tc(const moe_config_t& c, const void* x, const void* Wg,
                              float* logits, cudaStream_t s) {
  using namespace tc;
  const int bn = (c.E + 31) / 32 * 32;
  CUtensorMap mA, mB;
  const uint64_t H = c.H, E = c.E, T = c.T;
  {
    uint64_t d[2] = {H, T}, st[1] = {H};
    uint32_t box[2] = {BK, BM};
    if (!make_map(&mA, x, 2, d, st, box, false)) return MOE_ERR_CUDA;
  }
  {
    uint64_t d[2] = {H, E}, st[1] = {H};
    uint32_t box[2] = {BK, (uint32_t)bn};
    if (!make_map(&mB, Wg, 2, d, st, box, true)) return MOE_ERR_CUDA;
  }
  Params P{};
  P.n_rows = c.T;
  P.k = 1;
  P.N = c.E;
  P.K = c.H;
  P.n_tiles = 1;
  P.m_tiles = ceil_div(c.T, BM);
  P.block_m = BM;
  P.out = logits;
  P.ld_out = c.E;
  const int tiles = P.m_tiles;
  switch (bn) {
    case 32: return launch<kRouter, 32, 4>(mA, mB, mB, P, tiles, s);
    case 64: return launch<kRouter, 64, 4>(mA, mB, mB, P, tiles, s);
    case 96: return launch<kRouter, 96, 4>(mA, mB, mB, P, tiles, s);
    case 128: return launch<kRouter, 128, 4>(mA, mB, mB, P, tiles, s);
    case 160: return launch<kRouter, 160, 4>(mA, mB, mB, P, tiles, s);
    case 192: return launch<kRouter, 192, 4>(mA, mB, mB, P, tiles, s);
    case 224: return launch<kRouter, 224, 4>(mA, mB, mB, P, tiles, s);
    case 256: return launch<kRouter, 256, 4>(mA, mB, mB, P, tiles, s);
    default: return MOE_ERR_UNSUPPORTED;
  }
}

}  // namespace moe
