// tc_ptx.cuh — inline-PTX building blocks of the tensor-core kernels (internal header):
// mbarriers with bounded waits, TMA tile copies, 16-byte cp.async, cluster barriers and
// remote arrivals, tcgen05 (TMEM allocation, MMA, commit, TMEM loads) for one CTA or a CTA
// pair, shared-memory matrix descriptors, and the host-side tensor-map encoder.
#pragma once

#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace moe {
namespace ptx {

constexpr int BM = 128;     // rows of one CTA's MMA tile (TMEM lanes)
constexpr int BK = 64;      // 64 bf16 = 128 bytes = one swizzle row
constexpr int UMMA_K = 16;  // K of one kind::f16 MMA
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per pipeline wait

__device__ __forceinline__ uint32_t su32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------- mbarriers
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count));
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
// Arrive on the mbarrier at the same shared-memory offset in cluster CTA `rank`.
__device__ __forceinline__ void mbar_arrive_cta(uint64_t* b, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(su32(b)), "r"(rank));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait with a suspend-time hint: a thread whose phase is not complete sleeps in hardware
// until the phase completes or about `ns` nanoseconds pass, issuing nothing meanwhile.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* b, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of parity `parity`. Returns false (after raising the CTA's
// abort flag and writing kStatusTimeout to *status) when it runs out of time, or when
// another role of the CTA has aborted. sleep_ns > 0 suspends the thread between polls (for
// roles whose spinning would take issue slots from warps doing arithmetic).
static __device__ __noinline__ bool wait_slow(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                       int* status, uint32_t sleep_ns = 0) {
  const uint64_t t0 = gtimer();
  for (uint32_t it = 1;; ++it) {
    if (sleep_ns ? mbar_try_wait_sleep(b, parity, sleep_ns) : mbar_try_wait(b, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (gtimer() - t0 > kTimeoutNs) {
        *abort_flag = 1;
        atomicExch(status, kStatusTimeout);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool wait_bounded(uint64_t* b, uint32_t parity,
                                             volatile int* abort_flag, int* status) {
  if (mbar_try_wait(b, parity)) return true;
  return wait_slow(b, parity, abort_flag, status);
}
constexpr uint32_t kSleepNs = 1000;  // suspend hint of the sleeping waits
__device__ __forceinline__ bool wait_bounded_sleep(uint64_t* b, uint32_t parity,
                                                   volatile int* abort_flag, int* status) {
  if (mbar_try_wait(b, parity)) return true;
  return wait_slow(b, parity, abort_flag, status, kSleepNs);
}

// ------------------------------------------------------------------- cluster
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------------------- copies
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
// Pair forms: the copy lands in this CTA's shared memory and completes its bytes on the
// mbarrier at shared::cluster address `mbar`, which may belong to the peer CTA of the pair.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(su32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void tma_2d_pair(void* dst, const CUtensorMap* tm, uint32_t mbar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(su32(dst)),
      "l"((uint64_t)tm), "r"(c0), "r"(c1), "r"(mbar)
      : "memory");
}
__device__ __forceinline__ void tma_3d_pair(void* dst, const CUtensorMap* tm, uint32_t mbar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(su32(dst)),
      "l"((uint64_t)tm), "r"(c0), "r"(c1), "r"(c2), "r"(mbar)
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)tm) : "memory");
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

// ------------------------------------------------------------------- tcgen05
// CG = 1: one CTA owns its MMAs and TMEM; CG = 2: a CTA pair (cluster ranks 2i, 2i+1) runs
// M=256 MMAs, each CTA holding 128 rows of A, half of B and its 128 rows of D in its TMEM.
// Every tcgen05 instruction of a kernel uses the same CG.
template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  if (CG == 1)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(slot)),
                 "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(slot)),
                 "r"(ncols)
                 : "memory");
}
template <int CG>
__device__ __forceinline__ void tmem_relinquish() {
  if (CG == 1)
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  else
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  if (CG == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate.
template <int CG>
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  if (CG == 1)
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// One arrival on `bar` (this CTA) once every MMA issued so far by this thread is done.
template <int CG>
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  if (CG == 1)
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            su32(bar))
        : "memory");
  else
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            su32(bar))
        : "memory");
}
// Pair form: one arrival on the mbarrier at `bar`'s offset in every CTA of `cta_mask`.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(su32(bar)),
      "h"(cta_mask)
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
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of 128 bytes,
// 8-row swizzle atoms 1024 bytes apart (stride byte offset). Tile bases are 1024-aligned;
// stepping K by 16 elements inside the atom advances the start address by 32 bytes.
__host__ __device__ constexpr uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // bits 0-13: start address / 16
  d |= (uint64_t)1 << 16;                    // bits 16-29: leading byte offset (unused)
  d |= (uint64_t)(1024 >> 4) << 32;          // bits 32-45: stride byte offset / 16
  d |= (uint64_t)1 << 46;                    // bits 46-47: descriptor version 1
  d |= (uint64_t)2 << 61;                    // bits 61-63: 128-byte swizzle
  return d;
}
// The same descriptor as its two 32-bit words: the high word is one constant for every
// operand, the low word (start address / 16, plus the leading-offset field) differs. A
// descriptor `off` bytes (a multiple of 16) past another is its low word plus off / 16.
constexpr uint32_t kSw128DescHi = (1024u >> 4) | (1u << 14) | (2u << 29);
__host__ __device__ constexpr uint32_t sw128_desc_lo(uint32_t saddr) {
  return ((saddr & 0x3FFFFu) >> 4) | (1u << 16);
}
static_assert((uint32_t)(sw128_desc(0x2C40u) >> 32) == kSw128DescHi &&
                  (uint32_t)sw128_desc(0x2C40u) == sw128_desc_lo(0x2C40u),
              "split descriptor words");
// tcgen05.mma (cta_group::1, kind::f16) with both operand descriptors given by their low words.
__device__ __forceinline__ void umma_bf16_lo(uint32_t d_tmem, uint32_t alo, uint32_t blo,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 ad, bd;\n mov.b64 ad, {%1, %5};\n mov.b64 bd, {%2, %5};\n"
      " setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(alo), "r"(blo), "r"(idesc), "r"(accumulate), "r"(kSw128DescHi)
      : "memory");
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

// ------------------------------------------------------------------- FP8 E4M3 weights
// E4M3 -> bf16 with integer operations only. An E4M3 byte s.eeee.mmm moved into the bf16
// bit pattern s.0000eeee.mmm0000 is, read as bf16, the code's value times 2^-120, for
// subnormal codes too (E4M3 exponent 0 lands in the bf16 subnormal range with the same
// mantissa). The bf16 subnormals take part in the bf16 multiply below without flushing.
// (The NaN code 0x7F is not propagated; weights hold finite codes.)
// Per 16-bit half holding a code b in its low byte, (b & 0x7F) << 4 | (b & 0x80) << 8 equals
// 16 b + 240 (b & 0x80): times 16 puts the magnitude in place and the sign at bit 11, and
// 15 * 0x800 more carries that bit to bit 15 (no half overflows into the next). Written as
// multiply-adds, half of the work runs on the FMA pipe instead of the integer ALU, which
// the conversion otherwise saturates.
__device__ __forceinline__ void e4m3x4_to_bf16x4_lowexp(uint32_t x, uint32_t& p01, uint32_t& p23) {
  const uint32_t a = __byte_perm(x, 0u, 0x4140u);  // [0 b1 0 b0]
  const uint32_t b = __byte_perm(x, 0u, 0x4342u);  // [0 b3 0 b2]
  p01 = a * 16u + (a & 0x00800080u) * 240u;
  p23 = b * 16u + (b & 0x00800080u) * 240u;
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// General scale: exact fp32 products, one rounding to bf16.
__device__ __forceinline__ uint32_t bf16x2_lowexp_scale_f32(uint32_t p, float sc) {
  const float lo = __uint_as_float(p << 16) * 0x1p120f;
  const float hi = __uint_as_float(p & 0xFFFF0000u) * 0x1p120f;
  return pack_bf16(lo * sc, hi * sc);
}

// Sixteen E4M3 codes (raw bytes) times their block scale sc, as eight packed bf16 pairs: the
// operand a bf16 MMA reads in place of the weights. A power-of-two scale below 2^8 (or 0)
// times 2^120 is an exact bf16, so one packed bf16 multiply per two weights is exact; any
// other scale takes exact fp32 products and one rounding.
__device__ __forceinline__ void e4m3x16_scaled_bf16(const uint4& q, float sc, uint32_t (&v)[8]) {
  const float scb = sc * 0x1p120f;
  const bool fast = (__float_as_uint(sc) & 0x807FFFFFu) == 0 && sc < 0x1p8f;
  const uint32_t sc2 = (__float_as_uint(scb) >> 16) * 0x10001u;
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
}

// ------------------------------------------------------------------- host: tensor maps
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// bf16 tensor map with 128-byte swizzle, or (fp8) a byte map without swizzle whose rows of
// BK codes land densely; dims/strides in elements (dim 0 innermost).
inline bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides_elems, const uint32_t* box, bool weights,
                     bool fp8 = false) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[3], gstr[2];
  cuuint32_t bdim[3], estr[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) gstr[i] = strides_elems[i] * (fp8 ? 1 : 2);
  CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank,
                  const_cast<void*>(base), gdim, gstr, bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  fp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                  weights ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace ptx
}  // namespace moe
