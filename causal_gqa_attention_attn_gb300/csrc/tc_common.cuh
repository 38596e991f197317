// sm_103a building blocks written as inline PTX: mbarrier, TMA tile loads,
// tcgen05 (TMEM allocation, MMA kind::tf32, TMEM loads/stores), and the
// shared-memory / instruction descriptors of the tensor-core MMA.
//
// Shared-memory operand layout used throughout (the 128-byte swizzle):
//   an fp32 tile of R rows x 128 columns is stored as d/32 column "panels",
//   each panel R rows x 32 floats (128 B per row), rows packed, with the
//   16-byte chunk index of each row XOR-ed with (row % 8). That is exactly
//   what a TMA load with CU_TENSOR_MAP_SWIZZLE_128B and a 32-float box
//   writes, and it is an 8-row x 128-byte swizzle atom stack that the MMA
//   reads K-major (K along the 128-byte rows): SBO = 1024 B between 8-row
//   groups; a K step of 8 floats advances the start by 32 B; the next panel
//   holds the next 32 K values.
// Every TF32 operand here is K-major: on this part the kind::tf32 MMA gave
// all-zero results with the transpose (MN-major) bits set, so where a
// contraction needs the other orientation the code stages a transposed copy.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gqa {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// The same with acquire at cluster scope, for barriers that the other CTA of
// a pair arrives on.
__device__ __forceinline__ bool mbar_try_wait_cl(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait. Gives up after ~kWaitCycles SM cycles (or as soon as another
// thread of the CTA gave up: *abort != 0), records `site` in the global status
// word and returns false; the caller then leaves its loop. A correct run never
// comes near the bound (waits here are microseconds).
constexpr long long kWaitCycles = 4000000000LL;

template <bool kCluster = false>
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint32_t* status, uint32_t site,
                                          long long limit = kWaitCycles) {
  auto poll = [&]() { return kCluster ? mbar_try_wait_cl(bar, parity) : mbar_try_wait(bar, parity); };
  if (poll()) return true;
  const long long t0 = clock64();
  while (true) {
    if (poll()) return true;
    if (*abort) return false;
    if (clock64() - t0 > limit) {
      *abort = 1;
      atomicOr(status, 0x80000000u | site);
      return false;
    }
  }
}

// The same wait by every lane of a warp; the result is made warp-uniform.
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint32_t* status, uint32_t site) {
  const bool ok = mbar_wait<kCluster>(bar, parity, abort, status, site);
  return __all_sync(0xffffffffu, ok);
}

// One lane of a converged warp (the same one each time): issue point for
// TMA, MMA and commit instructions whose operands the warp computed.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\t@p mov.u32 %0, 1;\n\t}"
      : "+r"(pred));
  return pred != 0;
}

// Contiguous copy global -> this CTA's shared memory by the TMA unit
// (cp.async.bulk): both addresses 16-byte aligned, bytes a multiple of 16;
// completes on bar (its transaction count).
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------------------
// TMA tile loads (no multicast)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            int w, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------------------
// Thread-block clusters
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA in the cluster: release this CTA's prior shared
// memory writes (e.g. mbarrier inits) and wait for all CTAs to arrive.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// shared::cluster address of the variable at `p`'s offset in CTA `rank`
__device__ __forceinline__ uint32_t mapa_u32(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
// Arrive on the mbarrier at a shared::cluster address (the other CTA of a
// pair), relaxed. Every use hands over data that is already complete before
// the arrive issues and is read only by tcgen05 MMAs issued after the waiter
// observes the phase: TMEM written or read by the sender is finished
// (tcgen05.wait::st / ::ld, then tcgen05.fence::before_thread_sync), or the
// sender observed its own TMA barrier complete; the receiver issues the MMA
// after tcgen05.fence::after_thread_sync. The arrive orders execution only,
// and carries no data. (A release arrive to the other CTA of the pair cost
// ~320 cycles of blocking on this part, a relaxed one ~5; the release cost
// is what made the SM-pair kernel slower than one SM.)
__device__ __forceinline__ void mbar_arrive_cl(uint32_t bar_cl) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cl)
               : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, fences, MMA, commit
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
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

// D[tmem] (+)= A[smem] . B[smem]^T   (kind::tf32, fp32 accumulate)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] . B[smem]^T
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Accumulating form with a constant predicate (K steps after the first).
__device__ __forceinline__ void mma_ts_acc(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc) {
  asm volatile("tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, 1;" ::"r"(d_tmem),
               "r"(a_tmem), "l"(b_desc), "r"(idesc)
               : "memory");
}
__device__ __forceinline__ void mma_ss_acc(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc) {
  asm volatile("tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, 1;" ::"r"(d_tmem),
               "l"(a_desc), "l"(b_desc), "r"(idesc)
               : "memory");
}

// Arrive on `bar` once every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------------------
// The same tcgen05 operations for a CTA group of CG = 1 (one SM) or CG = 2 (an
// SM pair of a 2-CTA cluster; a kernel uses one group size for all of its
// tcgen05 instructions). With CG = 2:
//  - alloc / dealloc / relinquish run in one warp of each CTA of the pair and
//    give both CTAs the same TMEM columns;
//  - an MMA is issued by one thread of the even CTA. M = 256: A rows 0-127
//    come from the even CTA and 128-255 from the odd one (same TMEM columns
//    or shared-memory offset in each), B rows [0, N/2) from the even CTA's
//    shared memory and [N/2, N) from the odd CTA's (same offset), and each
//    CTA's TMEM receives its 128 rows of D, all N columns;
//  - a commit arrives on the barrier at the same offset in both CTAs.
// (Checked on this part with a probe against an fp64 product: TS and SS
// forms, N = 32, 64, 128.)
// ---------------------------------------------------------------------------
template <int CG>
__device__ __forceinline__ void tmem_alloc_g(uint32_t* dst_smem, uint32_t ncols) {
  if constexpr (CG == 1) {
    tmem_alloc(dst_smem, ncols);
  } else {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
  }
}
template <int CG>
__device__ __forceinline__ void tmem_relinquish_g() {
  if constexpr (CG == 1) tmem_relinquish();
  else asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
template <int CG>
__device__ __forceinline__ void tmem_dealloc_g(uint32_t taddr, uint32_t ncols) {
  if constexpr (CG == 1) {
    tmem_dealloc(taddr, ncols);
  } else {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
  }
}
template <int CG>
__device__ __forceinline__ void mma_ts_g(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  if constexpr (CG == 1) {
    mma_ts(d_tmem, a_tmem, b_desc, idesc, accumulate);
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}
template <int CG>
__device__ __forceinline__ void mma_ts_acc_g(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc) {
  if constexpr (CG == 1) {
    mma_ts_acc(d_tmem, a_tmem, b_desc, idesc);
  } else {
    asm volatile("tcgen05.mma.cta_group::2.kind::tf32 [%0], [%1], %2, %3, 1;" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b_desc), "r"(idesc)
                 : "memory");
  }
}
template <int CG>
__device__ __forceinline__ void mma_ss_g(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  if constexpr (CG == 1) {
    mma_ss(d_tmem, a_desc, b_desc, idesc, accumulate);
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}
template <int CG>
__device__ __forceinline__ void mma_ss_acc_g(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc) {
  if constexpr (CG == 1) {
    mma_ss_acc(d_tmem, a_desc, b_desc, idesc);
  } else {
    asm volatile("tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, 1;" ::"r"(d_tmem),
                 "l"(a_desc), "l"(b_desc), "r"(idesc)
                 : "memory");
  }
}
// Arrive on `bar` (CG = 1) or on the barrier at its offset in both CTAs of the
// pair (CG = 2) once every MMA this thread issued so far has completed.
template <int CG>
__device__ __forceinline__ void mma_commit_g(uint64_t* bar) {
  if constexpr (CG == 1) {
    mma_commit(bar);
  } else {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"((uint16_t)3)
        : "memory");
  }
}

// Shared-memory matrix descriptor, 128-byte swizzle, sm_100 descriptor version.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo & 0x3FFFFu) >> 4) << 16;
  d |= (uint64_t)((sbo & 0x3FFFFu) >> 4) << 32;
  d |= (uint64_t)1 << 46;   // descriptor version
  d |= (uint64_t)2 << 61;   // 128-byte swizzle
  return d;
}

// Descriptor increment for K step `ks` (8 fp32 = 32 bytes) of a K-major
// operand stored as 128-byte panels of `panel_bytes` each: the start address
// field is (address >> 4) in the low 14 bits, and shared-memory addresses stay
// below 256 KB, so adding to the descriptor never carries out of the field.
__host__ __device__ constexpr uint64_t desc_off(int ks, int panel_bytes) {
  return (uint64_t)(((ks / 4) * panel_bytes + (ks % 4) * 32) >> 4);
}

// Instruction descriptor: kind::tf32, fp32 D, M x N, operand majorness.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N, bool a_mn_major,
                                                  bool b_mn_major) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// Round to TF32 (10 mantissa bits; the low 13 bits of the fp32 pattern
// cleared), to nearest with ties away from zero, for operands this code
// writes once per tile (the TMEM copies of Q, dO and K). (The tensor core
// itself keeps the top 19 bits of an fp32 operand, that is truncates; the
// per-element softmax outputs P and dS go to it unrounded, as the TMA-loaded
// operands do.) On the sign-magnitude
// bit pattern, adding half a TF32 unit in the last place (bit 12) and then
// truncating rounds the magnitude to nearest, ties up; a mantissa carry moves
// into the exponent, which is the correctly rounded next binade. Two integer
// operations on the ALU pipe, where a conversion instruction per element
// would queue behind the softmax's exponentials. (Finite inputs; the
// softmax never produces an infinity or NaN operand.)
__host__ __device__ __forceinline__ uint32_t tf32_rna_bits(uint32_t u) {
  return (u + 0x1000u) & 0xffffe000u;
}
__device__ __forceinline__ float to_tf32(float x) {
  return __uint_as_float(tf32_rna_bits(__float_as_uint(x)));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// TMEM <-> registers, 32 lanes x 32 bits, 16 or 32 consecutive columns
// ---------------------------------------------------------------------------
#define GQA_R16(p) \
  "=f"(p[0]), "=f"(p[1]), "=f"(p[2]), "=f"(p[3]), "=f"(p[4]), "=f"(p[5]), "=f"(p[6]), \
      "=f"(p[7]), "=f"(p[8]), "=f"(p[9]), "=f"(p[10]), "=f"(p[11]), "=f"(p[12]), "=f"(p[13]), \
      "=f"(p[14]), "=f"(p[15])
#define GQA_W16(p) \
  "f"(p[0]), "f"(p[1]), "f"(p[2]), "f"(p[3]), "f"(p[4]), "f"(p[5]), "f"(p[6]), "f"(p[7]), \
      "f"(p[8]), "f"(p[9]), "f"(p[10]), "f"(p[11]), "f"(p[12]), "f"(p[13]), "f"(p[14]), \
      "f"(p[15])

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : GQA_R16(v)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : GQA_R16(v), GQA_R16((v + 16))
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      GQA_W16(v)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      GQA_W16(v), GQA_W16((v + 16))
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Byte offset of element (row, col) of an R-row panel stack written by a
// SWIZZLE_128B TMA load of 32-float boxes (col in [0, 32 * n_panels)).
__host__ __device__ constexpr uint32_t sw128_offset(uint32_t row, uint32_t col, uint32_t rows) {
  return (col / 32) * rows * 128u + row * 128u +
         ((((col % 32) / 4) ^ (row % 8)) * 16u) + (col % 4) * 4u;
}

}  // namespace tc
}  // namespace gqa
