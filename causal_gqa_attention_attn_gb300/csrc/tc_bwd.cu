// Tensor-core backward (tcgen05, kind::tf32, fp32 accumulation in TMEM).
//
// Two kernels, both warp-specialised: two TMA producer warps, one MMA warp
// (one elected lane issues every MMA and commit) and two compute warpgroups
// (eight warps; a warp reads and writes the 32 TMEM lanes of its quadrant,
// the two warpgroups split the columns of each tile), with every operand
// resident on chip. By default both run on SM pairs (cta_group::2, M = 256).
//
//  tc_query_major (grid: query slabs x kv heads). A slab is 128 rows =
//    (128 / G) queries x the G query heads of one kv group, so the whole group
//    shares each K/V chunk. Q and dO of the slab sit in TMEM as the A operands;
//    K/V chunks stream through a TMA ring (128-byte swizzle).
//    Pass 1 over the visible chunks: S = Q K^T, dP = dO V^T, D += rowsum(P dP)
//    (backward_attention.wgsl, attention_backward Pass A). Pass 2: the same
//    S, dP, then dS = scale P (dP - D) written back to TMEM over S and
//    dQ += dS K (Pass B), with B = the matching chunk of K^T (a transposed
//    copy of K in the workspace: the TF32 MMA reads both operands K-major).
//    At d = 128 on SM pairs pass 2 goes by chunk in four cycled TMEM slots
//    and reads K from K', a row-permuted copy (QmCfg::CYC), and by default
//    the two passes are one (QmCfg::SP): the walk accumulates U = sum P dP K
//    and W = sum P K beside D = rowsum(P dP), and dQ = scale (U - D W), since
//    dS K = scale (P dP - D P) K. Four contractions per chunk instead of five.
//    dQ and D are owned writes (no atomics). Its prologue also writes the
//    transposed copies Q^T and dO^T that the key-major kernel reads, and
//    each row's record for it (lse log2 e, scale D, query, seg).
//
//  tc_key_major (grid: key tiles x kv heads): dK and dV of 128 keys, summed
//    over the G heads of the group, from S^T = K Q^T and dP^T = V dO^T
//    (attention_backward_short_dKdV's key-major ownership); see below.
//
// Rows of a slab are ordered query-major: row r = (r / G)-th query, head
// g*G + r % G, which is also the memory order of Q / dO / dQ for a group.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdlib.h>

#include <atomic>
#include <type_traits>

#include "common.cuh"
#include "tc_common.cuh"

namespace gqa {
namespace {

using namespace tc;

// Warp roles: two TMA producer warps (one issuing stream reached ~43 B/clk
// per SM on this part, two ~71), one MMA warp, two compute warpgroups.
constexpr int kProducerWarps = 2;
constexpr int kMmaWarp = kProducerWarps;
constexpr int kFirstCompute = kProducerWarps + 1;
constexpr int kComputeWarps = 8;
constexpr int kThreads = 32 * (kFirstCompute + kComputeWarps);
constexpr uint32_t kTmemCols = 512;

// Status-word sites of bounded waits (ORed into the workspace status word).
enum : uint32_t {
  kSiteQmProducer = 1u << 0, kSiteQmMma = 1u << 1, kSiteQmCompute = 1u << 2,
  kSiteKmProducer = 1u << 4, kSiteKmMma = 1u << 5, kSiteKmCompute = 1u << 6,
  kSiteKmLayout = 1u << 7,   // dynamic shared memory not 1 KB aligned (nothing ran)
};

// ---------------------------------------------------------------------------
// Query-major configuration. Both passes stream K / V (and K^T in pass 2) in
// chunks of BK1 keys, one TMA box per tensor, chunk and CTA (on this part a
// box costs about the same TMA time from 8 KB up to 32 KB, so few large boxes
// keep the copies ahead). The boxes go through a ring of NUNIT equal units
// with a full / empty barrier each: a pass-1 chunk takes two units (K, V), a
// pass-2 chunk three (K, V, K^T). Pass 1 runs N = BK1 MMAs; pass 2 splits a
// chunk into sub-chunks of BK2 keys so that the softmax of one sub-chunk
// overlaps the MMAs of the next.
//
// C = CTA group. With C = 2 an SM pair runs M = 256 rows (two slabs) with
// cta_group::2 MMAs: each CTA stages half of every B operand (its BK1/2 keys
// of a K / V chunk, its d/2 rows of a K^T chunk), so each SM's shared memory
// takes half the TMA writes and half the tensor-core reads per flop (the two
// together are what limits the one-SM kernel). An MMA with N columns takes
// rows [0, N/2) of B from the even CTA and [N/2, N) from the odd one, so a
// pass-2 sub-chunk h is made of keys h*BK2/2 + [0, BK2/2) of each CTA's half
// (a fixed permutation of the chunk's keys, undone by key_of()).
// ---------------------------------------------------------------------------
template <int D_, int C_, bool SP_ = false>
struct QmCfg {
  static constexpr int D = D_, C = C_;
  static constexpr bool SP = SP_;
  static constexpr int BK1 = 64;                            // keys per chunk
  static constexpr int BK2 = (D == 128) ? 32 : 64;          // keys per pass-2 sub-chunk
  static constexpr int NSUB = BK1 / BK2;
  static constexpr int HALF1 = BK1 / C, HALF2 = BK2 / C;    // this CTA's keys of a chunk / sub-chunk
  static constexpr int PANELS = D / 32;
  static constexpr int KV_PANEL_BYTES = HALF1 * 128;        // K / V unit: HALF1 rows x 32 floats per panel
  static constexpr int UNIT_BYTES = PANELS * KV_PANEL_BYTES;
  static constexpr int KT_ROWS = D / C;                     // K^T unit: d/C rows x 32 keys per panel
  static constexpr int KT_PANELS = BK1 / 32;
  static constexpr int KT_PANEL_BYTES = KT_ROWS * 128;
  static_assert(KT_PANELS * KT_PANEL_BYTES == UNIT_BYTES, "K^T unit size");
  // SP (single pass, below): the slab's dO rows in shared memory ahead of
  // the ring, 128 rows x 32 floats per panel, as the A operand of dP
  static constexpr int DO_PANEL_BYTES = 128 * 128;
  static constexpr int DO_BYTES = SP ? PANELS * DO_PANEL_BYTES : 0;
  static constexpr int OFF_DO = 0, OFF_RING = DO_BYTES;
  // (SP: 9 units, three chunks: the producers stay about two chunks ahead
  // of the MMAs that read them)
  static constexpr int RING_BUDGET = (SP ? 144 : 192) * 1024;
  static constexpr int NUNIT = (RING_BUDGET / UNIT_BYTES < 12) ? RING_BUDGET / UNIT_BYTES : 12;
  static_assert(NUNIT >= 6, "ring depth");
  // + alignment slack; at least 120 KB so that one CTA (holding all 512 TMEM
  // columns) runs per SM and a second never waits in tcgen05.alloc
  static constexpr int SMEM_BYTES = (DO_BYTES + NUNIT * UNIT_BYTES + 1024 > 120 * 1024)
                                        ? DO_BYTES + NUNIT * UNIT_BYTES + 1024
                                        : 120 * 1024;
  // 227 KB per CTA, of which the static barriers and row sums take 2 KB
  static_assert(SMEM_BYTES <= 225 * 1024, "shared memory budget (with the static barriers)");
  // TMEM columns: Q | dO | dQ | stages. A pass-1 stage holds S and dP of a
  // chunk (2 BK1 columns); when two do not fit beside dQ, stage 1 of pass 1
  // uses the dQ columns, which pass 1 does not touch. The two pass-2 stages
  // (2 BK2 columns each) lie inside the pass-1 stage columns.
  // SP: Q | U | W | four slots, U and W in the dO and dQ columns.
  static constexpr uint32_t T_Q = 0, T_DO = D, T_DQ = 2 * D, T_ST = 3 * D;
  static constexpr uint32_t T_U = D, T_W = 2 * D;
  static constexpr uint32_t W1 = 2 * BK1, W2 = 2 * BK2;
  static constexpr bool P1_IN_DQ = T_ST + 2 * W1 > 512;
  static constexpr uint32_t p1_stage(int st) { return st == 0 ? T_ST : (P1_IN_DQ ? T_DQ : T_ST + W1); }
  static constexpr uint32_t p2_stage(int st) { return T_ST + st * W2; }
  static_assert(T_ST + W1 <= 512 && T_ST + 2 * W2 <= 512, "TMEM budget");
  static_assert(!P1_IN_DQ || (W1 <= D && 2 * W2 <= W1), "pass-1 stage 1 must fit the dQ columns");
  static_assert(P1_IN_DQ || W2 == W1, "pass-2 stages coincide with pass-1 stages");
  static_assert(KV_PANEL_BYTES % 1024 == 0 && KT_PANEL_BYTES % 1024 == 0 &&
                    (HALF2 * 128) % 1024 == 0 && HALF2 % 8 == 0,
                "panels must keep 1 KB swizzle alignment");
  // key offset (in the chunk) of column n of pass-2 sub-chunk h
  static __device__ __forceinline__ int key_of(int h, int n) {
    return (n / HALF2) * HALF1 + h * HALF2 + (n % HALF2);
  }
  // CYC (d = 128 on SM pairs): pass 2 goes by chunk, in the four 32-column
  // slots of the pass-1 stage-0 columns, cycled by halves of a chunk as in
  // the key-major kernel (slot functions below). Half h = keys 32 h + [0, 32)
  // of the chunk: S of a half by its own N = 32 MMA, dP of the chunk by one
  // N = 64 MMA into two adjacent slots (half 0 below half 1). For S of half
  // h to hold key 32 h + c in column c, the K chunk is read from K' (a copy
  // of K whose rows are permuted within each 64-key chunk): rows 16 h + i of
  // CTA r's unit are keys 32 h + 16 r + i. Pass 1's N = 64 S then holds key
  // c in column c for c in [0, 16) and [48, 64), key c + 16 for [16, 32) and
  // key c - 16 for [32, 48); V (and so dP) stays in key order.
  static constexpr bool CYC = (D == 128 && C == 2);
  static constexpr uint32_t t_slot(int sl) { return T_ST + 32 * sl; }
  static constexpr int c_first(int p) { return p; }
  static constexpr int c_s_slot(int p, int h) { return p == 0 ? 3 * h : 3 - h; }
  static constexpr int c_dp_slot(int p, int h) { return 1 - p + h; }
  static_assert(!CYC || (BK1 == 64 && HALF1 == 32 && T_ST + 128 <= 512 && P1_IN_DQ),
                "chunk-level pass 2: 64-key chunks, four slots in the pass-1 stage-0 columns");
  // SP (single pass, CYC shapes without a given D): one walk over the chunks
  // accumulates U = sum_k P dP K and W = sum_k P K beside D = rowsum(P dP);
  // the epilogue forms dQ = scale (U - D W). Per chunk: S halves (A = Q in
  // TMEM), dP (A = dO in shared memory: SS), then per half W += P K (A = P
  // over S) and U += (P dP) K (A = P dP over dP), with the slots cycled as in
  // the key-major kernel (W in the role of dV, U in that of dK).
  static_assert(!SP || (CYC && DO_PANEL_BYTES % 1024 == 0), "single pass: d = 128 on SM pairs");
  // the epilogue's dQ box (128 rows x d floats) at shared-memory offset 0:
  // the dO tile (SP) or the ring's first units
  static_assert(128 * D * 4 <= (SP ? DO_BYTES : NUNIT * UNIT_BYTES), "dQ box in idle shared memory");
};

struct QmBarriers {
  uint64_t full[12], empty[12], s_full[2], s_free[2], qdo_ready, dq_done;
  uint32_t tmem_base;
  int abort;
  unsigned kmin;
  float dx[2][128];   // partial row sums of P dP from the two compute warpgroups
};

__device__ __forceinline__ uint32_t lane_base(uint32_t tmem, int warp) {
  return tmem + ((uint32_t)(32 * (warp & 3)) << 16);
}

// Arrive on a barrier of the MMA-issuing CTA: this CTA's own (C = 1) or the
// even CTA's of the pair (C = 2, a remote arrive at cluster scope).
template <int C>
__device__ __forceinline__ void arrive_issuer(uint64_t* bar) {
  if constexpr (C == 1) mbar_arrive(bar);
  else mbar_arrive_cl(mapa_u32(bar, 0));
}

// Programmatic dependent launch (the query-major, key-major and part-sum
// kernels are launched as dependents of the kernel before them): let the
// next kernel of the stream start once every CTA of this one runs, and wait
// until the previous kernel has completed with its writes visible. Both are
// no-ops for a kernel not launched as a dependent.
// Make this thread's ordinary shared-memory writes visible to the async
// proxy (the tensor core's operand reads), before the barrier arrive that
// hands them over.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Release at cluster scope ahead of a relaxed remote arrive: the writes this
// thread has made or observed become visible to the CTA that acquires the
// barrier.
__device__ __forceinline__ void fence_acq_rel_cluster() {
  asm volatile("fence.acq_rel.cluster;" ::: "memory");
}

// The dQ tile leaves through the TMA unit: dst += the box at src (shared
// memory, in the tensor map's box layout), one add per element, as a
// read-modify-write would make, without the reads (dQ may be formed by a
// reduction; dK and dV keep their owned read-modify-writes, no global
// atomics). Coordinates are never negative here; rows past the tensor's end
// are not written.
__device__ __forceinline__ void tma_reduce_add_4d(const CUtensorMap* map, const void* src, int x, int y,
                                                  int z, int w) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          map),
      "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}
// Close this thread's bulk group and wait until its boxes have been read out
// of shared memory (the writes to global memory complete with the kernel).
__device__ __forceinline__ void bulk_commit_wait_read() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void pdl_launch_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_prev() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// GD: D is given (precomputed from O, attn_bwd_o): pass 1 is skipped.
// SP: the single pass of QmCfg (d = 128 on SM pairs, D not given).
template <int D, int C, bool GD, bool SP>
__global__ void __launch_bounds__(kThreads, 1)
    tc_query_major(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                   const __grid_constant__ CUtensorMap mapKt, const __grid_constant__ CUtensorMap mapDQ,
                   const float* __restrict__ Q, const float* __restrict__ dO,
                   const float* __restrict__ LSE, const uint32_t* __restrict__ seg,
                   float* __restrict__ Dws, float* __restrict__ Qt,
                   float* __restrict__ dOt, long long ld_qt, float4* __restrict__ kmeta,
                   long long ld_meta, uint32_t* __restrict__ status, Shape sh,
                   const RopeParams rope, int slab_major) {
  using Cfg = QmCfg<D, C, SP>;
  static_assert(!SP || !GD, "the single pass forms D itself");
  constexpr int NU = Cfg::NUNIT;
  constexpr bool kCl = C > 1;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int smem_shift = (int)(smem - smem_raw);   // 0 .. 1023
  __shared__ QmBarriers bars;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = sh.G, QR = 128 / G;
  // Dispatch order (CTAs start x-fastest), as for the key-major kernel:
  // kv-head-major, grid (slab groups * C, Hk), when the grid is four or more
  // waves deep (the CTAs running together stream one head's K / V chunks);
  // slab-major, grid (C * Hk, slab groups), below that (the longest rows of
  // every kv head first). Slab groups are counted from the end of the
  // sequence: longest rows first.
  const int sg = slab_major ? (int)blockIdx.y : (int)blockIdx.x / C;
  const int g = slab_major ? (int)blockIdx.x / C : (int)blockIdx.y;
  const int n_pad = (slab_major ? (int)gridDim.y : (int)gridDim.x / C) * C;   // slabs, padded to a multiple of C
  const uint32_t rank = (C > 1) ? cluster_ctarank() : 0u;
  const bool issuer = rank == 0;                         // issues the group's MMAs
  const int top_slab = n_pad - 1 - sg * C;               // the group's last slab
  const int slab = top_slab - (int)rank;
  const int q0 = slab * QR;
  const int S = sh.S, H = sh.H;
  // The key-major kernel may start once every CTA of this one runs. Until
  // this kernel waits (pdl_wait_prev), it reads only the call's inputs: the
  // K' / K^T copies and the per-block records of the kernel before are read
  // after the producers' waits, D (given O) after the compute warps'.
  pdl_launch_next();

  if (threadIdx.x == 0) {
    for (int i = 0; i < NU; ++i) {
      mbar_init(&bars.full[i], 1);        // armed by this CTA's producer warp (its bytes)
      mbar_init(&bars.empty[i], 1);       // released by the issuer's MMA commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.s_free[i], C * kComputeWarps);   // every compute warp of each CTA
    }
    mbar_init(&bars.qdo_ready, C * kComputeWarps);
    mbar_init(&bars.dq_done, 1);
    bars.abort = 0;
    bars.kmin = 0xffffffffu;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc_g<C>(&bars.tmem_base, kTmemCols);
    tmem_relinquish_g<C>();
  }
  __syncthreads();
  // smallest document start over the group's queries -> first chunk; both
  // CTAs of a pair walk the same chunk range (the union of their slabs')
  if (warp >= kFirstCompute) {
    const int r = 32 * (warp & 3) + lane;
    unsigned v = 0xffffffffu;
    for (int i = 0; i < C; ++i) {
      const int q = (top_slab - i) * QR + r / G;
      if (q < S) v = min(v, __ldg(seg + q));
    }
    for (int o = 16; o >= 1; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) atomicMin(&bars.kmin, v);
  }
  tc_fence_before();
  __syncthreads();
  if (C > 1) cluster_sync();   // the issuer's barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  const int q_last = min(top_slab * QR + QR, S) - 1;
  const int kc0 = (int)(min(bars.kmin, (unsigned)q_last) / Cfg::BK1);
  const int nk = q_last / Cfg::BK1 - kc0 + 1;          // chunks per pass
  const int p2_base = (GD || SP) ? 0 : 2 * nk;         // first pass-2 unit
  const int n_units = p2_base + 3 * nk;                // 2 per pass-1 chunk, 3 per pass-2 chunk
  const int n_sub = Cfg::NSUB * nk;                    // pass-2 sub-chunks
  volatile int* abort = &bars.abort;

  // The producer and MMA warps run their loops with all 32 lanes (waits
  // included) so that addresses and descriptors are warp-uniform; one elected
  // lane issues each TMA / MMA / commit. Issuing from a single thread inside a
  // divergent branch cost 3-10x more cycles per MMA on this part.
  if (warp < kProducerWarps) {
    // ---------------- TMA producers: warp pw loads this CTA's part of the units i with i % 2 == pw ----------------
    const int pw = warp;
    // debug build: the group's K / V / K^T rows exist and the last chunk
    // starts inside the sequence (recorded only: a box outside the tensor
    // reads the fill value)
    (void)GQA_DCHECK(status, g < sh.Hk && kc0 >= 0 && (kc0 + nk - 1) * Cfg::BK1 < S, kChkTcQmLoad);
    if (elect_one()) {
      tma_prefetch_desc(&mapK);
      tma_prefetch_desc(&mapV);
      tma_prefetch_desc(&mapKt);
    }
    __syncwarp();
    pdl_wait_prev();                       // K' and K^T of the kernel before
    for (int i = pw; i < n_units; i += 2) {
      const int u = i % NU;
      if (i >= NU &&
          !warp_wait<kCl>(&bars.empty[u], ((i / NU) - 1) & 1, abort, status, kSiteQmProducer))
        break;
      // unit i: pass-1 chunk i/2 (K, V) or pass-2 chunk (i - 2nk)/3 (K, V, K^T)
      const bool p1 = i < p2_base;
      const int chunk = p1 ? i / 2 : (i - p2_base) / 3;
      const int kind = p1 ? i % 2 : (i - p2_base) % 3;
      const int key0 = (kc0 + chunk) * Cfg::BK1;
      unsigned char* dst = smem + Cfg::OFF_RING + u * Cfg::UNIT_BYTES;
      if (elect_one()) {
        mbar_arrive_expect_tx(&bars.full[u], Cfg::UNIT_BYTES);
        if (kind == 2)
          tma_load_3d(dst, &mapKt, 0, g * D + (int)rank * Cfg::KT_ROWS, key0 / 32, &bars.full[u]);
        else
          tma_load_3d(dst, kind == 0 ? &mapK : &mapV, 0, key0 + (int)rank * Cfg::HALF1,
                      g * Cfg::PANELS, &bars.full[u]);
      }
      __syncwarp();
    }
    // leave only once every load this warp issued has landed
    const int i_lo = max(0, n_units - NU);
    for (int i = i_lo + (((i_lo & 1) != pw) ? 1 : 0); i < n_units; i += 2)
      warp_wait<kCl>(&bars.full[i % NU], (i / NU) & 1, abort, status, kSiteQmProducer);
  } else if (warp == kMmaWarp && issuer) {
    // ---------------- MMA issuer ----------------
    // It waits on one barrier per step and never on a copy: the compute warps
    // of both CTAs wait for the units that the MMAs issued after their next
    // hand-back will read (each on its own CTA's copy barrier: its half of
    // the unit) before they arrive on it (qdo_ready, s_free). A satisfied
    // mbarrier wait costs the issuing warp ~100-150 cycles, and this warp,
    // not the tensor core, paced the dQ pass; the compute warps wait while
    // they would otherwise idle.
    constexpr uint32_t id_s1 = idesc_tf32(128 * C, Cfg::BK1, false, false);   // pass 1 S, dP: N = BK1
    constexpr uint32_t id_s2 = idesc_tf32(128 * C, Cfg::BK2, false, false);   // pass 2 S, dP: N = BK2
    constexpr uint32_t id_q = idesc_tf32(128 * C, D, false, false);           // dQ: N = d
    const uint64_t desc0 = sdesc(smem_u32(smem + Cfg::OFF_RING), 16, 1024);
    auto unit_desc = [&](int i) { return desc0 + (uint64_t)(((i % NU) * Cfg::UNIT_BYTES) >> 4); };
    int use0 = 0, use1 = 0;       // pass-1 uses of each TMEM stage (s_free phases)
    // wait until the previous use of stage st has been released by its warpgroup(s)
    auto stage_free = [&](int st) {
      const int u = st ? use1 : use0;
      return u == 0 || warp_wait<kCl>(&bars.s_free[st], (u - 1) & 1, abort, status, kSiteQmMma);
    };
    // S = Q K^T and dP = dO V^T into (ts, ts + n)
    auto issue_sdp = [&](uint32_t ts, uint32_t n, uint32_t id, uint64_t bk, uint64_t bv) {
      tc_fence_after();
      mma_ts_g<C>(ts, tmem + Cfg::T_Q, bk, id, 0u);
      mma_ts_g<C>(ts + n, tmem + Cfg::T_DO, bv, id, 0u);
#pragma unroll
      for (int ks = 1; ks < D / 8; ++ks) {
        const uint64_t o = desc_off(ks, Cfg::KV_PANEL_BYTES);
        mma_ts_acc_g<C>(ts, tmem + Cfg::T_Q + 8 * ks, bk + o, id);
        mma_ts_acc_g<C>(ts + n, tmem + Cfg::T_DO + 8 * ks, bv + o, id);
      }
    };
    bool ok = warp_wait<kCl>(&bars.qdo_ready, 0, abort, status, kSiteQmMma);
    // ---- pass 1: chunk c in stage c & 1 ----
    for (int c = 0; ok && !GD && !SP && c < nk; ++c) {
      const int st = c & 1;
      const int ust = st ? use1 : use0;   // the stage's earlier uses (its release to wait for)
      // K, V of chunk c: covered by qdo_ready (c < 2) or by chunk c-2's release of the stage
      if (ust > 0 && !warp_wait<kCl>(&bars.s_free[st], (ust - 1) & 1, abort, status, kSiteQmMma)) {
        ok = false;
        break;
      }
      if (elect_one()) {
        issue_sdp(tmem + Cfg::p1_stage(st), Cfg::BK1, id_s1, unit_desc(2 * c), unit_desc(2 * c + 1));
        mma_commit_g<C>(&bars.s_full[st]);
        mma_commit_g<C>(&bars.empty[(2 * c) % NU]);
        mma_commit_g<C>(&bars.empty[(2 * c + 1) % NU]);
      }
      __syncwarp();
      if (st) ++use1; else ++use0;
    }
    if constexpr (SP) {
    // ---- single pass by chunk j (QmCfg::SP): per chunk, with f = its first
    // half and l the other: wait f's P / P dP, issue W_f(j), U_f(j) and, into
    // the two slots they read, dP(j+1); wait l's, issue U_l(j), S of (j+1)'s
    // first half into l's dP slot, W_l(j), then S of (j+1)'s second half into
    // l's S slot. MMAs run in issue order, so no slot is rewritten before the
    // MMA that reads it.
    constexpr uint32_t id_h = idesc_tf32(128 * C, 32, false, false);
    const uint64_t a_do = sdesc(smem_u32(smem + Cfg::OFF_DO), 16, 1024);   // the slab's dO rows
    auto s_half = [&](int j, int h) {
      const uint32_t d = tmem + Cfg::t_slot(Cfg::c_s_slot(j & 1, h));
      const uint64_t bk = unit_desc(3 * j) + (uint64_t)((h * 16 * 128) >> 4);
      mma_ts_g<C>(d, tmem + Cfg::T_Q, bk, id_h, 0u);
#pragma unroll
      for (int ks = 1; ks < D / 8; ++ks)
        mma_ts_acc_g<C>(d, tmem + Cfg::T_Q + 8 * ks, bk + desc_off(ks, Cfg::KV_PANEL_BYTES), id_h);
    };
    // dP of chunk j into its two dP slots (N = 64; SS: A = dO)
    auto dp_pair = [&](int j) {
      const uint32_t d = tmem + Cfg::t_slot(Cfg::c_dp_slot(j & 1, 0));
      const uint64_t bv = unit_desc(3 * j + 1);
      mma_ss_g<C>(d, a_do, bv, id_s1, 0u);
#pragma unroll
      for (int ks = 1; ks < D / 8; ++ks)
        mma_ss_acc_g<C>(d, a_do + desc_off(ks, Cfg::DO_PANEL_BYTES), bv + desc_off(ks, Cfg::KV_PANEL_BYTES),
                        id_s1);
    };
    // acc += X_h K_h over half h of chunk j: K steps 4h + i (keys 32 h + 8 i
    // ..), X at column 8 i of slot sl, B = the K^T unit (panel h). Chunk 0 is
    // even, so its half 0 issues the first (overwriting) MMA.
    auto acc_half = [&](int j, int h, uint32_t acc, int sl) {
      const uint32_t a = tmem + Cfg::t_slot(sl);
      const uint64_t bkt = unit_desc(3 * j + 2);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        mma_ts_g<C>(tmem + acc, a + 8 * i, bkt + desc_off(4 * h + i, Cfg::KT_PANEL_BYTES), id_q,
                    (j > 0 || h > 0 || i > 0) ? 1u : 0u);
    };
    auto w_half = [&](int j, int h) { acc_half(j, h, Cfg::T_W, Cfg::c_s_slot(j & 1, h)); };
    auto u_half = [&](int j, int h) { acc_half(j, h, Cfg::T_U, Cfg::c_dp_slot(j & 1, h)); };
    // chunk 0 (qdo_ready covers dO in shared memory and its K', V units)
    if (ok && elect_one()) {
      tc_fence_after();
      dp_pair(0);
      s_half(0, Cfg::c_first(0));
      mma_commit_g<C>(&bars.s_full[0]);
      s_half(0, Cfg::c_first(0) ^ 1);
      mma_commit_g<C>(&bars.s_full[1]);
      mma_commit_g<C>(&bars.empty[0]);
      mma_commit_g<C>(&bars.empty[1]);
    }
    __syncwarp();
    for (int j = 0; ok && j < nk; ++j) {
      const bool more = j + 1 < nk;
      const int hf = Cfg::c_first(j & 1), hl = hf ^ 1;   // chunk j+1 hands hl back first
      const int ik = 3 * j;
      // first half back (which also covers K^T of chunk j and K', V of j+1)
      if (!warp_wait<kCl>(&bars.s_free[0], j & 1, abort, status, kSiteQmMma)) {
        ok = false;
        break;
      }
      if (elect_one()) {
        tc_fence_after();
        w_half(j, hf);
        u_half(j, hf);
        if (more) dp_pair(j + 1);
      }
      __syncwarp();
      if (!warp_wait<kCl>(&bars.s_free[1], j & 1, abort, status, kSiteQmMma)) {
        ok = false;
        break;
      }
      if (elect_one()) {
        tc_fence_after();
        u_half(j, hl);
        if (more) {
          s_half(j + 1, hl);
          mma_commit_g<C>(&bars.s_full[0]);
        }
        w_half(j, hl);
        mma_commit_g<C>(&bars.empty[(ik + 2) % NU]);
        if (more) {
          s_half(j + 1, hf);
          mma_commit_g<C>(&bars.s_full[1]);
          mma_commit_g<C>(&bars.empty[(ik + 3) % NU]);
          mma_commit_g<C>(&bars.empty[(ik + 4) % NU]);
        }
      }
      __syncwarp();
    }
    } else if constexpr (Cfg::CYC) {
    // ---- pass 2 by chunk j (QmCfg::CYC): per chunk, with f = its first half
    // and l the other: wait f's dS, issue dQ_f(j) and, into the two slots
    // that frees (dQ_f reads f's S slot; its dP slot is free once the
    // softmax read it), dP(j+1); wait l's dS, issue S of (j+1)'s first half
    // into l's dP slot, dQ_l(j), then S of (j+1)'s second half into l's S
    // slot. MMAs run in issue order, so no slot is rewritten before the MMA
    // that reads it.
    constexpr uint32_t id_h = idesc_tf32(128 * C, 32, false, false);
    // S of half h of chunk j (B = rows 16h.. of each CTA's K' unit)
    auto s_half = [&](int j, int h) {
      const uint32_t d = tmem + Cfg::t_slot(Cfg::c_s_slot(j & 1, h));
      const uint64_t bk = unit_desc(p2_base + 3 * j) + (uint64_t)((h * 16 * 128) >> 4);
      mma_ts_g<C>(d, tmem + Cfg::T_Q, bk, id_h, 0u);
#pragma unroll
      for (int ks = 1; ks < D / 8; ++ks)
        mma_ts_acc_g<C>(d, tmem + Cfg::T_Q + 8 * ks, bk + desc_off(ks, Cfg::KV_PANEL_BYTES), id_h);
    };
    // dP of chunk j into its two dP slots (N = 64)
    auto dp_pair = [&](int j) {
      const uint32_t d = tmem + Cfg::t_slot(Cfg::c_dp_slot(j & 1, 0));
      const uint64_t bv = unit_desc(p2_base + 3 * j + 1);
      mma_ts_g<C>(d, tmem + Cfg::T_DO, bv, id_s1, 0u);
#pragma unroll
      for (int ks = 1; ks < D / 8; ++ks)
        mma_ts_acc_g<C>(d, tmem + Cfg::T_DO + 8 * ks, bv + desc_off(ks, Cfg::KV_PANEL_BYTES), id_s1);
    };
    // dQ += dS_h K_h: K steps 4h + i (keys 32 h + 8 i ..), dS at column 8 i
    // of the half's S slot, B = the K^T unit (panel h). Chunk 0 is even, so
    // its half 0 issues the first (overwriting) MMA.
    auto dq_half = [&](int j, int h) {
      const uint32_t a = tmem + Cfg::t_slot(Cfg::c_s_slot(j & 1, h));
      const uint64_t bkt = unit_desc(p2_base + 3 * j + 2);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        mma_ts_g<C>(tmem + Cfg::T_DQ, a + 8 * i, bkt + desc_off(4 * h + i, Cfg::KT_PANEL_BYTES), id_q,
                    (j > 0 || h > 0 || i > 0) ? 1u : 0u);
    };
    // prologue: the slots lie in pass-1 stage 0's columns and dQ in stage
    // 1's, so both are released first (their releases cover chunk 0's K', V)
    if (ok) ok = stage_free(0) && stage_free(1);
    if (ok && elect_one()) {
      tc_fence_after();
      dp_pair(0);
      s_half(0, Cfg::c_first(0));
      mma_commit_g<C>(&bars.s_full[0]);
      s_half(0, Cfg::c_first(0) ^ 1);
      mma_commit_g<C>(&bars.s_full[1]);
      mma_commit_g<C>(&bars.empty[p2_base % NU]);
      mma_commit_g<C>(&bars.empty[(p2_base + 1) % NU]);
    }
    __syncwarp();
    for (int j = 0; ok && j < nk; ++j) {
      const bool more = j + 1 < nk;
      const int hf = Cfg::c_first(j & 1), hl = hf ^ 1;   // chunk j+1 hands hl back first
      const int ik = p2_base + 3 * j;
      // first half back (which also covers K^T of chunk j and K', V of j+1)
      if (!warp_wait<kCl>(&bars.s_free[0], (use0 + j) & 1, abort, status, kSiteQmMma)) {
        ok = false;
        break;
      }
      if (elect_one()) {
        tc_fence_after();
        dq_half(j, hf);
        if (more) dp_pair(j + 1);
      }
      __syncwarp();
      if (!warp_wait<kCl>(&bars.s_free[1], (use1 + j) & 1, abort, status, kSiteQmMma)) {
        ok = false;
        break;
      }
      if (elect_one()) {
        tc_fence_after();
        if (more) {
          s_half(j + 1, hl);
          mma_commit_g<C>(&bars.s_full[0]);
        }
        dq_half(j, hl);
        mma_commit_g<C>(&bars.empty[(ik + 2) % NU]);
        if (more) {
          s_half(j + 1, hf);
          mma_commit_g<C>(&bars.s_full[1]);
          mma_commit_g<C>(&bars.empty[(ik + 3) % NU]);
          mma_commit_g<C>(&bars.empty[(ik + 4) % NU]);
        }
      }
      __syncwarp();
    }
    } else {
    // ---- pass 2: sub-chunk s (chunk s / NSUB, part s % NSUB) in stage s & 1 ----
    // dQ(s) and S / dP of sub-chunk s + 2 (the same stage: MMAs run in issue
    // order, so the stage is rewritten only after dQ(s) has read dS(s)) go out
    // as one burst once the softmax has handed dS(s) back; the tensor core's
    // order is the same as issuing them apart, with one wait and one burst
    // fewer per sub-chunk on the issuing warp.
    static_assert(!Cfg::P1_IN_DQ || Cfg::NSUB >= 2,
                  "the prologue must release both pass-1 stages before the first dQ");
    // S / dP of sub-chunk s2 into stage s2 & 1, with its commits
    auto sdp2 = [&](int s2) {
      const int j = s2 / Cfg::NSUB, h = s2 % Cfg::NSUB, ik = p2_base + 3 * j;
      const uint64_t off = (uint64_t)((h * Cfg::HALF2 * 128) >> 4);   // rows h*HALF2.. of each panel
      issue_sdp(tmem + Cfg::p2_stage(s2 & 1), Cfg::BK2, id_s2, unit_desc(ik) + off, unit_desc(ik + 1) + off);
      mma_commit_g<C>(&bars.s_full[s2 & 1]);
      if (h == Cfg::NSUB - 1) {
        mma_commit_g<C>(&bars.empty[ik % NU]);
        mma_commit_g<C>(&bars.empty[(ik + 1) % NU]);
      }
    };
    // prologue: sub-chunks 0 and 1, each after the last pass-1 use of its stage
    // (whose release covers their K, V units; qdo_ready does for a stage
    // that pass 1 did not use)
    for (int s = 0; ok && s < 2 && s < n_sub; ++s) {
      if (!stage_free(s & 1)) { ok = false; break; }
      if (elect_one()) sdp2(s);   // issue_sdp fences after the waits
      __syncwarp();
    }
    for (int s = 0; ok && s < n_sub; ++s) {
      const int st = s & 1, j = s / Cfg::NSUB, h = s % Cfg::NSUB, s2 = s + 2;
      const int ikt = p2_base + 3 * j + 2;
      const int u = (st ? use1 : use0) + (s >> 1);      // this sub-chunk's use of stage st
      // dS(s) handed back (which also covers K^T of s's chunk and K, V of s2's)
      if (!warp_wait<kCl>(&bars.s_free[st], u & 1, abort, status, kSiteQmMma)) {
        ok = false;
        break;
      }
      const uint32_t a_ds = tmem + Cfg::p2_stage(st), d_q = tmem + Cfg::T_DQ;
      const uint64_t bkt = unit_desc(ikt);
      if (elect_one()) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < Cfg::BK2 / 8; ++kk) {
          // K step kk: columns 8kk.. of the sub-chunk = keys key_of(h, 8kk).. of the chunk
          const int key = Cfg::key_of(h, 8 * kk);
          const uint64_t o = (uint64_t)(((key / 32) * Cfg::KT_PANEL_BYTES + (key % 32) * 4) >> 4);
          if (kk == 0) mma_ts_g<C>(d_q, a_ds, bkt + o, id_q, s > 0 ? 1u : 0u);
          else mma_ts_acc_g<C>(d_q, a_ds + 8 * kk, bkt + o, id_q);
        }
        if (h == Cfg::NSUB - 1) mma_commit_g<C>(&bars.empty[ikt % NU]);
        if (s2 < n_sub) sdp2(s2);
      }
      __syncwarp();
    }
    }   // CYC
    if (elect_one()) mma_commit_g<C>(&bars.dq_done);   // also drains every MMA issued above
    __syncwarp();
    // no MMA of the group may still run when the CTAs leave
    warp_wait<kCl>(&bars.dq_done, 0, abort, status, kSiteQmMma);
  } else if (warp >= kFirstCompute) {
    // ---------------- compute: two warpgroups, one TMEM lane (= one row) per thread ----------------
    // Each warpgroup keeps a partial row sum of P dP over its columns of the
    // pass-1 chunks (SP: of the single pass), and the two partials are added
    // through shared memory before the first dS (SP: the epilogue) needs D.
    const int wg = (warp - kFirstCompute) >> 2;
    const int r = 32 * (warp & 3) + lane;
    const int qi = r / G, q = q0 + qi;
    const int h = g * G + r % G;
    // (debug build: the row's Q / dO / dQ range and its LSE / D index lie in
    // the tensors; a row that fails is treated as padding)
    const bool valid = q < S && GQA_DCHECK(status, h < H && g < sh.Hk, kChkTcQmLoad);
    const uint32_t tl = lane_base(tmem, warp);
    const long long row_off = (long long)q * H * D + (long long)h * D;
    // This CTA's copies of units [lo, lo + cnt) (those that exist) have
    // landed: waited for by every compute warp before the hand-back after
    // which the MMA warp issues the MMAs that read them.
    auto units_landed = [&](int lo, int cnt) {
      bool okw = true;
      for (int i = lo; okw && i < lo + cnt && i < n_units; ++i)
        okw = warp_wait<kCl>(&bars.full[i % NU], (i / NU) & 1, abort, status, kSiteQmCompute);
      return okw;
    };
    // K, V units of pass-2 sub-chunk s2's chunk (CYC: of chunk s2)
    auto p2_kv = [&](int s2) { return p2_base + 3 * (Cfg::CYC ? s2 : s2 / Cfg::NSUB); };
    bool ok = true;
    // Q (warpgroup 0) or dO (warpgroup 1) rows into TMEM, rounded to TF32:
    // the A operands of S and dP (SP: dO into shared memory instead, in the
    // 128-byte-swizzled layout a TMA load of 32-float boxes would give). The
    // same rows go, unrounded, to the transposed copy Q^T / dO^T that the
    // key-major kernel reads (column q0*G + r of kv group g; a warp's 32 rows
    // are 32 adjacent columns, so each store instruction writes 128
    // contiguous bytes). Rows past the sequence write the zero padding columns.
    {
      const float* src = (wg == 0) ? Q : dO;
      float* xt = (wg == 0) ? Qt : dOt;
      const long long col = (long long)q0 * G + r;
      const bool in_ld = col < ld_qt && GQA_DCHECK(status, g < sh.Hk && col >= 0, kChkTcQmStore);
      const uint32_t col0 = (wg == 0) ? Cfg::T_Q : Cfg::T_DO;
      float v[32];
      for (int cc = 0; cc < D; cc += 32) {
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          float4 x = valid ? __ldg(reinterpret_cast<const float4*>(src + row_off + cc + i))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
          if (in_ld) {
            float* p = xt + (long long)(g * D + cc + i) * ld_qt + col;
            p[0] = x.x; p[ld_qt] = x.y; p[2 * ld_qt] = x.z; p[3 * ld_qt] = x.w;
          }
          v[i] = to_tf32(x.x); v[i + 1] = to_tf32(x.y); v[i + 2] = to_tf32(x.z); v[i + 3] = to_tf32(x.w);
        }
        if (SP && wg == 1) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(smem_raw + smem_shift + Cfg::OFF_DO + sw128_offset(r, cc + i, 128)) =
                make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        } else {
          tmem_st32(tl + col0 + cc, v);
        }
      }
      if (SP && wg == 1) fence_proxy_async_smem();   // dO, read by the tensor core
      tmem_st_wait();
      tc_fence_before();
      pdl_wait_prev();                     // the kernel before (D when given) has completed
      // the units of the MMAs issued after qdo_ready: pass-1 chunks 0 and 1,
      // and pass-2 sub-chunk st's K, V for a stage st that pass 1 leaves
      // unused (CYC: pass-2 chunk 0 is issued after both stages' last pass-1
      // releases, or right away when pass 1 is skipped)
      ok = GD || SP || units_landed(0, 2 * min(nk, 2));
      if constexpr (Cfg::CYC) {
        if (ok && (GD || SP)) ok = units_landed(p2_kv(0), 2);
      } else {
        for (int st = 0; st < 2; ++st)
          if (ok && (GD || st >= nk) && st < n_sub) ok = units_landed(p2_kv(st), 2);
      }
      __syncwarp();
      // SP: the warp's dO rows (each lane fenced its own) are released with
      // the arrive
      if (SP && wg == 1 && lane == 0) fence_acq_rel_cluster();
      if (ok && lane == 0) arrive_issuer<C>(&bars.qdo_ready);
    }
    const float sl2 = sh.scale * kLog2e;
    const float lse2 = valid ? __ldg(LSE + (long long)q * H + h) * kLog2e : 0.f;
    const int segq = valid ? (int)__ldg(seg + q) : 0;
    float Dpart = 0.f;
    // Both warpgroups take every chunk / sub-chunk, warpgroup wg the columns
    // [wg*W/2, (wg+1)*W/2) of it: the softmax of a chunk then finishes in
    // half the time, which is what the MMA warp waits for before dQ.
    // ---- pass 1: D = rowsum(P dP) ----
    constexpr int H1 = Cfg::BK1 / 2, H2 = Cfg::BK2 / 2;
    static_assert(H1 == 32 && (H2 == 16 || H2 == 32), "column split");
    for (int c = 0; ok && !GD && !SP && c < nk; ++c) {
      const int st = c & 1;
      // units of the MMAs issued after this chunk's release of stage st:
      // chunk c + 2's K, V, or after the stage's last pass-1 use, those of
      // pass-2 sub-chunk st
      if (!(c + 2 < nk ? units_landed(2 * (c + 2), 2)
                       : (Cfg::CYC ? units_landed(p2_kv(0), 2) : (st >= n_sub || units_landed(p2_kv(st), 2))))) {
        ok = false;
        break;
      }
      if (!mbar_wait<kCl>(&bars.s_full[st], (c >> 1) & 1, abort, status, kSiteQmCompute)) { ok = false; break; }
      tc_fence_after();
      const int k0 = (kc0 + c) * Cfg::BK1 + wg * H1;          // this warpgroup's first key
      // every key of these columns visible to this row: no per-element mask
      const bool full = valid && k0 >= segq && k0 + H1 - 1 <= q;
      const uint32_t ts = tl + Cfg::p1_stage(st) + wg * H1;
      float sv[32], dp[32];
      if constexpr (Cfg::CYC) {
        // keys 32 wg + [0, 32) of the chunk: S columns 16 wg + [0, 16) and
        // 32 + 16 wg + [0, 16) (K' order), dP columns 32 wg + [0, 32)
        const uint32_t s0 = tl + Cfg::p1_stage(st) + 16 * wg;
        tmem_ld16(s0, sv);
        tmem_ld16(s0 + 32, sv + 16);
      } else {
        tmem_ld32(ts, sv);
      }
      tmem_ld32(ts + Cfg::BK1, dp);
      tmem_ld_wait();
      if (full) {
#pragma unroll
        for (int j = 0; j < 32; ++j) Dpart = fmaf(ex2(fmaf(sv[j], sl2, -lse2)), dp[j], Dpart);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int key = k0 + j;
          const bool vis = valid && key >= segq && key <= q;
          Dpart = fmaf(vis ? ex2(fmaf(sv[j], sl2, -lse2)) : 0.f, dp[j], Dpart);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_issuer<C>(&bars.s_free[st]);
    }
    // both warpgroups' partial sums (each has finished reading the pass-1
    // stages), or the given D
    // (SP: both formed after the single pass)
    auto sum_d = [&]() {
      bars.dx[wg][r] = Dpart;
      tc_fence_before();
      asm volatile("bar.sync 2, 256;" ::: "memory");
      return bars.dx[0][r] + bars.dx[1][r];
    };
    // the key-major kernel's record of this row's column (the column of
    // Q^T / dO^T; padding rows get a record that masks the column out)
    auto write_record = [&](float Dr) {
      if (wg == 0) {
        const long long col = (long long)q0 * G + r;
        if (col < ld_meta && GQA_DCHECK(status, g < sh.Hk && col >= 0, kChkTcQmStore))
          kmeta[(long long)g * ld_meta + col] =
              valid ? make_float4(lse2, sh.scale * Dr, __int_as_float(q), __int_as_float(segq))
                    : make_float4(0.f, 0.f, __int_as_float(-1), __int_as_float(0x7fffffff));
      }
    };
    float Drow = 0.f;
    if constexpr (GD) {
      Drow = valid ? Dws[(long long)q * H + h] : 0.f;
      write_record(Drow);
    } else if constexpr (!SP) {
      Drow = sum_d();
      write_record(Drow);
    }
    if constexpr (SP) {
      // ---- single pass: P over S and P dP over dP, D += rowsum(P dP) ----
      // By chunk j, its halves in hand-over order (QmCfg: c_first): half h of
      // warpgroup wg is columns 16 wg + [0, 16) of the half's S and dP slots,
      // keys 32 h + 16 wg + [0, 16) of the chunk. The first half's S (and the
      // chunk's dP) is ready with s_full[0], the second's with s_full[1].
      for (int j = 0; ok && j < nk; ++j) {
        // units of the MMAs issued after this chunk's hand-backs: K^T of
        // chunk j, and K', V of chunk j + 1
        if (!(units_landed(3 * j + 2, 1) && (j + 1 >= nk || units_landed(p2_kv(j + 1), 2)))) {
          ok = false;
          break;
        }
        const int p = j & 1, kc = (kc0 + j) * Cfg::BK1;
        for (int i = 0; i < 2; ++i) {
          const int hh = Cfg::c_first(p) ^ i;
          if (!mbar_wait<kCl>(&bars.s_full[i], j & 1, abort, status, kSiteQmCompute)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int k0 = kc + 32 * hh + 16 * wg;
          const bool full = valid && k0 >= segq && k0 + 15 <= q;
          const uint32_t ts = tl + Cfg::t_slot(Cfg::c_s_slot(p, hh)) + 16 * wg;
          const uint32_t tdp = tl + Cfg::t_slot(Cfg::c_dp_slot(p, hh)) + 16 * wg;
          float sv[16], dp[16];
          tmem_ld16(ts, sv);
          tmem_ld16(tdp, dp);
          tmem_ld_wait();
          if (full) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const float pj = ex2(fmaf(sv[jj], sl2, -lse2));
              const float x = pj * dp[jj];
              Dpart += x;
              sv[jj] = pj;
              dp[jj] = x;
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int key = k0 + jj;
              const bool vis = valid && key >= segq && key <= q;
              const float pj = vis ? ex2(fmaf(sv[jj], sl2, -lse2)) : 0.f;
              const float x = pj * dp[jj];
              Dpart += x;
              sv[jj] = pj;
              dp[jj] = x;
            }
          }
          tmem_st16(ts, sv);
          tmem_st16(tdp, dp);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive_issuer<C>(&bars.s_free[i]);
        }
      }
      // every compute warp gets here (a failed wait only skips work)
      Drow = sum_d();
      write_record(Drow);
    } else if constexpr (Cfg::CYC) {
      // by chunk j, its halves in hand-over order (QmCfg: c_first): half h of
      // warpgroup wg is columns 16 wg + [0, 16) of the half's S and dP slots,
      // keys 32 h + 16 wg + [0, 16) of the chunk. The first half's S (and the
      // chunk's dP) is ready with s_full[0], the second's with s_full[1].
      for (int j = 0; ok && j < nk; ++j) {
        // units of the MMAs issued after this chunk's hand-backs: K^T of
        // chunk j, and K', V of chunk j + 1
        if (!(units_landed(p2_base + 3 * j + 2, 1) && (j + 1 >= nk || units_landed(p2_kv(j + 1), 2)))) {
          ok = false;
          break;
        }
        const int p = j & 1, kc = (kc0 + j) * Cfg::BK1;
        for (int i = 0; i < 2; ++i) {
          const int hh = Cfg::c_first(p) ^ i;
          const int u1 = GD ? 0 : (i == 0 ? (nk + 1) / 2 : nk / 2);   // pass-1 uses of s_full[i]
          if (!mbar_wait<kCl>(&bars.s_full[i], (u1 + j) & 1, abort, status, kSiteQmCompute)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int k0 = kc + 32 * hh + 16 * wg;
          const bool full = valid && k0 >= segq && k0 + 15 <= q;
          const uint32_t ts = tl + Cfg::t_slot(Cfg::c_s_slot(p, hh)) + 16 * wg;
          float sv[16], dp[16];
          tmem_ld16(ts, sv);
          tmem_ld16(tl + Cfg::t_slot(Cfg::c_dp_slot(p, hh)) + 16 * wg, dp);
          tmem_ld_wait();
          if (full) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
              sv[jj] = sh.scale * ex2(fmaf(sv[jj], sl2, -lse2)) * (dp[jj] - Drow);
          } else {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int key = k0 + jj;
              const bool vis = valid && key >= segq && key <= q;
              const float pj = vis ? ex2(fmaf(sv[jj], sl2, -lse2)) : 0.f;
              sv[jj] = sh.scale * pj * (dp[jj] - Drow);
            }
          }
          tmem_st16(ts, sv);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive_issuer<C>(&bars.s_free[i]);
        }
      }
    } else {
    // ---- pass 2: dS = scale P (dP - D) over S, for dQ += dS K ----
    for (int s = 0; ok && s < n_sub; ++s) {
      const int st = s & 1;
      // units of the MMAs issued after dS(s) is handed back: K^T of s's
      // chunk (at its first sub-chunk) and K, V of sub-chunk s + 2's chunk
      // (when s + 2 starts a chunk)
      if (!((s % Cfg::NSUB != 0 || units_landed(p2_base + 3 * (s / Cfg::NSUB) + 2, 1)) &&
            (s + 2 >= n_sub || (s + 2) % Cfg::NSUB != 0 || units_landed(p2_kv(s + 2), 2)))) {
        ok = false;
        break;
      }
      const int u1 = GD ? 0 : (st ? nk / 2 : (nk + 1) / 2);   // pass-1 uses of this stage
      if (!mbar_wait<kCl>(&bars.s_full[st], (u1 + (s >> 1)) & 1, abort, status, kSiteQmCompute)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int kc = (kc0 + s / Cfg::NSUB) * Cfg::BK1, hh = s % Cfg::NSUB;
      const int n0 = wg * H2;                                  // this warpgroup's first column
      // these columns' keys lie in [kc + key_of(hh, n0), kc + key_of(hh, n0 + H2 - 1)]
      const bool full = valid && kc + Cfg::key_of(hh, n0) >= segq &&
                        kc + Cfg::key_of(hh, n0 + H2 - 1) <= q;
      const uint32_t ts = tl + Cfg::p2_stage(st) + n0;
      float sv[H2], dp[H2];
      if constexpr (H2 == 16) {
        tmem_ld16(ts, sv);
        tmem_ld16(ts + Cfg::BK2, dp);
      } else {
        tmem_ld32(ts, sv);
        tmem_ld32(ts + Cfg::BK2, dp);
      }
      tmem_ld_wait();
      if (full) {
#pragma unroll
        for (int j = 0; j < H2; ++j)
          sv[j] = sh.scale * ex2(fmaf(sv[j], sl2, -lse2)) * (dp[j] - Drow);
      } else {
#pragma unroll
        for (int j = 0; j < H2; ++j) {
          const int key = kc + Cfg::key_of(hh, n0 + j);
          const bool vis = valid && key >= segq && key <= q;
          const float pj = vis ? ex2(fmaf(sv[j], sl2, -lse2)) : 0.f;
          sv[j] = sh.scale * pj * (dp[j] - Drow);
        }
      }
      if constexpr (H2 == 16) tmem_st16(ts, sv);
      else tmem_st32(ts, sv);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_issuer<C>(&bars.s_free[st]);
    }
    }   // CYC
    // epilogue: the tile's contribution to dQ (warpgroup wg: half wg of the
    // columns), NaN-guarded and, with rope.on, rotated by the RoPE backward of
    // row q, goes to shared memory at offset 0 (the dO tile or the ring's
    // first units, idle once the last MMA has completed) in the layout of the
    // dQ tensor map's box (the slab's 128 rows, d/32 swizzled panels); one
    // thread then adds the box to dQ with a TMA reduce. Padding rows write
    // zeros, and the box's rows past the sequence are not written. D to the
    // workspace.
    const bool ep = ok && mbar_wait<kCl>(&bars.dq_done, 0, abort, status, kSiteQmCompute);
    if (ep) {
      tc_fence_after();
      for (int cc = wg * (D / 2); cc < (wg + 1) * (D / 2); cc += 16) {
        float v[16];
        if constexpr (SP) {
          // dQ = scale (U - D W)
          float w[16];
          tmem_ld16(tl + Cfg::T_U + cc, v);
          tmem_ld16(tl + Cfg::T_W + cc, w);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = sh.scale * fmaf(-Drow, w[i], v[i]);
        } else {
          tmem_ld16(tl + Cfg::T_DQ + cc, v);
          tmem_ld_wait();
        }
        if (valid) {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = (v[i] == v[i]) ? v[i] : 0.f;
          if (rope.on) {
            const long long tpos = (long long)q + rope.pos_offset;
#pragma unroll
            for (int j = 0; j < 8; ++j) rope_rotate(v[2 * j], v[2 * j + 1], tpos, cc / 2 + j, rope);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          *reinterpret_cast<float4*>(smem_raw + smem_shift + sw128_offset(r, cc + i, 128)) =
              make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
      }
      fence_proxy_async_smem();   // the box, read by the TMA unit
      if (!GD && valid && wg == 0) Dws[(long long)q * H + h] = Drow;
    }
    // every compute thread (a failed wait skips only work); no box is added
    // after a failed wait
    asm volatile("bar.sync 2, 256;" ::: "memory");
    if (warp == kFirstCompute && lane == 0 && *abort == 0 && q0 < S &&
        GQA_DCHECK(status, g < sh.Hk && q0 >= 0, kChkTcQmStore)) {
      tma_reduce_add_4d(&mapDQ, smem, 0, g * G, q0, 0);
      bulk_commit_wait_read();
    }
  }
  tc_fence_before();
  __syncthreads();
  // both CTAs of a pair are done with every copy and MMA of the group before
  // its TMEM is freed and before either leaves
  if (C > 1) cluster_sync();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc_g<C>(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// Key-major kernel: dK and dV for 128 keys of one kv head, summed over the
// query heads of its group (no atomics: the CTA owns these rows).
//
// Per (query, head) block of NQ columns (NQ/G queries x G heads):
//   S^T  = K . Q^T        A = K (TMEM, loaded once),   B = Q block   (smem)
//   dP^T = V . dO^T       A = V (smem, loaded once),   B = dO block  (smem)
//   P^T, dS^T = scale P (dP - D) written back to TMEM over S^T / dP^T
//   dV  += P^T . dO       A = P^T (TMEM),  B = dO^T block (smem, K-major copy)
//   dK  += dS^T . Q       A = dS^T (TMEM), B = Q^T block  (smem, K-major copy)
// Blocks alternate between two TMEM stages, so block n's softmax runs while
// the tensor core does S^T / dP^T of block n+1 and dV / dK of block n-1 (at
// d = 128 on SM pairs, one stage of four slots cycled by halves of a block:
// below); both compute warpgroups take every block, half its columns each. Q / dO blocks
// and Q^T / dO^T blocks stream through their own shared-memory stages (a
// block's copies take thousands of cycles to land while the tensor core is
// busy). Blocks are visited from the end of the sequence down to the tile's
// first query: CTAs that run at the same time then read the same blocks at
// about the same time, so the per-group Q / dO / Q^T / dO^T stream (larger
// than L2 at 16k tokens) is served mostly from L2.
//
// C = CTA group. With C = 2 an SM pair takes two adjacent key tiles (M = 256)
// with cta_group::2 MMAs: each CTA stages half of every B operand (NQ/2
// columns of a Q / dO block, d/2 rows of a Q^T / dO^T block), which halves
// the TMA writes and the B-operand reads per SM. Those, with the reads of V
// as the A operand of dP^T, are what limits the one-SM kernel: its
// shared-memory traffic per block is about twice what the tensor core needs
// of it per flop. The pair walks the union of the two tiles' query blocks.
// ---------------------------------------------------------------------------
template <int D_, int C_, bool W_ = false>
struct KmCfg {
  static constexpr int D = D_, C = C_;
  // (query, head) columns per block: 64, or 32 at d = 128 unless W (wide:
  // SM pairs only, one TMEM stage)
  static constexpr int NQ = (D == 128 && !W_) ? 32 : 64;
  static constexpr int NQH = NQ / C;                      // this CTA's columns of a Q / dO block
  static constexpr int DH = D / C;                        // this CTA's rows of a Q^T / dO^T block
  static constexpr int V_PANEL_BYTES = 128 * 128;         // 128 keys x 32 floats
  static constexpr int V_BYTES = (D / 32) * V_PANEL_BYTES;
  static constexpr int BLK_PANEL_BYTES = NQH * 128;       // Q / dO block panel: NQH rows x 32 floats
  static constexpr int BLK_BYTES = (D / 32) * BLK_PANEL_BYTES;
  static constexpr int T_PANEL_BYTES = DH * 128;          // Q^T / dO^T panel: d/C rows x 32 columns
  static constexpr int T_PANELS = NQ / 32;
  static_assert(T_PANELS * T_PANEL_BYTES == BLK_BYTES, "transposed block size");
  static_assert(BLK_PANEL_BYTES % 1024 == 0 && T_PANEL_BYTES % 1024 == 0,
                "panels must keep 1 KB swizzle alignment");
  // shared memory: V | Q dO stages | Q^T dO^T stages. With C = 1 the layout
  // is 224 KB at d = 128 and has no alignment slack (the kernel checks that
  // its dynamic shared memory starts 1 KB aligned and reports an error
  // otherwise); with C = 2 the halved blocks leave room for deeper staging
  // and the slack.
  static constexpr int NSQ = (C == 1) ? 3 : (NQ * D > 4096 ? 2 : 4);
  static constexpr int NST = (C == 1) ? 2 : (NQ * D > 4096 ? 2 : 4);
  static constexpr int SLACK = (C == 1) ? 0 : 1024;
  static constexpr int OFF_V = 0, OFF_QDO = V_BYTES, OFF_T = OFF_QDO + NSQ * 2 * BLK_BYTES;
  static constexpr int off_q(int b) { return OFF_QDO + b * 2 * BLK_BYTES; }
  static constexpr int off_do(int b) { return OFF_QDO + b * 2 * BLK_BYTES + BLK_BYTES; }
  static constexpr int off_qt(int b) { return OFF_T + b * 2 * BLK_BYTES; }
  static constexpr int off_dot(int b) { return OFF_T + b * 2 * BLK_BYTES + BLK_BYTES; }
  // per Q^T / dO^T stage: the block's column records (NQ x 16 bytes: lse
  // log2 e, scale D, query, seg) and its 16-byte max-seg record, copied with
  // the stage's tiles
  static constexpr int META_BYTES = NQ * 16;
  static constexpr int META_STRIDE = (META_BYTES + 16 + 127) / 128 * 128;
  static constexpr int OFF_META = OFF_T + NST * 2 * BLK_BYTES;
  static constexpr int off_meta(int b) { return OFF_META + b * META_STRIDE; }
  static constexpr int END = OFF_META + NST * META_STRIDE;
  static constexpr int SMEM_BYTES = (END + SLACK > 120 * 1024) ? END + SLACK : 120 * 1024;
  // 227 KB per CTA, of which the static barriers take under 1 KB
  static_assert(SMEM_BYTES <= 226 * 1024, "shared memory budget (with the static barriers)");
  // TMEM columns: K | dK | dV | NS stages of S^T dP^T (two where they fit;
  // at d = 128 with 64-column blocks one: 3 x 128 + 2 x 64 = 512)
  static constexpr int NS = (3 * D + 4 * NQ <= 512) ? 2 : 1;
  static constexpr uint32_t T_K = 0, T_DK = D, T_DV = 2 * D;
  static constexpr uint32_t t_s(int b) { return 3 * D + b * 2 * NQ; }
  static constexpr uint32_t t_dp(int b) { return 3 * D + b * 2 * NQ + NQ; }
  static_assert(3 * D + 2 * NS * NQ <= 512, "TMEM budget");
  // W: the stage is four slots of 32 columns. A block has two halves of 32
  // columns, E = block columns [0, 32) and O = [32, 64) (h = 0, 1), each with
  // an S^T slot and a dP^T slot; the dP^T slots of a block are adjacent (E
  // below O: one N = 64 MMA). Block parity p:
  //   p = 0: S_E 0, dP_E 1, dP_O 2, S_O 3; half E is handed back first
  //   p = 1: dP_E 0, dP_O 1, S_O 2, S_E 3; half O is handed back first
  // The first half's two slots are adjacent and take the next block's dP^T;
  // the second half's take the next block's S^T halves.
  static constexpr int w_first(int p) { return p; }
  static constexpr int w_s_slot(int p, int h) { return p == 0 ? 3 * h : 3 - h; }
  static constexpr int w_dp_slot(int p, int h) { return 1 - p + h; }
  static constexpr uint32_t t_slot(int sl) { return 3 * D + 32 * sl; }
  // W: each CTA's Q tile is two sub-tiles of 16 rows, sub-tile h = block
  // columns 32 h + 16 rank + [0, 16), so that S^T of half h (an N = 32 MMA
  // taking 16 B rows from each CTA) holds block column 32 h + c in column c
  static constexpr int QSUB_BYTES = BLK_BYTES / 2;
  static constexpr int QSUB_PANEL_BYTES = BLK_PANEL_BYTES / 2;
  static_assert(!W_ || (NS == 1 && NQ == 64 && C == 2 && QSUB_PANEL_BYTES % 1024 == 0),
                "slot cycling: one stage of 64-column blocks on SM pairs");
};

struct KmBarriers {
  uint64_t v_full, k_ready;
  uint64_t qdo_full[4], qdo_empty[4];   // Q, dO blocks of each stage
  uint64_t t_full[4], t_empty[4];       // Q^T, dO^T blocks of each stage
  uint64_t s_full[2], p_ready[2], acc_done;
  uint32_t tmem_base;
  int abort;
};

// Visible query blocks of a key tile (or of an SM pair's two tiles), from the
// last block down to qb0, found 32 at a time: lane i of the warp tests block
// base - i and a ballot gives every lane the batch's mask. The next batch's
// per-block loads are issued a batch ahead, so no loop waits on them.
// Every lane of the warp calls next() together.
struct BlockWalk {
  const uint32_t* minseg;
  unsigned k_hi;
  int qb0, base;
  uint32_t mask;
  unsigned pend;   // this lane's min seg of the batch below `base`, in flight
  __device__ unsigned load(int b) const {
    const int qb = b - (int)(threadIdx.x % 32);
    return qb >= qb0 ? __ldg(minseg + qb) : 0xffffffffu;
  }
  __device__ BlockWalk(const uint32_t* m, unsigned kh, int q0, int nqb)
      : minseg(m), k_hi(kh), qb0(q0), base(nqb - 1) {
    mask = __ballot_sync(0xffffffffu, load(base) <= k_hi);
    pend = load(base - 32);
  }
  // next visible block, or -1 after the last
  __device__ int next() {
    while (mask == 0) {
      base -= 32;
      if (base < qb0) return -1;
      mask = __ballot_sync(0xffffffffu, pend <= k_hi);
      pend = load(base - 32);
    }
    const int i = __ffs(mask) - 1;
    mask &= mask - 1;
    return base - i;
  }
};

template <int D, int C, bool W>
__global__ void __launch_bounds__(kThreads, 1)
    tc_key_major(const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapQ,
                 const __grid_constant__ CUtensorMap mapDO, const __grid_constant__ CUtensorMap mapQt,
                 const __grid_constant__ CUtensorMap mapDOt, const float* __restrict__ K,
                 const float4* __restrict__ kmeta, long long ld_meta,
                 const uint32_t* __restrict__ blk_minseg, const uint4* __restrict__ blk_maxseg,
                 float* __restrict__ dK,
                 float* __restrict__ dV, uint32_t* __restrict__ status, Shape sh,
                 const RopeParams rope, int band, int n_split, float* __restrict__ parts) {
  using Cfg = KmCfg<D, C, W>;
  constexpr int NQ = Cfg::NQ, NS = Cfg::NS;
  constexpr bool kCl = C > 1;
  static_assert(Cfg::NSQ <= 4 && Cfg::NST <= 4 && NS <= 2, "barrier arrays");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ KmBarriers bars;
  unsigned char* smem = smem_raw;
  if constexpr (C == 1) {
    if ((smem_u32(smem) & 1023u) != 0) {  // the layout has no alignment slack
      if (threadIdx.x == 0) atomicOr(status, 0x80000000u | kSiteKmLayout);
      return;
    }
  } else {
    // the same offset in both CTAs of the pair (same kernel, same static layout)
    smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~uintptr_t(1023));
  }
  const int smem_shift = (int)(smem - smem_raw);   // 0 .. 1023
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = sh.G, QB = NQ / G;        // queries per block
  const int S = sh.S;
  const uint32_t rank = (C > 1) ? cluster_ctarank() : 0u;
  const bool issuer = rank == 0;          // issues the group's MMAs
  // Dispatch order: grid (C * band, Hk / band * n_tg), CTAs start x-fastest:
  // kv heads in bands of `band`, and within a band the tile groups heaviest
  // first (the first keys, seen by every later query), each tile group for
  // all heads of the band. band = 1: head after head, so the CTAs running
  // together share one head's Q / dO / Q^T / dO^T stream in L2 (16k causal:
  // 2.0 GB of DRAM reads per launch); band = Hk: the heaviest tiles of every
  // head first, which matters when the grid is only a few waves deep (packed
  // 4k documents: 1.12 -> 0.99 ms; at 16k it read 13.7 GB). The host picks.
  // With n_split > 1 (a grid under one wave deep) y also carries the part
  // of the tile pair's query walk this CTA takes (innermost).
  const int n_tg = ((S + 127) / 128 + C - 1) / C;
  const int yy = (int)blockIdx.y / n_split, part = (int)blockIdx.y % n_split;
  const int tg = yy % n_tg;
  const int g = (yy / n_tg) * band + (int)blockIdx.x / C;
  const int kg0 = tg * C * 128;                            // the group's first key
  const int k0 = kg0 + (int)rank * 128;
  const int k_hi = min(kg0 + 128 * C, S) - 1;             // the group's last key
  const int qb0 = kg0 / QB, nqb = (S + QB - 1) / QB;

  if (threadIdx.x == 0) {
    // A copy barrier is armed by this CTA's producer warp (its half of the
    // tile); the compute warps of each CTA wait on their own CTA's.
    const uint32_t nfull = 1;
    mbar_init(&bars.v_full, nfull);
    mbar_init(&bars.k_ready, C * kComputeWarps);          // every compute warp of each CTA
    for (int b = 0; b < Cfg::NSQ; ++b) {
      mbar_init(&bars.qdo_full[b], nfull);   // producer warp 0 arms both tiles
      mbar_init(&bars.qdo_empty[b], 1);      // released by the issuer's MMA commit
    }
    for (int b = 0; b < Cfg::NST; ++b) {
      mbar_init(&bars.t_full[b], nfull);     // producer warp 1 arms both tiles
      mbar_init(&bars.t_empty[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.s_full[b], 1);
      mbar_init(&bars.p_ready[b], C * kComputeWarps);
    }
    mbar_init(&bars.acc_done, 1);
    bars.abort = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc_g<C>(&bars.tmem_base, kTmemCols);
    tmem_relinquish_g<C>();
  }
  tc_fence_before();
  __syncthreads();
  if (C > 1) cluster_sync();   // the issuer's barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  volatile int* abort = &bars.abort;
  // this CTA's part of the query blocks [qb0, nqb) (all of them when n_split = 1)
  const int pb0 = qb0 + (int)((long long)(nqb - qb0) * part / n_split);
  const int pb1 = qb0 + (int)((long long)(nqb - qb0) * (part + 1) / n_split);
  // The per-block records (blk_minseg / blk_maxseg) come from two kernels
  // back and the column records, Q^T and dO^T from the query-major kernel, so
  // every role waits (pdl_wait_prev) before its block walk; before that only
  // the call's inputs are read (K into TMEM, V).
  pdl_launch_next();

  if (warp < kProducerWarps) {
    // ---------------- TMA producers: warp 0 loads Q and dO, warp 1 Q^T, dO^T and V ----------------
    // Each warp waits only for its own tiles' release: Q / dO of a stage are
    // free once its S^T / dP^T ran, Q^T / dO^T once its dV / dK ran. With
    // C = 2 this CTA loads its half of each block.
    const int pw = warp;
    // debug build: the group's heads and rows exist (recorded only, as above)
    (void)GQA_DCHECK(status, g < sh.Hk && (g + 1) * G <= sh.H && kg0 < S, kChkTcKmLoad);
    if (elect_one()) {
      if (pw == 0) {
        tma_prefetch_desc(&mapQ);
        tma_prefetch_desc(&mapDO);
      } else {
        tma_prefetch_desc(&mapQt);
        tma_prefetch_desc(&mapDOt);
        tma_prefetch_desc(&mapV);
        mbar_arrive_expect_tx(&bars.v_full, Cfg::V_BYTES);
        tma_load_3d(smem + Cfg::OFF_V, &mapV, 0, k0, g * (D / 32), &bars.v_full);
      }
    }
    __syncwarp();
    pdl_wait_prev();
    BlockWalk walk(blk_minseg, (unsigned)k_hi, pb0, pb1);
    uint64_t* full = pw == 0 ? bars.qdo_full : bars.t_full;
    uint64_t* empty = pw == 0 ? bars.qdo_empty : bars.t_empty;
    const int ns = pw == 0 ? Cfg::NSQ : Cfg::NST;      // this warp's stages
    int n = 0;
    for (int qb = walk.next(); qb >= 0; qb = walk.next()) {
      const int b = n % ns;
      const int q0 = qb * QB;
      if (n >= ns && !warp_wait<kCl>(&empty[b], ((n / ns) - 1) & 1, abort, status, kSiteKmProducer)) break;
      if (elect_one()) {
        mbar_arrive_expect_tx(&full[b], 2 * Cfg::BLK_BYTES + (pw == 1 ? Cfg::META_BYTES + 16 : 0));
        if (pw == 0) {   // 4-D boxes (32 dims, G heads, QB/C queries, d/32 panels)
          const int qh = q0 + (int)rank * (QB / C);
          if constexpr (W) {
            // Q as two sub-tiles of 16 (query, head) rows: boxes of (32 dims,
            // min(G, 16) heads, 16 / min(G, 16) queries, d/32 panels)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int c0 = 32 * h + 16 * (int)rank;
              tma_load_4d(smem + Cfg::off_q(b) + h * Cfg::QSUB_BYTES, &mapQ, 0, g * G + c0 % G,
                          q0 + c0 / G, 0, &full[b]);
            }
          } else {
            tma_load_4d(smem + Cfg::off_q(b), &mapQ, 0, g * G, qh, 0, &full[b]);
          }
          tma_load_4d(smem + Cfg::off_do(b), &mapDO, 0, g * G, qh, 0, &full[b]);
        } else {         // d/C rows x NQ (query, head) columns, in 32-column panels
          const int row = g * D + (int)rank * Cfg::DH;
          tma_load_3d(smem + Cfg::off_qt(b), &mapQt, 0, row, (q0 * G) / 32, &full[b]);
          tma_load_3d(smem + Cfg::off_dot(b), &mapDOt, 0, row, (q0 * G) / 32, &full[b]);
          // block qb's column records start at column qb * NQ = q0 * G
          bulk_load(smem + Cfg::off_meta(b), kmeta + (long long)g * ld_meta + (long long)qb * NQ,
                    Cfg::META_BYTES, &full[b]);
          bulk_load(smem + Cfg::off_meta(b) + Cfg::META_BYTES, blk_maxseg + qb, 16, &full[b]);
        }
      }
      __syncwarp();
      ++n;
    }
    // leave only once every load this warp issued has landed
    if (pw == 1) warp_wait<kCl>(&bars.v_full, 0, abort, status, kSiteKmProducer);
    for (int m = max(0, n - ns); m < n; ++m)
      warp_wait<kCl>(&full[m % ns], (m / ns) & 1, abort, status, kSiteKmProducer);
  } else if (warp == kMmaWarp && issuer) {
    pdl_wait_prev();
    BlockWalk walk(blk_minseg, (unsigned)k_hi, pb0, pb1);
    // ---------------- MMA issuer (warp-converged, elected issue) ----------------
    // One barrier per step and never a copy: the compute warps of both CTAs
    // wait for the copies that the MMAs issued after their next hand-back
    // read (each on its own CTA's barriers) before they arrive on it (k_ready,
    // p_ready), as in the query-major kernel.
    constexpr uint32_t id_s = idesc_tf32(128 * C, NQ, false, false);
    constexpr uint32_t id_g = idesc_tf32(128 * C, D, false, false);
    // V and the Q / dO tiles of blocks 0 .. NS-1 are covered by k_ready
    bool ok = warp_wait<kCl>(&bars.k_ready, 0, abort, status, kSiteKmMma);
    const uint64_t desc0 = sdesc(smem_u32(smem), 16, 1024);
    const uint64_t av = desc0 + (uint64_t)(Cfg::OFF_V >> 4);
    // S^T = K Q^T of block n into TMEM stage n % NS (TS: A = K in TMEM)
    auto s_mma = [&](int n) {
      const uint32_t d = tmem + Cfg::t_s(n % NS);
      const uint64_t bq = desc0 + (uint64_t)(Cfg::off_q(n % Cfg::NSQ) >> 4);
      mma_ts_g<C>(d, tmem + Cfg::T_K, bq, id_s, 0u);
#pragma unroll
      for (int ks = 1; ks < D / 8; ++ks)
        mma_ts_acc_g<C>(d, tmem + Cfg::T_K + 8 * ks, bq + desc_off(ks, Cfg::BLK_PANEL_BYTES), id_s);
    };
    // dP^T = V dO^T of block n (SS: A = V in shared memory), then the commits
    // that hand the stage to the softmax and free the Q / dO tiles
    auto dp_mma = [&](int n) {
      const int bs = n % Cfg::NSQ;
      const uint32_t d = tmem + Cfg::t_dp(n % NS);
      const uint64_t bdo = desc0 + (uint64_t)(Cfg::off_do(bs) >> 4);
      mma_ss_g<C>(d, av, bdo, id_s, 0u);
#pragma unroll
      for (int ks = 1; ks < D / 8; ++ks)
        mma_ss_acc_g<C>(d, av + desc_off(ks, Cfg::V_PANEL_BYTES), bdo + desc_off(ks, Cfg::BLK_PANEL_BYTES), id_s);
      mma_commit_g<C>(&bars.s_full[n % NS]);
      mma_commit_g<C>(&bars.qdo_empty[bs]);
    };
    // dV += P^T dO of block m (A = P^T over S^T in TMEM, B = its dO^T tile)
    auto dv_mma = [&](int m) {
      const uint32_t a_p = tmem + Cfg::t_s(m % NS);
      const uint64_t bdot = desc0 + (uint64_t)(Cfg::off_dot(m % Cfg::NST) >> 4);
      mma_ts_g<C>(tmem + Cfg::T_DV, a_p, bdot, id_g, m > 0 ? 1u : 0u);
#pragma unroll
      for (int kk = 1; kk < NQ / 8; ++kk)
        mma_ts_acc_g<C>(tmem + Cfg::T_DV, a_p + 8 * kk, bdot + desc_off(kk, Cfg::T_PANEL_BYTES), id_g);
    };
    // dK += dS^T Q of block m (A = dS^T over dP^T), then free its Q^T / dO^T tiles
    auto dk_mma = [&](int m) {
      const int bt = m % Cfg::NST;
      const uint32_t a_ds = tmem + Cfg::t_dp(m % NS);
      const uint64_t bqt = desc0 + (uint64_t)(Cfg::off_qt(bt) >> 4);
      mma_ts_g<C>(tmem + Cfg::T_DK, a_ds, bqt, id_g, m > 0 ? 1u : 0u);
#pragma unroll
      for (int kk = 1; kk < NQ / 8; ++kk)
        mma_ts_acc_g<C>(tmem + Cfg::T_DK, a_ds + 8 * kk, bqt + desc_off(kk, Cfg::T_PANEL_BYTES), id_g);
      mma_commit_g<C>(&bars.t_empty[bt]);
    };
    // Blocks are pulled from the walk one ahead of their use: exists(n) tells
    // whether the tile (pair) has an n-th visible block.
    int fetched = 0;
    bool done = false;
    auto exists = [&](int n) {
      while (!done && fetched <= n) {
        if (walk.next() < 0) done = true;
        else ++fetched;
      }
      return n < fetched;
    };
    // S^T / dP^T of blocks 0 .. NS-1, then per block m one burst: dV(m),
    // S^T(m+NS), dK(m), dP^T(m+NS). Block m + NS uses block m's TMEM stage;
    // MMAs run in issue order, so S^T(m+NS) overwrites P^T only after dV(m)
    // and dP^T(m+NS) overwrites dS^T only after dK(m) have been issued. The
    // slow shared-memory-A dP^T MMAs come last in the burst, keeping the
    // tensor core's queue long while the issuing warp waits for the next
    // block (this order ran the whole backward ~8% faster than dV, dK, then
    // S^T / dP^T alternating by K step). One wait on the softmax and one
    // burst per block. With one stage (64-column blocks at d = 128) the
    // tensor core idles while a block's softmax runs, but each dP^T MMA reads
    // its shared-memory A operand (V, 4 KB per K step) for 64 columns instead
    // of 32.
    if constexpr (NS == 1) {
      // One TMEM stage of four 32-column slots (KmCfg: w_s_slot, w_dp_slot),
      // handed over by halves. Per block m, with f its first half and l the
      // other: wait half f's softmax, issue dV_f(m), dK_f(m) and, into the
      // two slots those free, dP^T(m+1) (one N = 64 MMA: V, its shared-memory
      // A operand, is read once per 64 columns); wait half l's, issue dK_l(m),
      // S^T of block m+1's first half (into the slot dK_l freed), dV_l(m),
      // then S^T of m+1's second half (into the slot dV_l freed). The next
      // block's softmax can start as soon as its first S^T half lands, and
      // the tensor core still holds dV_l(m) and the second S^T half then.
      constexpr uint32_t id_h = idesc_tf32(128 * C, NQ / 2, false, false);
      // S^T of half h of block n (TS: A = K; B = sub-tile h of the Q tile)
      auto s_half = [&](int n, int h) {
        const uint32_t d = tmem + Cfg::t_slot(Cfg::w_s_slot(n & 1, h));
        const uint64_t bq = desc0 + (uint64_t)((Cfg::off_q(n % Cfg::NSQ) + h * Cfg::QSUB_BYTES) >> 4);
        mma_ts_g<C>(d, tmem + Cfg::T_K, bq, id_h, 0u);
#pragma unroll
        for (int ks = 1; ks < D / 8; ++ks)
          mma_ts_acc_g<C>(d, tmem + Cfg::T_K + 8 * ks, bq + desc_off(ks, Cfg::QSUB_PANEL_BYTES), id_h);
      };
      // dP^T of block n into its two adjacent dP^T slots (SS: A = V)
      auto dp_pair = [&](int n) {
        const uint32_t d = tmem + Cfg::t_slot(Cfg::w_dp_slot(n & 1, 0));
        const uint64_t bdo = desc0 + (uint64_t)(Cfg::off_do(n % Cfg::NSQ) >> 4);
        mma_ss_g<C>(d, av, bdo, id_s, 0u);
#pragma unroll
        for (int ks = 1; ks < D / 8; ++ks)
          mma_ss_acc_g<C>(d, av + desc_off(ks, Cfg::V_PANEL_BYTES), bdo + desc_off(ks, Cfg::BLK_PANEL_BYTES), id_s);
      };
      // dV += P^T dO and dK += dS^T Q over half h of block m: K steps 4h + i
      // (block columns 32 h + 8 i ..), P^T at column 8 i of the half's S^T
      // slot, dS^T at column 8 i of its dP^T slot. Block 0 is even, so its
      // half E issues the first (overwriting) MMA of each accumulator.
      auto dv_half = [&](int m, int h) {
        const uint64_t bdot = desc0 + (uint64_t)(Cfg::off_dot(m % Cfg::NST) >> 4);
        const uint32_t a = tmem + Cfg::t_slot(Cfg::w_s_slot(m & 1, h));
#pragma unroll
        for (int i = 0; i < 4; ++i)
          mma_ts_g<C>(tmem + Cfg::T_DV, a + 8 * i, bdot + desc_off(4 * h + i, Cfg::T_PANEL_BYTES), id_g,
                      (m > 0 || h > 0 || i > 0) ? 1u : 0u);
      };
      auto dk_half = [&](int m, int h) {
        const uint64_t bqt = desc0 + (uint64_t)(Cfg::off_qt(m % Cfg::NST) >> 4);
        const uint32_t a = tmem + Cfg::t_slot(Cfg::w_dp_slot(m & 1, h));
#pragma unroll
        for (int i = 0; i < 4; ++i)
          mma_ts_g<C>(tmem + Cfg::T_DK, a + 8 * i, bqt + desc_off(4 * h + i, Cfg::T_PANEL_BYTES), id_g,
                      (m > 0 || h > 0 || i > 0) ? 1u : 0u);
      };
      // block 0: dP^T, then its S^T halves in hand-over order (E first), each
      // followed by the commit its softmax waits for
      if (ok && exists(0) && elect_one()) {
        tc_fence_after();
        dp_pair(0);
        s_half(0, Cfg::w_first(0));
        mma_commit_g<C>(&bars.s_full[0]);
        s_half(0, Cfg::w_first(0) ^ 1);
        mma_commit_g<C>(&bars.s_full[1]);
        mma_commit_g<C>(&bars.qdo_empty[0]);
      }
      __syncwarp();
      for (int m = 0; ok && exists(m); ++m) {
        const bool more = exists(m + 1);
        const int hf = Cfg::w_first(m & 1), hl = hf ^ 1;   // block m+1 hands hl back first
        // the first half's hand-over also covers block m's Q^T / dO^T tiles
        // and block m+1's Q / dO tiles
        if (!warp_wait<kCl>(&bars.p_ready[0], m & 1, abort, status, kSiteKmMma)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          tc_fence_after();
          dv_half(m, hf);
          dk_half(m, hf);
          if (more) dp_pair(m + 1);
        }
        __syncwarp();
        if (!warp_wait<kCl>(&bars.p_ready[1], m & 1, abort, status, kSiteKmMma)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          tc_fence_after();
          dk_half(m, hl);
          if (more) {
            s_half(m + 1, hl);
            mma_commit_g<C>(&bars.s_full[0]);
          }
          dv_half(m, hl);
          mma_commit_g<C>(&bars.t_empty[m % Cfg::NST]);
          if (more) {
            s_half(m + 1, hf);
            mma_commit_g<C>(&bars.s_full[1]);
            mma_commit_g<C>(&bars.qdo_empty[(m + 1) % Cfg::NSQ]);
          }
        }
        __syncwarp();
      }
    } else {
    for (int n = 0; ok && n < NS && exists(n); ++n) {
      if (elect_one()) {
        tc_fence_after();
        s_mma(n);
        dp_mma(n);
      }
      __syncwarp();
    }
    for (int m = 0; ok && exists(m); ++m) {
      const int n2 = m + NS;
      const bool more = exists(n2);
      // block m's softmax (which also covers its Q^T / dO^T tiles and block
      // m+NS's Q / dO tiles)
      if (!warp_wait<kCl>(&bars.p_ready[m % NS], (m / NS) & 1, abort, status, kSiteKmMma)) {
        ok = false;
        break;
      }
      if (elect_one()) {
        tc_fence_after();
        dv_mma(m);
        if (more) s_mma(n2);
        dk_mma(m);
        if (more) dp_mma(n2);
      }
      __syncwarp();
    }
    }   // NS == 2
    if (elect_one()) mma_commit_g<C>(&bars.acc_done);   // also drains every MMA issued above
    __syncwarp();
    // no MMA of the group may still run when the CTAs leave
    warp_wait<kCl>(&bars.acc_done, 0, abort, status, kSiteKmMma);
  } else if (warp >= kFirstCompute) {
    // ---------------- compute: thread = key (TMEM lane) ----------------
    // (the odd CTA's MMA warp has no role and skips to the end)
    const int wg = (warp - kFirstCompute) >> 2;
    const int r = 32 * (warp & 3) + lane;
    const int key = k0 + r;
    const uint32_t tl = lane_base(tmem, warp);
    // (debug build: this kv head's K / dK / dV columns exist)
    const bool g_ok = GQA_DCHECK(status, g < sh.Hk, kChkTcKmLoad);
    {
      // K rows into TMEM (A of S^T), rounded to TF32; warpgroup wg: half wg of the columns
      float v[16];
      const float* krow = K + (long long)key * sh.Hk * D + (long long)g * D;
      for (int cc = wg * (D / 2); cc < (wg + 1) * (D / 2); cc += 16) {   // D/2 >= 16
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          float4 x = (key < S && g_ok) ? __ldg(reinterpret_cast<const float4*>(krow + cc + i))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
          v[i] = to_tf32(x.x); v[i + 1] = to_tf32(x.y); v[i + 2] = to_tf32(x.z); v[i + 3] = to_tf32(x.w);
        }
        tmem_st16(tl + Cfg::T_K + cc, v);
      }
      tmem_st_wait();
      tc_fence_before();
    }
    pdl_wait_prev();
    BlockWalk walk(blk_minseg, (unsigned)k_hi, pb0, pb1);
    // Copies the MMA warp reads after this warp's next hand-back, waited for
    // on this CTA's barriers: V and the Q / dO tiles of blocks 0 .. NS-1
    // before k_ready; per block n, its Q^T / dO^T tiles and block n+NS's
    // Q / dO tiles before p_ready(n). `ahead` walks NS blocks in front.
    BlockWalk ahead(blk_minseg, (unsigned)k_hi, pb0, pb1);
    int n_ahead = 0;                       // blocks the lookahead has found
    bool ok = warp_wait<kCl>(&bars.v_full, 0, abort, status, kSiteKmCompute);
    for (; ok && n_ahead < NS && ahead.next() >= 0; ++n_ahead)
      ok = warp_wait<kCl>(&bars.qdo_full[n_ahead % Cfg::NSQ], (n_ahead / Cfg::NSQ) & 1, abort, status,
                          kSiteKmCompute);
    __syncwarp();
    if (ok && lane == 0) arrive_issuer<C>(&bars.k_ready);
    // Both warpgroups take every block, warpgroup wg the columns
    // [wg*NQ/2, (wg+1)*NQ/2) of it: the softmax of a block then finishes in
    // half the time, which is what the MMA warp waits for before dV / dK.
    const float sl2 = sh.scale * kLog2e;
    constexpr int HQ = NQ / 2;
    static_assert(HQ == 16 || HQ == 32, "column split");
    // Block n's column records (lse log2 e, scale D, query, seg; written by
    // the query-major kernel) and its max-seg record arrive with its Q^T /
    // dO^T tiles (t_full), in that stage's shared memory, which the MMAs
    // release only after this block's last hand-back: the loop makes no
    // global load of its own. With one stage (W) warpgroup wg takes columns
    // 16 wg + [0, 16) of each half (records 32 h + 16 wg ..), else columns
    // HQ wg + [0, HQ).
    // A failed bounded wait clears ok, and the remaining iterations skip
    // their work.
    int n = 0;
    for (int qb = walk.next(); qb >= 0; qb = walk.next(), ++n) {
      const int st = n % NS;          // TMEM stage
      // the copies read by the MMAs issued after this block's hand-back
      // (blocks 0 .. n_ahead-1 are known to exist)
      if (n_ahead == n + NS && ahead.next() >= 0) ++n_ahead;
      const bool more = n_ahead > n + NS;
      if (ok)
        ok = warp_wait(&bars.t_full[n % Cfg::NST], (n / Cfg::NST) & 1, abort, status, kSiteKmCompute) &&
             (!more || warp_wait(&bars.qdo_full[(n + NS) % Cfg::NSQ], ((n + NS) / Cfg::NSQ) & 1, abort,
                                      status, kSiteKmCompute));
      if (ok) ok = warp_wait<kCl>(&bars.s_full[st], (n / NS) & 1, abort, status, kSiteKmCompute);
      if (ok) {
      tc_fence_after();
      // the block's records, addressed from the shared array itself (an
      // offset, not a cast address) so that they are read as shared memory
      const int rec_off = smem_shift + Cfg::off_meta(n % Cfg::NST);
      const float4* rec = reinterpret_cast<const float4*>(smem_raw + rec_off);
      const unsigned maxseg = *reinterpret_cast<const unsigned*>(smem_raw + rec_off + Cfg::META_BYTES);
      // every (key, column) of the block visible: key <= first query and >= every seg
      const int q_first = qb * QB;
      const bool full = key <= q_first && key >= (int)maxseg && q_first + QB - 1 < S;
      // P^T = 2^(s log2e scale - lse log2e) and dS^T = P (scale dP - scale D)
      // over NC columns: S^T at TMEM column ts, dP^T at tdp, the columns'
      // records at mt. Both go to the tensor core unrounded (it keeps the top
      // 19 bits of each): a rounding here would add two ALU operations per
      // element to the softmax, which the next MMAs wait for.
      auto softmax_cols = [&](auto nc, uint32_t ts, uint32_t tdp, const float4* mt) {
        constexpr int NC = decltype(nc)::value;
        float sv[NC], dp[NC];
        if constexpr (NC == 16) {
          tmem_ld16(ts, sv);
          tmem_ld16(tdp, dp);
        } else {
          tmem_ld32(ts, sv);
          tmem_ld32(tdp, dp);
        }
        tmem_ld_wait();
        if (full) {
#pragma unroll
          for (int j = 0; j < NC; ++j) {
            const float4 m = mt[j];
            const float pj = ex2(fmaf(sv[j], sl2, -m.x));
            sv[j] = pj;
            dp[j] = pj * fmaf(dp[j], sh.scale, -m.y);
          }
        } else {
#pragma unroll
          for (int j = 0; j < NC; ++j) {
            const float4 m = mt[j];
            const int q = __float_as_int(m.z), sq = __float_as_int(m.w);
            const bool vis = key <= q && key >= sq;        // q = -1 for padding columns
            const float pj = vis ? ex2(fmaf(sv[j], sl2, -m.x)) : 0.f;
            sv[j] = pj;
            dp[j] = pj * fmaf(dp[j], sh.scale, -m.y);
          }
        }
        if constexpr (NC == 16) {
          tmem_st16(ts, sv);
          tmem_st16(tdp, dp);
        } else {
          tmem_st32(ts, sv);
          tmem_st32(tdp, dp);
        }
        tmem_st_wait();
        tc_fence_before();
      };
      if constexpr (NS == 1) {
        // two hand-overs per block, in the order of KmCfg::w_first: half h of
        // warpgroup wg is columns 16 wg + [0, 16) of the half's S^T and dP^T
        // slots (block columns 32 h + 16 wg + [0, 16): records 32 h + 16 wg ..).
        // The first half's S^T slot is ready with s_full[0] (which also
        // covers the block's dP^T), the second's with s_full[1].
        const int p = n & 1;
        for (int i = 0; i < 2; ++i) {
          const int h = Cfg::w_first(p) ^ i;
          if (i == 1) {
            if (!warp_wait<kCl>(&bars.s_full[1], (n / NS) & 1, abort, status, kSiteKmCompute)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          softmax_cols(std::integral_constant<int, 16>{}, tl + Cfg::t_slot(Cfg::w_s_slot(p, h)) + 16 * wg,
                       tl + Cfg::t_slot(Cfg::w_dp_slot(p, h)) + 16 * wg, rec + 32 * h + 16 * wg);
          __syncwarp();
          if (lane == 0) arrive_issuer<C>(&bars.p_ready[i]);
        }
      } else {
        softmax_cols(std::integral_constant<int, HQ>{}, tl + Cfg::t_s(st) + wg * HQ,
                     tl + Cfg::t_dp(st) + wg * HQ, rec + wg * HQ);
        __syncwarp();
        if (lane == 0) arrive_issuer<C>(&bars.p_ready[st]);
      }
      }
    }
    // epilogue: warpgroup 0 adds dK (rotated by the RoPE backward of the key's
    // position when rope.on), warpgroup 1 adds dV (owned rows, NaN-guarded).
    // With n_split > 1 each part stores its partial sums instead (zeros when
    // it saw no block); km_split_reduce adds them up.
    if (ok && mbar_wait<kCl>(&bars.acc_done, 0, abort, status, kSiteKmCompute)) {
      tc_fence_after();
      const long long row = (long long)key * sh.Hk * D + (long long)g * D;
      float* dst_row = (wg == 0 ? dK : dV) + row;
      const uint32_t src = tl + (wg == 0 ? Cfg::T_DK : Cfg::T_DV);
      float* part_row = parts + ((size_t)(wg * n_split + part) * S) * ((size_t)sh.Hk * D) + row;
      for (int cc = 0; cc < D; cc += 32) {
        float a[32];
        tmem_ld32(src + cc, a);
        tmem_ld_wait();
        if (n_split > 1) {
          if (key < S && g_ok &&
              GQA_DCHECK(status, (size_t)(wg * n_split + part + 1) * S * ((size_t)sh.Hk * D) >=
                                     (size_t)(wg * n_split + part) * S * ((size_t)sh.Hk * D) + row + D &&
                                 wg * n_split + part < 2 * n_split,
                         kChkTcKmStore)) {
            float4* pp = reinterpret_cast<float4*>(part_row + cc);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              pp[i] = n > 0 ? make_float4(a[4 * i], a[4 * i + 1], a[4 * i + 2], a[4 * i + 3])
                            : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        } else if (key < S && n > 0 && g_ok &&
                   GQA_DCHECK(status, row + D <= (long long)S * sh.Hk * D, kChkTcKmStore)) {
#pragma unroll
          for (int i = 0; i < 32; ++i) a[i] = (a[i] == a[i]) ? a[i] : 0.f;
          if (wg == 0 && rope.on) {
            const long long tpos = (long long)key + rope.pos_offset;
#pragma unroll
            for (int j = 0; j < 16; ++j) rope_rotate(a[2 * j], a[2 * j + 1], tpos, cc / 2 + j, rope);
          }
          float4* pk = reinterpret_cast<float4*>(dst_row + cc);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float4 o = pk[i];
            o.x += a[4 * i];
            o.y += a[4 * i + 1];
            o.z += a[4 * i + 2];
            o.w += a[4 * i + 3];
            pk[i] = o;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // both CTAs of a pair are done with every copy and MMA of the group before
  // its TMEM is freed and before either leaves
  if (C > 1) cluster_sync();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc_g<C>(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// Group transpose: X [S][Hk*Gx][d] (row-major, head h = g*Gx + h') to
// Xt [Hk*d][ld] with Xt[g*d + e][q*Gx + h'] = X[q][(g*Gx + h')*d + e].
// With Gx = 1 this is K^T per kv head; with Gx = G it lays the (query, head)
// rows of a kv group out as the contiguous K dimension of a K-major operand.
// ld is S*Gx rounded up to 32; the grid covers all ld columns.
// With Xp (Gx = 1 only) it also writes K' for the query-major kernel: X with
// its rows permuted within each 64-row chunk, row 64c + 32r + 16a + i = row
// 64c + 32a + 16r + i of X (r, a in {0, 1}, i < 16), rows rows_p (S rounded
// up to 64) in all, those past S zero.
// With ms.seg, a last z slice of the grid (blockIdx.z == Hk) instead forms
// the key-major kernel's per-block seg minima and 16-byte max records (one
// warp per block of ms.tile queries, grid-stride), so that the backward's
// metadata costs no launch of its own.
// ---------------------------------------------------------------------------
constexpr int kTrRows = 64;   // rows r of X per CTA of the transpose (one K' chunk)

struct MinsegJob {
  const uint32_t* seg = nullptr;   // null: no job
  int tile = 0, n_tiles = 0;
  uint32_t* out_min = nullptr;
  uint4* out_max = nullptr;
};

__global__ void __launch_bounds__(256) group_transpose(const float* __restrict__ X,
                                                       float* __restrict__ Xt, int S, int Hk,
                                                       int Gx, int d, long long ld,
                                                       float* __restrict__ Xp, long long rows_p,
                                                       MinsegJob ms) {
  // the query-major kernel (a programmatic dependent) may start its prologue,
  // which reads none of this kernel's outputs, once every CTA here runs
  pdl_launch_next();
  if (ms.seg != nullptr && (int)blockIdx.z == Hk) {
    const int lane = threadIdx.x, wib = threadIdx.y;      // blockDim (32, 8)
    const int n_warps = (int)(gridDim.x * gridDim.y) * 8;
    for (int w = (int)(blockIdx.y * gridDim.x + blockIdx.x) * 8 + wib; w < ms.n_tiles; w += n_warps) {
      unsigned mn = 0xffffffffu, mx = 0u;
      for (int i = lane; i < ms.tile; i += 32) {
        const int q = w * ms.tile + i;
        if (q < S) {
          const unsigned x = __ldg(ms.seg + q);
          mn = min(mn, x);
          mx = max(mx, x);
        }
      }
      for (int o = 16; o >= 1; o >>= 1) {
        mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      }
      if (lane == 0) {
        ms.out_min[w] = mn;
        ms.out_max[w] = make_uint4(mx, 0u, 0u, 0u);
      }
    }
    return;
  }
  __shared__ float tile[kTrRows][33];
  constexpr int PER = kTrRows / 8;                        // rows per thread (blockDim.y = 8)
  const int g = blockIdx.z, e0 = blockIdx.y * 32;
  const int r0 = blockIdx.x * kTrRows, nrows = S * Gx;    // S * Gx < 2^31 (checked by the API)
  const long long row_stride = (long long)Hk * Gx * d;
  // all of this thread's loads first (coalesced: 32 consecutive e per row)
  float v[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int r = r0 + threadIdx.y + 8 * k;
    v[k] = 0.f;
    if (r < nrows) {
      const int q = r / Gx, hh = r - q * Gx;
      v[k] = __ldg(X + q * row_stride + (long long)(g * Gx + hh) * d + e0 + threadIdx.x);
    }
  }
#pragma unroll
  for (int k = 0; k < PER; ++k) tile[threadIdx.y + 8 * k][threadIdx.x] = v[k];
  __syncthreads();
  if (Xp != nullptr) {
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int i = threadIdx.y + 8 * k;                  // K' row in the chunk: 32r + 16a + (i % 16)
      const int src = 32 * ((i >> 4) & 1) + 16 * (i >> 5) + (i & 15);
      const long long rp = (long long)r0 + i;
      if (rp < rows_p) Xp[rp * row_stride + (long long)g * d + e0 + threadIdx.x] = tile[src][threadIdx.x];
    }
  }
  // columns nrows .. ld-1 are padding: written as zeros (the panel view of
  // the copy reads them as ordinary elements, masked to zero weight)
#pragma unroll
  for (int i = threadIdx.y; i < 32; i += 8) {
    float* dst = Xt + (long long)(g * d + e0 + i) * ld;
#pragma unroll
    for (int c = 0; c < kTrRows; c += 32) {
      const long long r = (long long)r0 + c + threadIdx.x;
      if (r < ld) dst[r] = tile[c + threadIdx.x][i];
    }
  }
}

// dK += R^T(sum of the key-major parts' dK), dV += sum of their dV: one
// float4 per thread, parts added in order (a fixed order: deterministic),
// NaN -> 0 on the sums as in the unsplit epilogue. parts holds [2][n_split]
// planes of [S][Hk * d] (dK planes, then dV planes). When a bounded wait of
// the backward gave up (status word set), a part that aborted has not written
// its slice and the planes may hold an earlier call's sums: nothing is added.
__global__ void __launch_bounds__(256) km_split_reduce(const float* __restrict__ parts,
                                                       float* __restrict__ dK,
                                                       float* __restrict__ dV, int S, int hkd,
                                                       int d, int n_split, const RopeParams rope,
                                                       const uint32_t* __restrict__ status) {
  pdl_wait_prev();                         // the key-major kernel's parts
  const long long n4 = (long long)S * hkd / 4;
  const long long i4 = (long long)blockIdx.x * 256 + threadIdx.x;
  if (i4 >= 2 * n4 || *status != 0u) return;
  const bool is_v = i4 >= n4;
  const long long e = (is_v ? i4 - n4 : i4) * 4;        // element index in [S][Hk * d]
  const size_t plane = (size_t)S * hkd;
  const float* src = parts + (is_v ? (size_t)n_split * plane : 0) + e;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int p = 0; p < n_split; ++p) {
    const float4 x = __ldg(reinterpret_cast<const float4*>(src + (size_t)p * plane));
    acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
  }
  acc.x = (acc.x == acc.x) ? acc.x : 0.f;
  acc.y = (acc.y == acc.y) ? acc.y : 0.f;
  acc.z = (acc.z == acc.z) ? acc.z : 0.f;
  acc.w = (acc.w == acc.w) ? acc.w : 0.f;
  if (!is_v && rope.on) {
    const long long key = e / hkd;
    const int c = (int)(e % hkd) % d;                  // column in the head (even)
    const long long tpos = key + rope.pos_offset;
    rope_rotate(acc.x, acc.y, tpos, c / 2, rope);
    rope_rotate(acc.z, acc.w, tpos, c / 2 + 1, rope);
  }
  float4* o = reinterpret_cast<float4*>((is_v ? dV : dK) + e);
  float4 cur = *o;
  cur.x += acc.x; cur.y += acc.y; cur.z += acc.z; cur.w += acc.w;
  *o = cur;
}

// D[i, h] = sum_e dO[i, h, e] * O[i, h, e]: one warp per (query, head) row,
// float4 loads. Equal to sum_j P_ij dP_ij when O is the forward's output for
// the same LSE (O_i = sum_j P_ij v_j, so dO_i . O_i = sum_j P_ij dO_i . v_j).
__global__ void __launch_bounds__(256) row_dot_kernel(const float* __restrict__ dO,
                                                      const float* __restrict__ O,
                                                      float* __restrict__ Dws, long long rows,
                                                      int d) {
  const long long row = (long long)blockIdx.x * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= rows) return;
  const float4* a = reinterpret_cast<const float4*>(dO + row * d);
  const float4* b = reinterpret_cast<const float4*>(O + row * d);
  float acc = 0.f;
  for (int v = lane; v < d / 4; v += 32) {
    const float4 x = __ldg(a + v), y = __ldg(b + v);
    acc = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, acc))));
  }
  for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) Dws[row] = acc;
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// arrives on, with a short limit, and must give up and record the site.
__global__ void wait_selftest_kernel(uint32_t* status, long long limit) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
    mbar_wait(&bar, 0, &abort_flag, status, 1u << 12, limit);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// The driver's tensor-map encoder, looked up once per process (a function-
// local static: initialised by exactly one thread).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

gqa_status encode(CUtensorMap* m, const float* base, int rank, const cuuint64_t* dims,
                  const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = encode_fn();
  if (fn == nullptr) return set_error(GQA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (cuuint32_t)rank,
                        const_cast<float*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(GQA_ERR_CUDA, "cuTensorMapEncodeTiled (rank %d) failed (%d)", rank, (int)r);
  return GQA_OK;
}

// Panel view of a row-major matrix with `rows` rows `ld` floats apart and
// `n_panels` 32-float panels per row: dims (32 floats, rows, panels), panel
// stride 128 B. One box (32, box_rows, box_panels) fills box_panels
// consecutive swizzled panels of box_rows x 128 B each in shared memory.
gqa_status map_panels(CUtensorMap* m, const float* base, long long ld, long long rows,
                      long long n_panels, int box_rows, int box_panels) {
  const cuuint64_t dims[3] = {32, (cuuint64_t)rows, (cuuint64_t)n_panels};
  const cuuint64_t strides[2] = {(cuuint64_t)ld * sizeof(float), 128};
  const cuuint32_t box[3] = {32, (cuuint32_t)box_rows, (cuuint32_t)box_panels};
  return encode(m, base, 3, dims, strides, box);
}

// (query, head) view of X [S][Hx][d]: dims (32 floats, Hx heads, S queries,
// d/32 panels); a box (32, bh, bq, d/32) fills d/32 panels of bq*bh rows
// (query-major, head-minor) x 128 B.
gqa_status map_heads(CUtensorMap* m, const float* base, int d, int Hx, int S, int bh, int bq) {
  const cuuint64_t dims[4] = {32, (cuuint64_t)Hx, (cuuint64_t)S, (cuuint64_t)(d / 32)};
  const cuuint64_t strides[3] = {(cuuint64_t)d * sizeof(float), (cuuint64_t)Hx * d * sizeof(float), 128};
  const cuuint32_t box[4] = {32, (cuuint32_t)bh, (cuuint32_t)bq, (cuuint32_t)(d / 32)};
  return encode(m, base, 4, dims, strides, box);
}

// Launch with a (cluster, 1, 1) thread-block cluster.
template <class... KArgs, class... Args>
gqa_status launch_clustered(void (*kern)(KArgs...), dim3 grid, int cluster, int smem,
                            cudaStream_t st, const char* what, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // a programmatic dependent of the stream's previous kernel (the kernels
  // launched here wait in pdl_wait_prev before they read its outputs)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  note_launch();
  if (e != cudaSuccess) return set_error(GQA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return check_launch(what);
}

// SMs of the current device (cached per device).
int sm_count() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 148;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

template <int D, int C, bool W>
gqa_status km_launch_c(const float* Q, const float* K, const float* V, const float* dO,
                       float* dK, float* dV, const float* Qt, const float* dOt, long long ld_qt,
                       const float4* kmeta, long long ld_meta, const uint32_t* blk_minseg,
                       const uint4* blk_maxseg, uint32_t* status, const Shape& sh,
                       cudaStream_t st, const RopeParams& rope, int n_split, float* parts) {
  using Cfg = KmCfg<D, C, W>;
  const int QB = Cfg::NQ / sh.G;
  CUtensorMap mv, mq, mdo, mqt, mdot;
  gqa_status r;
  const long long kv_panels = (long long)sh.Hk * D / 32;
  if ((r = map_panels(&mv, V, (long long)sh.Hk * D, sh.S, kv_panels, 128, D / 32)) != GQA_OK) return r;
  // W: Q in sub-tiles of 16 (query, head) rows (G divides 32 on SM pairs)
  const int qbh = W ? (sh.G < 16 ? sh.G : 16) : sh.G;
  if ((r = map_heads(&mq, Q, D, sh.H, sh.S, qbh, W ? 16 / qbh : QB / C)) != GQA_OK) return r;
  if ((r = map_heads(&mdo, dO, D, sh.H, sh.S, sh.G, QB / C)) != GQA_OK) return r;
  if ((r = map_panels(&mqt, Qt, ld_qt, (long long)sh.Hk * D, ld_qt / 32, Cfg::DH, Cfg::T_PANELS)) != GQA_OK) return r;
  if ((r = map_panels(&mdot, dOt, ld_qt, (long long)sh.Hk * D, ld_qt / 32, Cfg::DH, Cfg::T_PANELS)) != GQA_OK) return r;
  if (cudaFuncSetAttribute(tc_key_major<D, C, W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg::SMEM_BYTES) != cudaSuccess)
    return check_launch("key-major smem attribute");
  const int n_tiles = (sh.S + 127) / 128;
  const int n_tg = (n_tiles + C - 1) / C;
  // one CTA per SM (the kernel holds all of TMEM): all heads in one band
  // below four waves, else bands of two heads (one when Hk is odd)
  const bool few_waves = (long long)n_tg * C * sh.Hk < 4LL * sm_count();
  const int band = few_waves ? sh.Hk : (sh.Hk % 2 == 0 ? 2 : 1);
  const dim3 grid(C * band, (sh.Hk / band) * n_tg * n_split);
  r = launch_clustered(tc_key_major<D, C, W>, grid, C, Cfg::SMEM_BYTES, st,
                                  "tensor-core key-major", mv, mq, mdo, mqt, mdot, K, kmeta, ld_meta,
                                  blk_minseg, blk_maxseg, dK, dV, status, sh, rope, band, n_split,
                                  parts);
  if (r != GQA_OK || n_split == 1) return r;
  const long long n4 = (long long)sh.S * sh.Hk * D / 4;
  // a programmatic dependent of the key-major kernel (it waits first)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((2 * n4 + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, km_split_reduce, (const float*)parts, dK, dV, sh.S,
                                           sh.Hk * D, D, n_split, rope, (const uint32_t*)status);
  note_launch();
  if (e != cudaSuccess) return set_error(GQA_ERR_CUDA, "key-major part sums: %s", cudaGetErrorString(e));
  return check_launch("key-major part sums");
}

gqa_status transpose_launch(const float* X, float* Xt, int S, int Hk, int Gx, int d, long long ld,
                            cudaStream_t st, float* Xp = nullptr, long long rows_p = 0,
                            MinsegJob ms = MinsegJob{}) {
  // ld >= S * Gx; with Xp (Gx = 1) the grid's 64-row tiles also cover rows_p
  // = S rounded up to 64 (ld is S rounded up to 32); with ms.seg one more z
  // slice forms the per-block seg records
  dim3 grid((unsigned)((ld + kTrRows - 1) / kTrRows), d / 32, Hk + (ms.seg != nullptr ? 1 : 0));
  group_transpose<<<grid, dim3(32, 8), 0, st>>>(X, Xt, S, Hk, Gx, d, ld, Xp, rows_p, ms);
  note_launch();
  return check_launch("group transpose");
}

// CTA group of both backward kernels: 2 (SM pairs, cta_group::2: half the
// shared-memory traffic per SM per flop) by default; GQA_TC_CTA_GROUP=1
// selects one SM per slab / key tile. Read once per process.
int cta_group() {
  static int c = [] {
    const char* e = getenv("GQA_TC_CTA_GROUP");
    return (e != nullptr && atoi(e) == 1) ? 1 : 2;
  }();
  return c;
}

// Key-major block width at d = 128 on SM pairs: 64 (query, head) columns
// with one TMEM stage (the default), or 32 with two (GQA_KM_NARROW=1). Read
// once per process.
bool km_wide() {
  static bool w = [] {
    const char* e = getenv("GQA_KM_NARROW");
    return !(e != nullptr && atoi(e) == 1);
  }();
  return w;
}

// The key-major kernel runs on SM pairs when the pair's half block holds
// whole queries (G divides NQ/2), else on one SM per key tile.
int km_cta_group(const Shape& sh) {
  const int nqh = (sh.d == 128) ? (km_wide() ? KmCfg<128, 2, true>::NQH : KmCfg<128, 2>::NQH)
                                : KmCfg<64, 2>::NQH;
  return (cta_group() == 2 && nqh % sh.G == 0) ? 2 : 1;
}

// (query, head) columns per key-major block of the configuration that runs
// this shape (the per-block seg minima are formed for blocks of NQ / G queries).
int km_nq(const Shape& sh) {
  if (sh.d != 128) return KmCfg<64, 1>::NQ;
  if (km_cta_group(sh) == 2 && km_wide()) return KmCfg<128, 2, true>::NQ;
  return KmCfg<128, 1>::NQ;
}

// Parts the key-major kernel splits each tile (pair)'s query walk into: 1
// when its grid fills at least one wave (one CTA per SM), else enough parts,
// at most four, to fill about four waves. Each part writes partial dK / dV
// sums to the workspace; km_split_reduce adds them up. (Packed 4k documents,
// a 1.7-wave grid: unsplit 839 us, two parts 857 us; packed 2k documents, 0.4
// waves: four parts 94 us, unsplit 134 us.)
int km_split_for(const Shape& sh, int n_sm) {
  const int C = km_cta_group(sh);
  const long long ctas = (long long)(((sh.S + 127) / 128 + C - 1) / C) * C * sh.Hk;
  const long long target = 4LL * n_sm;
  if (ctas >= n_sm) return 1;
  const long long n = target / ctas;
  return (int)(n < 1 ? 1 : (n > 4 ? 4 : n));
}
// The workspace holds the parts of the split a device with kWsSmBound SMs
// would take (km_split_for grows with the SM count), so that the workspace
// size depends on the shape alone; a device with more SMs than that is held
// to that split.
constexpr int kWsSmBound = 192;
int km_split_ws(const Shape& sh) { return km_split_for(sh, kWsSmBound); }
int km_split(const Shape& sh) {
  const int a = km_split_for(sh, sm_count()), b = km_split_ws(sh);
  return a < b ? a : b;
}
template <int D>
gqa_status km_launch(const float* Q, const float* K, const float* V, const float* dO,
                     const float* LSE, const uint32_t* seg, float* dK, float* dV, const float* Qt,
                     const float* dOt, long long ld_qt, const float4* kmeta, long long ld_meta,
                     const uint32_t* blk_minseg, const uint32_t* blk_maxseg, uint32_t* status,
                     const Shape& sh, cudaStream_t st, const RopeParams& rope, float* parts) {
  (void)LSE;
  (void)seg;   // both reach the key-major kernel through the column records
  const int n_split = km_split(sh);
  const uint4* bmax = reinterpret_cast<const uint4*>(blk_maxseg);   // 16-byte records
#define GQA_KM_ARGS Q, K, V, dO, dK, dV, Qt, dOt, ld_qt, kmeta, ld_meta, blk_minseg, bmax, status, sh, st, \
                    rope, n_split, parts
  if (km_cta_group(sh) == 2) {
    if constexpr (D == 128) {
      if (km_wide()) return km_launch_c<D, 2, true>(GQA_KM_ARGS);
    }
    return km_launch_c<D, 2, false>(GQA_KM_ARGS);
  }
  return km_launch_c<D, 1, false>(GQA_KM_ARGS);
#undef GQA_KM_ARGS
}

// Query-major form at d = 128 on SM pairs without a given D: the single
// pass (QmCfg::SP, the default) or the two passes (GQA_QM_TWO_PASS=1). Read
// once per process.
bool qm_single_pass() {
  static bool sp = [] {
    const char* e = getenv("GQA_QM_TWO_PASS");
    return !(e != nullptr && atoi(e) == 1);
  }();
  return sp;
}

template <int D, int C, bool GD, bool SP = false>
gqa_status qm_launch_c(const float* Q, const float* K, const float* V, const float* dO,
                       const float* LSE, const uint32_t* seg, float* dQ, const float* Kt,
                       long long ld_kt, const float* Kp, long long rows_kp, float4* kmeta,
                       long long ld_meta, float* Dws, float* Qt, float* dOt, long long ld_qt,
                       uint32_t* status, const Shape& sh, cudaStream_t st, const RopeParams& rope) {
  using Cfg = QmCfg<D, C, SP>;
  CUtensorMap mk, mv, mkt, mdq;
  gqa_status r;
  const long long kv_panels = (long long)sh.Hk * D / 32;
  // CYC: K chunks from K' (rows permuted within 64-key chunks, padded to rows_kp)
  if (Cfg::CYC && (Kp == nullptr || rows_kp < sh.S))
    return set_error(GQA_ERR_INVALID_ARG, "query-major: K' missing from the workspace");
  if ((r = map_panels(&mk, Cfg::CYC ? Kp : K, (long long)sh.Hk * D, Cfg::CYC ? rows_kp : sh.S, kv_panels,
                      Cfg::HALF1, D / 32)) != GQA_OK)
    return r;
  if ((r = map_panels(&mv, V, (long long)sh.Hk * D, sh.S, kv_panels, Cfg::HALF1, D / 32)) != GQA_OK) return r;
  if ((r = map_panels(&mkt, Kt, ld_kt, (long long)sh.Hk * D, ld_kt / 32, Cfg::KT_ROWS, Cfg::KT_PANELS)) != GQA_OK) return r;
  // the epilogue's reduce into dQ: one slab's (query, head) rows per box
  if ((r = map_heads(&mdq, dQ, D, sh.H, sh.S, sh.G, 128 / sh.G)) != GQA_OK) return r;
  if (cudaFuncSetAttribute(tc_query_major<D, C, GD, SP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg::SMEM_BYTES) != cudaSuccess)
    return check_launch("query-major smem attribute");
  const int QR = 128 / sh.G;
  const int n_slabs = (sh.S + QR - 1) / QR;
  const int n_sg = (n_slabs + C - 1) / C;
  // one CTA per SM (the kernel holds all of TMEM): slab-major below four waves
  const int slab_major = (long long)n_sg * C * sh.Hk < 4LL * sm_count() ? 1 : 0;
  const dim3 grid = slab_major ? dim3(C * sh.Hk, n_sg) : dim3(n_sg * C, sh.Hk);
  return launch_clustered(tc_query_major<D, C, GD, SP>, grid, C, Cfg::SMEM_BYTES, st,
                          "tensor-core query-major", mk, mv, mkt, mdq, Q, dO, LSE, seg, Dws, Qt, dOt,
                          ld_qt, kmeta, ld_meta, status, sh, rope, slab_major);
}

template <int D>
gqa_status qm_launch(const float* Q, const float* K, const float* V, const float* dO,
                     const float* LSE, const uint32_t* seg, float* dQ, const float* Kt,
                     long long ld_kt, const float* Kp, long long rows_kp, float4* kmeta,
                     long long ld_meta, float* Dws, float* Qt, float* dOt, long long ld_qt,
                     uint32_t* status, const Shape& sh, cudaStream_t st, const RopeParams& rope,
                     bool given_d) {
#define GQA_QM_ARGS Q, K, V, dO, LSE, seg, dQ, Kt, ld_kt, Kp, rows_kp, kmeta, ld_meta, Dws, Qt, dOt, ld_qt, \
                    status, sh, st, rope
  if (given_d) {
    if (cta_group() == 1) return qm_launch_c<D, 1, true>(GQA_QM_ARGS);
    return qm_launch_c<D, 2, true>(GQA_QM_ARGS);
  }
  if (cta_group() == 1) return qm_launch_c<D, 1, false>(GQA_QM_ARGS);
  if constexpr (QmCfg<D, 2>::CYC) {
    if (qm_single_pass()) return qm_launch_c<D, 2, false, true>(GQA_QM_ARGS);
  }
  return qm_launch_c<D, 2, false>(GQA_QM_ARGS);
#undef GQA_QM_ARGS
}

}  // namespace

gqa_status wait_selftest(void* workspace, long long limit_cycles, cudaStream_t st) {
  if (cudaMemsetAsync(workspace, 0, kWsHeader, st) != cudaSuccess)
    return check_launch("self-test status reset");
  wait_selftest_kernel<<<1, 32, 0, st>>>(reinterpret_cast<uint32_t*>(workspace), limit_cycles);
  note_launch();
  return check_launch("wait self-test");
}

gqa_status tc_map_panels(CUtensorMap* m, const float* base, long long ld, long long rows,
                         long long n_panels, int box_rows, int box_panels) {
  return map_panels(m, base, ld, rows, n_panels, box_rows, box_panels);
}

gqa_status tc_transpose(const float* X, float* Xt, int S, int Hk, int Gx, int d, long long ld,
                        cudaStream_t st) {
  return transpose_launch(X, Xt, S, Hk, Gx, d, ld, st);
}

TcWsLayout tc_ws_layout(int S, int H, int Hk, int d) {
  TcWsLayout t;
  const WsLayout base = ws_layout(S, H);
  const long long G = H / Hk;
  t.ld_kt = ((long long)S + 31) / 32 * 32;
  t.ld_qt = ((long long)S * G + 31) / 32 * 32;
  t.kt_off = base.total;
  t.qt_off = t.kt_off + align256((size_t)Hk * d * t.ld_kt * sizeof(float));
  t.dot_off = t.qt_off + align256((size_t)Hk * d * t.ld_qt * sizeof(float));
  t.blk_off = t.dot_off + align256((size_t)Hk * d * t.ld_qt * sizeof(float));
  t.blkmax_off = t.blk_off + align256((size_t)S * sizeof(uint32_t));
  // K' (rows permuted within 64-key chunks) for the query-major kernel at d = 128
  t.rows_kp = (d == 128) ? ((long long)S + 63) / 64 * 64 : 0;
  t.kp_off = t.blkmax_off + align256((size_t)S * 4 * sizeof(uint32_t));   // 16-byte max-seg records
  // the key-major kernel's per-column records (lse log2 e, scale D, query, seg)
  t.ld_meta = ((long long)S * G + 63) / 64 * 64;
  t.meta_off = t.kp_off + align256((size_t)t.rows_kp * Hk * d * sizeof(float));
  t.part_off = t.meta_off + align256((size_t)Hk * t.ld_meta * 4 * sizeof(float));
  // the key-major kernel's partial dK / dV when it splits its walk
  const Shape sh{S, H, Hk, d, (int)G, 1.f};
  const int n_split = tc_supported(sh) ? km_split_ws(sh) : 1;
  const size_t parts = n_split > 1 ? (size_t)2 * n_split * S * Hk * d * sizeof(float) : 0;
  t.total = t.part_off + align256(parts);
  return t;
}

bool tc_supported(const Shape& sh) {
  // G must divide the query-major slab (128 rows) and the key-major block
  // (NQ columns: 32 at d = 128, 64 below)
  const int nq = (sh.d == 128) ? KmCfg<128, 1>::NQ : KmCfg<64, 1>::NQ;
  return (sh.d == 32 || sh.d == 64 || sh.d == 128) && sh.G >= 1 && sh.G <= nq &&
         (nq % sh.G) == 0;
}

gqa_status tc_bwd(const float* Q, const float* K, const float* V, const float* dO,
                  const float* LSE, const uint32_t* seg, float* dQ, float* dK, float* dV,
                  const Shape& sh, char* ws, cudaStream_t st, const RopeParams& rope,
                  const float* O) {
  const WsLayout L = ws_layout(sh.S, sh.H);
  const TcWsLayout T = tc_ws_layout(sh.S, sh.H, sh.Hk, sh.d);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  float* Dws = reinterpret_cast<float*>(ws + L.d_off);
  float* Kt = reinterpret_cast<float*>(ws + T.kt_off);
  float* Qt = reinterpret_cast<float*>(ws + T.qt_off);
  float* dOt = reinterpret_cast<float*>(ws + T.dot_off);
  uint32_t* blk = reinterpret_cast<uint32_t*>(ws + T.blk_off);
  uint32_t* blk_max = reinterpret_cast<uint32_t*>(ws + T.blkmax_off);
  float* parts = reinterpret_cast<float*>(ws + T.part_off);
  const int QB = km_nq(sh) / sh.G;
  gqa_status r;
  float4* kmeta = reinterpret_cast<float4*>(ws + T.meta_off);
  // One launch: K^T and K' for the query-major kernel, and (its last z slice)
  // the per-block seg min / max records for the key-major one. Q^T, dO^T and
  // the column records are written by the query-major kernel itself.
  float* Kp = T.rows_kp > 0 ? reinterpret_cast<float*>(ws + T.kp_off) : nullptr;
  MinsegJob ms;
  ms.seg = seg;
  ms.tile = QB;
  ms.n_tiles = (sh.S + QB - 1) / QB;
  ms.out_min = blk;
  ms.out_max = reinterpret_cast<uint4*>(blk_max);
  if ((r = transpose_launch(K, Kt, sh.S, sh.Hk, 1, sh.d, T.ld_kt, st, Kp, T.rows_kp, ms)) != GQA_OK) return r;
  // with O given, D = rowsum(dO * O) replaces the query-major kernel's pass 1
  if (O != nullptr) {
    const long long rows = (long long)sh.S * sh.H;
    row_dot_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(dO, O, Dws, rows, sh.d);
    note_launch();
    if ((r = check_launch("row dot (D from O)")) != GQA_OK) return r;
  }
  profile_before(st, "tc_query_major+tc_key_major");
  switch (sh.d) {
    case 32:
      r = qm_launch<32>(Q, K, V, dO, LSE, seg, dQ, Kt, T.ld_kt, Kp, T.rows_kp, kmeta, T.ld_meta, Dws, Qt, dOt, T.ld_qt, status, sh, st, rope,
                        O != nullptr);
      if (r == GQA_OK)
        r = km_launch<32>(Q, K, V, dO, LSE, seg, dK, dV, Qt, dOt, T.ld_qt, kmeta, T.ld_meta, blk, blk_max, status, sh, st, rope,
                           parts);
      break;
    case 64:
      r = qm_launch<64>(Q, K, V, dO, LSE, seg, dQ, Kt, T.ld_kt, Kp, T.rows_kp, kmeta, T.ld_meta, Dws, Qt, dOt, T.ld_qt, status, sh, st, rope,
                        O != nullptr);
      if (r == GQA_OK)
        r = km_launch<64>(Q, K, V, dO, LSE, seg, dK, dV, Qt, dOt, T.ld_qt, kmeta, T.ld_meta, blk, blk_max, status, sh, st, rope,
                           parts);
      break;
    default:
      r = qm_launch<128>(Q, K, V, dO, LSE, seg, dQ, Kt, T.ld_kt, Kp, T.rows_kp, kmeta, T.ld_meta, Dws, Qt, dOt, T.ld_qt, status, sh, st, rope,
                        O != nullptr);
      if (r == GQA_OK)
        r = km_launch<128>(Q, K, V, dO, LSE, seg, dK, dV, Qt, dOt, T.ld_qt, kmeta, T.ld_meta, blk, blk_max, status, sh, st, rope,
                           parts);
      break;
  }
  profile_after(st);
  return r;
}

}  // namespace gqa
