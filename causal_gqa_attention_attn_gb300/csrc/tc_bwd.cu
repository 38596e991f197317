// Tensor-core backward (tcgen05, kind::tf32, fp32 accumulation in TMEM).
//
// Two kernels, both warp-specialised (TMA producer warp, MMA warp, four
// compute warps that own the 128 TMEM lanes), with every operand resident on
// chip:
//
//  tc_query_major (grid: query slabs x kv heads). A slab is 128 rows =
//    (128 / G) queries x the G query heads of one kv group, so the whole group
//    shares each K/V chunk. Q and dO of the slab sit in TMEM as the A operands;
//    K/V chunks of BK keys stream through a TMA ring (128-byte swizzle).
//    Pass 1 over the visible chunks: S = Q K^T, dP = dO V^T, D += rowsum(P dP)
//    (backward_attention.wgsl, attention_backward Pass A). Pass 2: the same
//    S, dP, then dS = scale P (dP - D) written back to TMEM over S and
//    dQ += dS K (Pass B), with B = the matching chunk of K^T (a transposed
//    copy of K in the workspace: the TF32 MMA reads both operands K-major).
//    dQ and D are owned writes (no atomics).
//
//  tc_key_major (grid: key tiles x kv heads): added below.
//
// Rows of a slab are ordered query-major: row r = (r / G)-th query, head
// g*G + r % G, which is also the memory order of Q / dO / dQ for a group.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdlib.h>

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
};

// ---------------------------------------------------------------------------
// Query-major configuration
// ---------------------------------------------------------------------------
template <int D_>
struct QmCfg {
  static constexpr int D = D_;
  static constexpr int BK = (D == 128) ? 32 : 64;          // keys per chunk
  static constexpr int PANELS = D / 32;
  static constexpr int PANEL_BYTES = BK * 128;             // BK rows x 32 floats
  static constexpr int TILE_BYTES = PANELS * PANEL_BYTES;  // one K or V chunk
  static constexpr int KT_PANELS = BK / 32;                // K^T chunk: d rows x BK keys
  static constexpr int KT_PANEL_BYTES = D * 128;
  static_assert(KT_PANELS * KT_PANEL_BYTES == TILE_BYTES, "K^T chunk size");
  static constexpr int SLOT_BYTES = 3 * TILE_BYTES;        // K, V, K^T
  static constexpr int NSLOT = (4 * SLOT_BYTES <= 200 * 1024) ? 4 : 3;
  // + alignment slack; at least 120 KB so that one CTA (holding all 512 TMEM
  // columns) runs per SM and a second never waits in tcgen05.alloc
  static constexpr int SMEM_BYTES =
      (NSLOT * SLOT_BYTES + 1024 > 120 * 1024) ? NSLOT * SLOT_BYTES + 1024 : 120 * 1024;
  // TMEM columns
  static constexpr uint32_t T_Q = 0, T_DO = D, T_DQ = 2 * D, T_ST = 3 * D;
  static constexpr uint32_t t_s(int st) { return T_ST + st * 2 * BK; }
  static constexpr uint32_t t_dp(int st) { return T_ST + st * 2 * BK + BK; }
  static_assert(3 * D + 4 * BK <= 512, "TMEM budget");
  static_assert(PANEL_BYTES % 1024 == 0, "panels must keep 1 KB swizzle alignment");
};

struct QmBarriers {
  uint64_t kv_full[4], kv_empty[4], s_full[2], s_free[2], qdo_ready, dq_done;
  uint32_t tmem_base;
  int abort;
  unsigned kmin;
  float dx[2][128];   // partial row sums of P dP from the two compute warpgroups
};

__device__ __forceinline__ uint32_t lane_base(uint32_t tmem, int warp) {
  return tmem + ((uint32_t)(32 * (warp & 3)) << 16);
}

template <int D, int C>
__global__ void __launch_bounds__(kThreads, 1)
    tc_query_major(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                   const __grid_constant__ CUtensorMap mapKt,
                   const float* __restrict__ Q, const float* __restrict__ dO,
                   const float* __restrict__ LSE, const uint32_t* __restrict__ seg,
                   float* __restrict__ dQ, float* __restrict__ Dws, uint32_t* __restrict__ status,
                   Shape sh) {
  using Cfg = QmCfg<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ QmBarriers bars;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = sh.G, QR = 128 / G;
  const int n_pad = gridDim.x;                           // slabs, padded to a multiple of C
  const int slab = n_pad - 1 - (int)blockIdx.x;          // longest rows first
  const uint32_t rank = (C > 1) ? cluster_ctarank() : 0u;
  const int top_slab = n_pad - 1 - ((int)blockIdx.x - (int)rank);   // cluster's last slab
  const uint16_t all_ctas = (uint16_t)((1u << C) - 1u);
  const int g = blockIdx.y;
  const int q0 = slab * QR;
  const int S = sh.S, H = sh.H;

  if (threadIdx.x == 0) {
    for (int i = 0; i < Cfg::NSLOT; ++i) {
      mbar_init(&bars.kv_full[i], kProducerWarps);   // each producer arms its own bytes
      mbar_init(&bars.kv_empty[i], C);      // every CTA of the cluster releases a slot
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.s_free[i], kComputeWarps / 2);   // one warpgroup per stage
    }
    mbar_init(&bars.qdo_ready, kComputeWarps);
    mbar_init(&bars.dq_done, 1);
    bars.abort = 0;
    bars.kmin = 0xffffffffu;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  // smallest document start over the cluster's queries -> first chunk; all
  // CTAs of a cluster walk the same chunk range (the union of their slabs')
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
  tc_fence_after();
  if (C > 1) cluster_sync();   // peers' barriers are initialised before any multicast
  const uint32_t tmem = bars.tmem_base;
  const int q_last = min(top_slab * QR + QR, S) - 1;
  const int kc0 = (int)(min(bars.kmin, (unsigned)q_last) / Cfg::BK);
  const int kc1 = q_last / Cfg::BK;
  const int nk = kc1 - kc0 + 1;
  const int total = 2 * nk;
  volatile int* abort = &bars.abort;

  // The producer and MMA warps run their loops with all 32 lanes (waits
  // included) so that addresses and descriptors are warp-uniform; one elected
  // lane issues each TMA / MMA / commit. Issuing from a single thread inside a
  // divergent branch cost 3-10x more cycles per MMA on this part.
  if (warp < kProducerWarps) {
    // ---------------- TMA producers: warp 0 loads K (and K^T in pass 2), warp 1 loads V ----------------
    const int pw = warp;
    if (elect_one()) {
      if (pw == 0) { tma_prefetch_desc(&mapK); tma_prefetch_desc(&mapKt); }
      else tma_prefetch_desc(&mapV);
    }
    __syncwarp();
    for (int c = 0; c < total; ++c) {
      const int slot = c % Cfg::NSLOT;
      if (c >= Cfg::NSLOT &&
          !warp_wait(&bars.kv_empty[slot], ((c / Cfg::NSLOT) - 1) & 1, abort, status, kSiteQmProducer))
        break;
      const int key0 = (kc0 + c % nk) * Cfg::BK;
      unsigned char* sk = smem + slot * Cfg::SLOT_BYTES;
      unsigned char* sv = sk + Cfg::TILE_BYTES;
      const bool pass2 = c >= nk;
      if (elect_one()) {
        const uint32_t bytes = (pw == 0) ? (pass2 ? 2 : 1) * Cfg::TILE_BYTES : Cfg::TILE_BYTES;
        mbar_arrive_expect_tx(&bars.kv_full[slot], bytes);
        // one box per tile (all its 128-byte panels); tile i of the chunk is
        // loaded by cluster rank i % C into every CTA
        auto load = [&](int i, void* dst, const CUtensorMap* m, int y, int z) {
          if (C == 1) tma_load_3d(dst, m, 0, y, z, &bars.kv_full[slot]);
          else if (i % C == (int)rank) tma_load_3d_mc(dst, m, 0, y, z, &bars.kv_full[slot], all_ctas);
        };
        if (pw == 0) {
          load(0, sk, &mapK, key0, g * Cfg::PANELS);
          if (pass2) load(2, sv + Cfg::TILE_BYTES, &mapKt, g * D, key0 / 32);
        } else {
          load(1, sv, &mapV, key0, g * Cfg::PANELS);
        }
      }
      __syncwarp();
    }
    // leave only once every load this CTA issued has landed
    for (int c = max(0, total - Cfg::NSLOT); c < total; ++c)
      warp_wait(&bars.kv_full[c % Cfg::NSLOT], (c / Cfg::NSLOT) & 1, abort, status, kSiteQmProducer);
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t id_s = idesc_tf32(128, Cfg::BK, false, false);   // S, dP: N = BK keys
    constexpr uint32_t id_q = idesc_tf32(128, D, false, false);         // dQ: N = d, B = K^T chunk
    bool ok = warp_wait(&bars.qdo_ready, 0, abort, status, kSiteQmMma);
    bool first_dq = true;
    const uint64_t desc0 = sdesc(smem_u32(smem), 16, 1024);
    // a slot is free once this CTA's MMAs that read it are done, in every CTA
    auto release = [&](int slot) {
      if (C == 1) mma_commit(&bars.kv_empty[slot]);
      else mma_commit_mc(&bars.kv_empty[slot], all_ctas);
    };
    auto issue_dq = [&](int cc) -> bool {
      const int st = cc & 1, slot = cc % Cfg::NSLOT;
      if (!warp_wait(&bars.s_free[st], (cc / 2) & 1, abort, status, kSiteQmMma)) return false;
      const uint64_t bkt = desc0 + (uint64_t)((slot * Cfg::SLOT_BYTES + 2 * Cfg::TILE_BYTES) >> 4);
      const uint32_t a_ds = tmem + Cfg::t_s(st), d_q = tmem + Cfg::T_DQ;
      const uint32_t acc0 = first_dq ? 0u : 1u;
      if (elect_one()) {
        tc_fence_after();
        mma_ts(d_q, a_ds, bkt, id_q, acc0);
#pragma unroll
        for (int kk = 1; kk < Cfg::BK / 8; ++kk)
          mma_ts_acc(d_q, a_ds + 8 * kk, bkt + desc_off(kk, Cfg::KT_PANEL_BYTES), id_q);
        release(slot);
      }
      __syncwarp();
      first_dq = false;
      return true;
    };
    for (int c = 0; ok && c < total; ++c) {
      const int slot = c % Cfg::NSLOT, st = c & 1;
      const bool pass2 = c >= nk;
      if (!warp_wait(&bars.kv_full[slot], (c / Cfg::NSLOT) & 1, abort, status, kSiteQmMma)) break;
      if (c >= 2 && !warp_wait(&bars.s_free[st], ((c - 2) / 2) & 1, abort, status, kSiteQmMma))
        break;
      const uint64_t bk = desc0 + (uint64_t)((slot * Cfg::SLOT_BYTES) >> 4);
      const uint64_t bv = bk + ((uint64_t)Cfg::TILE_BYTES >> 4);
      const uint32_t d_s = tmem + Cfg::t_s(st), d_dp = tmem + Cfg::t_dp(st);
      const uint32_t a_q = tmem + Cfg::T_Q, a_do = tmem + Cfg::T_DO;
      if (elect_one()) {
        tc_fence_after();
        mma_ts(d_s, a_q, bk, id_s, 0u);
        mma_ts(d_dp, a_do, bv, id_s, 0u);
#pragma unroll
        for (int ks = 1; ks < D / 8; ++ks) {
          const uint64_t off = desc_off(ks, Cfg::PANEL_BYTES);
          mma_ts_acc(d_s, a_q + 8 * ks, bk + off, id_s);
          mma_ts_acc(d_dp, a_do + 8 * ks, bv + off, id_s);
        }
        mma_commit(&bars.s_full[st]);
        if (!pass2) release(slot);
      }
      __syncwarp();
      if (pass2 && c > nk && !issue_dq(c - 1)) { ok = false; break; }
    }
    if (ok) ok = issue_dq(total - 1);
    if (elect_one()) mma_commit(&bars.dq_done);     // also drains every MMA issued above
    __syncwarp();
  } else {
    // ---------------- compute: two warpgroups, one TMEM lane (= one row) per thread ----------------
    // Warpgroup wg handles the chunks that use TMEM stage wg (c % 2 == wg), so
    // two chunks are in flight at once; each keeps a partial row sum of P dP
    // over its pass-1 chunks, and the two partials are added through shared
    // memory before the first dS is formed.
    const int wg = (warp - kFirstCompute) >> 2;
    const int r = 32 * (warp & 3) + lane;
    const int qi = r / G, q = q0 + qi;
    const int h = g * G + r % G;
    const bool valid = q < S;
    const uint32_t tl = lane_base(tmem, warp);
    const long long row_off = (long long)q * H * D + (long long)h * D;
    // Q (warpgroup 0) or dO (warpgroup 1) rows into TMEM, rounded to TF32:
    // the A operands of S and dP
    {
      const float* src = (wg == 0) ? Q : dO;
      const uint32_t col0 = (wg == 0) ? Cfg::T_Q : Cfg::T_DO;
      float v[32];
      for (int cc = 0; cc < D; cc += 32) {
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          float4 x = valid ? __ldg(reinterpret_cast<const float4*>(src + row_off + cc + i))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
          v[i] = to_tf32(x.x); v[i + 1] = to_tf32(x.y); v[i + 2] = to_tf32(x.z); v[i + 3] = to_tf32(x.w);
        }
        tmem_st32(tl + col0 + cc, v);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.qdo_ready);
    }
    const float sl2 = sh.scale * kLog2e;
    const float lse2 = valid ? __ldg(LSE + (long long)q * H + h) * kLog2e : 0.f;
    const int segq = valid ? (int)__ldg(seg + q) : 0;
    float Dpart = 0.f, Drow = 0.f;
    bool have_D = false, ok = true;
    auto combine_D = [&]() {
      bars.dx[wg][r] = Dpart;
      asm volatile("bar.sync 2, 256;" ::: "memory");
      Drow = bars.dx[0][r] + bars.dx[1][r];
      have_D = true;
    };
    const uint32_t ts = tl + Cfg::t_s(wg), tdp = tl + Cfg::t_dp(wg);
    for (int c = wg; c < total; c += 2) {
      const bool pass2 = c >= nk;
      if (pass2 && !have_D) combine_D();
      const int k0 = (kc0 + c % nk) * Cfg::BK;
      if (!mbar_wait(&bars.s_full[wg], (c / 2) & 1, abort, status, kSiteQmCompute)) { ok = false; break; }
      tc_fence_after();
      // every key of the chunk visible to this row: no per-element mask
      const bool full = valid && k0 >= segq && k0 + Cfg::BK - 1 <= q;
#pragma unroll
      for (int jb = 0; jb < Cfg::BK; jb += 32) {
        float sv[32], dp[32];
        tmem_ld32(ts + jb, sv);
        tmem_ld32(tdp + jb, dp);
        tmem_ld_wait();
        if (!pass2) {
          if (full) {
#pragma unroll
            for (int j = 0; j < 32; ++j) Dpart = fmaf(ex2(fmaf(sv[j], sl2, -lse2)), dp[j], Dpart);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int key = k0 + jb + j;
              const bool vis = valid && key >= segq && key <= q;
              Dpart = fmaf(vis ? ex2(fmaf(sv[j], sl2, -lse2)) : 0.f, dp[j], Dpart);
            }
          }
        } else {
          if (full) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              sv[j] = to_tf32(sh.scale * ex2(fmaf(sv[j], sl2, -lse2)) * (dp[j] - Drow));
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int key = k0 + jb + j;
              const bool vis = valid && key >= segq && key <= q;
              const float pj = vis ? ex2(fmaf(sv[j], sl2, -lse2)) : 0.f;
              sv[j] = to_tf32(sh.scale * pj * (dp[j] - Drow));
            }
          }
          tmem_st32(ts + jb, sv);
        }
      }
      if (pass2) tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.s_free[wg]);
    }
    if (!have_D) combine_D();   // a warpgroup without pass-2 chunks still joins the exchange
    // epilogue: dQ += accumulated tile (warpgroup wg: half wg of the columns), D to the workspace
    if (ok && mbar_wait(&bars.dq_done, 0, abort, status, kSiteQmCompute)) {
      tc_fence_after();
      for (int cc = wg * (D / 2); cc < (wg + 1) * (D / 2); cc += 16) {
        float v[16];
        tmem_ld16(tl + Cfg::T_DQ + cc, v);
        tmem_ld_wait();
        if (valid) {
          float4* dst = reinterpret_cast<float4*>(dQ + row_off + cc);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float4 o = dst[i];
            o.x += (v[4 * i] == v[4 * i]) ? v[4 * i] : 0.f;
            o.y += (v[4 * i + 1] == v[4 * i + 1]) ? v[4 * i + 1] : 0.f;
            o.z += (v[4 * i + 2] == v[4 * i + 2]) ? v[4 * i + 2] : 0.f;
            o.w += (v[4 * i + 3] == v[4 * i + 3]) ? v[4 * i + 3] : 0.f;
            dst[i] = o;
          }
        }
      }
      if (valid && wg == 0) Dws[(long long)q * H + h] = Drow;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
  if (C > 1) cluster_sync();   // no CTA leaves while a peer may still signal it
}

// ---------------------------------------------------------------------------
// Key-major kernel: dK and dV for 128 keys of one kv head, summed over the
// query heads of its group (no atomics: the CTA owns these rows).
//
// Per (query, head) block of NQ rows (NQ/G queries x G heads):
//   S^T  = K . Q^T        A = K (TMEM, loaded once),   B = Q block   (smem)
//   dP^T = V . dO^T       A = V (smem, loaded once),   B = dO block  (smem)
//   P^T, dS^T = scale P (dP - D) written back to TMEM over S^T / dP^T
//   dV  += P^T . dO       A = P^T (TMEM),  B = dO^T block (smem, K-major copy)
//   dK  += dS^T . Q       A = dS^T (TMEM), B = Q^T block  (smem, K-major copy)
// The four streamed tiles each have a full/empty barrier pair, so the next
// block's Q/dO load while dV/dK of this block run, and its Q^T/dO^T load
// while its S^T/dP^T run. Blocks are visited from the end of the sequence
// down to the tile's first query: CTAs that run at the same time then read
// the same blocks at about the same time, so the per-group Q / dO / Q^T /
// dO^T stream (larger than L2 at 16k tokens) is served mostly from L2.
// ---------------------------------------------------------------------------
template <int D_>
struct KmCfg {
  static constexpr int D = D_;
  static constexpr int NQ = (D == 128) ? 64 : 128;        // (query, head) rows per block
  static constexpr int V_PANEL_BYTES = 128 * 128;         // 128 keys x 32 floats
  static constexpr int V_BYTES = (D / 32) * V_PANEL_BYTES;
  static constexpr int BLK_PANEL_BYTES = NQ * 128;        // Q / dO block panel: NQ rows x 32 floats
  static constexpr int BLK_BYTES = (D / 32) * BLK_PANEL_BYTES;
  static constexpr int T_PANEL_BYTES = D * 128;           // Q^T / dO^T panel: d rows x 32 columns
  static constexpr int T_PANELS = NQ / 32;
  static_assert(T_PANELS * T_PANEL_BYTES == BLK_BYTES, "transposed block size");
  // shared memory: V | Q | dO | Q^T | dO^T
  static constexpr int OFF_V = 0, OFF_Q = V_BYTES, OFF_DO = OFF_Q + BLK_BYTES,
                       OFF_QT = OFF_DO + BLK_BYTES, OFF_DOT = OFF_QT + BLK_BYTES,
                       END = OFF_DOT + BLK_BYTES;
  static constexpr int SMEM_BYTES = (END + 1024 > 120 * 1024) ? END + 1024 : 120 * 1024;
  // TMEM columns
  static constexpr uint32_t T_K = 0, T_DK = D, T_DV = 2 * D, T_S = 3 * D, T_DP = 3 * D + NQ;
  static_assert(3 * D + 2 * NQ <= 512, "TMEM budget");
};

struct KmBarriers {
  uint64_t v_full, k_ready;
  uint64_t full[4], empty[4];     // Q, dO, Q^T, dO^T blocks
  uint64_t s_full, p_ready, acc_done;
  uint32_t tmem_base;
  int abort;
};

template <int D, int C>
__global__ void __launch_bounds__(kThreads, 1)
    tc_key_major(const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapQ,
                 const __grid_constant__ CUtensorMap mapDO, const __grid_constant__ CUtensorMap mapQt,
                 const __grid_constant__ CUtensorMap mapDOt, const float* __restrict__ K,
                 const float* __restrict__ LSE, const float* __restrict__ Dws,
                 const uint32_t* __restrict__ seg, const uint32_t* __restrict__ blk_minseg,
                 const uint32_t* __restrict__ blk_maxseg, float* __restrict__ dK,
                 float* __restrict__ dV, uint32_t* __restrict__ status, Shape sh) {
  using Cfg = KmCfg<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ KmBarriers bars;
  __shared__ float4 meta[2][Cfg::NQ];     // per block column: (lse*log2e, D, query, seg)
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = sh.G, QB = Cfg::NQ / G;   // queries per block
  const int S = sh.S, H = sh.H;
  const int k0 = blockIdx.x * 128, g = blockIdx.y;
  const uint32_t rank = (C > 1) ? cluster_ctarank() : 0u;
  const uint16_t all_ctas = (uint16_t)((1u << C) - 1u);
  // all CTAs of a cluster (adjacent key tiles) walk the union of their blocks
  const int k0_first = ((int)blockIdx.x - (int)rank) * 128;
  const int k_hi = min(k0_first + 128 * C, S) - 1;
  const int qb0 = k0_first / QB, nqb = (S + QB - 1) / QB;

  if (threadIdx.x == 0) {
    mbar_init(&bars.v_full, 1);
    mbar_init(&bars.k_ready, kComputeWarps);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars.full[i], 1);
      mbar_init(&bars.empty[i], C);       // every CTA of the cluster releases a tile
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.p_ready, kComputeWarps);
    mbar_init(&bars.acc_done, 1);
    bars.abort = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (C > 1) cluster_sync();   // peers' barriers are initialised before any multicast
  const uint32_t tmem = bars.tmem_base;
  volatile int* abort = &bars.abort;
  auto visible = [&](int qb) { return __ldg(blk_minseg + qb) <= (unsigned)k_hi; };

  if (warp < kProducerWarps) {
    // ---------------- TMA producers: warp 0 loads Q and Q^T, warp 1 dO, dO^T and V ----------------
    const int pw = warp;
    const CUtensorMap* maps[4] = {&mapQ, &mapDO, &mapQt, &mapDOt};
    if (elect_one()) {
      tma_prefetch_desc(maps[pw]);
      tma_prefetch_desc(maps[pw + 2]);
      if (pw == 1) {
        tma_prefetch_desc(&mapV);
        mbar_arrive_expect_tx(&bars.v_full, Cfg::V_BYTES);
        tma_load_3d(smem + Cfg::OFF_V, &mapV, 0, k0, g * (D / 32), &bars.v_full);
      }
    }
    __syncwarp();
    const int offs[4] = {Cfg::OFF_Q, Cfg::OFF_DO, Cfg::OFF_QT, Cfg::OFF_DOT};
    int n = 0;
    bool ok = true;
    for (int qb = nqb - 1; ok && qb >= qb0; --qb) {
      if (!visible(qb)) continue;
      const int q0 = qb * QB;
      // one box per tile; tile t is loaded by cluster rank t % C into every CTA
      for (int t = pw; t < 4; t += 2) {
        if (n > 0 && !warp_wait(&bars.empty[t], (n - 1) & 1, abort, status, kSiteKmProducer)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          mbar_arrive_expect_tx(&bars.full[t], Cfg::BLK_BYTES);
          if (C == 1 || t % C == (int)rank) {
            unsigned char* dst = smem + offs[t];
            if (t < 2) {          // Q / dO block: 4-D box (32 dims, G heads, QB queries, d/32 panels)
              if (C == 1) tma_load_4d(dst, maps[t], 0, g * G, q0, 0, &bars.full[t]);
              else tma_load_4d_mc(dst, maps[t], 0, g * G, q0, 0, &bars.full[t], all_ctas);
            } else {              // Q^T / dO^T block: d rows x NQ (query, head) columns, in panels
              if (C == 1) tma_load_3d(dst, maps[t], 0, g * D, (q0 * G) / 32, &bars.full[t]);
              else tma_load_3d_mc(dst, maps[t], 0, g * D, (q0 * G) / 32, &bars.full[t], all_ctas);
            }
          }
        }
        __syncwarp();
      }
      ++n;
    }
    // leave only once every load this warp issued has landed
    if (pw == 1) warp_wait(&bars.v_full, 0, abort, status, kSiteKmProducer);
    if (n > 0)
      for (int t = pw; t < 4; t += 2) warp_wait(&bars.full[t], (n - 1) & 1, abort, status, kSiteKmProducer);
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer (warp-converged, elected issue) ----------------
    constexpr uint32_t id_s = idesc_tf32(128, Cfg::NQ, false, false);
    constexpr uint32_t id_g = idesc_tf32(128, D, false, false);
    bool ok = warp_wait(&bars.v_full, 0, abort, status, kSiteKmMma) &&
              warp_wait(&bars.k_ready, 0, abort, status, kSiteKmMma);
    auto release = [&](int t) {     // tile t is free once every CTA's MMAs read it
      if (C == 1) mma_commit(&bars.empty[t]);
      else mma_commit_mc(&bars.empty[t], all_ctas);
    };
    const uint64_t desc0 = sdesc(smem_u32(smem), 16, 1024);
    const uint64_t av = desc0 + (uint64_t)(Cfg::OFF_V >> 4), bq = desc0 + (uint64_t)(Cfg::OFF_Q >> 4),
                   bdo = desc0 + (uint64_t)(Cfg::OFF_DO >> 4),
                   bqt = desc0 + (uint64_t)(Cfg::OFF_QT >> 4),
                   bdot = desc0 + (uint64_t)(Cfg::OFF_DOT >> 4);
    int n = 0;
    for (int qb = nqb - 1; ok && qb >= qb0; --qb) {
      if (!visible(qb)) continue;
      const uint32_t par = n & 1;
      if (!warp_wait(&bars.full[0], par, abort, status, kSiteKmMma) ||
          !warp_wait(&bars.full[1], par, abort, status, kSiteKmMma)) { ok = false; break; }
      if (elect_one()) {
        tc_fence_after();
        mma_ts(tmem + Cfg::T_S, tmem + Cfg::T_K, bq, id_s, 0u);
        mma_ss(tmem + Cfg::T_DP, av, bdo, id_s, 0u);
#pragma unroll
        for (int ks = 1; ks < D / 8; ++ks) {
          const uint64_t ob = desc_off(ks, Cfg::BLK_PANEL_BYTES);
          mma_ts_acc(tmem + Cfg::T_S, tmem + Cfg::T_K + 8 * ks, bq + ob, id_s);
          mma_ss_acc(tmem + Cfg::T_DP, av + desc_off(ks, Cfg::V_PANEL_BYTES), bdo + ob, id_s);
        }
        mma_commit(&bars.s_full);
        release(0);
        release(1);
      }
      __syncwarp();
      if (!warp_wait(&bars.p_ready, par, abort, status, kSiteKmMma) ||
          !warp_wait(&bars.full[2], par, abort, status, kSiteKmMma) ||
          !warp_wait(&bars.full[3], par, abort, status, kSiteKmMma)) { ok = false; break; }
      const uint32_t acc0 = (n > 0) ? 1u : 0u;
      if (elect_one()) {
        tc_fence_after();
        mma_ts(tmem + Cfg::T_DV, tmem + Cfg::T_S, bdot, id_g, acc0);
        mma_ts(tmem + Cfg::T_DK, tmem + Cfg::T_DP, bqt, id_g, acc0);
#pragma unroll
        for (int kk = 1; kk < Cfg::NQ / 8; ++kk) {
          const uint64_t ot = desc_off(kk, Cfg::T_PANEL_BYTES);
          mma_ts_acc(tmem + Cfg::T_DV, tmem + Cfg::T_S + 8 * kk, bdot + ot, id_g);
          mma_ts_acc(tmem + Cfg::T_DK, tmem + Cfg::T_DP + 8 * kk, bqt + ot, id_g);
        }
        release(2);
        release(3);
      }
      __syncwarp();
      ++n;
    }
    if (elect_one()) mma_commit(&bars.acc_done);
    __syncwarp();
  } else {
    // ---------------- compute: thread = key (TMEM lane); warpgroup wg owns half the columns ----------------
    const int wg = (warp - kFirstCompute) >> 2;
    const int r = 32 * (warp & 3) + lane;
    const int key = k0 + r;
    const uint32_t tl = lane_base(tmem, warp);
    const int ct = threadIdx.x - 32 * kFirstCompute;       // 0..255 among compute threads
    {
      float v[16];
      const float* krow = K + (long long)key * sh.Hk * D + (long long)g * D;
      for (int cc = wg * (D / 2); cc < (wg + 1) * (D / 2); cc += 16) {   // D/2 >= 16
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          float4 x = (key < S) ? __ldg(reinterpret_cast<const float4*>(krow + cc + i))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
          v[i] = to_tf32(x.x); v[i + 1] = to_tf32(x.y); v[i + 2] = to_tf32(x.z); v[i + 3] = to_tf32(x.w);
        }
        tmem_st16(tl + Cfg::T_K + cc, v);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.k_ready);
    }
    const float sl2 = sh.scale * kLog2e;
    constexpr int HALF = Cfg::NQ / 2;
    const int cbase = wg * HALF;
    int n = 0;
    bool ok = true;
    for (int qb = nqb - 1; qb >= qb0; --qb) {
      if (!visible(qb)) continue;
      // column metadata of this block (double-buffered; one named barrier per block)
      if (ct < Cfg::NQ) {
        const int q = qb * QB + ct / G, h = g * G + ct % G;
        float4 m = make_float4(0.f, 0.f, __int_as_float(-1), __int_as_float(0x7fffffff));
        if (q < S)
          m = make_float4(__ldg(LSE + (long long)q * H + h) * kLog2e, Dws[(long long)q * H + h],
                          __int_as_float(q), __int_as_float((int)__ldg(seg + q)));
        meta[n & 1][ct] = m;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (!mbar_wait(&bars.s_full, n & 1, abort, status, kSiteKmCompute)) { ok = false; break; }
      tc_fence_after();
      // every (key, column) of the block visible: key <= first query and >= every seg
      const int q_first = qb * QB;
      const bool full = key <= q_first && key >= (int)__ldg(blk_maxseg + qb) &&
                        q_first + QB - 1 < S;
#pragma unroll
      for (int cb = 0; cb < HALF; cb += 32) {
        float sv[32], dp[32];
        tmem_ld32(tl + Cfg::T_S + cbase + cb, sv);
        tmem_ld32(tl + Cfg::T_DP + cbase + cb, dp);
        tmem_ld_wait();
        if (full) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float4 m = meta[n & 1][cbase + cb + j];
            const float pj = ex2(fmaf(sv[j], sl2, -m.x));
            sv[j] = to_tf32(pj);
            dp[j] = to_tf32(sh.scale * pj * (dp[j] - m.y));
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float4 m = meta[n & 1][cbase + cb + j];
            const int q = __float_as_int(m.z), sq = __float_as_int(m.w);
            const bool vis = key <= q && key >= sq;        // q = -1 for padding columns
            const float pj = vis ? ex2(fmaf(sv[j], sl2, -m.x)) : 0.f;
            sv[j] = to_tf32(pj);
            dp[j] = to_tf32(sh.scale * pj * (dp[j] - m.y));
          }
        }
        tmem_st32(tl + Cfg::T_S + cbase + cb, sv);
        tmem_st32(tl + Cfg::T_DP + cbase + cb, dp);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.p_ready);
      ++n;
    }
    // epilogue: warpgroup 0 adds dK, warpgroup 1 adds dV (owned rows)
    if (ok && mbar_wait(&bars.acc_done, 0, abort, status, kSiteKmCompute)) {
      tc_fence_after();
      const long long row = (long long)key * sh.Hk * D + (long long)g * D;
      float* dst_row = (wg == 0 ? dK : dV) + row;
      const uint32_t src = tl + (wg == 0 ? Cfg::T_DK : Cfg::T_DV);
      for (int cc = 0; cc < D; cc += 32) {
        float a[32];
        tmem_ld32(src + cc, a);
        tmem_ld_wait();
        if (key < S && n > 0) {
          float4* pk = reinterpret_cast<float4*>(dst_row + cc);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float4 o = pk[i];
            o.x += (a[4 * i] == a[4 * i]) ? a[4 * i] : 0.f;
            o.y += (a[4 * i + 1] == a[4 * i + 1]) ? a[4 * i + 1] : 0.f;
            o.z += (a[4 * i + 2] == a[4 * i + 2]) ? a[4 * i + 2] : 0.f;
            o.w += (a[4 * i + 3] == a[4 * i + 3]) ? a[4 * i + 3] : 0.f;
            pk[i] = o;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
  if (C > 1) cluster_sync();   // no CTA leaves while a peer may still signal it
}

// ---------------------------------------------------------------------------
// Group transpose: X [S][Hk*Gx][d] (row-major, head h = g*Gx + h') to
// Xt [Hk*d][ld] with Xt[g*d + e][q*Gx + h'] = X[q][(g*Gx + h')*d + e].
// With Gx = 1 this is K^T per kv head; with Gx = G it lays the (query, head)
// rows of a kv group out as the contiguous K dimension of a K-major operand.
// ld is S*Gx rounded up to 32; the grid covers all ld columns.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) group_transpose(const float* __restrict__ X,
                                                       float* __restrict__ Xt, int S, int Hk,
                                                       int Gx, int d, long long ld) {
  __shared__ float tile[32][33];
  const int g = blockIdx.z, e0 = blockIdx.y * 32;
  const long long r0 = (long long)blockIdx.x * 32, nrows = (long long)S * Gx;
  const long long row_stride = (long long)Hk * Gx * d;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const long long r = r0 + i;
    float v = 0.f;
    if (r < nrows) {
      const long long q = r / Gx, hh = r % Gx;
      v = __ldg(X + q * row_stride + (g * Gx + hh) * d + e0 + threadIdx.x);
    }
    tile[i][threadIdx.x] = v;
  }
  __syncthreads();
  // columns nrows .. ld-1 are padding: written as zeros (the panel view of
  // the copy reads them as ordinary elements, masked to zero weight)
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const long long r = r0 + threadIdx.x;
    if (r < ld) Xt[(long long)(g * d + e0 + i) * ld + r] = tile[threadIdx.x][i];
  }
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
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
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
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  note_launch();
  if (e != cudaSuccess) return set_error(GQA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return check_launch(what);
}

// Cluster size for the streamed-operand multicast (1, 2 or 4; default 1:
// measured on the 16k workload, 2 and 4 gave no gain). GQA_TC_CLUSTER
// overrides it (tuning).
int cluster_size() {
  static int c = [] {
    const char* e = getenv("GQA_TC_CLUSTER");
    const int v = e ? atoi(e) : 1;
    return (v == 1 || v == 2 || v == 4) ? v : 1;
  }();
  return c;
}

template <int D, int C>
gqa_status km_launch_c(const CUtensorMap& mv, const CUtensorMap& mq, const CUtensorMap& mdo,
                       const CUtensorMap& mqt, const CUtensorMap& mdot, const float* K,
                       const float* LSE, const float* Dws, const uint32_t* seg,
                       const uint32_t* blk_minseg, const uint32_t* blk_maxseg, float* dK,
                       float* dV, uint32_t* status, const Shape& sh, cudaStream_t st) {
  using Cfg = KmCfg<D>;
  if (cudaFuncSetAttribute(tc_key_major<D, C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg::SMEM_BYTES) != cudaSuccess)
    return check_launch("key-major smem attribute");
  const int n_tiles = (sh.S + 127) / 128;
  dim3 grid((n_tiles + C - 1) / C * C, sh.Hk);
  return launch_clustered(tc_key_major<D, C>, grid, C, Cfg::SMEM_BYTES, st, "tensor-core key-major",
                          mv, mq, mdo, mqt, mdot, K, LSE, Dws, seg, blk_minseg, blk_maxseg, dK, dV,
                          status, sh);
}

template <int D>
gqa_status km_launch(const float* Q, const float* K, const float* V, const float* dO,
                     const float* LSE, const uint32_t* seg, float* dK, float* dV, const float* Qt,
                     const float* dOt, long long ld_qt, const float* Dws, const uint32_t* blk_minseg,
                     const uint32_t* blk_maxseg, uint32_t* status, const Shape& sh,
                     cudaStream_t st) {
  using C = KmCfg<D>;
  const int QB = C::NQ / sh.G;
  CUtensorMap mv, mq, mdo, mqt, mdot;
  gqa_status r;
  const long long kv_panels = (long long)sh.Hk * D / 32;
  if ((r = map_panels(&mv, V, (long long)sh.Hk * D, sh.S, kv_panels, 128, D / 32)) != GQA_OK) return r;
  if ((r = map_heads(&mq, Q, D, sh.H, sh.S, sh.G, QB)) != GQA_OK) return r;
  if ((r = map_heads(&mdo, dO, D, sh.H, sh.S, sh.G, QB)) != GQA_OK) return r;
  if ((r = map_panels(&mqt, Qt, ld_qt, (long long)sh.Hk * D, ld_qt / 32, D, C::T_PANELS)) != GQA_OK) return r;
  if ((r = map_panels(&mdot, dOt, ld_qt, (long long)sh.Hk * D, ld_qt / 32, D, C::T_PANELS)) != GQA_OK) return r;
  switch (cluster_size()) {
    case 1: return km_launch_c<D, 1>(mv, mq, mdo, mqt, mdot, K, LSE, Dws, seg, blk_minseg, blk_maxseg, dK, dV, status, sh, st);
    case 4: return km_launch_c<D, 4>(mv, mq, mdo, mqt, mdot, K, LSE, Dws, seg, blk_minseg, blk_maxseg, dK, dV, status, sh, st);
    default: return km_launch_c<D, 2>(mv, mq, mdo, mqt, mdot, K, LSE, Dws, seg, blk_minseg, blk_maxseg, dK, dV, status, sh, st);
  }
}

gqa_status transpose_launch(const float* X, float* Xt, int S, int Hk, int Gx, int d, long long ld,
                            cudaStream_t st) {
  const long long nrows = (long long)S * Gx;
  dim3 grid((unsigned)((nrows + 31) / 32), d / 32, Hk);
  group_transpose<<<grid, dim3(32, 8), 0, st>>>(X, Xt, S, Hk, Gx, d, ld);
  note_launch();
  return check_launch("group transpose");
}

template <int D, int C>
gqa_status qm_launch_c(const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mkt,
                       const float* Q, const float* dO, const float* LSE, const uint32_t* seg,
                       float* dQ, float* Dws, uint32_t* status, const Shape& sh, cudaStream_t st) {
  using Cfg = QmCfg<D>;
  if (cudaFuncSetAttribute(tc_query_major<D, C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg::SMEM_BYTES) != cudaSuccess)
    return check_launch("query-major smem attribute");
  const int QR = 128 / sh.G;
  const int n_slabs = (sh.S + QR - 1) / QR;
  dim3 grid((n_slabs + C - 1) / C * C, sh.Hk);
  return launch_clustered(tc_query_major<D, C>, grid, C, Cfg::SMEM_BYTES, st,
                          "tensor-core query-major", mk, mv, mkt, Q, dO, LSE, seg, dQ, Dws, status,
                          sh);
}

template <int D>
gqa_status qm_launch(const float* Q, const float* K, const float* V, const float* dO,
                     const float* LSE, const uint32_t* seg, float* dQ, const float* Kt,
                     long long ld_kt, float* Dws, uint32_t* status, const Shape& sh,
                     cudaStream_t st) {
  using C = QmCfg<D>;
  CUtensorMap mk, mv, mkt;
  gqa_status r;
  const long long kv_panels = (long long)sh.Hk * D / 32;
  if ((r = map_panels(&mk, K, (long long)sh.Hk * D, sh.S, kv_panels, C::BK, D / 32)) != GQA_OK) return r;
  if ((r = map_panels(&mv, V, (long long)sh.Hk * D, sh.S, kv_panels, C::BK, D / 32)) != GQA_OK) return r;
  if ((r = map_panels(&mkt, Kt, ld_kt, (long long)sh.Hk * D, ld_kt / 32, D, C::KT_PANELS)) != GQA_OK) return r;
  switch (cluster_size()) {
    case 1: return qm_launch_c<D, 1>(mk, mv, mkt, Q, dO, LSE, seg, dQ, Dws, status, sh, st);
    case 4: return qm_launch_c<D, 4>(mk, mv, mkt, Q, dO, LSE, seg, dQ, Dws, status, sh, st);
    default: return qm_launch_c<D, 2>(mk, mv, mkt, Q, dO, LSE, seg, dQ, Dws, status, sh, st);
  }
}

}  // namespace

gqa_status wait_selftest(void* workspace, long long limit_cycles, cudaStream_t st) {
  if (cudaMemsetAsync(workspace, 0, kWsHeader, st) != cudaSuccess)
    return check_launch("self-test status reset");
  wait_selftest_kernel<<<1, 32, 0, st>>>(reinterpret_cast<uint32_t*>(workspace), limit_cycles);
  note_launch();
  return check_launch("wait self-test");
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
  t.total = t.blkmax_off + align256((size_t)S * sizeof(uint32_t));
  return t;
}

bool tc_supported(const Shape& sh) {
  // G must divide the 128-row slab and the key-major (query, head) block
  const int nq = (sh.d == 128) ? 64 : 128;
  return (sh.d == 32 || sh.d == 64 || sh.d == 128) && sh.G >= 1 && sh.G <= nq &&
         (nq % sh.G) == 0;
}

gqa_status tc_bwd(const float* Q, const float* K, const float* V, const float* dO,
                  const float* LSE, const uint32_t* seg, float* dQ, float* dK, float* dV,
                  const Shape& sh, char* ws, cudaStream_t st) {
  const WsLayout L = ws_layout(sh.S, sh.H);
  const TcWsLayout T = tc_ws_layout(sh.S, sh.H, sh.Hk, sh.d);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  float* Dws = reinterpret_cast<float*>(ws + L.d_off);
  float* Kt = reinterpret_cast<float*>(ws + T.kt_off);
  float* Qt = reinterpret_cast<float*>(ws + T.qt_off);
  float* dOt = reinterpret_cast<float*>(ws + T.dot_off);
  uint32_t* blk = reinterpret_cast<uint32_t*>(ws + T.blk_off);
  uint32_t* blk_max = reinterpret_cast<uint32_t*>(ws + T.blkmax_off);
  const int QB = ((sh.d == 128) ? 64 : 128) / sh.G;
  gqa_status r;
  if ((r = tile_minseg(seg, sh.S, QB, blk, st, blk_max)) != GQA_OK) return r;
  if ((r = transpose_launch(K, Kt, sh.S, sh.Hk, 1, sh.d, T.ld_kt, st)) != GQA_OK) return r;
  if ((r = transpose_launch(Q, Qt, sh.S, sh.Hk, sh.G, sh.d, T.ld_qt, st)) != GQA_OK) return r;
  if ((r = transpose_launch(dO, dOt, sh.S, sh.Hk, sh.G, sh.d, T.ld_qt, st)) != GQA_OK) return r;
  profile_before(st, "tc_query_major+tc_key_major");
  switch (sh.d) {
    case 32:
      r = qm_launch<32>(Q, K, V, dO, LSE, seg, dQ, Kt, T.ld_kt, Dws, status, sh, st);
      if (r == GQA_OK)
        r = km_launch<32>(Q, K, V, dO, LSE, seg, dK, dV, Qt, dOt, T.ld_qt, Dws, blk, blk_max, status, sh, st);
      break;
    case 64:
      r = qm_launch<64>(Q, K, V, dO, LSE, seg, dQ, Kt, T.ld_kt, Dws, status, sh, st);
      if (r == GQA_OK)
        r = km_launch<64>(Q, K, V, dO, LSE, seg, dK, dV, Qt, dOt, T.ld_qt, Dws, blk, blk_max, status, sh, st);
      break;
    default:
      r = qm_launch<128>(Q, K, V, dO, LSE, seg, dQ, Kt, T.ld_kt, Dws, status, sh, st);
      if (r == GQA_OK)
        r = km_launch<128>(Q, K, V, dO, LSE, seg, dK, dV, Qt, dOt, T.ld_qt, Dws, blk, blk_max, status, sh, st);
      break;
  }
  profile_after(st);
  return r;
}

}  // namespace gqa
