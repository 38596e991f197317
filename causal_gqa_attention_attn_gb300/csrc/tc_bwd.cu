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

#include "common.cuh"
#include "tc_common.cuh"

namespace gqa {
namespace {

using namespace tc;

constexpr int kComputeWarps = 4;
constexpr int kThreads = 32 * (2 + kComputeWarps);   // producer, MMA, 4 compute warps
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
};

__device__ __forceinline__ uint32_t lane_base(uint32_t tmem, int warp) {
  return tmem + ((uint32_t)(32 * (warp & 3)) << 16);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    tc_query_major(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                   const __grid_constant__ CUtensorMap mapKt,
                   const float* __restrict__ Q, const float* __restrict__ dO,
                   const float* __restrict__ LSE, const uint32_t* __restrict__ seg,
                   float* __restrict__ dQ, float* __restrict__ Dws, uint32_t* __restrict__ status,
                   Shape sh) {
  using C = QmCfg<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ QmBarriers bars;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = sh.G, QR = 128 / G;
  const int n_slabs = (sh.S + QR - 1) / QR;
  const int slab = n_slabs - 1 - (int)blockIdx.x;        // longest rows first
  const int g = blockIdx.y;
  const int q0 = slab * QR;
  const int S = sh.S, H = sh.H;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(&bars.kv_full[i], 1);
      mbar_init(&bars.kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.s_free[i], kComputeWarps);
    }
    mbar_init(&bars.qdo_ready, kComputeWarps);
    mbar_init(&bars.dq_done, 1);
    bars.abort = 0;
    bars.kmin = 0xffffffffu;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  // smallest document start over the slab's queries -> first visible chunk
  if (warp >= 2) {
    const int r = 32 * (warp & 3) + lane;
    const int q = q0 + r / G;
    unsigned v = (q < S) ? __ldg(seg + q) : 0xffffffffu;
    for (int o = 16; o >= 1; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) atomicMin(&bars.kmin, v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  const int q_last = min(q0 + QR, S) - 1;
  const int kc0 = (int)(min(bars.kmin, (unsigned)q_last) / C::BK);
  const int kc1 = q_last / C::BK;
  const int nk = kc1 - kc0 + 1;
  const int total = 2 * nk;
  volatile int* abort = &bars.abort;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&mapK);
      tma_prefetch_desc(&mapV);
      tma_prefetch_desc(&mapKt);
      for (int c = 0; c < total; ++c) {
        const int slot = c % C::NSLOT;
        if (c >= C::NSLOT &&
            !mbar_wait(&bars.kv_empty[slot], ((c / C::NSLOT) - 1) & 1, abort, status, kSiteQmProducer))
          break;
        const int key0 = (kc0 + c % nk) * C::BK;
        unsigned char* sk = smem + slot * C::SLOT_BYTES;
        unsigned char* sv = sk + C::TILE_BYTES;
        const bool pass2 = c >= nk;
        mbar_arrive_expect_tx(&bars.kv_full[slot], (pass2 ? 3 : 2) * C::TILE_BYTES);
        for (int p = 0; p < C::PANELS; ++p) {
          tma_load_2d(sk + p * C::PANEL_BYTES, &mapK, g * D + 32 * p, key0, &bars.kv_full[slot]);
          tma_load_2d(sv + p * C::PANEL_BYTES, &mapV, g * D + 32 * p, key0, &bars.kv_full[slot]);
        }
        if (pass2) {
          unsigned char* skt = sv + C::TILE_BYTES;
          for (int p = 0; p < C::KT_PANELS; ++p)
            tma_load_2d(skt + p * C::KT_PANEL_BYTES, &mapKt, key0 + 32 * p, g * D, &bars.kv_full[slot]);
        }
      }
      // leave only once every load this CTA issued has landed
      for (int c = max(0, total - C::NSLOT); c < total; ++c)
        mbar_wait(&bars.kv_full[c % C::NSLOT], (c / C::NSLOT) & 1, abort, status, kSiteQmProducer);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_tf32(128, C::BK, false, false);   // S, dP: N = BK keys
      constexpr uint32_t id_q = idesc_tf32(128, D, false, false);       // dQ: N = d, B = K^T chunk
      bool ok = mbar_wait(&bars.qdo_ready, 0, abort, status, kSiteQmMma);
      bool first_dq = true;
      auto issue_dq = [&](int cc) -> bool {
        const int st = cc & 1, slot = cc % C::NSLOT;
        if (!mbar_wait(&bars.s_free[st], (cc / 2) & 1, abort, status, kSiteQmMma)) return false;
        tc_fence_after();
        const uint32_t ktbase = smem_u32(smem + slot * C::SLOT_BYTES + 2 * C::TILE_BYTES);
        for (int kk = 0; kk < C::BK / 8; ++kk) {
          const uint64_t b = sdesc(ktbase + (kk / 4) * C::KT_PANEL_BYTES + (kk % 4) * 32, 16, 1024);
          mma_ts(tmem + C::T_DQ, tmem + C::t_s(st) + 8 * kk, b, id_q, (first_dq && kk == 0) ? 0u : 1u);
        }
        first_dq = false;
        mma_commit(&bars.kv_empty[slot]);
        return true;
      };
      tc_fence_after();
      for (int c = 0; ok && c < total; ++c) {
        const int slot = c % C::NSLOT, st = c & 1;
        const bool pass2 = c >= nk;
        if (!mbar_wait(&bars.kv_full[slot], (c / C::NSLOT) & 1, abort, status, kSiteQmMma)) break;
        if (c >= 2 && !mbar_wait(&bars.s_free[st], ((c - 2) / 2) & 1, abort, status, kSiteQmMma))
          break;
        tc_fence_after();
        const uint32_t kbase = smem_u32(smem + slot * C::SLOT_BYTES);
        const uint32_t vbase = kbase + C::TILE_BYTES;
        for (int ks = 0; ks < D / 8; ++ks) {
          const uint32_t off = (ks / 4) * C::PANEL_BYTES + (ks % 4) * 32;
          mma_ts(tmem + C::t_s(st), tmem + C::T_Q + 8 * ks, sdesc(kbase + off, 16, 1024), id_s,
                 ks > 0);
          mma_ts(tmem + C::t_dp(st), tmem + C::T_DO + 8 * ks, sdesc(vbase + off, 16, 1024), id_s,
                 ks > 0);
        }
        mma_commit(&bars.s_full[st]);
        if (!pass2) mma_commit(&bars.kv_empty[slot]);
        if (pass2 && c > nk && !issue_dq(c - 1)) { ok = false; break; }
      }
      if (ok) ok = issue_dq(total - 1);
      mma_commit(&bars.dq_done);     // also drains every MMA issued above
    }
  } else {
    // ---------------- compute warps: one TMEM lane (= one row) per thread ----------------
    const int r = 32 * (warp & 3) + lane;
    const int qi = r / G, q = q0 + qi;
    const int h = g * G + r % G;
    const bool valid = q < S;
    const uint32_t tl = lane_base(tmem, warp);
    const long long row_off = (long long)q * H * D + (long long)h * D;
    // Q and dO rows into TMEM (rounded to TF32): the A operands of S and dP
    {
      float v[32];
      for (int cc = 0; cc < D; cc += 32) {
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          float4 x = valid ? __ldg(reinterpret_cast<const float4*>(Q + row_off + cc + i))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
          v[i] = to_tf32(x.x); v[i + 1] = to_tf32(x.y); v[i + 2] = to_tf32(x.z); v[i + 3] = to_tf32(x.w);
        }
        tmem_st32(tl + C::T_Q + cc, v);
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          float4 x = valid ? __ldg(reinterpret_cast<const float4*>(dO + row_off + cc + i))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
          v[i] = to_tf32(x.x); v[i + 1] = to_tf32(x.y); v[i + 2] = to_tf32(x.z); v[i + 3] = to_tf32(x.w);
        }
        tmem_st32(tl + C::T_DO + cc, v);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.qdo_ready);
    }
    const float sl2 = sh.scale * kLog2e;
    const float lse2 = valid ? __ldg(LSE + (long long)q * H + h) * kLog2e : 0.f;
    const int segq = valid ? (int)__ldg(seg + q) : 0;
    float Dacc = 0.f, Drow = 0.f;
    bool ok = true;
    for (int c = 0; c < total; ++c) {
      const int st = c & 1;
      const bool pass2 = c >= nk;
      const int k0 = (kc0 + c % nk) * C::BK;
      if (!mbar_wait(&bars.s_full[st], (c / 2) & 1, abort, status, kSiteQmCompute)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int jb = 0; jb < C::BK; jb += 32) {
        float s[32], dp[32];
        tmem_ld32(tl + C::t_s(st) + jb, s);
        tmem_ld32(tl + C::t_dp(st) + jb, dp);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int key = k0 + jb + j;
          const bool vis = valid && key >= segq && key <= q;
          const float p = vis ? ex2(fmaf(s[j], sl2, -lse2)) : 0.f;
          if (!pass2) {
            Dacc = fmaf(p, dp[j], Dacc);
          } else {
            s[j] = to_tf32(sh.scale * p * (dp[j] - Drow));
          }
        }
        if (pass2) tmem_st32(tl + C::t_s(st) + jb, s);
      }
      if (pass2) tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.s_free[st]);
      if (c == nk - 1) Drow = Dacc;
    }
    // epilogue: dQ += accumulated tile, D to the workspace
    if (ok && mbar_wait(&bars.dq_done, 0, abort, status, kSiteQmCompute)) {
      tc_fence_after();
      for (int cc = 0; cc < D; cc += 32) {
        float v[32];
        tmem_ld32(tl + C::T_DQ + cc, v);
        tmem_ld_wait();
        if (valid) {
          float4* dst = reinterpret_cast<float4*>(dQ + row_off + cc);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float4 o = dst[i];
            o.x += (v[4 * i] == v[4 * i]) ? v[4 * i] : 0.f;
            o.y += (v[4 * i + 1] == v[4 * i + 1]) ? v[4 * i + 1] : 0.f;
            o.z += (v[4 * i + 2] == v[4 * i + 2]) ? v[4 * i + 2] : 0.f;
            o.w += (v[4 * i + 3] == v[4 * i + 3]) ? v[4 * i + 3] : 0.f;
            dst[i] = o;
          }
        }
      }
      if (valid) Dws[(long long)q * H + h] = Drow;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
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
// while its S^T/dP^T run.
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

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    tc_key_major(const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapQ,
                 const __grid_constant__ CUtensorMap mapDO, const __grid_constant__ CUtensorMap mapQt,
                 const __grid_constant__ CUtensorMap mapDOt, const float* __restrict__ K,
                 const float* __restrict__ LSE, const float* __restrict__ Dws,
                 const uint32_t* __restrict__ seg, const uint32_t* __restrict__ blk_minseg,
                 float* __restrict__ dK, float* __restrict__ dV, uint32_t* __restrict__ status,
                 Shape sh) {
  using C = KmCfg<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ KmBarriers bars;
  __shared__ float4 meta[2][C::NQ];     // per block column: (lse*log2e, D, query, seg)
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = sh.G, QB = C::NQ / G;   // queries per block
  const int S = sh.S, H = sh.H;
  const int k0 = blockIdx.x * 128, g = blockIdx.y;
  const int k_hi = min(k0 + 128, S) - 1;
  const int qb0 = k0 / QB, nqb = (S + QB - 1) / QB;

  if (threadIdx.x == 0) {
    mbar_init(&bars.v_full, 1);
    mbar_init(&bars.k_ready, kComputeWarps);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars.full[i], 1);
      mbar_init(&bars.empty[i], 1);
    }
    mbar_init(&bars.s_full, 1);
    mbar_init(&bars.p_ready, kComputeWarps);
    mbar_init(&bars.acc_done, 1);
    bars.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  volatile int* abort = &bars.abort;
  auto visible = [&](int qb) { return __ldg(blk_minseg + qb) <= (unsigned)k_hi; };

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const CUtensorMap* maps[4] = {&mapQ, &mapDO, &mapQt, &mapDOt};
      for (int i = 0; i < 4; ++i) tma_prefetch_desc(maps[i]);
      tma_prefetch_desc(&mapV);
      mbar_arrive_expect_tx(&bars.v_full, C::V_BYTES);
      for (int p = 0; p < D / 32; ++p)
        tma_load_2d(smem + C::OFF_V + p * C::V_PANEL_BYTES, &mapV, g * D + 32 * p, k0, &bars.v_full);
      const int offs[4] = {C::OFF_Q, C::OFF_DO, C::OFF_QT, C::OFF_DOT};
      int n = 0;
      bool ok = true;
      for (int qb = qb0; ok && qb < nqb; ++qb) {
        if (!visible(qb)) continue;
        const int q0 = qb * QB;
        for (int t = 0; t < 4; ++t) {
          if (n > 0 && !mbar_wait(&bars.empty[t], (n - 1) & 1, abort, status, kSiteKmProducer)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars.full[t], C::BLK_BYTES);
          unsigned char* dst = smem + offs[t];
          if (t < 2) {          // Q / dO block: 3-D box (32 dims, G heads, QB queries)
            for (int p = 0; p < D / 32; ++p)
              tma_load_3d(dst + p * C::BLK_PANEL_BYTES, maps[t], 32 * p, g * G, q0, &bars.full[t]);
          } else {              // Q^T / dO^T block: d rows x NQ (query, head) columns
            for (int p = 0; p < C::T_PANELS; ++p)
              tma_load_2d(dst + p * C::T_PANEL_BYTES, maps[t], q0 * G + 32 * p, g * D, &bars.full[t]);
          }
        }
        ++n;
      }
      // leave only once every load this CTA issued has landed
      mbar_wait(&bars.v_full, 0, abort, status, kSiteKmProducer);
      if (n > 0)
        for (int t = 0; t < 4; ++t) mbar_wait(&bars.full[t], (n - 1) & 1, abort, status, kSiteKmProducer);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_tf32(128, C::NQ, false, false);
      constexpr uint32_t id_g = idesc_tf32(128, D, false, false);
      bool ok = mbar_wait(&bars.v_full, 0, abort, status, kSiteKmMma) &&
                mbar_wait(&bars.k_ready, 0, abort, status, kSiteKmMma);
      tc_fence_after();
      const uint32_t sv = smem_u32(smem + C::OFF_V), sq = smem_u32(smem + C::OFF_Q),
                     sdo = smem_u32(smem + C::OFF_DO), sqt = smem_u32(smem + C::OFF_QT),
                     sdot = smem_u32(smem + C::OFF_DOT);
      int n = 0;
      for (int qb = qb0; ok && qb < nqb; ++qb) {
        if (!visible(qb)) continue;
        const uint32_t par = n & 1;
        if (!mbar_wait(&bars.full[0], par, abort, status, kSiteKmMma) ||
            !mbar_wait(&bars.full[1], par, abort, status, kSiteKmMma)) { ok = false; break; }
        tc_fence_after();
        for (int ks = 0; ks < D / 8; ++ks) {
          const uint32_t pb = (ks / 4) * C::BLK_PANEL_BYTES + (ks % 4) * 32;
          mma_ts(tmem + C::T_S, tmem + C::T_K + 8 * ks, sdesc(sq + pb, 16, 1024), id_s, ks > 0);
          const uint32_t pv = (ks / 4) * C::V_PANEL_BYTES + (ks % 4) * 32;
          mma_ss(tmem + C::T_DP, sdesc(sv + pv, 16, 1024), sdesc(sdo + pb, 16, 1024), id_s, ks > 0);
        }
        mma_commit(&bars.s_full);
        mma_commit(&bars.empty[0]);
        mma_commit(&bars.empty[1]);
        if (!mbar_wait(&bars.p_ready, par, abort, status, kSiteKmMma) ||
            !mbar_wait(&bars.full[2], par, abort, status, kSiteKmMma) ||
            !mbar_wait(&bars.full[3], par, abort, status, kSiteKmMma)) { ok = false; break; }
        tc_fence_after();
        for (int kk = 0; kk < C::NQ / 8; ++kk) {
          const uint32_t pt = (kk / 4) * C::T_PANEL_BYTES + (kk % 4) * 32;
          const uint32_t acc = (n > 0 || kk > 0) ? 1u : 0u;
          mma_ts(tmem + C::T_DV, tmem + C::T_S + 8 * kk, sdesc(sdot + pt, 16, 1024), id_g, acc);
          mma_ts(tmem + C::T_DK, tmem + C::T_DP + 8 * kk, sdesc(sqt + pt, 16, 1024), id_g, acc);
        }
        mma_commit(&bars.empty[2]);
        mma_commit(&bars.empty[3]);
        ++n;
      }
      mma_commit(&bars.acc_done);
    }
  } else {
    // ---------------- compute warps: thread = key (TMEM lane) ----------------
    const int r = 32 * (warp & 3) + lane;
    const int key = k0 + r;
    const uint32_t tl = lane_base(tmem, warp);
    const int ct = threadIdx.x - 64;                       // 0..127 among compute threads
    {
      float v[32];
      const float* krow = K + (long long)key * sh.Hk * D + (long long)g * D;
      for (int cc = 0; cc < D; cc += 32) {
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          float4 x = (key < S) ? __ldg(reinterpret_cast<const float4*>(krow + cc + i))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
          v[i] = to_tf32(x.x); v[i + 1] = to_tf32(x.y); v[i + 2] = to_tf32(x.z); v[i + 3] = to_tf32(x.w);
        }
        tmem_st32(tl + C::T_K + cc, v);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.k_ready);
    }
    const float sl2 = sh.scale * kLog2e;
    int n = 0;
    bool ok = true;
    for (int qb = qb0; qb < nqb; ++qb) {
      if (!visible(qb)) continue;
      // column metadata of this block (double-buffered; one named barrier per block)
      if (ct < C::NQ) {
        const int q = qb * QB + ct / G, h = g * G + ct % G;
        float4 m = make_float4(0.f, 0.f, __int_as_float(-1), __int_as_float(0x7fffffff));
        if (q < S)
          m = make_float4(__ldg(LSE + (long long)q * H + h) * kLog2e, Dws[(long long)q * H + h],
                          __int_as_float(q), __int_as_float((int)__ldg(seg + q)));
        meta[n & 1][ct] = m;
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (!mbar_wait(&bars.s_full, n & 1, abort, status, kSiteKmCompute)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int cb = 0; cb < C::NQ; cb += 32) {
        float s[32], dp[32];
        tmem_ld32(tl + C::T_S + cb, s);
        tmem_ld32(tl + C::T_DP + cb, dp);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float4 m = meta[n & 1][cb + j];
          const int q = __float_as_int(m.z), sq = __float_as_int(m.w);
          const bool vis = key <= q && key >= sq;        // q = -1 for padding columns
          const float p = vis ? ex2(fmaf(s[j], sl2, -m.x)) : 0.f;
          s[j] = to_tf32(p);
          dp[j] = to_tf32(sh.scale * p * (dp[j] - m.y));
        }
        tmem_st32(tl + C::T_S + cb, s);
        tmem_st32(tl + C::T_DP + cb, dp);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.p_ready);
      ++n;
    }
    if (ok && mbar_wait(&bars.acc_done, 0, abort, status, kSiteKmCompute)) {
      tc_fence_after();
      const long long row = (long long)key * sh.Hk * D + (long long)g * D;
      for (int cc = 0; cc < D; cc += 32) {
        float a[32], b[32];
        tmem_ld32(tl + C::T_DK + cc, a);
        tmem_ld32(tl + C::T_DV + cc, b);
        tmem_ld_wait();
        if (key < S && n > 0) {
          float4* pk = reinterpret_cast<float4*>(dK + row + cc);
          float4* pv = reinterpret_cast<float4*>(dV + row + cc);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float4 o = pk[i], w = pv[i];
            o.x += (a[4 * i] == a[4 * i]) ? a[4 * i] : 0.f;
            o.y += (a[4 * i + 1] == a[4 * i + 1]) ? a[4 * i + 1] : 0.f;
            o.z += (a[4 * i + 2] == a[4 * i + 2]) ? a[4 * i + 2] : 0.f;
            o.w += (a[4 * i + 3] == a[4 * i + 3]) ? a[4 * i + 3] : 0.f;
            w.x += (b[4 * i] == b[4 * i]) ? b[4 * i] : 0.f;
            w.y += (b[4 * i + 1] == b[4 * i + 1]) ? b[4 * i + 1] : 0.f;
            w.z += (b[4 * i + 2] == b[4 * i + 2]) ? b[4 * i + 2] : 0.f;
            w.w += (b[4 * i + 3] == b[4 * i + 3]) ? b[4 * i + 3] : 0.f;
            pk[i] = o;
            pv[i] = w;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// Group transpose: X [S][Hk*Gx][d] (row-major, head h = g*Gx + h') to
// Xt [Hk*d][ld] with Xt[g*d + e][q*Gx + h'] = X[q][(g*Gx + h')*d + e].
// With Gx = 1 this is K^T per kv head; with Gx = G it lays the (query, head)
// rows of a kv group out as the contiguous K dimension of a K-major operand.
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
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const long long r = r0 + threadIdx.x;
    if (r < nrows) Xt[(long long)(g * d + e0 + i) * ld + r] = tile[threadIdx.x][i];
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

// 2-D fp32 map: `cols` contiguous elements per row, `rows` rows `ld` elements
// apart, box = 32 columns (128 bytes, the swizzle span) x box_rows rows.
gqa_status map_2d(CUtensorMap* m, const float* base, long long cols, long long rows,
                  long long ld, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return set_error(GQA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * sizeof(float)};
  cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(GQA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return GQA_OK;
}

// 3-D fp32 map over X [S][Hx][d]: box = 32 dims x `bh` heads x `bq` queries.
gqa_status map_3d(CUtensorMap* m, const float* base, int d, int Hx, int S, int bh, int bq) {
  auto fn = encode_fn();
  if (fn == nullptr) return set_error(GQA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)Hx, (cuuint64_t)S};
  cuuint64_t strides[2] = {(cuuint64_t)d * sizeof(float), (cuuint64_t)Hx * d * sizeof(float)};
  cuuint32_t box[3] = {32, (cuuint32_t)bh, (cuuint32_t)bq};
  cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(GQA_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (%d)", (int)r);
  return GQA_OK;
}

template <int D>
gqa_status km_launch(const float* Q, const float* K, const float* V, const float* dO,
                     const float* LSE, const uint32_t* seg, float* dK, float* dV, const float* Qt,
                     const float* dOt, long long ld_qt, const float* Dws, const uint32_t* blk_minseg,
                     uint32_t* status, const Shape& sh, cudaStream_t st) {
  using C = KmCfg<D>;
  const int QB = C::NQ / sh.G;
  CUtensorMap mv, mq, mdo, mqt, mdot;
  gqa_status r;
  if ((r = map_2d(&mv, V, (long long)sh.Hk * D, sh.S, (long long)sh.Hk * D, 128)) != GQA_OK) return r;
  if ((r = map_3d(&mq, Q, D, sh.H, sh.S, sh.G, QB)) != GQA_OK) return r;
  if ((r = map_3d(&mdo, dO, D, sh.H, sh.S, sh.G, QB)) != GQA_OK) return r;
  const long long cols = (long long)sh.S * sh.G;
  if ((r = map_2d(&mqt, Qt, cols, (long long)sh.Hk * D, ld_qt, D)) != GQA_OK) return r;
  if ((r = map_2d(&mdot, dOt, cols, (long long)sh.Hk * D, ld_qt, D)) != GQA_OK) return r;
  if (cudaFuncSetAttribute(tc_key_major<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::SMEM_BYTES) != cudaSuccess)
    return check_launch("key-major smem attribute");
  dim3 grid((sh.S + 127) / 128, sh.Hk);
  tc_key_major<D><<<grid, kThreads, C::SMEM_BYTES, st>>>(mv, mq, mdo, mqt, mdot, K, LSE, Dws, seg,
                                                         blk_minseg, dK, dV, status, sh);
  note_launch();
  return check_launch("tensor-core key-major");
}

gqa_status transpose_launch(const float* X, float* Xt, int S, int Hk, int Gx, int d, long long ld,
                            cudaStream_t st) {
  const long long nrows = (long long)S * Gx;
  dim3 grid((unsigned)((nrows + 31) / 32), d / 32, Hk);
  group_transpose<<<grid, dim3(32, 8), 0, st>>>(X, Xt, S, Hk, Gx, d, ld);
  note_launch();
  return check_launch("group transpose");
}

template <int D>
gqa_status qm_launch(const float* Q, const float* K, const float* V, const float* dO,
                     const float* LSE, const uint32_t* seg, float* dQ, const float* Kt,
                     long long ld_kt, float* Dws, uint32_t* status, const Shape& sh,
                     cudaStream_t st) {
  using C = QmCfg<D>;
  CUtensorMap mk, mv, mkt;
  gqa_status r;
  if ((r = map_2d(&mk, K, (long long)sh.Hk * D, sh.S, (long long)sh.Hk * D, C::BK)) != GQA_OK) return r;
  if ((r = map_2d(&mv, V, (long long)sh.Hk * D, sh.S, (long long)sh.Hk * D, C::BK)) != GQA_OK) return r;
  if ((r = map_2d(&mkt, Kt, sh.S, (long long)sh.Hk * D, ld_kt, D)) != GQA_OK) return r;
  if (cudaFuncSetAttribute(tc_query_major<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::SMEM_BYTES) != cudaSuccess)
    return check_launch("query-major smem attribute");
  const int QR = 128 / sh.G;
  dim3 grid((sh.S + QR - 1) / QR, sh.Hk);
  tc_query_major<D><<<grid, kThreads, C::SMEM_BYTES, st>>>(mk, mv, mkt, Q, dO, LSE, seg, dQ, Dws,
                                                           status, sh);
  note_launch();
  return check_launch("tensor-core query-major");
}

}  // namespace

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
  t.total = t.blk_off + align256((size_t)S * sizeof(uint32_t));
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
  const int QB = ((sh.d == 128) ? 64 : 128) / sh.G;
  gqa_status r;
  if ((r = tile_minseg(seg, sh.S, QB, blk, st)) != GQA_OK) return r;
  if ((r = transpose_launch(K, Kt, sh.S, sh.Hk, 1, sh.d, T.ld_kt, st)) != GQA_OK) return r;
  if ((r = transpose_launch(Q, Qt, sh.S, sh.Hk, sh.G, sh.d, T.ld_qt, st)) != GQA_OK) return r;
  if ((r = transpose_launch(dO, dOt, sh.S, sh.Hk, sh.G, sh.d, T.ld_qt, st)) != GQA_OK) return r;
  profile_before(st, "tc_query_major+tc_key_major");
  switch (sh.d) {
    case 32:
      r = qm_launch<32>(Q, K, V, dO, LSE, seg, dQ, Kt, T.ld_kt, Dws, status, sh, st);
      if (r == GQA_OK)
        r = km_launch<32>(Q, K, V, dO, LSE, seg, dK, dV, Qt, dOt, T.ld_qt, Dws, blk, status, sh, st);
      break;
    case 64:
      r = qm_launch<64>(Q, K, V, dO, LSE, seg, dQ, Kt, T.ld_kt, Dws, status, sh, st);
      if (r == GQA_OK)
        r = km_launch<64>(Q, K, V, dO, LSE, seg, dK, dV, Qt, dOt, T.ld_qt, Dws, blk, status, sh, st);
      break;
    default:
      r = qm_launch<128>(Q, K, V, dO, LSE, seg, dQ, Kt, T.ld_kt, Dws, status, sh, st);
      if (r == GQA_OK)
        r = km_launch<128>(Q, K, V, dO, LSE, seg, dK, dV, Qt, dOt, T.ld_qt, Dws, blk, status, sh, st);
      break;
  }
  profile_after(st);
  return r;
}

}  // namespace gqa
