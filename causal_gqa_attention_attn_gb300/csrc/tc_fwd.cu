// Tensor-core forward with the log-sum-exp (tcgen05, kind::tf32, fp32
// accumulation in TMEM): O and LSE for every (query, head), the setup the
// backward consumes (tang llm.rs, causal_attention_fused: row max, sum of
// exponentials, weighted V; the LSE as the backward_attention.wgsl header
// uses it: P = exp(scale q.k - LSE)).
//
// One CTA per (slab of 128/G queries, kv head), M = 128 rows = the slab's
// queries x the G heads of the group, the same layout as the backward's
// query-major kernel. Q sits in TMEM (A operand). Two passes over the slab's
// visible keys, in chunks of 64 keys streamed by TMA through a ring of units:
//  pass 1: S = Q K^T per chunk; the row max m and sum l of 2^(s log2e
//          scale - m) run online in registers, giving LSE = (m + log2 l) ln 2;
//  pass 2: S again, P = exp(scale s - LSE) written back to TMEM (A operand)
//          and O += P V (B = the chunk of V^T, a transposed copy in the
//          workspace: TF32 operands are read K-major only).
// Computing the LSE first keeps O free of the running rescale an online
// softmax needs; the price is a second Q K^T (three contractions per pair
// and head). O and LSE are overwritten.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "tc_common.cuh"

namespace gqa {
namespace {

using namespace tc;

constexpr int kFwdProducers = 2;
constexpr int kFwdMmaWarp = kFwdProducers;
constexpr int kFwdFirstCompute = kFwdProducers + 1;
constexpr int kFwdComputeWarps = 8;
constexpr int kFwdThreads = 32 * (kFwdFirstCompute + kFwdComputeWarps);
constexpr uint32_t kTmemColsFwd = 512;   // allocations are powers of two; one CTA per SM

enum : uint32_t { kSiteFwdProducer = 1u << 8, kSiteFwdMma = 1u << 9, kSiteFwdCompute = 1u << 10 };

template <int D_>
struct FwdCfg {
  static constexpr int D = D_;
  static constexpr int BK = 64;                             // keys per chunk
  static constexpr int PANELS = D / 32;
  static constexpr int K_PANEL_BYTES = BK * 128;            // K unit: BK rows x 32 floats per panel
  static constexpr int UNIT_BYTES = PANELS * K_PANEL_BYTES;
  static constexpr int VT_PANELS = BK / 32;                 // V^T unit: d rows x 32 keys per panel
  static constexpr int VT_PANEL_BYTES = D * 128;
  static_assert(VT_PANELS * VT_PANEL_BYTES == UNIT_BYTES, "V^T unit size");
  static constexpr int NUNIT = (192 * 1024 / UNIT_BYTES < 12) ? 192 * 1024 / UNIT_BYTES : 12;
  static constexpr int SMEM_BYTES =
      (NUNIT * UNIT_BYTES + 1024 > 120 * 1024) ? NUNIT * UNIT_BYTES + 1024 : 120 * 1024;
  // TMEM columns: Q | O | two S stages of BK columns
  static constexpr uint32_t T_Q = 0, T_O = D, T_ST = 2 * D;
  static constexpr uint32_t stage(int st) { return T_ST + st * BK; }
  static_assert(T_ST + 2 * BK <= 512, "TMEM budget");
};

struct FwdBarriers {
  uint64_t full[12], empty[12], s_full[2], s_free[2], q_ready, o_done;
  uint32_t tmem_base;
  int abort;
  unsigned kmin;
  float part[2][2][128];   // per warpgroup: running max and sum of each row
};

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
    tc_forward(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapVt,
               const float* __restrict__ Q, const uint32_t* __restrict__ seg,
               float* __restrict__ O, float* __restrict__ LSE, uint32_t* __restrict__ status,
               Shape sh) {
  using Cfg = FwdCfg<D>;
  constexpr int NU = Cfg::NUNIT, BK = Cfg::BK, HB = BK / 2;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ FwdBarriers bars;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = sh.G, QR = 128 / G;
  const int slab = (int)gridDim.x - 1 - (int)blockIdx.x;   // longest rows first
  const int g = blockIdx.y;
  const int q0 = slab * QR;
  const int S = sh.S, H = sh.H;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NU; ++i) {
      mbar_init(&bars.full[i], 1);
      mbar_init(&bars.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.s_free[i], kFwdComputeWarps);
    }
    mbar_init(&bars.q_ready, kFwdComputeWarps);
    mbar_init(&bars.o_done, 1);
    bars.abort = 0;
    bars.kmin = 0xffffffffu;
    fence_barrier_init();
  }
  if (warp == kFwdMmaWarp) {
    tmem_alloc(&bars.tmem_base, kTmemColsFwd);
    tmem_relinquish();
  }
  __syncthreads();
  if (warp >= kFwdFirstCompute) {   // smallest document start over the slab -> first chunk
    const int q = q0 + (32 * (warp & 3) + lane) / G;
    unsigned v = (q < S) ? __ldg(seg + q) : 0xffffffffu;
    for (int o = 16; o >= 1; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) atomicMin(&bars.kmin, v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  const int q_last = min(q0 + QR, S) - 1;
  const int kc0 = (int)(min(bars.kmin, (unsigned)q_last) / BK);
  const int nk = q_last / BK - kc0 + 1;                     // chunks per pass
  const int n_units = 3 * nk;                               // K (pass 1); K, V^T (pass 2)
  volatile int* abort = &bars.abort;

  if (warp < kFwdProducers) {
    // ---------------- TMA producers: warp pw loads the units i with i % 2 == pw ----------------
    const int pw = warp;
    if (elect_one()) {
      tma_prefetch_desc(&mapK);
      tma_prefetch_desc(&mapVt);
    }
    __syncwarp();
    for (int i = pw; i < n_units; i += 2) {
      const int u = i % NU;
      if (i >= NU && !warp_wait(&bars.empty[u], ((i / NU) - 1) & 1, abort, status, kSiteFwdProducer))
        break;
      const bool p1 = i < nk;
      const int chunk = p1 ? i : (i - nk) / 2;
      const bool vt = !p1 && ((i - nk) % 2 == 1);
      const int key0 = (kc0 + chunk) * BK;
      unsigned char* dst = smem + u * Cfg::UNIT_BYTES;
      if (elect_one()) {
        mbar_arrive_expect_tx(&bars.full[u], Cfg::UNIT_BYTES);
        if (vt) tma_load_3d(dst, &mapVt, 0, g * D, key0 / 32, &bars.full[u]);
        else tma_load_3d(dst, &mapK, 0, key0, g * Cfg::PANELS, &bars.full[u]);
      }
      __syncwarp();
    }
    const int i_lo = max(0, n_units - NU);
    for (int i = i_lo + (((i_lo & 1) != pw) ? 1 : 0); i < n_units; i += 2)
      warp_wait(&bars.full[i % NU], (i / NU) & 1, abort, status, kSiteFwdProducer);
  } else if (warp == kFwdMmaWarp) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t id_s = idesc_tf32(128, BK, false, false);   // S: N = BK keys
    constexpr uint32_t id_o = idesc_tf32(128, D, false, false);    // O: N = d
    const uint64_t desc0 = sdesc(smem_u32(smem), 16, 1024);
    auto unit_desc = [&](int i) { return desc0 + (uint64_t)(((i % NU) * Cfg::UNIT_BYTES) >> 4); };
    auto unit_wait = [&](int i) {
      return warp_wait(&bars.full[i % NU], (i / NU) & 1, abort, status, kSiteFwdMma);
    };
    int use0 = 0, use1 = 0;
    auto stage_free = [&](int st) {
      const int u = st ? use1 : use0;
      return u == 0 || warp_wait(&bars.s_free[st], (u - 1) & 1, abort, status, kSiteFwdMma);
    };
    auto issue_s = [&](uint32_t ts, uint64_t bk) {
      tc_fence_after();
      mma_ts(ts, tmem + Cfg::T_Q, bk, id_s, 0u);
#pragma unroll
      for (int ks = 1; ks < D / 8; ++ks)
        mma_ts_acc(ts, tmem + Cfg::T_Q + 8 * ks, bk + desc_off(ks, Cfg::K_PANEL_BYTES), id_s);
    };
    bool ok = warp_wait(&bars.q_ready, 0, abort, status, kSiteFwdMma);
    // ---- pass 1: S of chunk c in stage c & 1 ----
    for (int c = 0; ok && c < nk; ++c) {
      const int st = c & 1;
      if (!unit_wait(c) || !stage_free(st)) { ok = false; break; }
      if (elect_one()) {
        issue_s(tmem + Cfg::stage(st), unit_desc(c));
        mma_commit(&bars.s_full[st]);
        mma_commit(&bars.empty[c % NU]);
      }
      __syncwarp();
      if (st) ++use1; else ++use0;
    }
    // ---- pass 2: S of chunk c, then O += P V for chunk c-1 ----
    int o_use = 0;
    auto issue_o = [&](int c) -> bool {
      const int st = c & 1, ivt = nk + 2 * c + 1;
      if (!warp_wait(&bars.s_free[st], o_use & 1, abort, status, kSiteFwdMma) || !unit_wait(ivt))
        return false;
      const uint32_t a_p = tmem + Cfg::stage(st), d_o = tmem + Cfg::T_O;
      const uint64_t bvt = unit_desc(ivt);
      if (elect_one()) {
        tc_fence_after();
        mma_ts(d_o, a_p, bvt, id_o, c > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 1; kk < BK / 8; ++kk)
          mma_ts_acc(d_o, a_p + 8 * kk, bvt + desc_off(kk, Cfg::VT_PANEL_BYTES), id_o);
        mma_commit(&bars.empty[ivt % NU]);
      }
      __syncwarp();
      return true;
    };
    for (int c = 0; ok && c < nk; ++c) {
      const int st = c & 1, ik = nk + 2 * c;
      if (!unit_wait(ik)) { ok = false; break; }
      // the stage's previous use: pass 1 for c < 2, else chunk c-2 of this
      // pass, whose release issue_o(c-2) has already waited for
      if (c < 2 && !stage_free(st)) { ok = false; break; }
      if (elect_one()) {
        issue_s(tmem + Cfg::stage(st), unit_desc(ik));
        mma_commit(&bars.s_full[st]);
        mma_commit(&bars.empty[ik % NU]);
      }
      __syncwarp();
      const int this_use = st ? use1++ : use0++;
      if (c > 0 && !issue_o(c - 1)) { ok = false; break; }
      o_use = this_use;
    }
    if (ok && nk > 0) ok = issue_o(nk - 1);
    if (elect_one()) mma_commit(&bars.o_done);   // also drains every MMA issued above
    __syncwarp();
  } else {
    // ---------------- compute: one TMEM lane (= one row) per thread; both
    // warpgroups take every chunk, warpgroup wg its columns [wg*BK/2, (wg+1)*BK/2) ----------------
    const int wg = (warp - kFwdFirstCompute) >> 2;
    const int r = 32 * (warp & 3) + lane;
    const int qi = r / G, q = q0 + qi;
    const int h = g * G + r % G;
    const bool valid = q < S;
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const long long row_off = (long long)q * H * D + (long long)h * D;
    {
      // Q rows into TMEM, rounded to TF32 (warpgroup wg: half wg of the columns)
      float v[16];
      for (int cc = wg * (D / 2); cc < (wg + 1) * (D / 2); cc += 16) {
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          float4 x = valid ? __ldg(reinterpret_cast<const float4*>(Q + row_off + cc + i))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
          v[i] = to_tf32(x.x); v[i + 1] = to_tf32(x.y); v[i + 2] = to_tf32(x.z); v[i + 3] = to_tf32(x.w);
        }
        tmem_st16(tl + Cfg::T_Q + cc, v);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.q_ready);
    }
    const float sl2 = sh.scale * kLog2e;
    const int segq = valid ? (int)__ldg(seg + q) : 0;
    float m = -1e30f, l = 0.f;     // running max (log2 units) and sum over this warpgroup's keys
    bool ok = true;
    // ---- pass 1: row max and sum, online ----
    for (int c = 0; c < nk; ++c) {
      const int st = c & 1;
      if (!mbar_wait(&bars.s_full[st], (c >> 1) & 1, abort, status, kSiteFwdCompute)) { ok = false; break; }
      tc_fence_after();
      const int k0 = (kc0 + c) * BK + wg * HB;
      const bool full = valid && k0 >= segq && k0 + HB - 1 <= q;
      float sv[32];
      tmem_ld32(tl + Cfg::stage(st) + wg * HB, sv);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.s_free[st]);
      float mx = -1e30f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int key = k0 + j;
        const bool vis = full || (valid && key >= segq && key <= q);
        sv[j] = vis ? sv[j] * sl2 : -1e30f;
        mx = fmaxf(mx, sv[j]);
      }
      if (mx > m) {
        l *= ex2(m - mx);
        m = mx;
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) l += (sv[j] > -1e29f) ? ex2(sv[j] - m) : 0.f;
    }
    // both warpgroups' (max, sum) pairs -> the row's LSE (log2 units)
    bars.part[wg][0][r] = m;
    bars.part[wg][1][r] = l;
    asm volatile("bar.sync 2, 256;" ::: "memory");
    const float m0 = bars.part[0][0][r], m1 = bars.part[1][0][r];
    const float mm = fmaxf(m0, m1);
    const float ll = bars.part[0][1][r] * ex2(m0 - mm) + bars.part[1][1][r] * ex2(m1 - mm);
    const float lse2 = mm + __log2f(ll);
    // ---- pass 2: P = 2^(s*scale*log2e - lse2) over S, for O += P V ----
    for (int c = 0; ok && c < nk; ++c) {
      const int st = c & 1;
      const int uses_p1 = st ? nk / 2 : (nk + 1) / 2;
      if (!mbar_wait(&bars.s_full[st], (uses_p1 + (c >> 1)) & 1, abort, status, kSiteFwdCompute)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int k0 = (kc0 + c) * BK + wg * HB;
      const bool full = valid && k0 >= segq && k0 + HB - 1 <= q;
      const uint32_t ts = tl + Cfg::stage(st) + wg * HB;
      float sv[32];
      tmem_ld32(ts, sv);
      tmem_ld_wait();
      if (full) {
#pragma unroll
        for (int j = 0; j < 32; ++j) sv[j] = to_tf32(ex2(fmaf(sv[j], sl2, -lse2)));
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int key = k0 + j;
          const bool vis = valid && key >= segq && key <= q;
          sv[j] = vis ? to_tf32(ex2(fmaf(sv[j], sl2, -lse2))) : 0.f;
        }
      }
      tmem_st32(ts, sv);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.s_free[st]);
    }
    // epilogue: O (warpgroup wg: half wg of the columns) and LSE, overwritten
    if (ok && mbar_wait(&bars.o_done, 0, abort, status, kSiteFwdCompute)) {
      tc_fence_after();
      for (int cc = wg * (D / 2); cc < (wg + 1) * (D / 2); cc += 16) {
        float v[16];
        tmem_ld16(tl + Cfg::T_O + cc, v);
        tmem_ld_wait();
        if (valid) {
          float4* dst = reinterpret_cast<float4*>(O + row_off + cc);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
      }
      if (valid && wg == 0) LSE[(long long)q * H + h] = lse2 / kLog2e;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kFwdMmaWarp) tmem_dealloc(tmem, kTmemColsFwd);
}

template <int D>
gqa_status fwd_launch(const float* Q, const float* K, const float* Vt, long long ld_vt,
                      const uint32_t* seg, float* O, float* LSE, uint32_t* status, const Shape& sh,
                      cudaStream_t st) {
  using Cfg = FwdCfg<D>;
  CUtensorMap mk, mvt;
  gqa_status r;
  const long long kv_panels = (long long)sh.Hk * D / 32;
  if ((r = tc_map_panels(&mk, K, (long long)sh.Hk * D, sh.S, kv_panels, Cfg::BK, D / 32)) != GQA_OK) return r;
  if ((r = tc_map_panels(&mvt, Vt, ld_vt, (long long)sh.Hk * D, ld_vt / 32, D, Cfg::VT_PANELS)) != GQA_OK) return r;
  if (cudaFuncSetAttribute(tc_forward<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg::SMEM_BYTES) != cudaSuccess)
    return check_launch("forward smem attribute");
  const int QR = 128 / sh.G;
  dim3 grid((sh.S + QR - 1) / QR, sh.Hk);
  profile_before(st, "tc_forward");
  tc_forward<D><<<grid, kFwdThreads, Cfg::SMEM_BYTES, st>>>(mk, mvt, Q, seg, O, LSE, status, sh);
  note_launch();
  profile_after(st);
  return check_launch("tensor-core forward");
}

}  // namespace

bool tc_fwd_supported(const Shape& sh) {
  return (sh.d == 32 || sh.d == 64 || sh.d == 128) && sh.G >= 1 && sh.G <= 128 &&
         (128 % sh.G) == 0;
}

size_t tc_fwd_ws_bytes(int S, int Hk, int d) {
  const long long ld = ((long long)S + 31) / 32 * 32;
  return kWsHeader + align256((size_t)Hk * d * ld * sizeof(float));
}

gqa_status tc_fwd(const float* Q, const float* K, const float* V, const uint32_t* seg, float* O,
                  float* LSE, const Shape& sh, char* ws, cudaStream_t st) {
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  float* Vt = reinterpret_cast<float*>(ws + kWsHeader);
  const long long ld = ((long long)sh.S + 31) / 32 * 32;
  gqa_status r;
  if ((r = tc_transpose(V, Vt, sh.S, sh.Hk, 1, sh.d, ld, st)) != GQA_OK) return r;
  switch (sh.d) {
    case 32: return fwd_launch<32>(Q, K, Vt, ld, seg, O, LSE, status, sh, st);
    case 64: return fwd_launch<64>(Q, K, Vt, ld, seg, O, LSE, status, sh, st);
    default: return fwd_launch<128>(Q, K, Vt, ld, seg, O, LSE, status, sh, st);
  }
}

}  // namespace gqa
