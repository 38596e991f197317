// Tensor-core forward with the log-sum-exp (tcgen05, kind::tf32, fp32
// accumulation in TMEM): O and LSE for every (query, head), the setup the
// backward consumes (tang llm.rs, causal_attention_fused: row max, sum of
// exponentials, weighted V; the LSE as the backward_attention.wgsl header
// uses it: P = exp(scale q.k - LSE)).
//
// One CTA per (slab of 128/G queries, kv head), M = 128 rows = the slab's
// queries x the G heads of the group, the same layout as the backward's
// query-major kernel. Q sits in TMEM (A operand). One pass over the slab's
// visible keys in chunks of 64, streamed by TMA through a ring of units (K
// and V^T, a transposed copy in the workspace: TF32 operands are read K-major
// only), with an online softmax:
//   S = Q K^T of chunk c into TMEM stage c & 1;
//   the softmax warpgroup c & 1 (one thread per row, all 64 columns) keeps
//   its own running row max m and sum l, writes P = 2^(s scale log2e - m)
//   back over S (A operand) and the MMA warp adds P V into that warpgroup's
//   own O accumulator (O_0 for even chunks, O_1 for odd ones);
//   at the end the two (m, l, O) are combined: O = (O_0 2^(m_0 - m) +
//   O_1 2^(m_1 - m)) / (l_0 2^(m_0 - m) + l_1 2^(m_1 - m)), LSE = m + log2(...).
// The running max is raised (and O rescaled in TMEM) only when a chunk's max
// exceeds it by more than 2^8, so P stays below 256 and rescaling is rare.
// When the softmax of chunk c starts, the P V product of its warpgroup's
// previous chunk c - 2 has completed (issued before S(c), which has
// completed), so the rescale needs no extra hand-off. Two contractions per
// pair and head (Q K^T, P V). O and LSE are overwritten.
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
constexpr float kRescaleLog2 = 8.f;      // raise the running max only past 2^8

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
  // TMEM columns: Q | O_0 | O_1 | two S stages of BK columns
  static constexpr uint32_t T_Q = 0, T_ST = 3 * D;
  static constexpr uint32_t t_o(int w) { return D + w * D; }
  static constexpr uint32_t stage(int st) { return T_ST + st * BK; }
  static_assert(T_ST + 2 * BK <= 512, "TMEM budget");
};

struct FwdBarriers {
  uint64_t full[12], empty[12], s_full[2], p_ready[2], q_ready, o_done;
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
  constexpr int NU = Cfg::NUNIT, BK = Cfg::BK;
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
      mbar_init(&bars.p_ready[i], kFwdComputeWarps / 2);   // the four warps of warpgroup i
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
  const int nk = q_last / BK - kc0 + 1;                     // chunks
  const int n_units = 2 * nk;                               // unit 2c: K of chunk c, 2c + 1: its V^T
  volatile int* abort = &bars.abort;

  if (warp < kFwdProducers) {
    // ---------------- TMA producers: warp 0 loads the K units, warp 1 the V^T units ----------------
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
      const int key0 = (kc0 + i / 2) * BK;
      unsigned char* dst = smem + u * Cfg::UNIT_BYTES;
      if (elect_one()) {
        mbar_arrive_expect_tx(&bars.full[u], Cfg::UNIT_BYTES);
        if (pw == 1) tma_load_3d(dst, &mapVt, 0, g * D, key0 / 32, &bars.full[u]);
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
    // O_{c&1} += P(c) V(c): after the softmax of chunk c has written P
    auto issue_o = [&](int c) -> bool {
      const int st = c & 1, ivt = 2 * c + 1;
      if (!warp_wait(&bars.p_ready[st], (c >> 1) & 1, abort, status, kSiteFwdMma) || !unit_wait(ivt))
        return false;
      const uint32_t a_p = tmem + Cfg::stage(st), d_o = tmem + Cfg::t_o(st);
      const uint64_t bvt = unit_desc(ivt);
      if (elect_one()) {
        tc_fence_after();
        mma_ts(d_o, a_p, bvt, id_o, c >= 2 ? 1u : 0u);   // chunks 0 and 1 start their accumulators
#pragma unroll
        for (int kk = 1; kk < BK / 8; ++kk)
          mma_ts_acc(d_o, a_p + 8 * kk, bvt + desc_off(kk, Cfg::VT_PANEL_BYTES), id_o);
        mma_commit(&bars.empty[ivt % NU]);
      }
      __syncwarp();
      return true;
    };
    bool ok = warp_wait(&bars.q_ready, 0, abort, status, kSiteFwdMma);
    // S(c) into stage c & 1 (its previous P was read by O(c-2), issued before),
    // then O(c-1): the tensor core works on S(c) while the softmax of c-1 runs
    for (int c = 0; ok && c < nk; ++c) {
      const int st = c & 1, ik = 2 * c;
      if (!unit_wait(ik)) { ok = false; break; }
      if (elect_one()) {
        tc_fence_after();
        const uint32_t ts = tmem + Cfg::stage(st);
        const uint64_t bk = unit_desc(ik);
        mma_ts(ts, tmem + Cfg::T_Q, bk, id_s, 0u);
#pragma unroll
        for (int ks = 1; ks < D / 8; ++ks)
          mma_ts_acc(ts, tmem + Cfg::T_Q + 8 * ks, bk + desc_off(ks, Cfg::K_PANEL_BYTES), id_s);
        mma_commit(&bars.s_full[st]);
        mma_commit(&bars.empty[ik % NU]);
      }
      __syncwarp();
      if (c > 0 && !issue_o(c - 1)) { ok = false; break; }
    }
    if (ok && nk > 0) ok = issue_o(nk - 1);
    if (elect_one()) mma_commit(&bars.o_done);   // also drains every MMA issued above
    __syncwarp();
  } else {
    // ---------------- compute: one TMEM lane (= one row) per thread; warpgroup
    // wg takes the chunks c with c & 1 == wg, all BK columns of them ----------------
    const int wg = (warp - kFwdFirstCompute) >> 2;
    const int r = 32 * (warp & 3) + lane;
    const int qi = r / G, q = q0 + qi;
    const int h = g * G + r % G;
    // (debug build: the row's Q / O range and LSE index lie in the tensors;
    // a row that fails is treated as padding)
    const bool valid = q < S && GQA_DCHECK(status, h < H && g < sh.Hk, kChkFwd);
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
    const uint32_t to = tl + Cfg::t_o(wg);
    float m = -1e30f, l = 0.f;     // running max (log2 units) and sum over this warpgroup's keys
    bool ok = true, has_o = false;
    for (int c = wg; c < nk; c += 2) {
      if (!mbar_wait(&bars.s_full[wg], (c >> 1) & 1, abort, status, kSiteFwdCompute)) { ok = false; break; }
      tc_fence_after();
      const int k0 = (kc0 + c) * BK;
      const bool full = valid && k0 >= segq && k0 + BK - 1 <= q;
      const uint32_t ts = tl + Cfg::stage(wg);
      float sv[BK];
      tmem_ld32(ts, sv);
      tmem_ld32(ts + 32, sv + 32);
      tmem_ld_wait();
      float mx = -1e30f;
      if (full) {
#pragma unroll
        for (int j = 0; j < BK; ++j) {
          sv[j] *= sl2;
          mx = fmaxf(mx, sv[j]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < BK; ++j) {
          const int key = k0 + j;
          const bool vis = valid && key >= segq && key <= q;
          sv[j] = vis ? sv[j] * sl2 : -1e30f;
          mx = fmaxf(mx, sv[j]);
        }
      }
      // raise the running max past 2^8 growth only; O of this warpgroup is
      // idle here (its last P V product completed before S(c) did)
      const bool raise = mx > m + kRescaleLog2;
      const float alpha = raise ? ex2(m - mx) : 1.f;
      if (raise) {
        l *= alpha;
        m = mx;
      }
      if (has_o && __any_sync(0xffffffffu, raise)) {
        for (int cc = 0; cc < D; cc += 32) {
          float ov[32];
          tmem_ld32(to + cc, ov);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] *= alpha;
          tmem_st32(to + cc, ov);
        }
      }
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < BK; ++j) {
        const float pj = (sv[j] > -1e29f) ? ex2(sv[j] - m) : 0.f;
        sum += pj;
        sv[j] = pj;
      }
      l += sum;
      tmem_st32(ts, sv);
      tmem_st32(ts + 32, sv + 32);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.p_ready[wg]);
      has_o = true;
    }
    // both warpgroups' (max, sum) of each row -> its LSE (log2 units) and the
    // weights of the two O accumulators
    bars.part[wg][0][r] = m;
    bars.part[wg][1][r] = l;
    asm volatile("bar.sync 2, 256;" ::: "memory");
    const float m0 = bars.part[0][0][r], m1 = bars.part[1][0][r];
    const float mm = fmaxf(m0, m1);
    const float a0 = ex2(m0 - mm), a1 = ex2(m1 - mm);
    const float ll = bars.part[0][1][r] * a0 + bars.part[1][1][r] * a1;
    const float lse2 = mm + __log2f(ll);
    const float inv = 1.f / ll;
    // epilogue: O (warpgroup wg: half wg of the columns of both accumulators) and LSE
    if (ok && mbar_wait(&bars.o_done, 0, abort, status, kSiteFwdCompute)) {
      tc_fence_after();
      const bool has1 = nk >= 2;   // O_1 was written only if there is an odd chunk
      for (int cc = wg * (D / 2); cc < (wg + 1) * (D / 2); cc += 16) {
        float v0[16], v1[16];
        tmem_ld16(tl + Cfg::t_o(0) + cc, v0);
        if (has1) tmem_ld16(tl + Cfg::t_o(1) + cc, v1);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) v0[i] = (v0[i] * a0 + (has1 ? v1[i] * a1 : 0.f)) * inv;
        if (valid) {
          float4* dst = reinterpret_cast<float4*>(O + row_off + cc);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_float4(v0[4 * i], v0[4 * i + 1], v0[4 * i + 2], v0[4 * i + 3]);
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
