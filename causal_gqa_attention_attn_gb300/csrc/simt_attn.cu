// CUDA-core (fp32 FFMA) kernels for causal GQA attention: forward with LSE and
// the backward from a saved LSE. Exact fp32 products, no tensor cores.
//
// Tiling: 64 query rows x 64 keys per tile, 256 threads. Thread (ty, tx) =
// (tid / 16, tid % 16) owns rows 4*ty .. 4*ty+3 and columns tx + 16*j of a
// 64x64 score tile, so a row's 16 owners are one half-warp (row reductions are
// four xor-shuffles). Operand tiles live in shared memory with a row stride of
// DP + 1 floats (DP = head_dim rounded up to 32/64/128) so that the column
// walks of the micro-GEMMs hit distinct banks.
//
// Backward structure (two launches, no atomics, deterministic):
//   1. query-major  (grid: query tiles x heads): pass 1 over the row's keys
//      forms D_i = sum_j P_ij dP_ij (backward_attention.wgsl, attention_backward
//      Pass A), pass 2 recomputes P, dP, forms dS = scale P (dP - D) and
//      accumulates dQ_i = sum_j dS_ij k_j (Pass B). D goes to the workspace.
//   2. key-major    (grid: key tiles x kv heads): the owner of a key tile loops
//      over the query tiles that can see it and over the query heads of its
//      group, recomputes P and dS, and sums dV = P^T dO and dK = dS^T Q for
//      the whole group before one owned write (the key-major idea of
//      attention_backward_short_dKdV, without its O(S^2) scratch).
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"

namespace gqa {
namespace {

// RoPE backward on a gradient row held by the 16 threads of a half-warp:
// column c = tx + 16n, so pair (2p, 2p+1) sits in lanes tx and tx ^ 1. Every
// lane of the warp calls it (it shuffles).
__device__ __forceinline__ void rope_pair_shfl(float& v, int c, long long tpos, int tx,
                                               const RopeParams& rope) {
  const float other = __shfl_xor_sync(0xffffffffu, v, 1);
  float x0 = (tx & 1) ? other : v, x1 = (tx & 1) ? v : other;
  rope_rotate(x0, x1, tpos, c >> 1, rope);
  v = (tx & 1) ? x1 : x0;
}

constexpr int BT = 64;          // tile rows / cols
constexpr int NT = 256;         // threads per block
constexpr int PS = BT + 1;      // row stride of 64x64 score tiles

template <int DP>
struct Tile {
  float v[BT][DP + 1];
};

struct ScoreTile {
  float v[BT][PS];
};

// Load rows [r0, r0 + BT) of a row-major matrix (row stride ld floats), columns
// [col0, col0 + d), into a tile; rows >= nrow_valid and columns >= d read zero.
template <int DP>
__device__ __forceinline__ void load_tile(Tile<DP>& t, const float* __restrict__ X, long long ld,
                                          int col0, int r0, int nrow_valid, int d) {
  constexpr int C4 = DP / 4;
  for (int idx = threadIdx.x; idx < BT * C4; idx += NT) {
    const int r = idx / C4, c = (idx % C4) * 4;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < nrow_valid && c < d)
      x = __ldg(reinterpret_cast<const float4*>(X + (long long)(r0 + r) * ld + col0 + c));
    t.v[r][c + 0] = x.x;
    t.v[r][c + 1] = x.y;
    t.v[r][c + 2] = x.z;
    t.v[r][c + 3] = x.w;
  }
}

// acc[i][j] = sum_k A[4ty+i][k] * B[tx+16j][k]
template <int DP>
__device__ __forceinline__ void mm_abt(const Tile<DP>& A, const Tile<DP>& B, float acc[4][4]) {
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 8
  for (int k = 0; k < DP; ++k) {
    float a[4], b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = A.v[4 * ty + i][k];
#pragma unroll
    for (int j = 0; j < 4; ++j) b[j] = B.v[tx + 16 * j][k];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
  }
}

// out[i][n] += sum_c M[4ty+i][c] * X[c][tx+16n]
template <int DP>
__device__ __forceinline__ void mm_ab_acc(const ScoreTile& M, const Tile<DP>& X,
                                          float out[4][DP / 16]) {
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
#pragma unroll 4
  for (int c = 0; c < BT; ++c) {
    float m[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) m[i] = M.v[4 * ty + i][c];
#pragma unroll
    for (int n = 0; n < DP / 16; ++n) {
      const float x = X.v[c][tx + 16 * n];
#pragma unroll
      for (int i = 0; i < 4; ++i) out[i][n] = fmaf(m[i], x, out[i][n]);
    }
  }
}

__device__ __forceinline__ float half_warp_sum(float v) {
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float half_warp_max(float v) {
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Smallest seg over rows [r0, min(r0 + BT, S)) of a query tile (block-wide).
__device__ unsigned tile_min_seg(const uint32_t* __restrict__ seg, int r0, int S, unsigned* red) {
  unsigned v = 0xffffffffu;
  if (threadIdx.x < BT && r0 + (int)threadIdx.x < S) v = __ldg(seg + r0 + threadIdx.x);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x / 32] = v;
  __syncthreads();
  unsigned m = red[0];
  for (int w = 1; w < NT / 32; ++w) m = min(m, red[w]);
  __syncthreads();
  return m;
}

// ---------------------------------------------------------------------------
// Forward: O and LSE, online softmax over the row's visible key tiles.
// ---------------------------------------------------------------------------
template <int DP>
struct FwdSmem {
  Tile<DP> q, k, v;
  ScoreTile p;
  unsigned red[NT / 32];
};

template <int DP>
__global__ void __launch_bounds__(NT) fwd_kernel(const float* __restrict__ Q,
                                                 const float* __restrict__ K,
                                                 const float* __restrict__ V,
                                                 const uint32_t* __restrict__ seg,
                                                 float* __restrict__ O, float* __restrict__ LSE,
                                                 Shape sh) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  FwdSmem<DP>& sm = *reinterpret_cast<FwdSmem<DP>*>(smem_raw);
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  const int q0 = blockIdx.x * BT, h = blockIdx.y, g = h / sh.G;
  const int S = sh.S, d = sh.d;
  const long long ldq = (long long)sh.H * d, ldk = (long long)sh.Hk * d;
  const float sl2 = sh.scale * kLog2e;

  load_tile<DP>(sm.q, Q, ldq, h * d, q0, min(BT, S - q0), d);
  int row[4];
  unsigned rseg[4];
  float m[4], l[4], acc[4][DP / 16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    row[i] = q0 + 4 * ty + i;
    rseg[i] = row[i] < S ? __ldg(seg + row[i]) : 0u;
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int n = 0; n < DP / 16; ++n) acc[i][n] = 0.f;
  }
  const int kt0 = (int)(tile_min_seg(seg, q0, S, sm.red) / BT);
  const int kt1 = min(q0 + BT - 1, S - 1) / BT;
  for (int kt = kt0; kt <= kt1; ++kt) {
    const int k0 = kt * BT;
    load_tile<DP>(sm.k, K, ldk, g * d, k0, min(BT, S - k0), d);
    load_tile<DP>(sm.v, V, ldk, g * d, k0, min(BT, S - k0), d);
    __syncthreads();
    float s[4][4];
    mm_abt<DP>(sm.q, sm.k, s);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float tmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int key = k0 + tx + 16 * j;
        const bool ok = row[i] < S && key <= row[i] && (unsigned)key >= rseg[i];
        s[i][j] = ok ? s[i][j] * sl2 : -INFINITY;   // log2 domain
        tmax = fmaxf(tmax, s[i][j]);
      }
      tmax = half_warp_max(tmax);
      const float mn = fmaxf(m[i], tmax);
      const float corr = (mn == -INFINITY) ? 1.f : exp2f(m[i] - mn);
      float rs = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float p = (s[i][j] == -INFINITY) ? 0.f : exp2f(s[i][j] - mn);
        sm.p.v[4 * ty + i][tx + 16 * j] = p;
        rs += p;
      }
      l[i] = l[i] * corr + half_warp_sum(rs);
      m[i] = mn;
#pragma unroll
      for (int n = 0; n < DP / 16; ++n) acc[i][n] *= corr;
    }
    __syncthreads();
    mm_ab_acc<DP>(sm.p, sm.v, acc);
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (row[i] >= S) continue;
    const float inv = 1.f / l[i];
#pragma unroll
    for (int n = 0; n < DP / 16; ++n) {
      const int c = tx + 16 * n;
      if (c < d) O[(long long)row[i] * ldq + h * d + c] = acc[i][n] * inv;
    }
    if (tx == 0) LSE[(long long)row[i] * sh.H + h] = (m[i] + log2f(l[i])) / kLog2e;
  }
}

// ---------------------------------------------------------------------------
// Backward 1 (query-major): D for every (row, head) and dQ += dS K.
// ---------------------------------------------------------------------------
template <int DP>
struct QmSmem {
  Tile<DP> q, dout, k, v;
  ScoreTile ds;
  unsigned red[NT / 32];
};

template <int DP>
__global__ void __launch_bounds__(NT) bwd_query_major(
    const float* __restrict__ Q, const float* __restrict__ K, const float* __restrict__ V,
    const float* __restrict__ dO, const float* __restrict__ LSE, const uint32_t* __restrict__ seg,
    float* __restrict__ dQ, float* __restrict__ Dws, uint32_t* __restrict__ minseg64, Shape sh,
    const RopeParams rope, uint32_t* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  QmSmem<DP>& sm = *reinterpret_cast<QmSmem<DP>*>(smem_raw);
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  const int q0 = blockIdx.x * BT, h = blockIdx.y, g = h / sh.G;
  const int S = sh.S, d = sh.d;
  const long long ldq = (long long)sh.H * d, ldk = (long long)sh.Hk * d;
  const float sl2 = sh.scale * kLog2e;

  load_tile<DP>(sm.q, Q, ldq, h * d, q0, min(BT, S - q0), d);
  load_tile<DP>(sm.dout, dO, ldq, h * d, q0, min(BT, S - q0), d);
  int row[4];
  unsigned rseg[4];
  float lse2[4], Dp[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    row[i] = q0 + 4 * ty + i;
    rseg[i] = row[i] < S ? __ldg(seg + row[i]) : 0u;
    lse2[i] = row[i] < S ? __ldg(LSE + (long long)row[i] * sh.H + h) * kLog2e : 0.f;
    Dp[i] = 0.f;
  }
  const unsigned mseg = tile_min_seg(seg, q0, S, sm.red);
  if (h == 0 && threadIdx.x == 0) minseg64[blockIdx.x] = mseg;
  const int kt0 = (int)(mseg / BT);
  const int kt1 = min(q0 + BT - 1, S - 1) / BT;

  // Pass 1: D_i = sum_j P_ij dP_ij
  for (int kt = kt0; kt <= kt1; ++kt) {
    const int k0 = kt * BT;
    load_tile<DP>(sm.k, K, ldk, g * d, k0, min(BT, S - k0), d);
    load_tile<DP>(sm.v, V, ldk, g * d, k0, min(BT, S - k0), d);
    __syncthreads();
    float s[4][4], dp[4][4];
    mm_abt<DP>(sm.q, sm.k, s);
    mm_abt<DP>(sm.dout, sm.v, dp);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int key = k0 + tx + 16 * j;
        const bool ok = row[i] < S && key <= row[i] && (unsigned)key >= rseg[i];
        const float p = ok ? exp2f(s[i][j] * sl2 - lse2[i]) : 0.f;
        Dp[i] = fmaf(p, dp[i][j], Dp[i]);
      }
    __syncthreads();
  }
  float D[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    D[i] = half_warp_sum(Dp[i]);
    if (tx == 0 && row[i] < S &&
        GQA_DCHECK(status, h < sh.H && (long long)row[i] * sh.H + h < (long long)S * sh.H, kChkSimt))
      Dws[(long long)row[i] * sh.H + h] = D[i];
  }

  // Pass 2: dS = scale P (dP - D), dQ_i += sum_j dS_ij k_j
  float acc[4][DP / 16];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int n = 0; n < DP / 16; ++n) acc[i][n] = 0.f;
  for (int kt = kt0; kt <= kt1; ++kt) {
    const int k0 = kt * BT;
    load_tile<DP>(sm.k, K, ldk, g * d, k0, min(BT, S - k0), d);
    load_tile<DP>(sm.v, V, ldk, g * d, k0, min(BT, S - k0), d);
    __syncthreads();
    float s[4][4], dp[4][4];
    mm_abt<DP>(sm.q, sm.k, s);
    mm_abt<DP>(sm.dout, sm.v, dp);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int key = k0 + tx + 16 * j;
        const bool ok = row[i] < S && key <= row[i] && (unsigned)key >= rseg[i];
        const float p = ok ? exp2f(s[i][j] * sl2 - lse2[i]) : 0.f;
        sm.ds.v[4 * ty + i][tx + 16 * j] = ok ? sh.scale * p * (dp[i][j] - D[i]) : 0.f;
      }
    __syncthreads();
    mm_ab_acc<DP>(sm.ds, sm.k, acc);
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int n = 0; n < DP / 16; ++n) {
      const int c = tx + 16 * n;
      float v = acc[i][n];
      v = (v == v) ? v : 0.f;   // NaN guard on the final write, as the pages do
      if (rope.on) rope_pair_shfl(v, c, (long long)row[i] + rope.pos_offset, tx, rope);
      if (row[i] < S && c < d &&
          GQA_DCHECK(status, (long long)row[i] * ldq + h * d + c < (long long)S * ldq, kChkSimt))
        dQ[(long long)row[i] * ldq + h * d + c] += v;
    }
  }
}

// ---------------------------------------------------------------------------
// Backward 2 (key-major): dK, dV for a key tile, summed over the GQA group.
// ---------------------------------------------------------------------------
template <int DP>
struct KmSmem {
  Tile<DP> k, v, q, dout;
  ScoreTile pt, dst;
};

template <int DP>
__global__ void __launch_bounds__(NT) bwd_key_major(
    const float* __restrict__ Q, const float* __restrict__ K, const float* __restrict__ V,
    const float* __restrict__ dO, const float* __restrict__ LSE, const uint32_t* __restrict__ seg,
    const float* __restrict__ Dws, const uint32_t* __restrict__ minseg64, float* __restrict__ dK,
    float* __restrict__ dV, Shape sh, const RopeParams rope, uint32_t* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  KmSmem<DP>& sm = *reinterpret_cast<KmSmem<DP>*>(smem_raw);
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  const int k0 = blockIdx.x * BT, g = blockIdx.y;
  const int S = sh.S, d = sh.d;
  const long long ldq = (long long)sh.H * d, ldk = (long long)sh.Hk * d;
  const float sl2 = sh.scale * kLog2e;
  const int k_hi = min(k0 + BT, S) - 1;

  load_tile<DP>(sm.k, K, ldk, g * d, k0, min(BT, S - k0), d);
  load_tile<DP>(sm.v, V, ldk, g * d, k0, min(BT, S - k0), d);
  float dk[4][DP / 16], dv[4][DP / 16];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int n = 0; n < DP / 16; ++n) dk[i][n] = dv[i][n] = 0.f;

  const int nqt = (S + BT - 1) / BT;
  for (int qt = k0 / BT; qt < nqt; ++qt) {
    if ((int)__ldg(minseg64 + qt) > k_hi) continue;      // no row of this tile sees these keys
    const int q0 = qt * BT;
    int qrow[4];
    unsigned qseg[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      qrow[j] = q0 + tx + 16 * j;
      qseg[j] = qrow[j] < S ? __ldg(seg + qrow[j]) : 0u;
    }
    for (int h = g * sh.G; h < (g + 1) * sh.G; ++h) {
      __syncthreads();   // previous iteration's readers of q, dout, pt, dst are done
      load_tile<DP>(sm.q, Q, ldq, h * d, q0, min(BT, S - q0), d);
      load_tile<DP>(sm.dout, dO, ldq, h * d, q0, min(BT, S - q0), d);
      float lse2[4], Dq[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        lse2[j] = qrow[j] < S ? __ldg(LSE + (long long)qrow[j] * sh.H + h) * kLog2e : 0.f;
        Dq[j] = qrow[j] < S ? Dws[(long long)qrow[j] * sh.H + h] : 0.f;
      }
      __syncthreads();
      float s[4][4], dp[4][4];
      mm_abt<DP>(sm.k, sm.q, s);       // S^T: rows = keys, cols = queries
      mm_abt<DP>(sm.v, sm.dout, dp);   // dP^T
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int key = k0 + 4 * ty + i;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const bool ok = qrow[j] < S && key <= qrow[j] && (unsigned)key >= qseg[j];
          const float p = ok ? exp2f(s[i][j] * sl2 - lse2[j]) : 0.f;
          sm.pt.v[4 * ty + i][tx + 16 * j] = p;
          sm.dst.v[4 * ty + i][tx + 16 * j] = ok ? sh.scale * p * (dp[i][j] - Dq[j]) : 0.f;
        }
      }
      __syncthreads();
      mm_ab_acc<DP>(sm.pt, sm.dout, dv);
      mm_ab_acc<DP>(sm.dst, sm.q, dk);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int key = k0 + 4 * ty + i;
#pragma unroll
    for (int n = 0; n < DP / 16; ++n) {
      const int c = tx + 16 * n;
      float a = dk[i][n];
      const float b = dv[i][n];
      a = (a == a) ? a : 0.f;
      if (rope.on) rope_pair_shfl(a, c, (long long)key + rope.pos_offset, tx, rope);
      if (key < S && c < d &&
          GQA_DCHECK(status, g < sh.Hk && (long long)key * ldk + g * d + c < (long long)S * ldk,
                     kChkSimt)) {
        const long long o = (long long)key * ldk + g * d + c;
        dK[o] += a;
        dV[o] += (b == b) ? b : 0.f;
      }
    }
  }
}

template <class Kern>
cudaError_t allow_smem(Kern k, size_t bytes) {
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int DP>
gqa_status fwd_launch(const float* Q, const float* K, const float* V, const uint32_t* seg,
                      float* O, float* LSE, const Shape& sh, cudaStream_t st) {
  const size_t smem = sizeof(FwdSmem<DP>);
  if (allow_smem(fwd_kernel<DP>, smem) != cudaSuccess) return check_launch("fwd smem attribute");
  dim3 grid((sh.S + BT - 1) / BT, sh.H);
  fwd_kernel<DP><<<grid, NT, smem, st>>>(Q, K, V, seg, O, LSE, sh);
  note_launch();
  return check_launch("simt forward");
}

template <int DP>
gqa_status bwd_launch(const float* Q, const float* K, const float* V, const float* dO,
                      const float* LSE, const uint32_t* seg, float* dQ, float* dK, float* dV,
                      const Shape& sh, char* ws, cudaStream_t st, const RopeParams& rope) {
  const WsLayout L = ws_layout(sh.S, sh.H);
  float* Dws = reinterpret_cast<float*>(ws + L.d_off);
  uint32_t* minseg = reinterpret_cast<uint32_t*>(ws + L.minseg64);
  const size_t s1 = sizeof(QmSmem<DP>), s2 = sizeof(KmSmem<DP>);
  if (allow_smem(bwd_query_major<DP>, s1) != cudaSuccess) return check_launch("bwd smem attribute");
  if (allow_smem(bwd_key_major<DP>, s2) != cudaSuccess) return check_launch("bwd smem attribute");
  const int nt = (sh.S + BT - 1) / BT;
  profile_before(st, "simt_bwd_query_major+key_major");
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  bwd_query_major<DP><<<dim3(nt, sh.H), NT, s1, st>>>(Q, K, V, dO, LSE, seg, dQ, Dws, minseg, sh, rope,
                                                      status);
  note_launch();
  gqa_status r = check_launch("simt backward (query-major)");
  if (r != GQA_OK) return r;
  bwd_key_major<DP><<<dim3(nt, sh.Hk), NT, s2, st>>>(Q, K, V, dO, LSE, seg, Dws, minseg, dK, dV, sh, rope,
                                                      status);
  note_launch();
  profile_after(st);
  return check_launch("simt backward (key-major)");
}

// Smallest (and optionally largest) seg over each `tile`-row query tile (one warp per tile).
__global__ void tile_minseg_kernel(const uint32_t* __restrict__ seg, int S, int tile,
                                   uint32_t* __restrict__ out, uint32_t* __restrict__ out_max,
                                   int n_tiles) {
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) / 32, lane = threadIdx.x % 32;
  if (w >= n_tiles) return;
  unsigned v = 0xffffffffu, m = 0u;
  for (int i = lane; i < tile; i += 32) {
    const int q = w * tile + i;
    if (q < S) {
      const unsigned x = __ldg(seg + q);
      v = min(v, x);
      m = max(m, x);
    }
  }
  for (int o = 16; o >= 1; o >>= 1) {
    v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  }
  if (lane == 0) {
    out[w] = v;
    if (out_max) out_max[w] = m;
  }
}

#ifdef GQA_CHECKS
// Debug build: flags seg[s] > s (the precondition every path relies on).
__global__ void seg_check_kernel(const uint32_t* __restrict__ seg, int S, uint32_t* status) {
  for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < S; s += gridDim.x * blockDim.x)
    if (__ldg(seg + s) > (uint32_t)s) atomicOr(status, kStatusCheck | kChkSeg);
}
#endif

}  // namespace

gqa_status debug_check_seg(const uint32_t* seg, int S, void* ws, cudaStream_t st) {
#ifdef GQA_CHECKS
  if (S <= 0) return GQA_OK;
  const int blocks = (S + 255) / 256 < 1024 ? (S + 255) / 256 : 1024;
  seg_check_kernel<<<blocks, 256, 0, st>>>(seg, S, reinterpret_cast<uint32_t*>(ws));
  note_launch();
  return check_launch("seg check (debug build)");
#else
  (void)seg; (void)S; (void)ws; (void)st;
  return GQA_OK;
#endif
}

gqa_status tile_minseg(const uint32_t* seg, int S, int tile, uint32_t* out, cudaStream_t st,
                       uint32_t* out_max) {
  const int n_tiles = (S + tile - 1) / tile;
  const int warps_per_block = 8;
  tile_minseg_kernel<<<(n_tiles + warps_per_block - 1) / warps_per_block, 32 * warps_per_block, 0,
                       st>>>(seg, S, tile, out, out_max, n_tiles);
  note_launch();
  return check_launch("tile min seg");
}


gqa_status simt_fwd_lse(const float* Q, const float* K, const float* V, const uint32_t* seg,
                        float* O, float* LSE, const Shape& sh, cudaStream_t st) {
  if (sh.d <= 32) return fwd_launch<32>(Q, K, V, seg, O, LSE, sh, st);
  if (sh.d <= 64) return fwd_launch<64>(Q, K, V, seg, O, LSE, sh, st);
  return fwd_launch<128>(Q, K, V, seg, O, LSE, sh, st);
}

gqa_status simt_bwd(const float* Q, const float* K, const float* V, const float* dO,
                    const float* LSE, const uint32_t* seg, float* dQ, float* dK, float* dV,
                    const Shape& sh, char* ws, cudaStream_t st, const RopeParams& rope) {
  if (sh.d <= 32) return bwd_launch<32>(Q, K, V, dO, LSE, seg, dQ, dK, dV, sh, ws, st, rope);
  if (sh.d <= 64) return bwd_launch<64>(Q, K, V, dO, LSE, seg, dQ, dK, dV, sh, ws, st, rope);
  return bwd_launch<128>(Q, K, V, dO, LSE, seg, dQ, dK, dV, sh, ws, st, rope);
}

}  // namespace gqa
