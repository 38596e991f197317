// Single-launch backward for short sequences (seq_len <= 2048 and a bounded
// amount of work): the whole backward of causal GQA attention from a saved LSE
// in ONE cooperative launch, for shapes where the two tensor-core kernels and
// their set-up launches are bound by latency, not by arithmetic.
//
// The pages' short path (backward_attention.wgsl, attention_backward_short and
// attention_backward_short_dKdV) also exists for short sequences; it keeps
// P and dS for every (query, key, head) in an O(S^2 H) scratch buffer. Here
// nothing of size S^2 is kept: the work is cut into cells (query tile of 32
// rows, key tile of 32 keys, query head) and the kernel runs three phases
// separated by grid-wide barriers (all CTAs are co-resident: cooperative
// launch; every wait is bounded):
//   A. per visible cell: S = Q K^T, dP = dO V^T, P = exp(scale s - LSE), and
//      the cell's share of D_i = sum_j P_ij dP_ij (a partial row sum);
//   B. per visible cell: D_i = the row's partials summed in key-tile order,
//      S and dP again, dS = scale P (dP - D), and the cell's partial
//      gradients dQ = dS K, dK = dS^T Q, dV = P^T dO (each 32 x d);
//   C. per output tile and group of rows (512 / DP rows, one float4 per
//      thread): the partials summed in a fixed order (dQ over key tiles; dK,
//      dV over the group's query heads, then query tiles), NaN -> 0, the
//      RoPE backward where asked, and one += into dQ / dK / dV.
// Deterministic (fixed summation order, no atomics on data); fp32 FFMA on
// CUDA cores, exact fp32 products.
#include <cuda_runtime.h>
#include <math.h>

#include <atomic>

#include "common.cuh"

namespace gqa {
namespace {

constexpr int kT = 32;           // query-tile rows = key-tile keys
constexpr int kThr = 128;        // threads per CTA
constexpr int kMaxTiles = 64;    // seq_len <= 2048
constexpr long long kGridWaitCycles = 2000000000LL;   // ~1 s at 2 GHz
constexpr uint32_t kSiteBarrier1 = 0x100u, kSiteBarrier2 = 0x200u, kSiteSelftest = 0x400u;
constexpr size_t kBarrierOffset = 128;                 // barrier counter: header byte 128

// Thread t: tr = t / 8 (0..15), tc = t % 8. In a 32 x 32 score tile it holds
// rows tr + 16 i (i < 2) and columns tc + 8 j (j < 4); the 8 threads of a row
// are 8 consecutive lanes (row sums: three xor-shuffles). In a 32 x DP
// gradient tile it holds rows tr + 16 i and the float4 column groups
// tc + 8 n (n < DP / 32).
template <int DP>
struct ShortSmem {
  float q[kT][DP + 4];      // Q rows of the query tile, head h (row stride DP+4: float4 loads
  float dout[kT][DP + 4];   // dO rows                          of 8 rows hit 32 distinct banks)
  float k[kT][DP + 4];      // K rows of the key tile, kv head h / G
  float v[kT][DP + 4];      // V rows
  float p[kT][kT + 1];      // P  [query][key]
  float ds[kT][kT + 1];     // dS [query][key]
  float dsum[kT];           // D of the query tile's rows
  float lse2[kT];           // LSE * log2(e)
  uint32_t seg[kT];
  uint32_t tmin[kMaxTiles]; // smallest seg of each query tile (phases B, C)
  int ok;
};

struct ShortArgs {
  const float *Q, *K, *V, *dO, *LSE;
  const uint32_t* seg;
  float *dQ, *dK, *dV;
  uint32_t* status;      // header word 0
  unsigned* barrier;     // header byte 128
  uint32_t* tminseg;     // [nt]
  float* dpart;          // [H][ntri][32]
  float *dqp, *dkp, *dvp;   // [H][ntri][32][DP]
  int nt, ntri;
};

__device__ __forceinline__ int tri_index(int qt, int kt) { return qt * (qt + 1) / 2 + kt; }

// (qt, kt) of a lower-triangle index t = qt (qt + 1) / 2 + kt, kt <= qt.
__device__ __forceinline__ void tri_decode(int t, int& qt, int& kt) {
  int q = (int)((sqrtf(8.f * (float)t + 1.f) - 1.f) * 0.5f);
  while (q * (q + 1) / 2 > t) --q;
  while ((q + 1) * (q + 2) / 2 <= t) ++q;
  qt = q;
  kt = t - q * (q + 1) / 2;
}

// Key tile kt holds a key that a row of query tile qt may see.
__device__ __forceinline__ bool visible(int qt, int kt, uint32_t tmin) {
  return kt <= qt && tmin <= (uint32_t)(kt * kT + kT - 1);
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier of a cooperative launch. Thread 0 of each CTA arrives
// (release: fence, then the counter add) and waits (acquire) for `target`
// arrivals. Bounded: after `limit` SM cycles it records `site` in the status
// word and returns false; it also returns false as soon as another CTA has
// given up (status word non-zero).
__device__ bool grid_barrier(const ShortArgs& a, unsigned target, uint32_t site, int* ok_flag,
                             long long limit = kGridWaitCycles) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    __threadfence();
    atomicAdd(a.barrier, 1u);
    if (ld_acquire(a.barrier) < target) {
      const long long t0 = clock64();
      while (ld_acquire(a.barrier) < target) {
        if (*(volatile uint32_t*)a.status != 0u) { ok = 0; break; }
        if (clock64() - t0 > limit) {
          atomicOr(a.status, 0x80000000u | site);
          ok = 0;
          break;
        }
      }
    }
    __threadfence();
    *ok_flag = ok;
  }
  __syncthreads();
  return *ok_flag != 0;
}

// 16-byte asynchronous copy global -> shared (cp.async, L2 only); with
// valid == false nothing is read and the 16 bytes are zero-filled.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
               :: "r"(s), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Start copying rows [r0, r0 + 32) of a row-major matrix (row stride ld),
// columns [col0, col0 + d), into a tile; rows >= nvalid and columns >= d are
// zero-filled. All four tiles of a cell are in flight at once; the caller
// waits with cp_async_wait_all() and a CTA barrier.
template <int DP>
__device__ __forceinline__ void load_rows_async(float (*dst)[DP + 4], const float* __restrict__ X,
                                                long long ld, int col0, int r0, int nvalid, int d) {
  constexpr int C4 = DP / 4;
  for (int idx = threadIdx.x; idx < kT * C4; idx += kThr) {
    const int r = idx / C4, c = (idx % C4) * 4;
    const bool ok = r < nvalid && c < d;
    cp_async16(&dst[r][c], ok ? X + (long long)(r0 + r) * ld + col0 + c : X, ok);
  }
}

// Sum of the float4s at p + u * stride, u in [0, n), in order of u, with
// eight loads in flight (the partials were written by other CTAs before a
// grid barrier: loads through L2 only).
__device__ __forceinline__ float4 sum_strided(const float* __restrict__ p, size_t stride, int n) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int u0 = 0; u0 < n; u0 += 8) {
    float4 x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      x[u] = (u0 + u < n) ? __ldcg(reinterpret_cast<const float4*>(p + (size_t)(u0 + u) * stride))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      acc.x += x[u].x; acc.y += x[u].y; acc.z += x[u].z; acc.w += x[u].w;
    }
  }
  return acc;
}

// acc[i][j] = sum_k A[tr + 16i][k] B[tc + 8j][k]
template <int DP>
__device__ __forceinline__ void mm_abt(const float (*A)[DP + 4], const float (*B)[DP + 4],
                                       float acc[2][4]) {
  const int tr = threadIdx.x / 8, tc = threadIdx.x % 8;
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 4
  for (int k = 0; k < DP; k += 4) {
    const float4 a0 = *reinterpret_cast<const float4*>(&A[tr][k]);
    const float4 a1 = *reinterpret_cast<const float4*>(&A[tr + 16][k]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 b = *reinterpret_cast<const float4*>(&B[tc + 8 * j][k]);
      acc[0][j] = fmaf(a0.x, b.x, fmaf(a0.y, b.y, fmaf(a0.z, b.z, fmaf(a0.w, b.w, acc[0][j]))));
      acc[1][j] = fmaf(a1.x, b.x, fmaf(a1.y, b.y, fmaf(a1.z, b.z, fmaf(a1.w, b.w, acc[1][j]))));
    }
  }
}

__device__ __forceinline__ void fma4(float4& o, float m, const float4& x) {
  o.x = fmaf(m, x.x, o.x);
  o.y = fmaf(m, x.y, o.y);
  o.z = fmaf(m, x.z, o.z);
  o.w = fmaf(m, x.w, o.w);
}

// out[i][n] = sum_c M[tr + 16i][c] X[c][4(tc + 8n) .. +3]        (kTrans = false)
// out[i][n] = sum_c M[c][tr + 16i] X[c][4(tc + 8n) .. +3]        (kTrans = true)
template <int DP, bool kTrans>
__device__ __forceinline__ void mm_score_rows(const float (*M)[kT + 1], const float (*X)[DP + 4],
                                              float4 out[2][DP / 32]) {
  const int tr = threadIdx.x / 8, tc = threadIdx.x % 8;
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int n = 0; n < DP / 32; ++n) out[i][n] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int c = 0; c < kT; ++c) {
    const float m0 = kTrans ? M[c][tr] : M[tr][c];
    const float m1 = kTrans ? M[c][tr + 16] : M[tr + 16][c];
#pragma unroll
    for (int n = 0; n < DP / 32; ++n) {
      const float4 x = *reinterpret_cast<const float4*>(&X[c][4 * (tc + 8 * n)]);
      fma4(out[0][n], m0, x);
      fma4(out[1][n], m1, x);
    }
  }
}

template <int DP>
__device__ __forceinline__ void store_partial(float* __restrict__ dst, const float4 out[2][DP / 32]) {
  const int tr = threadIdx.x / 8, tc = threadIdx.x % 8;
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int n = 0; n < DP / 32; ++n)
      *reinterpret_cast<float4*>(dst + (size_t)(tr + 16 * i) * DP + 4 * (tc + 8 * n)) = out[i][n];
}

// Smallest seg over the valid rows of query tile qt (every warp computes it).
__device__ __forceinline__ uint32_t tile_min_seg32(const uint32_t* __restrict__ seg, int q0, int S) {
  const int lane = threadIdx.x & 31;
  uint32_t v = (q0 + lane < S) ? __ldg(seg + q0 + lane) : 0xffffffffu;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float nan_to_zero(float x) { return (x == x) ? x : 0.f; }

template <int DP>
__global__ void __launch_bounds__(kThr) short_bwd_kernel(const ShortArgs a, const Shape sh,
                                                         const RopeParams rope) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  ShortSmem<DP>& sm = *reinterpret_cast<ShortSmem<DP>*>(smem_raw);
  const int S = sh.S, d = sh.d, G = sh.G;
  const long long ldq = (long long)sh.H * d, ldk = (long long)sh.Hk * d;
  const float sl2 = sh.scale * kLog2e;
  const int tr = threadIdx.x / 8, tc = threadIdx.x % 8;
  const int n_cells = sh.H * a.ntri;

  // ---- phase A: partial row sums of P * dP -----------------------------
  // The CTA's last visible cell keeps its tiles in shared memory and its P
  // and dP in registers: phase B, which walks the cells in reverse, starts
  // with that cell and reuses them.
  int kept = -1;
  float kp[2][4], kdp[2][4];
  for (int cell = blockIdx.x; cell < n_cells; cell += gridDim.x) {
    const int h = cell / a.ntri;
    int qt, kt;
    tri_decode(cell - h * a.ntri, qt, kt);
    const int q0 = qt * kT, k0 = kt * kT, g = h / G;
    const uint32_t tmin = tile_min_seg32(a.seg, q0, S);
    if (h == 0 && kt == qt && threadIdx.x == 0) a.tminseg[qt] = tmin;
    if (!visible(qt, kt, tmin)) continue;
    __syncthreads();   // the previous cell's readers of the tiles are done
    load_rows_async<DP>(sm.q, a.Q, ldq, h * d, q0, S - q0, d);
    load_rows_async<DP>(sm.dout, a.dO, ldq, h * d, q0, S - q0, d);
    load_rows_async<DP>(sm.k, a.K, ldk, g * d, k0, S - k0, d);
    load_rows_async<DP>(sm.v, a.V, ldk, g * d, k0, S - k0, d);
    if (threadIdx.x < kT) {
      const int row = q0 + threadIdx.x;
      sm.seg[threadIdx.x] = row < S ? __ldg(a.seg + row) : 0u;
      sm.lse2[threadIdx.x] = row < S ? __ldg(a.LSE + (long long)row * sh.H + h) * kLog2e : 0.f;
    }
    cp_async_wait_all();
    __syncthreads();
    float s[2][4], dp[2][4];
    mm_abt<DP>(sm.q, sm.k, s);
    mm_abt<DP>(sm.dout, sm.v, dp);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = tr + 16 * i, row = q0 + r;
      float part = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int key = k0 + tc + 8 * j;
        const bool ok = row < S && key <= row && (uint32_t)key >= sm.seg[r];
        const float p = ok ? exp2f(s[i][j] * sl2 - sm.lse2[r]) : 0.f;
        part = fmaf(p, dp[i][j], part);
        kp[i][j] = p;
        kdp[i][j] = dp[i][j];
      }
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
      part += __shfl_xor_sync(0xffffffffu, part, 4);
      if (tc == 0) a.dpart[(size_t)cell * kT + r] = part;
    }
    kept = cell;
  }
  if (!grid_barrier(a, gridDim.x, kSiteBarrier1, &sm.ok)) return;

  for (int t = threadIdx.x; t < a.nt; t += kThr) sm.tmin[t] = __ldcg(a.tminseg + t);
  __syncthreads();

  // ---- phase B: dS and the cells' partial gradients ----------------------
  const int last = (int)blockIdx.x < n_cells
                       ? (int)blockIdx.x + ((n_cells - 1 - (int)blockIdx.x) / (int)gridDim.x) * (int)gridDim.x
                       : -1;
  for (int cell = last; cell >= (int)blockIdx.x; cell -= gridDim.x) {
    const int h = cell / a.ntri;
    int qt, kt;
    tri_decode(cell - h * a.ntri, qt, kt);
    const uint32_t tmin = sm.tmin[qt];
    if (!visible(qt, kt, tmin)) continue;
    const int q0 = qt * kT, k0 = kt * kT, g = h / G;
    const bool reuse = cell == kept;   // first cell of this walk: tiles, P, dP still here
    if (!reuse) {
      __syncthreads();
      load_rows_async<DP>(sm.q, a.Q, ldq, h * d, q0, S - q0, d);
      load_rows_async<DP>(sm.dout, a.dO, ldq, h * d, q0, S - q0, d);
      load_rows_async<DP>(sm.k, a.K, ldk, g * d, k0, S - k0, d);
      load_rows_async<DP>(sm.v, a.V, ldk, g * d, k0, S - k0, d);
    }
    if (threadIdx.x < kT) {
      // D of row r: its partials over the visible key tiles k2 = tmin/32 .. qt
      // (consecutive cells), in order, eight loads in flight
      const int r = threadIdx.x, row = q0 + r;
      float D = 0.f;
      if (row < S) {
        const int k_lo = (int)(tmin / kT), n = qt - k_lo + 1;
        const float* p = a.dpart + ((size_t)h * a.ntri + tri_index(qt, k_lo)) * kT + r;
        for (int u0 = 0; u0 < n; u0 += 8) {
          float x[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) x[u] = (u0 + u < n) ? __ldcg(p + (size_t)(u0 + u) * kT) : 0.f;
#pragma unroll
          for (int u = 0; u < 8; ++u) D += x[u];
        }
      }
      sm.dsum[r] = D;
      if (!reuse) {
        sm.seg[r] = row < S ? __ldg(a.seg + row) : 0u;
        sm.lse2[r] = row < S ? __ldg(a.LSE + (long long)row * sh.H + h) * kLog2e : 0.f;
      }
    }
    if (!reuse) cp_async_wait_all();
    __syncthreads();
    float pv[2][4], dp[2][4];
    if (reuse) {
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          pv[i][j] = kp[i][j];
          dp[i][j] = kdp[i][j];
        }
    } else {
      float s[2][4];
      mm_abt<DP>(sm.q, sm.k, s);
      mm_abt<DP>(sm.dout, sm.v, dp);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = tr + 16 * i, row = q0 + r;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int key = k0 + tc + 8 * j;
          const bool ok = row < S && key <= row && (uint32_t)key >= sm.seg[r];
          pv[i][j] = ok ? exp2f(s[i][j] * sl2 - sm.lse2[r]) : 0.f;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = tr + 16 * i, row = q0 + r;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = tc + 8 * j, key = k0 + c;
        const bool ok = row < S && key <= row && (uint32_t)key >= sm.seg[r];
        sm.p[r][c] = pv[i][j];
        sm.ds[r][c] = ok ? sh.scale * pv[i][j] * (dp[i][j] - sm.dsum[r]) : 0.f;
      }
    }
    __syncthreads();
    const size_t off = (size_t)cell * kT * DP;
    // (debug build: the cell decodes to a tile pair of the triangle)
    const bool cell_ok = GQA_DCHECK(a.status, qt < a.nt && kt <= qt && h < sh.H, kChkShort);
    float4 out[2][DP / 32];
    mm_score_rows<DP, false>(sm.ds, sm.k, out);    // dQ partial = dS K
    if (cell_ok) store_partial<DP>(a.dqp + off, out);
    mm_score_rows<DP, true>(sm.ds, sm.q, out);     // dK partial = dS^T Q
    if (cell_ok) store_partial<DP>(a.dkp + off, out);
    mm_score_rows<DP, true>(sm.p, sm.dout, out);   // dV partial = P^T dO
    if (cell_ok) store_partial<DP>(a.dvp + off, out);
  }
  if (!grid_barrier(a, 2u * gridDim.x, kSiteBarrier2, &sm.ok)) return;

  // ---- phase C: fixed-order sums, RoPE, one += per output element -------
  // Items: (tensor, head or kv head, tile, row group) with 512 / DP rows per
  // item, so that each thread owns one float4 of one row.
  constexpr int Q4 = DP / 4;                 // float4 groups per row
  constexpr int RPI = kThr / Q4;             // rows per item
  constexpr int NRG = kT / RPI;              // row groups per tile
  const int per_head = a.nt * NRG;
  const int n_dq = sh.H * per_head, n_dk = sh.Hk * per_head;
  const int n_items = n_dq + 2 * n_dk;
  const size_t cell_stride = (size_t)kT * DP;
  const int rr = threadIdx.x / Q4, qd = threadIdx.x % Q4;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int kind = item < n_dq ? 0 : (item < n_dq + n_dk ? 1 : 2);   // dQ, dK, dV
    const int it = kind == 0 ? item : (kind == 1 ? item - n_dq : item - n_dq - n_dk);
    const int hh = it / per_head, rem = it % per_head;
    const int tile = rem / NRG, r = (rem % NRG) * RPI + rr;
    const int pos = tile * kT + r;             // row (dQ) or key (dK, dV)
    if (pos >= S || 4 * qd >= d) continue;
    if (!GQA_DCHECK(a.status, hh < (kind == 0 ? sh.H : sh.Hk) && tile < a.nt, kChkShort)) continue;
    float4 acc;
    if (kind == 0) {
      // dQ[pos, head hh]: partials over the visible key tiles (consecutive cells)
      const int k_lo = (int)(sm.tmin[tile] / kT);
      const float* p = a.dqp + ((size_t)hh * a.ntri + tri_index(tile, k_lo)) * cell_stride +
                       (size_t)r * DP + 4 * qd;
      acc = sum_strided(p, cell_stride, tile - k_lo + 1);
    } else {
      // dK / dV[pos, kv head hh]: over the group's heads, then the query
      // tiles that see key tile `tile`, eight loads in flight
      const float* src = (kind == 1 ? a.dkp : a.dvp) + (size_t)r * DP + 4 * qd;
      acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int h = hh * G; h < (hh + 1) * G; ++h) {
        const size_t base = (size_t)h * a.ntri;
        for (int q0t = tile; q0t < a.nt; q0t += 8) {
          float4 x[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int qt = q0t + u;
            x[u] = (qt < a.nt && visible(qt, tile, sm.tmin[qt]))
                       ? __ldcg(reinterpret_cast<const float4*>(src + (base + tri_index(qt, tile)) * cell_stride))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            acc.x += x[u].x; acc.y += x[u].y; acc.z += x[u].z; acc.w += x[u].w;
          }
        }
      }
    }
    acc.x = nan_to_zero(acc.x); acc.y = nan_to_zero(acc.y);
    acc.z = nan_to_zero(acc.z); acc.w = nan_to_zero(acc.w);
    if (rope.on && kind != 2) {
      const long long tpos = (long long)pos + rope.pos_offset;
      rope_rotate(acc.x, acc.y, tpos, 2 * qd, rope);
      rope_rotate(acc.z, acc.w, tpos, 2 * qd + 1, rope);
    }
    float* dst = kind == 0 ? a.dQ + (long long)pos * ldq
                           : (kind == 1 ? a.dK : a.dV) + (long long)pos * ldk;
    float4* o = reinterpret_cast<float4*>(dst + hh * d + 4 * qd);
    float4 cur = *o;
    cur.x += acc.x; cur.y += acc.y; cur.z += acc.z; cur.w += acc.w;
    *o = cur;
  }
}

// Failure-path self-test: two CTAs wait at a grid barrier for one arrival
// more than the grid makes, so the wait runs out after `limit` cycles.
__global__ void grid_barrier_selftest_kernel(const ShortArgs a, long long limit) {
  __shared__ int ok;
  grid_barrier(a, gridDim.x + 1u, kSiteSelftest, &ok, limit);
}

int padded_dim(int d) { return d <= 32 ? 32 : (d <= 64 ? 64 : 128); }

struct ShortLayout {
  size_t tmin_off, dpart_off, dqp_off, dkp_off, dvp_off, total;
  int nt, ntri;
};

ShortLayout short_layout(int S, int H, int d) {
  ShortLayout L;
  const int DP = padded_dim(d);
  L.nt = (S + kT - 1) / kT;
  L.ntri = L.nt * (L.nt + 1) / 2;
  const size_t cells = (size_t)H * L.ntri;
  const size_t part = align256(cells * kT * DP * sizeof(float));
  L.tmin_off = kWsHeader;
  L.dpart_off = L.tmin_off + align256((size_t)L.nt * sizeof(uint32_t));
  L.dqp_off = L.dpart_off + align256(cells * kT * sizeof(float));
  L.dkp_off = L.dqp_off + part;
  L.dvp_off = L.dkp_off + part;
  L.total = L.dvp_off + part;
  return L;
}

// Per device and head-dim variant: co-resident CTAs the cooperative launch
// may use (0 = not yet known; threads that race here compute the same value).
constexpr int kMaxDevices = 64;
std::atomic<int> g_capacity[kMaxDevices][3];

template <int DP>
gqa_status short_launch(const float* Q, const float* K, const float* V, const float* dO,
                        const float* LSE, const uint32_t* seg, float* dQ, float* dK, float* dV,
                        const Shape& sh, char* ws, cudaStream_t st, const RopeParams& rope) {
  const int vi = DP == 32 ? 0 : (DP == 64 ? 1 : 2);
  const size_t smem = sizeof(ShortSmem<DP>);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return check_launch("short path: device");
  if (dev < 0 || dev >= kMaxDevices) return set_error(GQA_ERR_UNSUPPORTED, "device ordinal %d", dev);
  int cap = g_capacity[dev][vi].load(std::memory_order_acquire);
  if (cap == 0) {
    if (cudaFuncSetAttribute(short_bwd_kernel<DP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return check_launch("short path: smem attribute");
    int per_sm = 0, n_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, short_bwd_kernel<DP>, kThr, smem) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return check_launch("short path: occupancy");
    if (per_sm <= 0) return set_error(GQA_ERR_CUDA, "short path: kernel cannot be resident");
    cap = per_sm * n_sm;
    g_capacity[dev][vi].store(cap, std::memory_order_release);   // after the smem attribute is set
  }
  const ShortLayout L = short_layout(sh.S, sh.H, sh.d);
  ShortArgs a;
  a.Q = Q; a.K = K; a.V = V; a.dO = dO; a.LSE = LSE; a.seg = seg;
  a.dQ = dQ; a.dK = dK; a.dV = dV;
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.barrier = reinterpret_cast<unsigned*>(ws + kBarrierOffset);
  a.tminseg = reinterpret_cast<uint32_t*>(ws + L.tmin_off);
  a.dpart = reinterpret_cast<float*>(ws + L.dpart_off);
  a.dqp = reinterpret_cast<float*>(ws + L.dqp_off);
  a.dkp = reinterpret_cast<float*>(ws + L.dkp_off);
  a.dvp = reinterpret_cast<float*>(ws + L.dvp_off);
  a.nt = L.nt;
  a.ntri = L.ntri;
  const long long cells = (long long)sh.H * L.ntri;
  const long long items = (long long)(sh.H + 2 * sh.Hk) * L.nt * (kT * DP / 512);
  long long grid = cells > items ? cells : items;
  if (grid > cap) grid = cap;
  Shape shv = sh;
  RopeParams rp = rope;
  void* args[] = {&a, &shv, &rp};
  profile_before(st, "short_bwd");
  const cudaError_t e = cudaLaunchCooperativeKernel((const void*)short_bwd_kernel<DP>,
                                                    dim3((unsigned)grid), dim3(kThr), args, smem, st);
  note_launch();
  profile_after(st);
  if (e != cudaSuccess) return set_error(GQA_ERR_CUDA, "short path launch: %s", cudaGetErrorString(e));
  return check_launch("short path");
}

}  // namespace

bool short_supported(const Shape& sh) {
  if (sh.S < 1 || sh.S > kT * kMaxTiles || sh.d > 128) return false;
  const long long nt = (sh.S + kT - 1) / kT;
  const long long work = nt * (nt + 1) / 2 * (long long)sh.H * padded_dim(sh.d) * kT * kT;
  return work <= kShortMaxWork;
}

size_t short_ws_bytes(int S, int H, int d) { return short_layout(S, H, d).total; }

gqa_status grid_barrier_selftest(void* workspace, long long limit_cycles, cudaStream_t st) {
  if (cudaMemsetAsync(workspace, 0, kWsHeader, st) != cudaSuccess)
    return check_launch("grid barrier self-test: status reset");
  ShortArgs a{};
  a.status = reinterpret_cast<uint32_t*>(workspace);
  a.barrier = reinterpret_cast<unsigned*>(static_cast<char*>(workspace) + kBarrierOffset);
  long long lim = limit_cycles;
  void* args[] = {&a, &lim};
  const cudaError_t e = cudaLaunchCooperativeKernel((const void*)grid_barrier_selftest_kernel,
                                                    dim3(2), dim3(32), args, 0, st);
  note_launch();
  if (e != cudaSuccess)
    return set_error(GQA_ERR_CUDA, "grid barrier self-test launch: %s", cudaGetErrorString(e));
  return check_launch("grid barrier self-test");
}

gqa_status short_bwd(const float* Q, const float* K, const float* V, const float* dO,
                     const float* LSE, const uint32_t* seg, float* dQ, float* dK, float* dV,
                     const Shape& sh, char* ws, cudaStream_t st, const RopeParams& rope) {
  switch (padded_dim(sh.d)) {
    case 32: return short_launch<32>(Q, K, V, dO, LSE, seg, dQ, dK, dV, sh, ws, st, rope);
    case 64: return short_launch<64>(Q, K, V, dO, LSE, seg, dQ, dK, dV, sh, ws, st, rope);
    default: return short_launch<128>(Q, K, V, dO, LSE, seg, dQ, dK, dV, sh, ws, st, rope);
  }
}

}  // namespace gqa
