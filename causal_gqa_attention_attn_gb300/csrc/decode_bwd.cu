// Decode-style attention backward from saved probabilities: one query per
// head against history_len cached keys (rullama training.rs,
// attention_backward_dq_chained: d_q and the staged d_scores [n_heads,
// history_len] from k_hist, v_hist, probs, d_out; attention_backward_dkv_chained:
// d_k_hist, d_v_hist from q, probs, d_out, d_scores). With G = H / Hk query
// heads per kv head g and scale sigma:
//   dP_hj = d_out_h . v_j,   D_h = sum_j probs_hj dP_hj
//   d_scores_hj = probs_hj (dP_hj - D_h)         (gradient of the scores sigma q.k)
//   d_q_h += sigma sum_j d_scores_hj k_j
//   d_k_j += sigma sum_{h in g} d_scores_hj q_h,   d_v_j += sum_{h in g} probs_hj d_out_h
//
// The work is two passes over the key history, so HBM decides the time:
// every key row is read once per pass for all G heads of its group. CTA =
// (block of 32 or 64 keys, kv head); a warp holds 4 or 8 key rows in
// registers, each lane d/32 columns of them.
//  decode_dp:   dP for the block's keys and the group's heads, staged in
//               d_scores; per-CTA partial sums of probs * dP; one owned +=
//               of the block's d_v rows (d_v needs no D). Reads V, d_v;
//               writes d_v.
//  decode_dsum: D_h = the partial sums added in a fixed order.
//  decode_dkv:  d_scores from the staged dP; one owned += of the block's d_k
//               rows; per-CTA partial d_q. Reads K, d_k; writes d_k (the two
//               passes move about the same bytes).
//  decode_dq:   d_q += the partials added in a fixed order.
// No atomics: results do not depend on scheduling.
// The last three launch as programmatic dependents of the one before (each
// kernel lets its successor start once all its CTAs run): decode_dkv loads
// its key and d_k rows, which no earlier kernel writes, before it waits for
// the staged dP and D; decode_dsum and decode_dq wait first.
#include <cuda_runtime.h>

#include "common.cuh"

namespace gqa {
namespace {

constexpr int kDecWarps = 8;
constexpr int kDecThreads = 32 * kDecWarps;
// key rows per warp: 8, or 4 for head_dim >= 96, so that the key rows and the
// dK / dV accumulators of decode_dkv leave registers for two CTAs per SM
__host__ __device__ constexpr int dec_kpw(int E) { return E >= 3 ? 4 : 8; }
__host__ __device__ constexpr int dec_keys(int E) { return kDecWarps * dec_kpw(E); }

struct DecWs {
  int nblk;
  size_t dpart, dsum, qpart, total;
};

DecWs dec_ws(int L, int H, int d) {
  DecWs w;
  const int keys = dec_keys(d / 32);
  w.nblk = (L + keys - 1) / keys;
  w.dpart = kWsHeader;
  w.dsum = w.dpart + align256((size_t)w.nblk * H * sizeof(float));
  w.qpart = w.dsum + align256((size_t)H * sizeof(float));
  w.total = w.qpart + align256((size_t)w.nblk * H * d * sizeof(float));
  return w;
}

// this lane's E consecutive columns of a row (16-byte aligned when E = 4),
// through the read-only path (RO) for data no kernel of the call writes
template <int E, bool RO = true>
__device__ __forceinline__ void load_cols(const float* p, float* v) {
  if constexpr (E == 4) {
    const float4 x = RO ? __ldg(reinterpret_cast<const float4*>(p)) : *reinterpret_cast<const float4*>(p);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  } else if constexpr (E == 2) {
    const float2 x = RO ? __ldg(reinterpret_cast<const float2*>(p)) : *reinterpret_cast<const float2*>(p);
    v[0] = x.x; v[1] = x.y;
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = RO ? __ldg(p + e) : p[e];
  }
}

// p[0 .. E) = v[0 .. E) (one vector store per lane when E = 2 or 4)
template <int E>
__device__ __forceinline__ void store_cols(float* p, const float* v) {
  if constexpr (E == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  } else if constexpr (E == 2) {
    *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) p[e] = v[e];
  }
}

// Programmatic dependent launch: let the next kernel of the stream start, and
// wait until the previous one has completed with its writes visible (both
// no-ops for a kernel not launched as a dependent).
__device__ __forceinline__ void pdl_launch_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_prev() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <int E>
__global__ void __launch_bounds__(kDecThreads) decode_dp(const float* __restrict__ V,
                                                         const float* __restrict__ probs,
                                                         const float* __restrict__ d_out,
                                                         float* __restrict__ dsc,
                                                         float* __restrict__ dpart,
                                                         float* __restrict__ dV, int L, int H,
                                                         int Hk, int G) {
  constexpr int D = 32 * E, KPW = dec_kpw(E);
  extern __shared__ float red[];                  // [kDecWarps][G] per-warp partial sums
  pdl_launch_next();
  const int g = blockIdx.y, blk = blockIdx.x;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int j0 = blk * dec_keys(E) + warp * KPW;
  // the warp's value rows and their d_v rows, loaded up front; d_v
  // accumulates onto the loaded rows and is stored once at the end
  float v[KPW][E], dv[KPW][E];
#pragma unroll
  for (int k = 0; k < KPW; ++k) {
    const int j = j0 + k;
    const long long off = ((long long)j * Hk + g) * D + lane * E;
    if (j < L) {
      load_cols<E>(V + off, v[k]);
      load_cols<E, false>(dV + off, dv[k]);    // rows this thread writes back below
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) v[k][e] = dv[k][e] = 0.f;
    }
  }
  constexpr int HC = 32 / KPW;                    // heads per chunk: one probs value per lane
  for (int c0 = 0; c0 < G; c0 += HC) {
    // lane l: probs of head c0 + l / KPW, key j0 + l % KPW (0 past the ends)
    const int lh = c0 + lane / KPW, lj = j0 + lane % KPW;
    const float pl = (lh < G && lj < L) ? __ldg(probs + (long long)(g * G + lh) * L + lj) : 0.f;
    for (int hh = c0; hh < G && hh < c0 + HC; ++hh) {
      const int h = g * G + hh;
      float o[E];
      load_cols<E>(d_out + (long long)h * D + lane * E, o);
      float mine = 0.f, psum = 0.f;               // lane k keeps dP of key k
#pragma unroll
      for (int k = 0; k < KPW; ++k) {
        float x = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) x = fmaf(o[e], v[k][e], x);
        x = warp_sum(x);
        if (lane == k) mine = x;
        const float p = __shfl_sync(0xffffffffu, pl, (hh - c0) * KPW + k);
        psum = fmaf(p, x, psum);
#pragma unroll
        for (int e = 0; e < E; ++e) dv[k][e] = fmaf(p, o[e], dv[k][e]);
      }
      if (lane < KPW && j0 + lane < L) dsc[(long long)h * L + j0 + lane] = mine;
      if (lane == 0) red[warp * G + hh] = psum;
    }
  }
#pragma unroll
  for (int k = 0; k < KPW; ++k) {
    const int j = j0 + k;
    if (j < L) store_cols<E>(dV + ((long long)j * Hk + g) * D + lane * E, dv[k]);
  }
  __syncthreads();
  for (int hh = threadIdx.x; hh < G; hh += kDecThreads) {
    float s = 0.f;
    for (int w = 0; w < kDecWarps; ++w) s += red[w * G + hh];
    dpart[(long long)blk * H + g * G + hh] = s;
  }
}

// D_h = the per-block partial sums added in a fixed order: thread t adds
// blocks t, t + 256, ..., each warp its 32 threads by a shuffle tree, then
// thread 0 the 8 warp sums in warp order.
__global__ void __launch_bounds__(256) decode_dsum(const float* __restrict__ dpart,
                                                   float* __restrict__ dsum, int nblk, int H) {
  __shared__ float part[8];
  pdl_launch_next();
  pdl_wait_prev();                                // decode_dp's partial sums
  const int h = blockIdx.x;
  float s = 0.f;
  for (int b = threadIdx.x; b < nblk; b += 256) s += dpart[(long long)b * H + h];
  s = warp_sum(s);
  if (threadIdx.x % 32 == 0) part[threadIdx.x / 32] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += part[w];
    dsum[h] = t;
  }
}

template <int E>
__global__ void __launch_bounds__(kDecThreads, E >= 3 ? 4 : 3) decode_dkv(
    const float* __restrict__ q, const float* __restrict__ K, const float* __restrict__ probs,
    const float* __restrict__ d_out, float* __restrict__ dsc, const float* __restrict__ dsum,
    float* __restrict__ dK, float* __restrict__ qpart, int L, int H, int Hk, int G, float scale) {
  constexpr int D = 32 * E, KPW = dec_kpw(E);
  constexpr int HC = 32 / KPW;                    // heads per chunk: one value per lane
  __shared__ float qred[HC][kDecWarps][D];        // per-warp partial d_q of a chunk's heads
  const int g = blockIdx.y, blk = blockIdx.x;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int j0 = blk * dec_keys(E) + warp * KPW;
  // the warp's key rows and their d_k rows, loaded up front; d_k accumulates
  // onto the loaded rows and is stored once
  float kr[KPW][E], dk[KPW][E];
#pragma unroll
  for (int k = 0; k < KPW; ++k) {
    const int j = j0 + k;
    const long long off = ((long long)j * Hk + g) * D + lane * E;
    if (j < L) {
      load_cols<E>(K + off, kr[k]);
      load_cols<E, false>(dK + off, dk[k]);   // rows this thread writes back below
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) kr[k][e] = dk[k][e] = 0.f;
    }
  }
  pdl_launch_next();
  pdl_wait_prev();                                // D and the staged dP of the earlier kernels
  for (int c0 = 0; c0 < G; c0 += HC) {
    // lane l: probs and the staged dP (decode_dp) of head c0 + l / KPW, key
    // j0 + l % KPW (0 past the ends), loaded before this chunk's d_scores
    // overwrite the staged values
    const int lh = c0 + lane / KPW, lj = j0 + lane % KPW;
    const bool lok = lh < G && lj < L;
    const float pl = lok ? __ldg(probs + (long long)(g * G + lh) * L + lj) : 0.f;
    const float dl = lok ? dsc[(long long)(g * G + lh) * L + lj] : 0.f;
    __syncwarp();
    for (int hh = c0; hh < G && hh < c0 + HC; ++hh) {
      const int h = g * G + hh;
      float qh[E], oh[E], qa[E];
      load_cols<E>(q + (long long)h * D + lane * E, qh);
      load_cols<E>(d_out + (long long)h * D + lane * E, oh);
#pragma unroll
      for (int e = 0; e < E; ++e) qa[e] = 0.f;
      const float Dh = __ldg(dsum + h);
      float mine = 0.f;                           // lane k keeps d_scores of key k
#pragma unroll
      for (int k = 0; k < KPW; ++k) {
        const int src = (hh - c0) * KPW + k;
        const float p = __shfl_sync(0xffffffffu, pl, src);
        const float dp = __shfl_sync(0xffffffffu, dl, src);
        const float ds = p * (dp - Dh);
        if (lane == k) mine = ds;
        const float sds = scale * ds;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          dk[k][e] = fmaf(sds, qh[e], dk[k][e]);
          qa[e] = fmaf(sds, kr[k][e], qa[e]);
        }
      }
      if (lane < KPW && j0 + lane < L) dsc[(long long)h * L + j0 + lane] = mine;
#pragma unroll
      for (int e = 0; e < E; ++e) qred[hh - c0][warp][lane * E + e] = qa[e];
    }
    // the chunk's partial d_q: warps added in a fixed order
    __syncthreads();
    const int nh = min(HC, G - c0);
    for (int t = threadIdx.x; t < nh * D; t += kDecThreads) {
      const int i = t / D, c = t % D;
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) sum += qred[i][w][c];
      qpart[((long long)blk * H + g * G + c0 + i) * D + c] = sum;
    }
    __syncthreads();
  }
#pragma unroll
  for (int k = 0; k < KPW; ++k) {
    const int j = j0 + k;
    if (j >= L) continue;
    store_cols<E>(dK + ((long long)j * Hk + g) * D + lane * E, dk[k]);
  }
}

// d_q[h, c] += sum over blocks of qpart[b, h, c]: grid (H, D / 32), warp w of
// 32 adds blocks b = w, w + 32, ... of its lane's column (eight loads in
// flight), then the 32 warp sums are added in warp order (a fixed order: the
// result does not depend on scheduling).
constexpr int kDqWarps = 32;
__global__ void __launch_bounds__(32 * kDqWarps) decode_dq(const float* __restrict__ qpart,
                                                           float* __restrict__ dq, int nblk, int H,
                                                           int D) {
  __shared__ float part[kDqWarps][33];
  pdl_wait_prev();                                // decode_dkv's partial d_q
  const int h = blockIdx.x, lane = threadIdx.x % 32, w = threadIdx.x / 32;
  const int c = blockIdx.y * 32 + lane;
  float s = 0.f;
  for (int b0 = w; b0 < nblk; b0 += 8 * kDqWarps) {
    float x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int b = b0 + u * kDqWarps;
      x[u] = b < nblk ? __ldg(qpart + ((long long)b * H + h) * D + c) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) s += x[u];
  }
  part[w][lane] = s;
  __syncthreads();
  if (w == 0) {
    float t = 0.f;
#pragma unroll 8
    for (int i = 0; i < kDqWarps; ++i) t += part[i][lane];
    dq[(long long)h * D + c] += t;
  }
}

// Launch as a programmatic dependent of the stream's previous kernel (it may
// start before that one completes and waits in griddepcontrol.wait).
template <class... KArgs, class... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int E>
gqa_status decode_launch(const float* q, const float* k_hist, const float* v_hist,
                         const float* probs, const float* d_out, float* d_scores, float* d_q,
                         float* d_k, float* d_v, int L, int H, int Hk, float scale, char* ws,
                         cudaStream_t st) {
  constexpr int D = 32 * E;
  const DecWs w = dec_ws(L, H, D);
  const int G = H / Hk;
  float* dpart = reinterpret_cast<float*>(ws + w.dpart);
  float* dsum = reinterpret_cast<float*>(ws + w.dsum);
  float* qpart = reinterpret_cast<float*>(ws + w.qpart);
  const dim3 grid((unsigned)w.nblk, (unsigned)Hk);
  const size_t red_bytes = (size_t)kDecWarps * G * sizeof(float);
  if (red_bytes > 48 * 1024 &&
      cudaFuncSetAttribute(decode_dp<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)red_bytes) != cudaSuccess)
    return check_launch("decode dP smem attribute");
  decode_dp<E><<<grid, kDecThreads, red_bytes, st>>>(v_hist, probs, d_out, d_scores, dpart, d_v,
                                                     L, H, Hk, G);
  note_launch();
  gqa_status r;
  if ((r = check_launch("decode dP")) != GQA_OK) return r;
  cudaError_t e = launch_dependent(decode_dsum, dim3((unsigned)H), dim3(256), 0, st,
                                   (const float*)dpart, dsum, w.nblk, H);
  note_launch();
  if (e != cudaSuccess) return set_error(GQA_ERR_CUDA, "decode D: %s", cudaGetErrorString(e));
  if ((r = check_launch("decode D")) != GQA_OK) return r;
  e = launch_dependent(decode_dkv<E>, grid, dim3(kDecThreads), 0, st, q, k_hist, probs, d_out,
                       d_scores, (const float*)dsum, d_k, qpart, L, H, Hk, G, scale);
  note_launch();
  if (e != cudaSuccess) return set_error(GQA_ERR_CUDA, "decode dK dV: %s", cudaGetErrorString(e));
  if ((r = check_launch("decode dK dV")) != GQA_OK) return r;
  e = launch_dependent(decode_dq, dim3((unsigned)H, D / 32), dim3(32 * kDqWarps), 0, st,
                       (const float*)qpart, d_q, w.nblk, H, D);
  note_launch();
  if (e != cudaSuccess) return set_error(GQA_ERR_CUDA, "decode dQ: %s", cudaGetErrorString(e));
  return check_launch("decode dQ");
}

}  // namespace

size_t decode_ws_bytes(int L, int H, int d) { return dec_ws(L, H, d).total; }

gqa_status decode_bwd(const float* q, const float* k_hist, const float* v_hist, const float* probs,
                      const float* d_out, float* d_scores, float* d_q, float* d_k, float* d_v,
                      int L, int H, int Hk, int d, float scale, char* ws, cudaStream_t st) {
  switch (d) {
    case 32: return decode_launch<1>(q, k_hist, v_hist, probs, d_out, d_scores, d_q, d_k, d_v, L, H, Hk, scale, ws, st);
    case 64: return decode_launch<2>(q, k_hist, v_hist, probs, d_out, d_scores, d_q, d_k, d_v, L, H, Hk, scale, ws, st);
    case 96: return decode_launch<3>(q, k_hist, v_hist, probs, d_out, d_scores, d_q, d_k, d_v, L, H, Hk, scale, ws, st);
    case 128: return decode_launch<4>(q, k_hist, v_hist, probs, d_out, d_scores, d_q, d_k, d_v, L, H, Hk, scale, ws, st);
    default: return set_error(GQA_ERR_UNSUPPORTED, "decode backward: head_dim %d not in {32, 64, 96, 128}", d);
  }
}

}  // namespace gqa
