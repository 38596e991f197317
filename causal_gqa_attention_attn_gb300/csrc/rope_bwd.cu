// Interleaved RoPE backward, in place (backward_attention.wgsl, rope_q_backward
// / rope_k_backward; tang llm.rs, interleaved_rope_backward). Memory-bound:
// one read and one write of the buffer. Each thread rotates two adjacent
// pairs (one float4).
//
// Angle accuracy: theta = t * base^(-2p/d) reaches ~1.6e4 rad at t = 16383,
// where an fp32 product alone would be off by ~1e-3 rad. The per-pair
// frequencies are computed on the host in fp64 (as the pages' f64 tables do)
// and the angle is reduced modulo 2*pi before fp32 sincosf:
//  - positions t < 2^15: in fp32, with the frequency split into two floats
//    (f = f_hi + f_lo) so that t*f_hi is carried exactly (product + FMA
//    error term), and 2*pi split into three constants with at most 11, 11
//    and 24 significant bits (Cody & Waite's argument reduction), so that
//    n*C1 and n*C2 are exact for the n < 2^13 quotients that occur;
//  - larger positions: the product and reduction in fp64 (a slow pipe on
//    this part, hence only there).
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"

namespace gqa {
namespace {

constexpr int kMaxPairs = 64;   // head_dim <= 128

struct RopeFreqs {
  double inv_freq[kMaxPairs];
  float f_hi[kMaxPairs], f_lo[kMaxPairs];
  float c1, c2, c3;   // 2*pi = c1 + c2 + c3 (<= 11, <= 11, 24 significant bits)
};

constexpr int kFastPosLimit = 1 << 15;

__device__ __forceinline__ void rot_fast(float& x0, float& x1, float t, float f_hi, float f_lo,
                                         const RopeFreqs& f) {
  const float p = t * f_hi;
  const float e = fmaf(t, f_hi, -p);               // t*f_hi = p + e exactly
  const float n = rintf(p * 0.15915494309189535f);  // nearest multiple of 2 pi
  float r = fmaf(-n, f.c1, p);
  r = fmaf(-n, f.c2, r);
  r = fmaf(-n, f.c3, r);
  r += fmaf(t, f_lo, e);
  float s, c;
  sincosf(r, &s, &c);
  const float a = x0, b = x1;
  x0 = a * c + b * s;
  x1 = -a * s + b * c;
}

__device__ __forceinline__ void rot(float& x0, float& x1, double theta) {
  // theta - 2 pi n with n = rint(theta / 2 pi); a multiply by the reciprocal
  // constant instead of a division (fp64 is a slow pipe on this part).
  const double two_pi = 6.283185307179586476925286766559;
  const double inv_two_pi = 0.15915494309189533576888376337251;
  const double r = fma(-two_pi, rint(theta * inv_two_pi), theta);
  float s, c;
  sincosf((float)r, &s, &c);
  const float a = x0, b = x1;
  x0 = a * c + b * s;
  x1 = -a * s + b * c;
}

__global__ void __launch_bounds__(256) rope_bwd_kernel(float* __restrict__ X, long long n_vec4,
                                                       int H, int d, int pos_offset,
                                                       RopeFreqs f) {
  const int v_per_head = d / 4;               // float4 per head
  const long long v_per_row = (long long)H * v_per_head;
  for (long long v = blockIdx.x * (long long)blockDim.x + threadIdx.x; v < n_vec4;
       v += (long long)gridDim.x * blockDim.x) {
    const long long s = v / v_per_row;
    const int p0 = (int)(v % v_per_head) * 2;  // first pair index in this float4
    const long long tpos = s + pos_offset;
    float4 x = reinterpret_cast<float4*>(X)[v];
    if (tpos < kFastPosLimit) {
      const float t = (float)tpos;
      rot_fast(x.x, x.y, t, f.f_hi[p0], f.f_lo[p0], f);
      rot_fast(x.z, x.w, t, f.f_hi[p0 + 1], f.f_lo[p0 + 1], f);
    } else {
      const double t = (double)tpos;
      rot(x.x, x.y, t * f.inv_freq[p0]);
      rot(x.z, x.w, t * f.inv_freq[p0 + 1]);
    }
    reinterpret_cast<float4*>(X)[v] = x;
  }
}

}  // namespace

gqa_status rope_bwd_launch(float* X, int S, int H, int d, int pos_offset, float base,
                           cudaStream_t st) {
  RopeFreqs f;
  for (int p = 0; p < kMaxPairs; ++p) {
    f.inv_freq[p] = (2 * p < d) ? pow((double)base, -(2.0 * p) / (double)d) : 0.0;
    f.f_hi[p] = (float)f.inv_freq[p];
    f.f_lo[p] = (float)(f.inv_freq[p] - (double)f.f_hi[p]);
  }
  {
    // split 2 pi: c1 a multiple of 2^-8 (<= 11 significant bits), c2 a multiple
    // of 2^-19 (<= 11 bits), c3 the fp32 rest; quotients n < 2^13 keep n*c1 and
    // n*c2 exact in fp32
    const double two_pi = 6.283185307179586476925286766559;
    const double c1 = nearbyint(two_pi * 256.0) / 256.0;
    const double c2 = nearbyint((two_pi - c1) * 524288.0) / 524288.0;
    f.c1 = (float)c1;
    f.c2 = (float)c2;
    f.c3 = (float)(two_pi - c1 - c2);
  }
  const long long n_vec4 = (long long)S * H * (d / 4);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (n_vec4 + 255) / 256;
  const long long cap = (long long)sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  rope_bwd_kernel<<<(unsigned)blocks, 256, 0, st>>>(X, n_vec4, H, d, pos_offset, f);
  note_launch();
  return check_launch("rope backward");
}

}  // namespace gqa
