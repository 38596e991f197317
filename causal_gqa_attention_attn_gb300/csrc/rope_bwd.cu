// Interleaved RoPE backward, in place (backward_attention.wgsl, rope_q_backward
// / rope_k_backward; tang llm.rs, interleaved_rope_backward). Memory-bound:
// one read and one write of the buffer. Each thread rotates two adjacent
// pairs (one float4).
//
// Angle accuracy: theta = t * base^(-2p/d) reaches ~1.6e4 rad at t = 16383,
// where an fp32 product alone would be off by ~1e-3 rad. The per-pair
// frequencies are computed on the host in fp64 (as the pages' f64 tables do),
// theta is formed and reduced modulo 2*pi on the device in fp64, and only the
// reduced angle (|r| <= pi) goes through fp32 sincosf.
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"

namespace gqa {
namespace {

constexpr int kMaxPairs = 64;   // head_dim <= 128

struct RopeFreqs {
  double inv_freq[kMaxPairs];
};

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
    const double t = (double)(s + pos_offset);
    float4 x = reinterpret_cast<float4*>(X)[v];
    rot(x.x, x.y, t * f.inv_freq[p0]);
    rot(x.z, x.w, t * f.inv_freq[p0 + 1]);
    reinterpret_cast<float4*>(X)[v] = x;
  }
}

}  // namespace

gqa_status rope_bwd_launch(float* X, int S, int H, int d, int pos_offset, float base,
                           cudaStream_t st) {
  RopeFreqs f;
  for (int p = 0; p < kMaxPairs; ++p)
    f.inv_freq[p] = (2 * p < d) ? pow((double)base, -(2.0 * p) / (double)d) : 0.0;
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
