// Interleaved RoPE backward, in place, and the host side of the rotation
// table (the rotation itself and its accuracy: rope_common.cuh). Memory-bound:
// one read and one write of the buffer. Each thread rotates two adjacent
// pairs (one float4).
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "rope_common.cuh"

namespace gqa {

RopeParams make_rope(int d, int pos_offset, float base) {
  RopeParams f{};
  f.on = 1;
  f.pos_offset = pos_offset;
  for (int p = 0; p < kMaxRopePairs; ++p) {
    f.inv_freq[p] = (2 * p < d) ? pow((double)base, -(2.0 * p) / (double)d) : 0.0;
    f.f_hi[p] = (float)f.inv_freq[p];
    f.f_lo[p] = (float)(f.inv_freq[p] - (double)f.f_hi[p]);
  }
  // split 2 pi: c1 a multiple of 2^-8 (<= 11 significant bits), c2 a multiple
  // of 2^-19 (<= 11 bits), c3 the fp32 rest; quotients n < 2^13 keep n*c1 and
  // n*c2 exact in fp32
  const double two_pi = 6.283185307179586476925286766559;
  const double c1 = nearbyint(two_pi * 256.0) / 256.0;
  const double c2 = nearbyint((two_pi - c1) * 524288.0) / 524288.0;
  f.c1 = (float)c1;
  f.c2 = (float)c2;
  f.c3 = (float)(two_pi - c1 - c2);
  return f;
}

namespace {

__global__ void __launch_bounds__(256) rope_bwd_kernel(float* __restrict__ X, long long n_vec4,
                                                       int H, int d, RopeParams f) {
  const int v_per_head = d / 4;               // float4 per head
  const long long v_per_row = (long long)H * v_per_head;
  for (long long v = blockIdx.x * (long long)blockDim.x + threadIdx.x; v < n_vec4;
       v += (long long)gridDim.x * blockDim.x) {
    const long long s = v / v_per_row;
    const int p0 = (int)(v % v_per_head) * 2;  // first pair index in this float4
    const long long tpos = s + f.pos_offset;
    float4 x = reinterpret_cast<float4*>(X)[v];
    rope_rotate(x.x, x.y, tpos, p0, f);
    rope_rotate(x.z, x.w, tpos, p0 + 1, f);
    reinterpret_cast<float4*>(X)[v] = x;
  }
}

}  // namespace

gqa_status rope_bwd_launch(float* X, int S, int H, int d, int pos_offset, float base,
                           cudaStream_t st) {
  const RopeParams f = make_rope(d, pos_offset, base);
  const long long n_vec4 = (long long)S * H * (d / 4);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (n_vec4 + 255) / 256;
  const long long cap = (long long)sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  rope_bwd_kernel<<<(unsigned)blocks, 256, 0, st>>>(X, n_vec4, H, d, f);
  note_launch();
  return check_launch("rope backward");
}

}  // namespace gqa
