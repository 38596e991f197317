// Interleaved RoPE backward rotation (backward_attention.wgsl, rope_q_backward
// / rope_k_backward; tang llm.rs, interleaved_rope_backward): pair p of a head
// at position t is rotated by the transpose of the forward rotation,
//   (x0, x1) <- (x0 cos a + x1 sin a, -x0 sin a + x1 cos a),  a = t * base^(-2p/d).
// Shared by the standalone in-place kernel and the epilogues of the fused
// backward (attn_bwd_rope).
//
// Angle accuracy: a reaches ~1.6e4 rad at t = 16383, where an fp32 product
// alone would be off by ~1e-3 rad. The per-pair frequencies are computed on
// the host in fp64 (as the pages' f64 tables do) and the angle is reduced
// modulo 2*pi before fp32 sincosf:
//  - positions t < 2^15: in fp32, with the frequency split into two floats
//    (f = f_hi + f_lo) so that t*f_hi is carried exactly (product + FMA
//    error term), and 2*pi split into three constants with at most 11, 11
//    and 24 significant bits (Cody & Waite's argument reduction), so that
//    n*C1 and n*C2 are exact for the n < 2^13 quotients that occur;
//  - larger positions: the product and reduction in fp64 (a slow pipe on
//    this part, hence only there).
#pragma once
#include <cuda_runtime.h>
#include <math.h>

namespace gqa {

constexpr int kMaxRopePairs = 64;           // head_dim <= 128
constexpr long long kRopeFastPosLimit = 1 << 15;

struct RopeParams {
  int on;                                   // 0: no rotation (plain backward)
  int pos_offset;                           // position of token 0
  double inv_freq[kMaxRopePairs];
  float f_hi[kMaxRopePairs], f_lo[kMaxRopePairs];
  float c1, c2, c3;                         // 2*pi = c1 + c2 + c3 (<= 11, <= 11, 24 significant bits)
};

// Host: the table for head_dim d and the given base (on = 1).
RopeParams make_rope(int d, int pos_offset, float base);
inline RopeParams no_rope() {
  RopeParams r{};
  r.on = 0;
  return r;
}

__device__ __forceinline__ void rope_rotate(float& x0, float& x1, long long tpos, int p,
                                            const RopeParams& f) {
  float r;
  if (tpos < kRopeFastPosLimit) {
    const float t = (float)tpos;
    const float hi = f.f_hi[p];
    const float prod = t * hi;
    const float e = fmaf(t, hi, -prod);                // t*hi = prod + e exactly
    const float n = rintf(prod * 0.15915494309189535f);  // nearest multiple of 2 pi
    r = fmaf(-n, f.c1, prod);
    r = fmaf(-n, f.c2, r);
    r = fmaf(-n, f.c3, r);
    r += fmaf(t, f.f_lo[p], e);
  } else {
    // theta - 2 pi n with n = rint(theta / 2 pi); a multiply by the reciprocal
    // constant instead of a division (fp64 is a slow pipe on this part)
    const double theta = (double)tpos * f.inv_freq[p];
    const double two_pi = 6.283185307179586476925286766559;
    const double inv_two_pi = 0.15915494309189533576888376337251;
    r = (float)fma(-two_pi, rint(theta * inv_two_pi), theta);
  }
  float s, c;
  sincosf(r, &s, &c);
  const float a = x0, b = x1;
  x0 = a * c + b * s;
  x1 = -a * s + b * c;
}

}  // namespace gqa
