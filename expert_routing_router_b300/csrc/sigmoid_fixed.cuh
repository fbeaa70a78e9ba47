// sigmoid_fixed.cuh -- the fp32 selection sigmoid S shared by the router (forward) and
// the router backward, so that both see the same s = S(l) for every logit.
//
// Ultralytics glossary "Expert Parallelism", section "Load balancing and capacity":
// DeepSeek-V3-style routing scores experts with a sigmoid and adds a selection-only
// bias.  Selection compares S(l) + bias across experts, so S is specified down to
// the bit to make the selection reproducible off the device.
#pragma once

namespace moe {

// fp32 sigmoid, evaluated as a fixed sequence of correctly rounded operations:
// clamp -l to [-20, 86]; n = rint(z*log2e); Cody & Waite (1980) reduction
// r = z - n*ln2_hi - n*ln2_lo with ln2_hi = 45426/65536; p = degree-7 Taylor
// polynomial of e^r in Horner form (one fused multiply-add per degree, coefficients
// 1/j! rounded to fp32); e = p * 2^n; S = 1 / (1 + e).  Any implementation of these
// steps returns the same bits, so selection on S + bias is reproducible off-device.
__device__ __forceinline__ float sigmoid_fixed(float l) {
  const float z = fminf(fmaxf(-l, -20.0f), 86.0f);
  const float n = rintf(__fmul_rn(z, 0x1.715476p+0f));
  float r = __fmaf_rn(-n, 0x1.62e4p-1f, z);
  r = __fmaf_rn(-n, 0x1.7f7d1cp-20f, r);
  float p = 0x1.a01a02p-13f;         // 1/7!
  p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);  // 1/6!
  p = __fmaf_rn(p, r, 0x1.111112p-7f);   // 1/5!
  p = __fmaf_rn(p, r, 0x1.555556p-5f);   // 1/4!
  p = __fmaf_rn(p, r, 0x1.555556p-3f);   // 1/3!
  p = __fmaf_rn(p, r, 0x1p-1f);          // 1/2!
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  const float two_n = __int_as_float((__float2int_rn(n) + 127) << 23);
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, __fmul_rn(p, two_n)));
}

}  // namespace moe
