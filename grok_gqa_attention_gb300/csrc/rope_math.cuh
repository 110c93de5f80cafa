// RoPE constants evaluated on the device, shared by the kernels that rotate:
// the fp32 inverse frequencies and the fp32 cos / sin of an fp32 phase.
//
// Grok-1 code-reading guide, ch. 4 "model.py close reading I", §4.3.1
// RotaryEmbedding: inv_freq = 1 / 10000^(2j/128) in fp32, phase = t * inv_freq
// in fp32, cos and sin of the phase.
#pragma once

#include "common.cuh"

namespace grok {

// cos and sin of an fp32 phase (0 <= phase < 65536), evaluated in fp64 and
// rounded once to fp32. Reduction by pi/2 (Cody-Waite): pi/2 is split into
// three doubles, the first two with 33 significant bits so that k * C1 and
// k * C2 are exact for k < 2^20, the third the remaining bits (pi/2 - C1 - C2 -
// C3 ~ 1e-37); each fused step rounds relative to its own result, so the
// reduced argument r (|r| <= pi/4, never below 2.7e-7 for a nonzero phase in
// this domain) carries about two ulps of relative error. sin and cos of r are
// Taylor polynomials through r^15 and r^14 (truncation below 2^-50 on
// |r| <= pi/4). The result is well inside the margin the fp32 rounding needs:
// for these phases every exact value lies at least 59 fp64 ulps from an fp32
// rounding midpoint, so the rounded table is the correctly rounded one.
__device__ __forceinline__ void rope_cos_sin(float phase, float& c_out, float& s_out) {
  constexpr double kTwoOverPi = 0x1.45f306dc9c883p-1;
  constexpr double C1 = 0x1.921fb54400000p+0;
  constexpr double C2 = 0x1.0b4611a600000p-34;
  constexpr double C3 = 0x1.3198a2e037073p-69;
  const double x = double(phase);
  const double k = rint(x * kTwoOverPi);
  double r = fma(-k, C1, x);
  r = fma(-k, C2, r);
  r = fma(-k, C3, r);
  const double r2 = r * r;
  // sin r = r + r^3 (-1/3! + r^2 (1/5! - ... + r^2 (-1/15!)))
  double sp = -1.0 / 1307674368000.0;
  sp = fma(sp, r2, 1.0 / 6227020800.0);
  sp = fma(sp, r2, -1.0 / 39916800.0);
  sp = fma(sp, r2, 1.0 / 362880.0);
  sp = fma(sp, r2, -1.0 / 5040.0);
  sp = fma(sp, r2, 1.0 / 120.0);
  sp = fma(sp, r2, -1.0 / 6.0);
  const double sr = fma(r * r2, sp, r);
  // cos r = 1 + r^2 (-1/2! + r^2 (1/4! - ... + r^2 (1/14!)))
  double cp = -1.0 / 87178291200.0;
  cp = fma(cp, r2, 1.0 / 479001600.0);
  cp = fma(cp, r2, -1.0 / 3628800.0);
  cp = fma(cp, r2, 1.0 / 40320.0);
  cp = fma(cp, r2, -1.0 / 720.0);
  cp = fma(cp, r2, 1.0 / 24.0);
  cp = fma(cp, r2, -0.5);
  const double cr = fma(r2, cp, 1.0);
  // phase = k pi/2 + r
  const int q = int(k) & 3;
  const double sv = (q == 0) ? sr : (q == 1) ? cr : (q == 2) ? -sr : -cr;
  const double cv = (q == 0) ? cr : (q == 1) ? -sr : (q == 2) ? -cr : sr;
  c_out = __double2float_rn(cv);
  s_out = __double2float_rn(sv);
}

// inv_freq[j] = 1 / RN32(10000^(2j/128)): the power in fp64 rounded once to
// fp32, then an fp32 division. 10000^(j/64) = 2^(j log2(10000) / 64); with
// log2(10000) rounded to double and exp2 within an ulp the power carries a
// few fp64 ulps of error, far inside the margin its fp32 rounding needs (every
// 10000^(j/64), j < 64, lies more than 4e6 fp64 ulps from an fp32 midpoint).
__device__ __forceinline__ float rope_inv_freq(int j) {
  constexpr double kLog2Base = 13.287712379549449;  // log2(10000)
  return __fdiv_rn(1.0f, __double2float_rn(exp2(double(j) * (kLog2Base / 64.0))));
}

}  // namespace grok
