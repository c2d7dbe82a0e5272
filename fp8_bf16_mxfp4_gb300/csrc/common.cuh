// Shared device/host helpers for libmxg (sm_103a only).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "mxg.h"

#define MXG_DEVINL __device__ __forceinline__

namespace mxg {

constexpr int kMaxExperts = 512;

// Global wait limit for bounded spins (nanoseconds); set from the host API.
uint64_t wait_timeout_ns();

// ---------------------------------------------------------------------------
// Status reporting: first error wins.
// ---------------------------------------------------------------------------
MXG_DEVINL void report(int32_t* st, int32_t code) {
  if (st != nullptr) atomicCAS(st, 0, code);
}

MXG_DEVINL uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// BF16 bit helpers.
// ---------------------------------------------------------------------------
MXG_DEVINL float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
MXG_DEVINL float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// max of |x| over the two bf16 halves of w, as a 15-bit magnitude pattern
// (for non-NaN values magnitude order equals integer order of the pattern).
MXG_DEVINL uint32_t bf16x2_absmax_bits(uint32_t w) {
  return max(w & 0x7FFFu, (w >> 16) & 0x7FFFu);
}

// The same over a 32-value block (16 words): the two 16-bit magnitude lanes
// are maxed side by side (unsigned 16-bit SIMD max) and folded at the end.
MXG_DEVINL uint32_t bf16x32_absmax_bits(const uint32_t* w) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = __vmaxu2(m, w[i] & 0x7FFF7FFFu);
  return max(m & 0xFFFFu, m >> 16);
}

// MX shared exponent from a BF16 magnitude pattern (OCP MX v1.0 rule with the
// -127 floor): floor(log2(amax)) - emax clamped to [-127, 127]; -127 for 0.
// With `round_up` (the TransformerEngine recipe of the PR #745 review: amax /
// maxval taken up to a power of two) it is the smallest e with maxval * 2^e >=
// amax: one more than the OCP exponent exactly when amax's mantissa exceeds
// maxval's, i.e. its 7 BF16 mantissa bits exceed `up_mant` (1.75 = 1 + 96/128
// for E4M3's 448, 1.5 = 1 + 64/128 for E2M1's 6).  A subnormal amax lands on
// the -127 floor under either rule.
MXG_DEVINL int mx_exponent_from_amax_bits(uint32_t amax, int emax, bool round_up = false, int up_mant = 0) {
  const int E = (int)(amax >> 7);
  const int m = (int)(amax & 0x7F);
  int fl;
  if (E != 0) {
    fl = E - 127;
  } else if (m != 0) {
    fl = -133 + (31 - __clz(m));  // subnormal: m * 2^-133
  } else {
    return -127;
  }
  int e = fl - emax + ((round_up && E != 0 && m > up_mant) ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^-e as an fp32 (e in [-127, 125] for finite BF16 input: always normal).
MXG_DEVINL float pow2_neg(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }

// ---------------------------------------------------------------------------
// Hardware conversions (RNE, saturating to the largest finite value).
// cvt.*x2 puts its first source operand in the high half of the result.
// ---------------------------------------------------------------------------
MXG_DEVINL uint32_t cvt_e2m1x8(const float* v) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

MXG_DEVINL uint32_t cvt_e4m3x4(float a0, float a1, float a2, float a3) {
  uint32_t r;
  asm("{\n\t.reg .b16 h0, h1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h0, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h1, %4, %3;\n\t"
      "mov.b32 %0, {h0, h1};\n\t}"
      : "=r"(r)
      : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
  return r;
}

}  // namespace mxg
