// silu.cuh -- the GroupNorm affine + SiLU + TF32 rounding of two elements
// (cortiq-engine "Module vae": GroupNorm followed by SiLU, x * sigmoid(x),
// before a conv; "VAE decode -> GPU handoff", "GPU plan": the conv operands
// in TF32).
#pragma once
#include <cstdint>

namespace vae {

// tf32(silu(x * a + b)) for two elements at a time, written for few issued
// instructions (timed on GB300, this per-element transform is what bounds
// the tensor-core head): packed f32x2 FMA-pipe operations for
// the affine, the exponent scaling, 1 + e and the Newton steps, and one
// special-function op per element. silu(u) = u / (1 + e^-u): e^-u by the
// exp2 unit (u clamped at -80, where silu is 0 to far below float resolution,
// so that 1 + e^-u stays finite); the reciprocal by Newton's iteration
// r <- r (2 - d r) from an integer-subtraction seed (relative error <= 5.1 %
// for d >= 1; two steps: <= 7e-6); then rounding to the nearest TF32 value,
// ties away from zero, on the bit pattern (add half of the unit of the 13
// dropped bits, clear them).
__device__ __forceinline__ uint64_t pk2(float x, float y) {
  return static_cast<uint64_t>(__float_as_uint(x)) |
         (static_cast<uint64_t>(__float_as_uint(y)) << 32);
}
__device__ __forceinline__ float lo2(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float hi2(uint64_t v) {
  return __uint_as_float(static_cast<uint32_t>(v >> 32));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float ex2_approx(float t) {
  float e;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(t));
  return e;
}
__device__ __forceinline__ uint32_t tf32_bits(uint32_t b) { return (b + 0x1000u) & 0xffffe000u; }

__device__ __forceinline__ float2 silu2_tf32(float x0, float x1, float a0, float a1, float b0,
                                             float b1) {
  const uint64_t u = fma2(pk2(x0, x1), pk2(a0, a1), pk2(b0, b1));
  const float nl2e = -1.4426950408889634f;  // -log2(e)
  const uint64_t t = mul2(pk2(fmaxf(lo2(u), -80.f), fmaxf(hi2(u), -80.f)), pk2(nl2e, nl2e));
  const uint64_t m1 = pk2(-1.f, -1.f), one = pk2(1.f, 1.f);
  const uint64_t nd = fma2(pk2(ex2_approx(lo2(t)), ex2_approx(hi2(t))), m1, m1);  // -(1 + e)
  // seed of 1 / d from -d's bits: 0xfef30000 - bits(-d) = 0x7ef30000 - bits(d)
  uint64_t r = static_cast<uint64_t>(0xfef30000u - static_cast<uint32_t>(nd)) |
               (static_cast<uint64_t>(0xfef30000u - static_cast<uint32_t>(nd >> 32)) << 32);
  r = fma2(r, fma2(nd, r, one), r);
  r = fma2(r, fma2(nd, r, one), r);
  const uint64_t y = mul2(u, r);
  return make_float2(__uint_as_float(tf32_bits(static_cast<uint32_t>(y))),
                     __uint_as_float(tf32_bits(static_cast<uint32_t>(y >> 32))));
}

}  // namespace vae
