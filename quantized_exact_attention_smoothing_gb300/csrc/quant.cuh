// quant.cuh -- the INT8 block quantiser's per-value step, shared by the
// preparation pass (Q and K) and by the forward kernel's in-kernel Q
// quantisation ("Experiment Log" page, entry "Phase 0 Import And
// Verification", stage "Q/K preparation").  Both produce the same bytes for
// the same value and scale.
#pragma once

#include <cstdint>

namespace sattn {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

constexpr float kRoundMagic = 12582912.0f;        // 1.5 * 2^23
constexpr float kTieMargin = 0.49993896484375f;   // 0.5 - 2^-14

// clamp(rint(fl(x / s)), -127, 127) by the IEEE division, as its
// two's-complement byte (the low bits of k + 1.5 * 2^23, which is exact for
// integers |k| < 2^22).
__device__ __forceinline__ uint32_t int8_code_div(float x, float s)
{
    const float k = fminf(fmaxf(rintf(__fdiv_rn(x, s)), -127.0f), 127.0f);
    return __float_as_uint(__fadd_rn(k, kRoundMagic)) & 0xffu;
}

// The same code without a division in the common case: q = fl(x * fl(1/s))
// lies within 3 ulp of fl(x / s) (two roundings of relative size 2^-24 each,
// plus that of the quotient), and |q| <= 127 * (1 + 2^-22), so an ulp of q is
// at most 2^-16.  When q is farther than 2^-14 from the nearest half-integer,
// fl(x / s) rounds to the same integer as q, rint(q) = fl(q + 1.5 * 2^23) -
// 1.5 * 2^23 (exact, ties to even, |q| < 2^22), and the clamp cannot bind
// (|q| < 127.5 whenever |x| <= amax and s = fl(amax / 127)), so the byte is
// the low byte of fl(q + 1.5 * 2^23).  Values near a rounding tie take the
// division.  BF16 inputs make them common (x / s = 127 x / amax often lands
// within an ulp of a half-integer: a few per thousand values of Gaussian
// data), so the branch is per value: a warp pays for the division only at
// the positions where one of its lanes needs it.  (Division-free exact tie
// decisions measured slower: short enough to be predicated, they are paid by
// every value.)
__device__ __forceinline__ uint32_t int8_code(float x, float s, float rs)
{
    const float q = __fmul_rn(x, rs);
    const float r = __fadd_rn(q, kRoundMagic);
    if (!(fabsf(__fsub_rn(q, __fsub_rn(r, kRoundMagic))) < kTieMargin))   // true for NaN / inf too
        return int8_code_div(x, s);
    return __float_as_uint(r) & 0xffu;
}

// int8_code of the eight BF16 values of one 16-byte chunk, as eight bytes in
// channel order.
__device__ __forceinline__ uint2 int8_codes8(const uint4 &a, float s, float rs)
{
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    uint32_t t[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        t[e] = int8_code((e & 1) ? bf16_hi(w[e >> 1]) : bf16_lo(w[e >> 1]), s, rs);
    return make_uint2(__byte_perm(__byte_perm(t[0], t[1], 0x0040u), __byte_perm(t[2], t[3], 0x0040u), 0x5410u),
                      __byte_perm(__byte_perm(t[4], t[5], 0x0040u), __byte_perm(t[6], t[7], 0x0040u), 0x5410u));
}

}  // namespace sattn
