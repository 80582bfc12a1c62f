// Per-row int8 code arithmetic shared by the quantization kernel and the
// decode W8A8 kernel that quantizes its own token rows: absmax of bf16
// vectors, and the round-half-even code of the IEEE quotient v / s computed
// through the correctly rounded reciprocal with an exact fallback near ties.
//
// Source: "Day 6 -- Quantize It Yourself", The mechanism, blocks 1 and 4
// (q = clamp(round(w / s)), s = absmax / 127, round to nearest).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace i8ql {
namespace {

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Packed |a| max of two bf16 pairs: the magnitude of each half is the larger
// magnitude (exact; the sign bit, an xor of the inputs', is ignored).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ float absmax8(const uint4& v, float a) {
    const uint32_t m = absmax_bf16x2(absmax_bf16x2(v.x, v.y), absmax_bf16x2(v.z, v.w));
    return fmaxf(a, fmaxf(fabsf(lo_bf16(m)), fabsf(hi_bf16(m))));
}

// The code of v is rint(fl32(v / s)).  Fast path: t = fl32(v * r) with
// r = fl32(1 / s) (correctly rounded).  Each of the two roundings is within
// half an ulp, so |t - v/s| <= |v/s| * (2^-23 + 2^-48), and fl32(v/s) is
// within |v/s| * 2^-24 of v/s; with |v/s| <= 127 * (1 + 2^-23) the two
// quotients differ by less than 2.3e-5.  rint changes value only at
// half-integers, so when t is farther than kNearTie = 2^-15 from the nearest
// half-integer, rint(t) == rint(fl32(v/s)).  Near-ties (and a reciprocal that
// overflowed, when s is subnormal) take the IEEE division.
//
// Rounding: adding 1.5 * 2^23 to |t| < 2^22 leaves round-half-even(t) in the
// low mantissa bits, so the low byte of the sum's bit pattern is the code in
// two's complement and subtracting 1.5 * 2^23 back gives it as a float.  The
// code never leaves [-127, 127] (|v/s| <= 127 * (1 + 2^-23)), so no clamp.
constexpr float kNearTie = 3.0517578125e-05f;  // 2^-15
constexpr float kRoundMagic = 12582912.0f;     // 1.5 * 2^23

struct RowScale {
    float s;      // the scale
    float r;      // fl32(1 / s)
    bool fast;    // r is finite
    uint64_t r2;  // (r, r) and the rounding constant, packed for f32x2 arithmetic
    uint64_t magic2;
};

// Codes of 8 values (two words of bf16 pairs) packed into two words.
__device__ __forceinline__ uint2 codes8(const uint4& v, const RowScale& rs) {
    float x[8] = {lo_bf16(v.x), hi_bf16(v.x), lo_bf16(v.y), hi_bf16(v.y),
                  lo_bf16(v.z), hi_bf16(v.z), lo_bf16(v.w), hi_bf16(v.w)};
    uint32_t b[8];
    float worst = 0.0f;  // largest |t - round(t)| over the 8 values
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        // per value, two at a time with the same IEEE single roundings:
        // t = x * r, m = t + magic, c = m - magic, d = t - c
        float d0, d1;
        asm("{\n\t.reg .b64 x, t, m, c, d;\n\t"
            "mov.b64 x, {%4, %5};\n\t"
            "mul.rn.f32x2 t, x, %6;\n\t"
            "add.rn.f32x2 m, t, %7;\n\t"
            "sub.rn.f32x2 c, m, %7;\n\t"
            "sub.rn.f32x2 d, t, c;\n\t"
            "mov.b64 {%0, %1}, m;\n\t"
            "mov.b64 {%2, %3}, d;\n\t}"
            : "=r"(b[i]), "=r"(b[i + 1]), "=f"(d0), "=f"(d1)
            : "f"(x[i]), "f"(x[i + 1]), "l"(rs.r2), "l"(rs.magic2));
        worst = fmaxf(worst, fmaxf(fabsf(d0), fabsf(d1)));
    }
    if (!rs.fast || worst > 0.5f - kNearTie) {
        // rare: some value lies next to a half-integer; take the division
#pragma unroll
        for (int i = 0; i < 8; ++i) b[i] = (uint32_t)__float2int_rn(__fdiv_rn(x[i], rs.s));
    }
    return make_uint2(__byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410),
                      __byte_perm(__byte_perm(b[4], b[5], 0x0040), __byte_perm(b[6], b[7], 0x0040), 0x5410));
}

__device__ __forceinline__ RowScale make_row_scale(float s) {
    RowScale rs;
    rs.s = s;
    rs.r = __frcp_rn(s);
    rs.fast = isfinite(rs.r);
    asm("mov.b64 %0, {%1, %1};" : "=l"(rs.r2) : "f"(rs.r));
    asm("mov.b64 %0, {%1, %1};" : "=l"(rs.magic2) : "f"(kRoundMagic));
    return rs;
}

}  // namespace
}  // namespace i8ql
