// det_math.cuh -- the profile's transcendental spellings as device functions:
// exp, log (used by the cross-entropy, SwiGLU, the rotary frequencies) and
// sin/cos (the rotary angles). Every operation is an explicitly rounded
// intrinsic; the library is built with -fmad=false -ftz=false, so nothing is
// contracted or flushed.
//
// exp and log ("mojolearn" PyPI page, section "What bitwise identity means, and
// why it is not the default": the spellings of exp and log are fixed by the
// profile): Cody-Waite reduction with a degree-7 Taylor polynomial for exp,
// and the atanh series arranged as in fdlibm for log.
// sin and cos: Cody-Waite reduction by pi/2 (three-float split, fmaf steps)
// with Taylor polynomials to degree 9 (sin) and 10 (cos), quadrant by k mod 4.
#pragma once

#include <stdint.h>

#include "det_internal.cuh"

namespace det {

// ---------------------------------------------------------------- exp / log
// exp constants: each the float nearest to its definition. LOG2E = 1/ln 2,
// LN2_HI = ln 2, LN2_LO = ln 2 - LN2_HI, C_k = 1/k!.
constexpr float kLog2e = 0x1.715476p+0f;
constexpr float kLn2Hi = 0x1.62e430p-1f;
constexpr float kLn2Lo = -0x1.05c610p-29f;
constexpr float kC2 = 0x1p-1f, kC3 = 0x1.555556p-3f, kC4 = 0x1.555556p-5f;
constexpr float kC5 = 0x1.111112p-7f, kC6 = 0x1.6c16c2p-10f, kC7 = 0x1.a01a02p-13f;
constexpr float kExpHi = 0x1.62e42ep+6f;   // largest float with a finite exp
constexpr float kExpLo = -104.0f;          // below: +0
// log constants: A_k = 2/k (k = 3..11 odd); the largest float below sqrt 2.
constexpr float kA3 = 0x1.555556p-1f, kA5 = 0x1.99999ap-2f, kA7 = 0x1.24924ap-2f;
constexpr float kA9 = 0x1.c71c72p-3f, kA11 = 0x1.745d18p-3f;
constexpr unsigned kSqrt2Bits = 0x3fb504f3u;

__device__ __forceinline__ float pow2i(int e) {   // 2^e, -126 <= e <= 127
    return __uint_as_float(unsigned(e + 127) << 23);
}

__device__ __forceinline__ float det_exp(float x) {
    if (x != x) return __fadd_rn(x, x);
    if (x > kExpHi) return __uint_as_float(0x7f800000u);
    if (x < kExpLo) return 0.0f;
    const float t = __fmul_rn(x, kLog2e);
    const float n = rintf(t);                 // round half to even
    float r = __fmaf_rn(-n, kLn2Hi, x);
    r = __fmaf_rn(-n, kLn2Lo, r);
    float p = kC7;
    p = __fmaf_rn(p, r, kC6);
    p = __fmaf_rn(p, r, kC5);
    p = __fmaf_rn(p, r, kC4);
    p = __fmaf_rn(p, r, kC3);
    p = __fmaf_rn(p, r, kC2);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const int ni = __float2int_rn(n);         // |n| <= 150, exact
    if (ni > 127) return __fmul_rn(__fadd_rn(p, p), pow2i(127));
    if (ni < -126) return __fmul_rn(__fmul_rn(p, pow2i(ni + 64)), pow2i(-64));
    return __fmul_rn(p, pow2i(ni));
}

// The fast forms below serve the row reductions (cross-entropy, the causal
// softmax), whose exp arguments are x - max <= 0.
namespace {
// exp for arguments d <= 0 (or -inf), never NaN, without branches: the same
// bits as det_exp(d) whenever the returned n satisfies n >= -125; otherwise the
// caller must use det_exp(d). n = rint(t) is formed as (t + 1.5 2^23) -
// 1.5 2^23, which rounds t to an integer with ties to even for |t| < 2^22; it
// can differ from rintf only in the sign of a zero n, which reaches the
// result only through r = d - n ln2 and the polynomial's products with r,
// where it is inert. For n >= -125 the scaling p 2^n is exact and is done on
// the exponent bits.
constexpr float kRoundMagic = 0x1.8p23f;

__device__ __forceinline__ float exp_le0_fast(float d, int &ni) {
    const float t = __fmul_rn(d, kLog2e);
    const float tm = __fadd_rn(t, kRoundMagic);
    ni = __float_as_int(tm) - __float_as_int(kRoundMagic);
    const float n = __fsub_rn(tm, kRoundMagic);
    float r = __fmaf_rn(-n, kLn2Hi, d);
    r = __fmaf_rn(-n, kLn2Lo, r);
    float p = kC7;
    p = __fmaf_rn(p, r, kC6);
    p = __fmaf_rn(p, r, kC5);
    p = __fmaf_rn(p, r, kC4);
    p = __fmaf_rn(p, r, kC3);
    p = __fmaf_rn(p, r, kC2);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    return __int_as_float(__float_as_int(p) + int(unsigned(ni) << 23));
}

// The general exp as an out-of-line call, for the rarely taken paths of the
// row reductions (deep underflow, -inf, non-finite maxima), so they cost no
// registers in the hot loops.
__device__ __noinline__ float det_exp_call(float x) { return det_exp(x); }

// exp_le0_fast on a pair: d = x - m, then the same rounded steps as the scalar
// routine on both halves at once; n ln2 enters as n (-LN2_HI), which is the
// same product as (-n) LN2_HI. Returns the pair and the two n.
// t = d LOG2E is formed by two scalar multiplies: a packed multiply whose
// result feeds a packed add was measured to round like a fused multiply-add
// (t not rounded on its own) at the ties of rint(t), which moves n there.
__device__ __forceinline__ f32x2 exp2_le0_fast(f32x2 x, f32x2 m2, int &n0, int &n1) {
    const f32x2 d = sub2(x, m2);
    float d0, d1;
    unpack2(d, d0, d1);
    const f32x2 t = pack2(__fmul_rn(d0, kLog2e), __fmul_rn(d1, kLog2e));
    const f32x2 tm = add2(t, splat2(kRoundMagic));
    const f32x2 n = sub2(tm, splat2(kRoundMagic));
    f32x2 r = fma2(n, splat2(-kLn2Hi), d);
    r = fma2(n, splat2(-kLn2Lo), r);
    f32x2 p = fma2(splat2(kC7), r, splat2(kC6));
    p = fma2(p, r, splat2(kC5));
    p = fma2(p, r, splat2(kC4));
    p = fma2(p, r, splat2(kC3));
    p = fma2(p, r, splat2(kC2));
    p = fma2(p, r, splat2(1.0f));
    p = fma2(p, r, splat2(1.0f));
    float t0, t1, p0, p1;
    unpack2(tm, t0, t1);
    unpack2(p, p0, p1);
    n0 = __float_as_int(t0) - __float_as_int(kRoundMagic);
    n1 = __float_as_int(t1) - __float_as_int(kRoundMagic);
    return pack2(__int_as_float(__float_as_int(p0) + int(unsigned(n0) << 23)),
                 __int_as_float(__float_as_int(p1) + int(unsigned(n1) << 23)));
}

// exp(v - m) for the 4 lanes of a granule; d <= 0 for every element of a row
// with a finite max. Rare deep-underflow elements take the general routine.
__device__ __forceinline__ float4 exp4(float4 v, float m) {
    const f32x2 m2 = splat2(m);
    int n0, n1, n2, n3;
    const f32x2 e01 = exp2_le0_fast(pack2(v.x, v.y), m2, n0, n1);
    const f32x2 e23 = exp2_le0_fast(pack2(v.z, v.w), m2, n2, n3);
    float4 e;
    unpack2(e01, e.x, e.y);
    unpack2(e23, e.z, e.w);
    if (min(min(n0, n1), min(n2, n3)) < -125) {
        if (n0 < -125) e.x = det_exp_call(__fsub_rn(v.x, m));
        if (n1 < -125) e.y = det_exp_call(__fsub_rn(v.y, m));
        if (n2 < -125) e.z = det_exp_call(__fsub_rn(v.z, m));
        if (n3 < -125) e.w = det_exp_call(__fsub_rn(v.w, m));
    }
    return e;
}

}  // namespace

__device__ __forceinline__ float det_log(float x) {
    if (x != x) return __fadd_rn(x, x);
    if (x < 0.0f) return __uint_as_float(0x7fc00000u);
    if (x == 0.0f) return __uint_as_float(0xff800000u);
    if (x == __uint_as_float(0x7f800000u)) return x;
    int e = 0;
    if (x < 0x1p-126f) { x = __fmul_rn(x, 0x1p23f); e = -23; }
    const unsigned b = __float_as_uint(x);
    e += int(b >> 23) - 127;
    unsigned fb = (b & 0x007fffffu) | 0x3f800000u;
    if (fb > kSqrt2Bits) { fb -= 0x00800000u; e += 1; }
    const float f = __uint_as_float(fb);
    const float u = __fsub_rn(f, 1.0f);
    const float s = __fdiv_rn(u, __fadd_rn(2.0f, u));
    const float z = __fmul_rn(s, s);
    float R = kA11;
    R = __fmaf_rn(R, z, kA9);
    R = __fmaf_rn(R, z, kA7);
    R = __fmaf_rn(R, z, kA5);
    R = __fmaf_rn(R, z, kA3);
    R = __fmul_rn(R, z);
    const float h = __fmul_rn(__fmul_rn(0.5f, u), u);
    const float lf = __fsub_rn(u, __fsub_rn(h, __fmul_rn(s, __fadd_rn(h, R))));
    const float ef = __int2float_rn(e);
    return __fmaf_rn(ef, kLn2Hi, __fmaf_rn(ef, kLn2Lo, lf));
}

// ---------------------------------------------------------------- sin / cos
// Constants: each the float nearest to its definition (2/pi; pi/2 split in
// three floats; the Taylor terms (-1)^k / (2k+1)! and (-1)^k / (2k)!).
constexpr float kTwoOverPi = 0x1.45f306p-1f;
constexpr float kPio2_1 = 0x1.921fb6p+0f, kPio2_2 = -0x1.777a5cp-25f;
constexpr float kPio2_3 = -0x1.ee59dap-50f;
constexpr float kS3 = -0x1.555556p-3f, kS5 = 0x1.111112p-7f;
constexpr float kS7 = -0x1.a01a02p-13f, kS9 = 0x1.71de3ap-19f;
constexpr float kCc2 = -0x1p-1f, kCc4 = 0x1.555556p-5f, kCc6 = -0x1.6c16c2p-10f;
constexpr float kCc8 = 0x1.a01a02p-16f, kCc10 = -0x1.27e4fcp-22f;
constexpr float kTrigMax = 0x1p20f;

// sin and cos of x together: k = rint(x 2/pi); r = x - k pi/2 (three fmaf
// steps); z = r^2; sin_r = fmaf(r, z Ps(z), r); cos_r = fmaf(Pc(z), z, 1);
// the quadrant k mod 4 picks the signs. 0 gives (x, 1); |x| > 2^20 and NaN
// give NaN.
__device__ __forceinline__ void det_sincos(float x, float &sn, float &cs) {
    if (x != x || fabsf(x) > kTrigMax) {
        sn = cs = __uint_as_float(0x7fc00000u);
        return;
    }
    if (x == 0.0f) {
        sn = x;
        cs = 1.0f;
        return;
    }
    const float k = rintf(__fmul_rn(x, kTwoOverPi));
    float r = __fmaf_rn(-k, kPio2_1, x);
    r = __fmaf_rn(-k, kPio2_2, r);
    r = __fmaf_rn(-k, kPio2_3, r);
    const float z = __fmul_rn(r, r);
    float ps = kS9;
    ps = __fmaf_rn(ps, z, kS7);
    ps = __fmaf_rn(ps, z, kS5);
    ps = __fmaf_rn(ps, z, kS3);
    const float s = __fmaf_rn(r, __fmul_rn(z, ps), r);
    float pc = kCc10;
    pc = __fmaf_rn(pc, z, kCc8);
    pc = __fmaf_rn(pc, z, kCc6);
    pc = __fmaf_rn(pc, z, kCc4);
    pc = __fmaf_rn(pc, z, kCc2);
    const float c = __fmaf_rn(pc, z, 1.0f);
    const int q = __float2int_rz(k) & 3;
    sn = q == 0 ? s : q == 1 ? c : q == 2 ? -s : -c;
    cs = q == 0 ? c : q == 1 ? -s : q == 2 ? -c : s;
}

}  // namespace det
