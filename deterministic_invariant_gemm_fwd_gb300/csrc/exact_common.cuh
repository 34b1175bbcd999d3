// exact_common.cuh - float64 building blocks of the exact tier shared by its
// kernels (exact_kbn.cu: any dtype; exact_int.cu: bf16 on the integer pipes).
#pragma once

#include <stdint.h>

namespace carbon {

// Exact widening of an fp32 bit pattern to float64.  Normal numbers are
// re-biased with integer operations; zeros keep their sign; subnormals,
// infinities and NaNs (rare) take the hardware conversion, which is exact.
__device__ __forceinline__ double widen(uint32_t f) {
    const uint32_t mag = f & 0x7fffffffu;
    if (mag - 0x00800000u < 0x7f000000u) {            // exponent field 1..254
        const uint32_t hi = (f & 0x80000000u) | ((mag >> 3) + (896u << 20));
        return __hiloint2double((int)hi, (int)(f << 29));
    }
    if (mag == 0u) return __hiloint2double((int)(f & 0x80000000u), 0);
    return (double)__uint_as_float(f);
}

// One KBN step with an exact product p = x * w.  key = (x_hi & EXP) +
// (w_hi & EXP): the sum of the operands' shifted exponent fields.
__device__ __forceinline__ void kbn_product_step(double &s, double &c, double x, double w,
                                                 uint32_t key) {
    const double t = __fma_rn(x, w, s);
    // E(s) > E(x) + E(w)  <=>  es_field + 1022 >= ex_field + ew_field
    const uint32_t es = ((uint32_t)__double2hiint(s) & 0x7ff00000u) + (1022u << 20);
    double a1, a2, b1, b2;
    asm("{\n\t.reg .pred sbig;\n\t"
        "setp.ge.u32 sbig, %4, %5;\n\t"
        "selp.f64 %0, %6, %7, sbig;\n\t"
        "selp.f64 %1, %8, %9, sbig;\n\t"
        "selp.f64 %2, %7, %6, sbig;\n\t"
        "selp.f64 %3, %9, %8, sbig;\n\t}"
        : "=d"(a1), "=d"(a2), "=d"(b1), "=d"(b2)
        : "r"(es), "r"(key), "d"(s), "d"(x), "d"(1.0), "d"(w));
    const double d = __fma_rn(a1, a2, -t);   // s - t   or   p - t   (exact)
    const double e = __fma_rn(b1, b2, d);    // + p     or   + s     (exact)
    c = __dadd_rn(c, e);
    s = t;
}

// One KBN step of the outer sum over chunk values (no product).  The
// magnitude test is exact: for non-NaN doubles the order of |a| equals the
// unsigned order of their bit patterns with the sign cleared.
__device__ __forceinline__ void kbn_value_step(double &S, double &C, double P) {
    const double t = __dadd_rn(S, P);
    const unsigned long long aS = (unsigned long long)__double_as_longlong(S) & 0x7fffffffffffffffull;
    const unsigned long long aP = (unsigned long long)__double_as_longlong(P) & 0x7fffffffffffffffull;
    const bool sbig = aS >= aP;
    const double u = sbig ? S : P;
    const double v = sbig ? P : S;
    C = __dadd_rn(C, __dadd_rn(__dadd_rn(u, -t), v));
    S = t;
}

// float64 -> bf16, round to nearest even, one rounding.
__device__ __forceinline__ unsigned short exact_round_bf16(double y) {
    const unsigned long long u = (unsigned long long)__double_as_longlong(y);
    const unsigned int sign = (unsigned int)(u >> 48) & 0x8000u;
    const unsigned long long mag = u & 0x7fffffffffffffffull;
    if (mag > 0x7ff0000000000000ull) return (unsigned short)(sign | 0x7fc0u);  // NaN
    const int E = (int)(mag >> 52) - 1023;
    if (E >= 128) return (unsigned short)(sign | 0x7f80u);                    // |y| >= 2^128
    if (E >= -126) {                                                          // bf16 normal range
        const unsigned long long lsb = (mag >> 45) & 1ull;
        const unsigned long long r = (mag + 0x00000fffffffffffull + lsb) >> 45;
        const int Ed = (int)(r >> 7);                                         // biased, after carry
        if (Ed - 1023 >= 128) return (unsigned short)(sign | 0x7f80u);
        return (unsigned short)(sign | ((unsigned int)(Ed - 1023 + 127) << 7) | (unsigned int)(r & 0x7f));
    }
    if (E < -134) return (unsigned short)sign;                                // below half the quantum
    // bf16 subnormal range: n = RNE(|y| / 2^-133), 0 <= n <= 128 (128 = min normal)
    const unsigned long long sig = (mag & 0x000fffffffffffffull) | 0x0010000000000000ull;
    const int shift = -81 - E;                                                // 46 .. 53
    const unsigned long long n = sig >> shift;
    const unsigned long long rem = sig & ((1ull << shift) - 1ull);
    const unsigned long long half = 1ull << (shift - 1);
    const unsigned long long nr = n + ((rem > half || (rem == half && (n & 1ull))) ? 1ull : 0ull);
    return (unsigned short)(sign | (unsigned int)nr);
}

}  // namespace carbon
