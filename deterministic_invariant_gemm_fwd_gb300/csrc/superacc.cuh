// superacc.cuh - device arithmetic of the correctly rounded tier: the exact
// sum of the products and the bias, rounded once to the output type (the
// superaccumulators of the Carbon README's "Roadmap": exact summation that
// needs no fixed order).
//
// Two forms of the exact sum are rounded here:
//  * a fixed-point accumulator of 32-bit digits, each held in an int64 so that
//    carries can wait until the end (the warp-per-output kernel of
//    superacc.cu: any input type, any magnitudes);
//  * a 128-bit integer times a power of two (the bf16 tensor-core path of
//    exact_tc.cu, whose exact sums live in an integer grain), with the bias
//    joined exactly.
#pragma once

#include <stdint.h>

#include "carbon_internal.h"

namespace carbon {
namespace sacc {

// Accumulator layout: digit k holds bits [32k, 32k + 32) of value * 2^kOff.
// Products of two fp32 values are integers below 2^48 times 2^e with
// e >= -298 and below 2^256 in magnitude; bf16 and fp16 products lie inside
// that range.  Digit kDigits - 1 keeps the sign after the carries.
constexpr int kDigits = 20;
constexpr int kOff = 320;

// Output format: precision, exponent bias, largest exponent, and the
// smallest quantum (of the subnormals) as a power of two.
template <int DT> struct Fmt;
template <> struct Fmt<CARBON_F32> { static constexpr int p = 24, bias = 127, emax = 127, qmin = -149; };
template <> struct Fmt<CARBON_BF16> { static constexpr int p = 8, bias = 127, emax = 127, qmin = -133; };
template <> struct Fmt<CARBON_F16> { static constexpr int p = 11, bias = 15, emax = 15, qmin = -24; };

// Class of an input: finite, +inf, -inf or NaN.
enum { kFinite = 0, kPosInf = 1, kNegInf = 2, kNaN = 4 };

// Input bits -> m * 2^e (m a signed integer below 2^p in magnitude) and class.
template <int DT>
__device__ __forceinline__ void decode_value(uint32_t h, long long &m, int &e, int &cls) {
    uint32_t ef, fr, sgn;
    if (DT == CARBON_F32) { ef = (h >> 23) & 0xffu; fr = h & 0x7fffffu; sgn = h >> 31; }
    else if (DT == CARBON_BF16) { ef = (h >> 7) & 0xffu; fr = h & 0x7fu; sgn = (h >> 15) & 1u; }
    else { ef = (h >> 10) & 0x1fu; fr = h & 0x3ffu; sgn = (h >> 15) & 1u; }
    constexpr uint32_t emask = DT == CARBON_F16 ? 0x1fu : 0xffu;
    constexpr int fbits = Fmt<DT>::p - 1;
    constexpr int e0 = Fmt<DT>::qmin;                  // exponent of the lowest bit of a subnormal
    if (ef == emask) {
        cls = fr ? kNaN : (sgn ? kNegInf : kPosInf);
        m = 0; e = 0;
        return;
    }
    cls = kFinite;
    const long long mag = ef ? (long long)((1u << fbits) | fr) : (long long)fr;
    m = sgn ? -mag : mag;
    e = (ef ? (int)ef - 1 : 0) + e0;
}

// IEEE class of a product of two classified values (m = 0 marks a zero).
__device__ __forceinline__ int product_class(int ca, long long ma, int cb, long long mb) {
    if ((ca | cb) & kNaN) return kNaN;
    if (ca == kFinite && cb == kFinite) return kFinite;
    // an infinity times zero is NaN; else an infinity with the product's sign
    const bool za = ca == kFinite && ma == 0, zb = cb == kFinite && mb == 0;
    if (za || zb) return kNaN;
    const bool na = ca == kNegInf || (ca == kFinite && ma < 0);
    const bool nb = cb == kNegInf || (cb == kFinite && mb < 0);
    return (na != nb) ? kNegInf : kPosInf;
}

// acc += m * 2^(pos - kOff), |m| < 2^48, 0 <= pos, pos + 48 < 32 * (kDigits - 1).
// Every digit takes a predicated addition (no dynamic register index).
__device__ __forceinline__ void add_scaled(long long (&acc)[kDigits], long long m, int pos) {
    const bool neg = m < 0;
    const unsigned long long u = neg ? 0ull - (unsigned long long)m : (unsigned long long)m;
    const int k = pos >> 5, s = pos & 31;
    const unsigned long long lo = u << s;                                  // bits 0..63 of u << s
    const unsigned long long hi = s ? (u >> (64 - s)) : 0ull;              // bits 64.. (< 2^15)
    long long d0 = (long long)(lo & 0xffffffffull), d1 = (long long)(lo >> 32), d2 = (long long)hi;
    if (neg) { d0 = -d0; d1 = -d1; d2 = -d2; }
#pragma unroll
    for (int d = 0; d < kDigits; ++d)
        acc[d] += d == k ? d0 : (d == k + 1 ? d1 : (d == k + 2 ? d2 : 0ll));
}

// Carries: digits 0 .. kDigits-2 into [0, 2^32), the top digit keeps the sign.
__device__ __forceinline__ void carry(long long (&acc)[kDigits]) {
#pragma unroll
    for (int d = 0; d + 1 < kDigits; ++d) {
        const long long c = acc[d] >> 32;              // floor division by 2^32
        acc[d] -= c * (1ll << 32);
        acc[d + 1] += c;
    }
}

// Output bits of sign * n * 2^qe, n < 2^(p+1) after rounding, qe >= qmin;
// n == 2^p (a carry out of the rounding) moves up one binade; overflow gives
// infinity.
template <int DT>
__device__ __forceinline__ uint32_t encode(bool neg, unsigned long long n, int qe) {
    constexpr int p = Fmt<DT>::p;
    const uint32_t sign = neg ? (DT == CARBON_F32 ? 0x80000000u : 0x8000u) : 0u;
    const uint32_t inf = DT == CARBON_F32 ? 0x7f800000u : (DT == CARBON_BF16 ? 0x7f80u : 0x7c00u);
    if (n == 0ull) return sign;
    if (n >> p) { n >>= 1; ++qe; }                     // exact: n was 2^p
    if (n < (1ull << (p - 1))) return sign | (uint32_t)n;   // subnormal (qe == qmin)
    const int E = qe + p - 1;                          // value in [2^E, 2^(E+1))
    if (E > Fmt<DT>::emax) return sign | inf;
    return sign | ((uint32_t)(E + Fmt<DT>::bias) << (p - 1)) | ((uint32_t)n & ((1u << (p - 1)) - 1u));
}

template <int DT>
__device__ __forceinline__ uint32_t nan_bits() {
    return DT == CARBON_F32 ? 0x7fc00000u : (DT == CARBON_BF16 ? 0x7fc0u : 0x7e00u);
}

template <int DT>
__device__ __forceinline__ uint32_t inf_bits(bool neg) {
    return DT == CARBON_F32 ? (neg ? 0xff800000u : 0x7f800000u)
                            : (DT == CARBON_BF16 ? (neg ? 0xff80u : 0x7f80u) : (neg ? 0xfc00u : 0x7c00u));
}

// Rounds the accumulator (already summed over the warp; destroyed) once to
// the output type.  cls: the OR of the terms' non-finite classes.  An exact
// zero gives +0.
template <int DT>
__device__ uint32_t round_acc(long long (&acc)[kDigits], int cls) {
    if ((cls & kNaN) || (cls & (kPosInf | kNegInf)) == (kPosInf | kNegInf)) return nan_bits<DT>();
    if (cls & (kPosInf | kNegInf)) return inf_bits<DT>((cls & kNegInf) != 0);
    carry(acc);
    const bool neg = acc[kDigits - 1] < 0;
    if (neg) {
#pragma unroll
        for (int d = 0; d < kDigits; ++d) acc[d] = -acc[d];
        carry(acc);
    }
    int top = -1;                                       // highest set bit
#pragma unroll
    for (int d = 0; d < kDigits; ++d)
        if (acc[d] != 0) top = 32 * d + 63 - __clzll(acc[d]);
    if (top < 0) return 0u;                             // exact zero: +0
    constexpr int p = Fmt<DT>::p;
    const int q = max(top - (p - 1), Fmt<DT>::qmin + kOff);   // bit of the quantum
    // bits q .. q + p (at most p + 1 of them) and the half and sticky bits below q
    unsigned long long n = 0ull;
    bool half = false, sticky = false;
#pragma unroll
    for (int d = 0; d < kDigits; ++d) {
        const unsigned long long v = (unsigned long long)acc[d];   // < 2^32 (top digit too, now)
        const int lo = 32 * d;                          // bit index of v's bit 0
        // part of v at or above q, aligned to q (digits above q + 40 are 0)
        if (lo + 32 > q && lo - q < 40) n |= (lo >= q) ? (v << (lo - q)) : (v >> (q - lo));
        // the half bit, q - 1
        if (q - 1 >= lo && q - 1 < lo + 32) half = (v >> (q - 1 - lo)) & 1ull;
        // sticky: bits below q - 1
        if (lo < q - 1) {
            const int nb = min(32, q - 1 - lo);
            sticky |= (v & ((nb == 32) ? 0xffffffffull : ((1ull << nb) - 1ull))) != 0ull;
        }
    }
    if (half && (sticky || (n & 1ull))) ++n;
    return encode<DT>(neg, n, q - kOff);
}

// S * 2^e rounded once to bf16 (|S| < 2^127).
__device__ __forceinline__ uint32_t round_i128_bf16(__int128 S, int e) {
    if (S == 0) return 0u;
    const bool neg = S < 0;
    const unsigned __int128 mag = neg ? (unsigned __int128)0 - (unsigned __int128)S : (unsigned __int128)S;
    const unsigned long long hi = (unsigned long long)(mag >> 64), lo = (unsigned long long)mag;
    const int nb = hi ? 128 - __clzll((long long)hi) : 64 - __clzll((long long)lo);
    const int q = max(nb - 1 + e - 7, Fmt<CARBON_BF16>::qmin);   // quantum exponent
    const int sh = q - e;                                         // bits below the quantum
    unsigned long long n;
    if (sh <= 0) {
        n = (unsigned long long)(mag << (-sh));                   // exact, below 2^8
    } else if (sh > nb) {
        n = 0ull;                                                 // below half the quantum
    } else {
        n = (unsigned long long)(mag >> sh);
        const bool half = (mag >> (sh - 1)) & 1;
        const bool sticky = sh > 1 && (mag & (((unsigned __int128)1 << (sh - 1)) - 1)) != 0;
        if (half && (sticky || (n & 1ull))) ++n;
    }
    return encode<CARBON_BF16>(neg, n, q);
}

// The exact value T * 2^G + b (T an integer below 2^70 in magnitude, b =
// bm * 2^be the bias with |bm| < 2^8, bm = 0 for none) rounded once to bf16.
// The two terms are aligned exactly in 128 bits unless one lies wholly below
// the other's grain by 20 bits or more.  Then the small term only decides on
// which side of the large one the sum falls, and a unit 20 bits below the
// large term's grain, with the small term's sign, rounds the same way: the
// large term L is a nonzero multiple of its grain 2^g, so every rounding
// midpoint and every power of two near L is a multiple of 2^(g - 8) (the bf16
// quantum in L's binade is at least 2^(g - 7), and at least 2^-133), and none
// lies strictly between L and L +- 2^(g - 20); both sums fall in that open
// interval, on the same side of L, in the same binade.
__device__ __forceinline__ uint32_t exact_sum_bf16(__int128 T, int G, int bm, int be, bool bias_bad,
                                                   uint32_t bias_bits) {
    if (bias_bad) return (bias_bits & 0x7fu) ? 0x7fc0u : bias_bits;   // T is finite: inf or NaN wins
    if (bm == 0) return round_i128_bf16(T, G);
    if (T == 0) return round_i128_bf16((__int128)bm, be);
    const __int128 sgnT = T < 0 ? -1 : 1;
    const int nbT = [&] {
        const unsigned __int128 mag = T < 0 ? (unsigned __int128)0 - (unsigned __int128)T : (unsigned __int128)T;
        const unsigned long long hi = (unsigned long long)(mag >> 64), lo = (unsigned long long)mag;
        return hi ? 128 - __clzll((long long)hi) : 64 - __clzll((long long)lo);
    }();
    if (be + 8 <= G - 20)                               // |b| < 2^(G - 20): b is a sticky unit
        return round_i128_bf16(T * ((__int128)1 << 20) + (bm < 0 ? -1 : 1), G - 20);
    if (nbT + G <= be - 20)                             // |T 2^G| < 2^(be - 20)
        return round_i128_bf16((__int128)bm * ((__int128)1 << 20) + sgnT, be - 20);
    // here -28 < be - G < nbT + 20 <= 86: both shifts below 2^94
    if (be >= G) return round_i128_bf16(T + (__int128)bm * ((__int128)1 << (be - G)), G);
    return round_i128_bf16(T * ((__int128)1 << (G - be)) + (__int128)bm, be);
}

}  // namespace sacc
}  // namespace carbon
