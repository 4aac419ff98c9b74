// The correctly rounded double quotient e / S of two integers, 1 <= e <= S <
// 2^50, in integer arithmetic: the value the IEEE double division (round to
// nearest, ties to even) gives, without the double-precision pipe (a small
// fraction of the fp32 rate on this GPU).
//
// Method: normalise both to 64 bits (e << a, S << s, top bits set), so that
// e / S = (En / Sn) 2^(s - a) with En / Sn in (1/2, 2). A reciprocal
// R = floor(2^127 / Sn), computed once per divisor, gives the estimate
// mulhi(En, R) of Q = floor(En 2^63 / Sn); the exact remainder
// En 2^63 - Q Sn corrects it (at most two steps), then the 53 leading bits of Q
// are rounded to nearest even with the bits below and the remainder as sticky.
// The same source compiles for the host, where the tests compare it with the
// hardware division.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define DS_XD __host__ __device__ __forceinline__
#else
#define DS_XD static inline
#endif

namespace ds {

struct ExactDivisor {
    unsigned long long sn;  // S << s, top bit set
    unsigned long long r;   // floor(2^127 / sn) - 2^63 (sn > 2^63) or 2^63 (sn == 2^63)
    int s;
};

DS_XD int clz64_(unsigned long long x) {
#if defined(__CUDA_ARCH__)
    return __clzll((long long)x);
#else
    return __builtin_clzll(x);
#endif
}

// Divisor set-up (once per S >= 1): restoring division of 2^127 by sn.
DS_XD ExactDivisor exact_divisor(unsigned long long S) {
    ExactDivisor d;
    d.s = clz64_(S);
    d.sn = S << d.s;
    // floor(2^127 / sn) lies in (2^63, 2^64] for sn in [2^63, 2^64)
    unsigned __int128 num = (unsigned __int128)1 << 127;
    const unsigned __int128 q = num / d.sn;
    d.r = (unsigned long long)(q - ((unsigned __int128)1 << 63));  // keeps the value below 2^64
    return d;
}

// RN(e / S) as a double, e in [1, S].
DS_XD double exact_div(unsigned long long e, const ExactDivisor &d) {
    const int a = clz64_(e);
    const unsigned long long en = e << a;
    // Q estimate: floor(en * floor(2^127 / sn) / 2^64) <= Q; the reciprocal is
    // 2^63 + d.r, so en * recip = en * 2^63 + en * d.r
    const unsigned __int128 prod = ((unsigned __int128)en << 63) + (unsigned __int128)en * d.r;
    unsigned long long q = (unsigned long long)(prod >> 64);
    // exact remainder of en * 2^63 - q * sn (fits: q <= Q < 2^64, remainder < 3 sn)
    const unsigned __int128 num = (unsigned __int128)en << 63;
    unsigned __int128 rem = num - (unsigned __int128)q * d.sn;
    while (rem >= d.sn) {
        rem -= d.sn;
        ++q;
    }
    // q = floor(en * 2^63 / sn), in [2^62, 2^64)
    const int L = 63 - clz64_(q);                 // 62 or 63
    const int sh = L - 52;                        // bits below the 53 kept
    unsigned long long mant = q >> sh;
    const unsigned long long below = q & ((1ull << sh) - 1);
    const unsigned long long half = 1ull << (sh - 1);
    const bool sticky = rem != 0;
    if (below > half || (below == half && (sticky || (mant & 1ull))) ) {
        ++mant;
    }
    // value = mant * 2^sh / 2^63 * 2^(s - a)
    int ex = sh - 63 + d.s - a;  // value = mant * 2^ex, mant in [2^52, 2^53]
    if (mant == (1ull << 53)) {
        mant >>= 1;
        ++ex;
    }
    const unsigned long long bits = ((unsigned long long)(ex + 52 + 1023) << 52) | (mant & ((1ull << 52) - 1));
#if defined(__CUDA_ARCH__)
    return __longlong_as_double((long long)bits);
#else
    double out;
    __builtin_memcpy(&out, &bits, 8);
    return out;
#endif
}

}  // namespace ds
