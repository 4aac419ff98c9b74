// The sampling spec shared by the Markov rollout and the verification kernels:
// counter-based uniforms, this library's own fp32 exp, the 2^32-scaled integer
// weights and keys of a logit row, argmax keys, and block reductions.
//
// Model cards: greedy or probabilistic draft sampling, top-p, an argmax match
// at temperature 0 ("Kimi-K3-DSpark-NVFP4", Quick Start / Sampling options);
// the target's distribution is preserved ("kimi-k3-dspark-gguf", intro). The
// cards give no numerics; every decision here is exact integer arithmetic so
// that a second implementation reproduces it bit for bit.
#pragma once

#include "internal.h"

namespace ds {

constexpr int kSampThreads = 512;
constexpr int kMaxSampBs = 32;

// ---------------------------------------------------------------------------
// Counter-based uniforms: Philox4x32-10, first output word.
// ---------------------------------------------------------------------------
DS_DEVINL uint32_t philox_word(unsigned long long seed, uint32_t seq, uint32_t step, uint32_t pos, uint32_t purpose) {
    uint32_t c0 = step, c1 = seq, c2 = pos, c3 = purpose;
    uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        if (round) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return c0;
}

// ---------------------------------------------------------------------------
// Own fp32 exp for x <= 0 (every step one IEEE operation).
// ---------------------------------------------------------------------------
DS_DEVINL float exp_hat(float x) {
    if (!(x >= -23.0f)) return 0.0f;
    // n = rint(x * log2(e)) (ties to even) by adding and removing 1.5 * 2^23: for
    // |x * log2(e)| < 2^22 the sum rounds to an integer and its low bits hold n
    // (the same integer as rintf, off the conversion pipe)
    const float t = __fadd_rn(__fmul_rn(x, 1.44269502162933349609375f), 12582912.0f);
    const float n = __fsub_rn(t, 12582912.0f);
    const int ni = __float_as_int(t) - 0x4B400000;
    float r = __fmaf_rn(-n, 0.693145751953125f, x);
    r = __fmaf_rn(-n, 1.428606765330187045037746429443359375e-06f, r);
    float p = 1.98412701138295233249664306640625e-04f;
    p = __fmaf_rn(p, r, 1.388888922519981861114501953125e-03f);
    p = __fmaf_rn(p, r, 8.333333767950534820556640625e-03f);
    p = __fmaf_rn(p, r, 4.16666679084300994873046875e-02f);
    p = __fmaf_rn(p, r, 1.66666671633720397949218750e-01f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    return __fmul_rn(p, __int_as_float((ni + 127) << 23));
}

// y = l / T, IEEE division (T == 1 gives l itself, bit for bit, without the division).
DS_DEVINL float div_T(float l, float T) { return T == 1.0f ? l : __fdiv_rn(l, T); }

// floor(e * 2^32) for e = 0 or a normal e in [0, 1] (the range of exp^(x), x <= 0),
// from the bits of e: e = M * 2^(ex - 150) with the 24-bit significand M, so
// e * 2^32 = M * 2^(ex - 118). The same integer as converting e * 2^32 (exact).
DS_DEVINL unsigned long long weight_bits(float e) {
    const uint32_t u = __float_as_uint(e);
    const int ex = (int)(u >> 23);
    if (ex < 95) return 0ull;  // e < 2^-32 (or zero)
    const unsigned long long M = (unsigned long long)((u & 0x7FFFFFu) | 0x800000u);
    return ex >= 118 ? M << (ex - 118) : M >> (118 - ex);
}

DS_DEVINL unsigned long long weight_of(float l, float T, float m) {
    const float y = div_T(l, T);
    const float e = exp_hat(__fsub_rn(y, m));
    return weight_bits(e);
}

DS_DEVINL unsigned long long key_of(unsigned long long E, int v) {
    return (E << 18) | (unsigned long long)((1u << 18) - 1u - (uint32_t)v);
}

// Order-preserving map of fp32 to uint32 (NaN excluded by the callers).
DS_DEVINL uint32_t f2ord(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
DS_DEVINL float ord2f(uint32_t o) { return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o); }

// Greedy key: larger value first, lower id on ties (-0 counts as +0).
DS_DEVINL unsigned long long argmax_key(float l, int v) {
    if (l == 0.0f) l = 0.0f;
    return ((unsigned long long)f2ord(l) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)v);
}
DS_DEVINL int argmax_token(unsigned long long key) { return (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull)); }

DS_DEVINL unsigned long long top_p_q32(float top_p) {
    if (!(top_p > 0.0f)) return 0ull;
    if (top_p >= 1.0f) return 1ull << 32;
    return (unsigned long long)((double)top_p * 4294967296.0);
}

// ---------------------------------------------------------------------------
// Block reductions
// ---------------------------------------------------------------------------
DS_DEVINL unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w > v ? w : v;
    }
    return v;
}
// Inclusive suffix sums over the lanes of a warp (lane l: sum of lanes >= l).
DS_DEVINL unsigned long long warp_suffix_u64(unsigned long long v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long w = __shfl_down_sync(0xffffffffu, v, o);
        if (lane + o < 32) v += w;
    }
    return v;
}
DS_DEVINL unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

DS_DEVINL unsigned long long block_max_u64(unsigned long long v, unsigned long long *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_max_u64(v);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    unsigned long long r = (threadIdx.x < (blockDim.x >> 5)) ? red[threadIdx.x] : 0ull;
    if (warp == 0) r = warp_max_u64(r);
    if (threadIdx.x == 0) red[32] = r;
    __syncthreads();
    return red[32];
}
DS_DEVINL unsigned long long block_sum_u64(unsigned long long v, unsigned long long *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum_u64(v);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    unsigned long long r = (threadIdx.x < (blockDim.x >> 5)) ? red[threadIdx.x] : 0ull;
    if (warp == 0) r = warp_sum_u64(r);
    if (threadIdx.x == 0) red[32] = r;
    __syncthreads();
    return red[32];
}


}  // namespace ds
