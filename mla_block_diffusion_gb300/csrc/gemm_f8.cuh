// Weight-only FP8 GEMM with the weights fed to the tensor core as they are stored.
//
//   y[m, n] = scale[n] * sum_k E4M3(q[n, k]) * x[m, k]     (x bf16, M <= 32 rows)
//
// Activation rows are padded to MR = 8, 16 or 32.
//
// Format ("Kimi-K3-DSpark-NVFP4", FP8 per-channel weight-only build): one E4M3
// code per weight and one fp32 scale per output channel.
//
// The E4M3 weight tile goes from HBM by TMA into shared memory and from there
// straight into tcgen05.mma kind::f8f6f4 as the A operand; nothing decodes it.
// The B operand is the activation tile written as a sum of two E4M3 numbers:
// for every activation row and 128-wide k chunk with largest magnitude in
// [2^E, 2^(E+1)), x * 2^(7-E) has magnitude below 256; hi = RN_E4M3(x 2^(7-E))
// keeps its 4 leading significant bits and lo = RN_E4M3((x 2^(7-E) - hi) 16)
// the remaining (at most 4) bits of the bf16 significand. Both are exact for
// every element within 2^13 of the chunk maximum (the E4M3 normal range), so
// hi 2^(E-7) + lo 2^(E-11) equals x; smaller elements keep an absolute error
// below 2^-21 of the chunk maximum. hi rows occupy B rows 0..MR-1 and lo rows
// MR..2MR-1 (N = 2 MR accumulator columns).
//
// Every chunk (4 MMAs of K = 32) has its own accumulator slot in tensor memory;
// the epilogue warps read it, multiply column m by 2^(E_m-7) (hi) or
// 2^(E_m-11) (lo) and add it into fp32 registers. Products of two E4M3 values
// are exact, so the result is the product of the decoded weights and the bf16
// activations up to fp32 summation order, as with the bf16 kernel.
//
// Roles (one CTA per SM, 12 warps): warp 0 TMA producer (weight tiles only, a
// ring of up to 12 16-KB stages, filled ahead of the dependency wait); warps 6,
// 7, 10 and 11 split the activation chunk of every fourth unit, read from L2
// into registers one unit ahead, into the E4M3 B tile and the factors of the
// unit's accumulator slot (eight slots: the split runs ahead of the MMAs and
// never holds a weight stage); warp 1 MMA issuer; warps 2-5 epilogue
// (per-chunk promotion, then the output functor, split partials or a pending
// slot as in the bf16 kernel).
#pragma once

#include "gemm.cuh"

namespace ds {

template <int MR>
struct GemmF8Cfg {
    static constexpr int kN = 2 * MR;                 // accumulator columns: hi rows, then lo rows
    static constexpr int kABytes = 128 * 128;         // 128 channels x 128 k, one byte each
    static constexpr int kBBytes = kN * 128;          // 2 MR rows x 128 k E4M3
    static constexpr int kSlots = 8;                  // accumulator slots (and E4M3 B tiles)
    static constexpr int kTmemCols = kSlots * kN <= 32 ? 32 : kSlots * kN <= 64 ? 64 : kSlots * kN <= 128 ? 128
                                     : kSlots * kN <= 256 ? 256 : 512;
    static constexpr int kXchgFloats = 64 * 17;
    static constexpr int kFixed = 1024 + kXchgFloats * 4 + kSlots * kN * 4 + kSlots * kBBytes + 1024;
    static constexpr int kStagesFit = (kGemmMaxSmem - kFixed) / kABytes;
    // 11 stages leave shared memory, and the register cap registers, for the
    // next kernel's CTAs to become resident beside this one before it ends
    static constexpr int kStages = kStagesFit > 11 ? 11 : kStagesFit;
    static constexpr int kMaxRegs = MR <= 8 ? 144 : 168;
    static constexpr int kSmemBytes = kFixed + kStages * kABytes;
    // split warps 6, 7, 10 and 11: only on the SM sub-partitions (warp % 4) of
    // neither the producer (warp 0) nor the MMA issuer (warp 1), whose single
    // threads would otherwise wait for issue slots behind the split arithmetic;
    // warps 8 and 9 only fill the numbering
    static constexpr int kSplitWarps = 4;
    static constexpr int kThreads = 192 + 32 * 6;
    // the split warps load the activation chunk of their next unit while
    // splitting the current one (register double buffer) where registers allow
    static constexpr bool kPrefetch = MR <= 16;
    static_assert(MR == 8 || MR == 16 || MR == 32, "activation rows padded to 8, 16 or 32");
    static_assert(kStages >= 8, "ring too shallow");
    static_assert(kBBytes % 1024 == 0, "1024-byte alignment");
    static_assert(kSlots * kN <= 512, "tensor memory");
};

// Instruction descriptor, kind::f8f6f4: E4M3 A and B, fp32 accumulator, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

DS_DEVINL void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Two floats to an f16 pair (round to nearest even): `even` in the low half.
DS_DEVINL uint32_t f32x2_to_f16x2(float even, float odd) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(odd), "f"(even));
    return d;
}
// An f16 pair to two E4M3 codes (round to nearest even, saturating), low half
// to the low byte.
DS_DEVINL uint32_t f16x2_to_e4m3x2(uint32_t h) {
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(d) : "r"(h));
    return d;
}
// Two E4M3 codes (low byte first) to an f16 pair.
DS_DEVINL uint32_t e4m3x2_to_f16x2_(uint32_t two) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)two));
    return h;
}
// (a - b) * 16 on f16 pairs.
DS_DEVINL uint32_t f16x2_sub_x16(uint32_t a, uint32_t b) {
    const __half2 d = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&b)),
                              __floats2half2_rn(16.f, 16.f));
    return *reinterpret_cast<const uint32_t *>(&d);
}

// The activation chunk of one unit in registers: pass p, lane l holds the 8
// bf16 values k = kc + 8 (l % 16) .. + 7 of row 2p + l / 16 (zero beyond M or K);
// passes whose rows all lie at or beyond M are not loaded.
template <int MR>
DS_DEVINL void load_chunk(uint4 (&xv)[MR / 2], const __nv_bfloat16 *act, int K, int M, int kc, int lane) {
    const int half = lane >> 4, c = lane & 15;
    const int k = kc + 8 * c;
#pragma unroll
    for (int pz = 0; pz < MR / 2; ++pz) {
        const int r = 2 * pz + half;
        xv[pz] = make_uint4(0u, 0u, 0u, 0u);
        if (2 * pz < M && r < M && k < K) xv[pz] = __ldcg((const uint4 *)(act + (size_t)r * K + k));
    }
}

// The chunk into the E4M3 B tile (2 MR rows x 128 bytes, 128-byte swizzled
// K-major) and the per-column promotion factors. Lanes 0-15 take row 2p, lanes
// 16-31 row 2p + 1; each lane 8 consecutive k. Rows at or beyond M are left
// as they are (zero since the kernel's start).
//
// Arithmetic: the chunk maximum is an integer maximum over the bf16 magnitude
// bits; x 2^(7-E) is exact in f16 (8 significant bits, at least 2^-17), hi is
// its E4M3 rounding, (x 2^(7-E) - hi) 16 is exact in f16 and lo its E4M3
// rounding.
template <int MR>
DS_DEVINL void split_chunk(const uint4 (&xv)[MR / 2], uint8_t *b8, float *sc, int lane, int M, bool &bad) {
    const int half = lane >> 4, c = lane & 15;
    const int chunk16 = c >> 1, byte_in = (c & 1) * 8;  // position of k = 8c in a 128-byte E4M3 row
    // every pass is computed (rows beyond M hold zeros) so that the compiler can
    // interleave the passes; only rows below M are stored
#pragma unroll
    for (int pz = 0; pz < MR / 2; ++pz) {
        const int r = 2 * pz + half;
        const int rl = MR + r;
        const uint32_t w[4] = {xv[pz].x, xv[pz].y, xv[pz].z, xv[pz].w};
        uint32_t mx = __vmaxu2(__vmaxu2(w[0] & 0x7FFF7FFFu, w[1] & 0x7FFF7FFFu),
                               __vmaxu2(w[2] & 0x7FFF7FFFu, w[3] & 0x7FFF7FFFu));
        mx = max(mx & 0xFFFFu, mx >> 16);
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        bad |= mx >= 0x7F80u;  // inf or NaN in the row's chunk
        int E = (int)(mx >> 7) - 127;  // exponent of the chunk maximum (bf16 field)
        E = E < -110 ? -110 : (E > 127 ? 127 : E);
        const float s = __uint_as_float((uint32_t)(127 + 7 - E) << 23);  // 2^(7 - E)
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const uint32_t a = f32x2_to_f16x2(__uint_as_float(w[t] << 16) * s, __uint_as_float(w[t] & 0xFFFF0000u) * s);
            hi[t] = f16x2_to_e4m3x2(a);
            lo[t] = f16x2_to_e4m3x2(f16x2_sub_x16(a, e4m3x2_to_f16x2_(hi[t])));
        }
        if (r >= M) continue;
        uint8_t *dhi = b8 + (r >> 3) * 1024 + (r & 7) * 128 + ((chunk16 ^ (r & 7)) << 4) + byte_in;
        uint8_t *dlo = b8 + (rl >> 3) * 1024 + (rl & 7) * 128 + ((chunk16 ^ (rl & 7)) << 4) + byte_in;
        *(uint2 *)dhi = make_uint2(hi[0] | (hi[1] << 16), hi[2] | (hi[3] << 16));
        *(uint2 *)dlo = make_uint2(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16));
        if (c == 0) {
            sc[r] = __uint_as_float((uint32_t)(127 + E - 7) << 23);   // 2^(E - 7)
            sc[rl] = __uint_as_float((uint32_t)(127 + E - 11) << 23); // 2^(E - 11)
        }
    }
}

template <int MR>
__global__ void __launch_bounds__(GemmF8Cfg<MR>::kThreads, 1) __maxnreg__(GemmF8Cfg<MR>::kMaxRegs)
    gemm_f8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                   const GemmParams p) {
    using C = GemmF8Cfg<MR>;
    constexpr int RS = C::kStages, R = C::kSlots, N = C::kN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;                              // [RS] weight tiles
    uint8_t *sB = sA + RS * C::kABytes;              // [R] E4M3 B tiles
    float *xchg = (float *)(sB + R * C::kBBytes);
    float *scl = xchg + C::kXchgFloats;              // [R][N] promotion factors
    uint64_t *full = (uint64_t *)(scl + R * N);      // [RS] weight tile landed
    uint64_t *empty = full + RS;                     // [RS] the tile's MMAs completed
    uint64_t *bfull = empty + RS;                    // [R] B tile and factors written
    uint64_t *afull = bfull + R;                     // [R] accumulator slot complete
    uint64_t *aempty = afull + R;                    // [R] slot read by the epilogue
    uint64_t *done = aempty + R;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    __shared__ int s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const long long u0 = gemm_unit_begin(cta, p.units, p.grid);
    const long long u1 = gemm_unit_begin(cta + 1, p.units, p.grid);

    if (threadIdx.x == 0) {
        for (int s = 0; s < RS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int j = 0; j < R; ++j) {
            mbar_init(&bfull[j], 1);
            mbar_init(&afull[j], 1);
            mbar_init(&aempty[j], 4);  // one arrival per epilogue warp
        }
        mbar_init(done, 1);
        s_abort = 0;
        fence_mbar_init();
    }
    if (threadIdx.x == 32) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmA2);
    }
    if (warp == 1) tmem_alloc(&s_tmem, C::kTmemCols);
    // B rows of activation rows at or beyond M, and their factors, stay zero
    for (int i = threadIdx.x; i < R * C::kBBytes / 16; i += C::kThreads) ((uint4 *)sB)[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < R * N; i += C::kThreads) scl[i] = 0.f;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    uint32_t armed = 0, armed_par = 0;
    pdl_trigger();

    auto load_weights = [&](long long u, int s, uint64_t pol) {
        const int tile = (int)(u / p.KB), kb = (int)(u % p.KB);
        uint8_t *a = sA + s * C::kABytes;
        // the codes' map has 16-bit elements: x counts byte pairs
        if (p.paired) {
            tma_load_2d_hint(a, &tmA, kb * 64, tile * 64, &full[s], pol);
            tma_load_2d_hint(a + 8192, &tmA2, kb * 64, tile * 64, &full[s], pol);
        } else {
            tma_load_2d_hint(a, &tmA, kb * 64, tile * 128, &full[s], pol);
            tma_load_2d_hint(a + 8192, &tmA, kb * 64, tile * 128 + 64, &full[s], pol);
        }
    };

    if (warp == 0) {
        // weights do not depend on the previous kernel: the whole ring is filled
        // before the dependency wait
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            const long long pre = min((long long)RS, u1 - u0);
            for (long long it = 0; it < pre; ++it) {
                mbar_arrive_expect_tx(&full[(int)it], C::kABytes);
                armed |= 1u << (int)it;
                load_weights(u0 + it, (int)it, pol);
            }
            l2_prefetch_share(p.pf, (unsigned int)cta, (unsigned int)p.grid);
            long long it = pre;
            for (long long u = u0 + pre; u < u1; ++u, ++it) {
                const int s = (int)(it % RS);
                const uint32_t round = (uint32_t)(it / RS);
                if (!mbar_wait_bounded(&empty[s], (round & 1u) ^ 1u, &s_abort)) break;
                mbar_arrive_expect_tx(&full[s], C::kABytes);
                armed |= 1u << s;
                armed_par = (armed_par & ~(1u << s)) | ((round & 1u) << s);
                load_weights(u, s, pol);
            }
        }
        pdl_wait();
    } else if (warp == 1) {
        pdl_wait();
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(128, N);
            bool ok = true;
            long long it = 0;
            for (long long u = u0; u < u1 && ok; ++u, ++it) {
                const int s = (int)(it % RS), j = (int)(it % R);
                const uint32_t ps = (uint32_t)(it / RS) & 1u, pj = (uint32_t)(it / R) & 1u;
                ok = mbar_wait_bounded(&bfull[j], pj, &s_abort) && mbar_wait_bounded(&aempty[j], pj ^ 1u, &s_abort) &&
                     mbar_wait_bounded(&full[s], ps, &s_abort);
                if (!ok) break;
                tc_fence_after();
                const uint64_t ad = sdesc_k_sw128(smem_u32(sA + s * C::kABytes));
                const uint64_t bd = sdesc_k_sw128(smem_u32(sB + j * C::kBBytes));
                const uint32_t d = tmem + (uint32_t)(j * N);
#pragma unroll
                for (int k = 0; k < 4; ++k) mma_e4m3(d, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), idesc, k > 0);
                mma_commit(&empty[s]);
                mma_commit(&afull[j]);
            }
            mma_commit(done);
            mbar_drain(done, 0);
        }
    } else if (warp >= 6 && (warp & 3) >= 2) {
        // split warps: split warp sw takes units sw, sw + 4, ...; the
        // activations come from L2 (written by the previous kernel) into registers
        pdl_wait();
        const int sw = warp < 8 ? warp - 6 : warp - 8;
        bool bad = false;
        uint4 xa[MR / 2], xb[MR / 2];
        // one unit: wait for its slot, split, publish; false once a wait gave up
        auto unit = [&](long long it, const uint4 (&xv)[MR / 2]) -> bool {
            const int j = (int)(it % R);
            const uint32_t pj = (uint32_t)(it / R) & 1u;
            const bool got = mbar_wait_bounded(&aempty[j], pj ^ 1u, &s_abort);
            if (!__all_sync(0xffffffffu, got)) return false;
            split_chunk<MR>(xv, sB + j * C::kBBytes, scl + j * N, lane, p.M, bad);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&bfull[j]);
            return true;
        };
        auto kc = [&](long long it) { return (int)((u0 + it) % p.KB) * 128; };
        constexpr long long W = C::kSplitWarps;
        long long it = sw;
        if (u0 + it < u1) load_chunk<MR>(xa, p.act, p.K, p.M, kc(it), lane);
        if (C::kPrefetch) {
            // two register buffers in turn: the next unit's chunk is in flight
            // while this one is split
            while (u0 + it < u1) {
                if (u0 + it + W < u1) load_chunk<MR>(xb, p.act, p.K, p.M, kc(it + W), lane);
                if (!unit(it, xa)) break;
                it += W;
                if (u0 + it >= u1) break;
                if (u0 + it + W < u1) load_chunk<MR>(xa, p.act, p.K, p.M, kc(it + W), lane);
                if (!unit(it, xb)) break;
                it += W;
            }
        } else {
            for (; u0 + it < u1; it += W) {
                if (!unit(it, xa)) break;
                if (u0 + it + W < u1) load_chunk<MR>(xa, p.act, p.K, p.M, kc(it + W), lane);
            }
        }
        if (bad) set_error(p.err, DSPARK_ERR_BAD_INPUT);
    } else if (warp >= 6) {
        pdl_wait();  // warps 8 and 9: no role
    } else {
        pdl_wait();
        // epilogue: warps 2..5, TMEM lane quadrant = warp % 4
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const int et = threadIdx.x - 64;
        const int nch = p.paired ? 64 : 128;
        const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
        long long u = u0, it = 0;
        bool ok = true;
        while (u < u1 && ok) {
            const int tile = (int)(u / p.KB);
            const long long tbeg = (long long)tile * p.KB, tend = tbeg + p.KB;
            const long long seg_end = min(u1, tend);
            const bool whole = (u == tbeg) && (seg_end == tend);
            float acc[MR];
#pragma unroll
            for (int m = 0; m < MR; ++m) acc[m] = 0.f;
            for (; u < seg_end; ++u, ++it) {
                const int j = (int)(it % R);
                const uint32_t pj = (uint32_t)(it / R) & 1u;
                const bool got = mbar_wait_bounded(&bfull[j], pj, &s_abort) && mbar_wait_bounded(&afull[j], pj, &s_abort);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t v[N];
#pragma unroll
                for (int c0 = 0; c0 < N; c0 += 16) tmem_ld16_issue(tl + (uint32_t)(j * N + c0), *(uint32_t(*)[16]) & v[c0]);
                float fs[N];
                const float *f = scl + j * N;
#pragma unroll
                for (int m = 0; m < N; m += 4) *(float4 *)&fs[m] = *(const float4 *)(f + m);
#pragma unroll
                for (int c0 = 0; c0 < N; c0 += 16) tmem_ld_wait_tied(*(uint32_t(*)[16]) & v[c0]);
                // the slot (accumulator columns and factors) is free once every warp has read it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&aempty[j]);
#pragma unroll
                for (int m = 0; m < MR; ++m) {
                    acc[m] = fmaf(__uint_as_float(v[m]), fs[m], acc[m]);
                    acc[m] = fmaf(__uint_as_float(v[MR + m]), fs[MR + m], acc[m]);
                }
            }
            // a warp that gave up makes the others give up at the same segment
            if (!named_bar_and(2, 128, ok)) break;
            // the channel's weight scale
            const bool second = p.paired && row >= 64;
            const int n_row = p.paired ? tile * 64 + (row & 63) : tile * 128 + row;
            const float rs = n_row < p.n_out ? gemm_row_scale(p, n_row, second) : 0.f;
#pragma unroll
            for (int m = 0; m < MR; ++m) acc[m] *= rs;
            const int slot = (tile == (int)(u0 / p.KB)) ? 2 * cta : 2 * cta + 1;
            constexpr int CW = MR < 16 ? MR : 16;  // columns per output pass
#pragma unroll
            for (int c0 = 0; c0 < MR; c0 += CW) {
                float v[16];
#pragma unroll
                for (int m = 0; m < 16; ++m) v[m] = m < CW ? acc[c0 + m] : 0.f;
                if (p.epi == EPI_PENDING) {
                    gemm_pending_store<MR>(p, slot, row, c0, v);
                } else if (whole) {
                    if (p.paired) {
                        if (q >= 2) {
#pragma unroll
                            for (int m = 0; m < CW; ++m) xchg[(row - 64) * 17 + m] = v[m];
                        }
                        named_bar_sync(1, 128);
                        const int n = tile * 64 + row;
                        if (q < 2 && n < p.n_out) {
#pragma unroll
                            for (int m = 0; m < CW; ++m)
                                if (c0 + m < p.M) gemm_store_swiglu(p, n, c0 + m, v[m], xchg[row * 17 + m]);
                        }
                        named_bar_sync(1, 128);
                    } else {
                        const int n = tile * 128 + row;
                        if (n < p.n_out) {
#pragma unroll
                            for (int m = 0; m < CW; ++m)
                                if (c0 + m < p.M) gemm_store(p, n, c0 + m, v[m]);
                        }
                    }
                } else {
                    float4 *dst = (float4 *)(p.partials + ((size_t)slot * 128 + row) * MR + c0);
#pragma unroll
                    for (int m = 0; m < CW / 4; ++m)
                        dst[m] = make_float4(v[4 * m], v[4 * m + 1], v[4 * m + 2], v[4 * m + 3]);
                }
            }
            if (!whole && p.epi != EPI_PENDING) {
                __threadfence();
                named_bar_sync(1, 128);
                const int c_lo = gemm_cta_of_unit(tbeg, p.units, p.grid);
                const int c_hi = gemm_cta_of_unit(tend - 1, p.units, p.grid);
                if (et == 0) {
                    const int old = atomicAdd(&p.counters[tile], 1);
                    s_last = (old == c_hi - c_lo);
                    if (s_last) p.counters[tile] = 0;
                }
                named_bar_sync(1, 128);
                if (s_last) {
                    __threadfence();
                    gemm_reduce_tile<MR, false, 4>(p, tile, c_lo, c_hi, et, nch);
                }
            }
        }
    }
    __syncthreads();
    if (s_abort) {
        if (threadIdx.x == 0) set_error(p.err, DSPARK_ERR_TIMEOUT);
        if (warp == 0 && lane == 0) {
            for (int s = 0; s < RS; ++s)
                if (armed & (1u << s)) mbar_drain(&full[s], (armed_par >> s) & 1u);
        }
        __syncthreads();
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

}  // namespace ds
