// Weight-only FP8 / NVFP4 variant of the skinny-M weight-streaming GEMM.
//
// Formats ("Kimi-K3-DSpark-NVFP4": FP8 per-channel weight-only is the recommended
// build; NVFP4 = compressed-tensors nvfp4-pack-quantized, group 16, E4M3 group
// scales, weight-only, "What is quantized to what": MLP, o_proj, q_b_proj,
// context_proj):
//   FP8:   w = E4M3(q) * scale[row]
//   NVFP4: w = E2M1(q) * E4M3(s_group) * global
// An E4M3 value, and an E2M1 value times its E4M3 group scale (at most 6
// significant bits, magnitude <= 2688), are exact in f16. So converter warps
// decode each raw tile exactly into f16 (one convert per pair for E4M3, a
// convert and a multiply for E2M1) and store it straight into tensor memory
// (row = lane, two k per 32-bit cell); the small activation tile is converted
// from bf16 to f16 in place (exact for |x| in [2^-14, 65504]; smaller
// magnitudes round to f16 subnormals, absolute error <= 2^-25; a larger one
// is reported as DSPARK_ERR_BAD_INPUT rather than overflowed silently);
// the tensor core runs kind::f16 with f16 operands and its A operand read from
// TMEM; the remaining per-row (FP8) or per-tensor (NVFP4) scale multiplies the
// fp32 accumulator row in the epilogue. The result is the exact product of the
// decoded weights and the activations (up to fp32 summation).
//
// Roles (one CTA per SM, 14 warps): warp 0 TMA producer (raw weight tiles,
// NVFP4 group scales, activation tiles into a ring of raw stages in shared
// memory); warps 6-13 converters in two groups of four (one warp per TMEM lane
// quadrant) taking alternate 64-wide k sub-blocks into a ring of up to 12 TMEM
// A stages; warp 1 MMA issuer; warps 2-5 epilogue. Work split, split-tile
// reduction and bounded waits are those of the bf16 kernel.
#pragma once

#include "gemm.cuh"

namespace ds {

template <int FMT>
struct QFmt;
template <>
struct QFmt<DSPARK_FMT_FP8> {
    static constexpr int kKR = 128;          // k per raw stage (128 bytes per row)
    static constexpr int kDataBytes = 128 * 128;
    static constexpr int kScaleBytes = 0;
};
template <>
struct QFmt<DSPARK_FMT_NVFP4> {
    static constexpr int kKR = 256;          // k per raw stage (128 bytes of packed codes per row)
    static constexpr int kDataBytes = 128 * 128;
    static constexpr int kScaleBytes = 128 * 16;  // 16 group scales per row
};
template <>
struct QFmt<DSPARK_FMT_MXFP4> {
    static constexpr int kKR = 512;          // k per raw stage (256 bytes of packed codes per row, two halves)
    static constexpr int kDataBytes = 2 * 128 * 128;
    static constexpr int kScaleBytes = 128 * 16;  // 16 power-of-two scales (groups of 32) per row
};

constexpr int kQConvThreads = 256;

template <int BN, int FMT>
struct GemmQCfg {
    static constexpr int kKR = QFmt<FMT>::kKR;
    static constexpr int kNSub = kKR / 64;
    static constexpr int kDataBytes = QFmt<FMT>::kDataBytes;
    static constexpr int kScaleBytes = QFmt<FMT>::kScaleBytes;
    static constexpr int kBBytes = BN * 128;
    static constexpr int kRawBytes = kDataBytes + kScaleBytes + kNSub * kBBytes;
    static constexpr int kTmemCols = 512;
    static constexpr int kACol0 = 2 * BN;                  // A stages follow the two accumulators
    static constexpr int kAFit = (kTmemCols - kACol0) / 32;
    static constexpr int kAStages = kAFit > 12 ? 12 : kAFit;
    static constexpr int kXchgFloats = 64 * 17;
    static constexpr int kFixed = 1024 + kXchgFloats * 4 + 1024;
    static constexpr int kRawFit = (kGemmMaxSmem - kFixed) / kRawBytes;
    static constexpr int kRawStages = kRawFit > 12 ? 12 : kRawFit;
    static constexpr int kSmemBytes = kFixed + kRawStages * kRawBytes;
    static constexpr int kThreads = 192 + kQConvThreads;
    static_assert(kRawStages >= 2 && kRawStages * kKR >= 384 && kAStages >= 4, "rings too shallow");
    static_assert(kRawBytes % 1024 == 0, "1024-byte stage alignment");
};

DS_DEVINL uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
    uint32_t d;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"((uint16_t)two_bytes));
    return d;
}
DS_DEVINL uint32_t e2m1x2_to_f16x2(uint32_t one_byte) {
    uint32_t d;
    asm("{\n\t.reg .b8 b;\n\tcvt.u8.u16 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(d) : "h"((uint16_t)one_byte));
    return d;
}
DS_DEVINL uint32_t mul_f16x2(uint32_t a, uint32_t b) {
    const __half2 r = __hmul2(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&b));
    return *reinterpret_cast<const uint32_t *>(&r);
}

// Byte offset of 16-byte chunk c of row r in a 128-row tile stored in the
// 128-byte-swizzled K-major layout (8-row atoms of 1024 bytes).
DS_DEVINL uint32_t sw128_off(int r, int c) { return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4)); }

// Row r of sub-block sb (64 k) of a raw stage, decoded to 32 f16 pairs (even k low).
// 2^(e - 127) of an E8M0 scale as an f16 pair, for e - 127 in [-22, 13], where
// every E2M1 value times the scale is exact in f16; other scales set *bad.
DS_DEVINL uint32_t e8m0_to_f16x2(uint32_t e, bool &bad) {
    const int k = (int)e - 127;
    uint32_t h;
    if (k < -22 || k > 13) {
        bad = true;
        h = 0u;
    } else {
        h = k >= -14 ? (uint32_t)(k + 15) << 10 : 1u << (k + 24);
    }
    return h * 0x10001u;
}

template <int FMT>
DS_DEVINL void convert_row(const uint8_t *raw, int sb, int r, uint32_t (&o)[32], bool &bad) {
    if (FMT == DSPARK_FMT_FP8) {
        // 128 E4M3 codes per row in 8 swizzled 16-byte chunks; sub-block sb = chunks 4sb..4sb+3
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 v = *(const uint4 *)(raw + sw128_off(r, 4 * sb + c));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                o[8 * c + 2 * t] = e4m3x2_to_f16x2(w[t] & 0xFFFFu);
                o[8 * c + 2 * t + 1] = e4m3x2_to_f16x2(w[t] >> 16);
            }
        }
    } else if (FMT == DSPARK_FMT_MXFP4) {
        // 512 E2M1 codes per row: two halves of 256 (128 bytes, 8 swizzled chunks of 32
        // codes each); sub-block sb = half sb / 4, chunks 2 (sb % 4), +1; 16 E8M0 scales per
        // row (one per 32 codes) follow the data
        const uint8_t *half = raw + (sb >> 2) * (128 * 128);
        const uint8_t *scales = raw + 2 * 128 * 128 + r * 16 + 2 * sb;
        const uint32_t sg[2] = {e8m0_to_f16x2(scales[0], bad), e8m0_to_f16x2(scales[1], bad)};
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const uint4 v = *(const uint4 *)(half + sw128_off(r, 2 * (sb & 3) + c));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
#pragma unroll
                for (int bt = 0; bt < 4; ++bt)
                    o[16 * c + 4 * t + bt] = mul_f16x2(e2m1x2_to_f16x2((w[t] >> (8 * bt)) & 0xFFu), sg[c]);
            }
        }
    } else {
        // 256 E2M1 codes per row (two per byte, even element low) in 8 swizzled chunks of
        // 32 codes; sub-block sb = chunks 2sb, 2sb+1; 16 E4M3 group scales per row follow
        const uint8_t *scales = raw + 128 * 128 + r * 16 + 4 * sb;
        const uint32_t s4 = *(const uint32_t *)scales;  // groups 4sb .. 4sb+3
        const uint32_t s01 = e4m3x2_to_f16x2(s4 & 0xFFFFu), s23 = e4m3x2_to_f16x2(s4 >> 16);
        const uint32_t sg[4] = {(s01 & 0xFFFFu) * 0x10001u, (s01 >> 16) * 0x10001u, (s23 & 0xFFFFu) * 0x10001u,
                                (s23 >> 16) * 0x10001u};
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const uint4 v = *(const uint4 *)(raw + sw128_off(r, 2 * sb + c));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
#pragma unroll
                for (int bt = 0; bt < 4; ++bt) {
                    const int e = 4 * t + bt;  // byte e of the chunk: elements 32c + 2e, +1
                    o[16 * c + e] = mul_f16x2(e2m1x2_to_f16x2((w[t] >> (8 * bt)) & 0xFFu), sg[2 * c + (e >> 3)]);
                }
            }
        }
    }
}

// bf16 -> f16 in place for the activation sub-tile (BN rows x 64 k, any layout).
// A magnitude above the f16 range sets DSPARK_ERR_BAD_INPUT.
template <int BN>
DS_DEVINL void bf16_tile_to_f16(uint8_t *tile, int gthr, int *err) {
    bool over = false;
#pragma unroll
    for (int j = 0; j < (BN * 8 + 127) / 128; ++j) {
        const int c = gthr + 128 * j;
        if (c < BN * 8) {
            uint4 *p = (uint4 *)(tile + 16 * c);
            uint4 v = *p;
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float lo = __uint_as_float(w[t] << 16), hi = __uint_as_float(w[t] & 0xFFFF0000u);
                over |= fmaxf(fabsf(lo), fabsf(hi)) > 65504.f;
                const __half2 h = __floats2half2_rn(lo, hi);
                w[t] = *reinterpret_cast<const uint32_t *>(&h);
            }
            *p = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    if (over) set_error(err, DSPARK_ERR_BAD_INPUT);
}

template <int BN, int FMT>
__global__ void __launch_bounds__(GemmQCfg<BN, FMT>::kThreads, 1)
    gemm_q_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                  const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmS2,
                  const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
    using C = GemmQCfg<BN, FMT>;
    constexpr int RS = C::kRawStages, CS = C::kAStages, NS = C::kNSub;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sRaw = smem;
    float *xchg = (float *)(sRaw + RS * C::kRawBytes);
    uint64_t *raw_full = (uint64_t *)(xchg + C::kXchgFloats);
    uint64_t *raw_empty = raw_full + RS;
    uint64_t *cvt_full = raw_empty + RS;
    uint64_t *cvt_empty = cvt_full + CS;
    uint64_t *tfull = cvt_empty + CS;
    uint64_t *tempty = tfull + 2;
    uint64_t *done = tempty + 2;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    __shared__ int s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const long long u0 = gemm_unit_begin(cta, p.units, p.grid);
    const long long u1 = gemm_unit_begin(cta + 1, p.units, p.grid);

    if (threadIdx.x == 0) {
        for (int s = 0; s < RS; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], 1);
        }
        for (int s = 0; s < CS; ++s) {
            mbar_init(&cvt_full[s], kQConvThreads / 2 / 32);  // one arrival per converter warp
            mbar_init(&cvt_empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        mbar_init(done, 1);
        s_abort = 0;
        fence_mbar_init();
    }
    if (threadIdx.x == 32) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmA2);
        tma_prefetch_desc(&tmB);
        if (FMT != DSPARK_FMT_FP8) {
            tma_prefetch_desc(&tmS);
            tma_prefetch_desc(&tmS2);
        }
    }
    if (warp == 1) tmem_alloc(&s_tmem, C::kTmemCols);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    uint32_t armed = 0, armed_par = 0;
    pdl_trigger();

    auto load_weights = [&](long long u, int s, uint64_t pol) {
        const int tile = (int)(u / p.KB), kr = (int)(u % p.KB);
        uint8_t *raw = sRaw + s * C::kRawBytes;
        const int row0 = p.paired ? tile * 64 : tile * 128;
        const int row1 = p.paired ? tile * 64 : tile * 128 + 64;
        const CUtensorMap *m1 = p.paired ? &tmA2 : &tmA;
        // the codes' map has 16-bit elements: x counts byte pairs
        tma_load_2d_hint(raw, &tmA, kr * (C::kDataBytes / 256), row0, &raw_full[s], pol);
        tma_load_2d_hint(raw + 8192, m1, kr * (C::kDataBytes / 256), row1, &raw_full[s], pol);
        if (FMT == DSPARK_FMT_MXFP4) {  // second half of the 256 packed bytes per row
            tma_load_2d_hint(raw + 16384, &tmA, kr * 128 + 64, row0, &raw_full[s], pol);
            tma_load_2d_hint(raw + 16384 + 8192, m1, kr * 128 + 64, row1, &raw_full[s], pol);
        }
        if (FMT != DSPARK_FMT_FP8) {
            const CUtensorMap *n1 = p.paired ? &tmS2 : &tmS;
            tma_load_2d_hint(raw + C::kDataBytes, &tmS, kr * 16, row0, &raw_full[s], pol);
            tma_load_2d_hint(raw + C::kDataBytes + 1024, n1, kr * 16, row1, &raw_full[s], pol);
        }
    };
    auto load_acts = [&](long long u, int s) {
        const int kr = (int)(u % p.KB);
        uint8_t *b = sRaw + s * C::kRawBytes + C::kDataBytes + C::kScaleBytes;
#pragma unroll
        for (int sb = 0; sb < NS; ++sb) tma_load_2d(b + sb * C::kBBytes, &tmB, (kr * NS + sb) * 64, 0, &raw_full[s]);
    };

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            const long long pre = min((long long)RS, u1 - u0);
            for (long long it = 0; it < pre; ++it) {
                mbar_arrive_expect_tx(&raw_full[(int)it], C::kRawBytes);
                armed |= 1u << (int)it;
                load_weights(u0 + it, (int)it, pol);
            }
            l2_prefetch_share(p.pf, (unsigned int)cta, (unsigned int)p.grid);
            pdl_wait();
            for (long long it = 0; it < pre; ++it) load_acts(u0 + it, (int)it);
            long long it = pre;
            for (long long u = u0 + pre; u < u1; ++u, ++it) {
                const int s = (int)(it % RS);
                const uint32_t round = (uint32_t)(it / RS);
                if (!mbar_wait_bounded(&raw_empty[s], (round & 1u) ^ 1u, &s_abort)) break;
                mbar_arrive_expect_tx(&raw_full[s], C::kRawBytes);
                armed |= 1u << s;
                armed_par = (armed_par & ~(1u << s)) | ((round & 1u) << s);
                load_weights(u, s, pol);
                load_acts(u, s);
            }
        } else {
            pdl_wait();
        }
    } else if (warp == 1) {
        pdl_wait();
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(128, BN);
            long long it = 0, u = u0, cit = 0;
            int seg = 0;
            bool ok = true;
            while (u < u1 && ok) {
                const int tile = (int)(u / p.KB);
                const long long seg_end = min(u1, (long long)(tile + 1) * p.KB);
                const int a = seg & 1;
                if (!mbar_wait_bounded(&tempty[a], (((uint32_t)seg >> 1) & 1u) ^ 1u, &s_abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(a * BN);
                bool first = true;
                for (; u < seg_end && ok; ++u, ++it) {
                    const int s = (int)(it % RS);
                    if (!mbar_wait_bounded(&raw_full[s], (uint32_t)(it / RS) & 1u, &s_abort)) {
                        ok = false;
                        break;
                    }
                    const uint8_t *b = sRaw + s * C::kRawBytes + C::kDataBytes + C::kScaleBytes;
                    for (int sb = 0; sb < NS; ++sb, ++cit) {
                        const int t = (int)(cit % CS);
                        if (!mbar_wait_bounded(&cvt_full[t], (uint32_t)(cit / CS) & 1u, &s_abort)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t at = tmem + (uint32_t)(C::kACol0 + 32 * t);
                        const uint64_t bd = sdesc_k_sw128(smem_u32(b + sb * C::kBBytes));
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_bf16_tmem_a(d, at + (uint32_t)(8 * k), bd + (uint64_t)(2 * k), idesc,
                                            (first && k == 0) ? 0u : 1u);
                        first = false;
                        mma_commit(&cvt_empty[t]);
                    }
                    if (ok) mma_commit(&raw_empty[s]);
                }
                if (!ok) break;
                mma_commit(&tfull[a]);
                ++seg;
            }
            mma_commit(done);
            mbar_drain(done, 0);
        }
    } else if (warp >= 6) {
        // converters: group g takes sub-blocks g, g+2, ...; warp w covers TMEM lanes 32*(w%4)..
        pdl_wait();
        const int g = (warp - 6) >> 2, qd = warp & 3, r = 32 * qd + lane;
        const int gthr = threadIdx.x - 192 - 128 * g;
        const long long total_sub = (u1 - u0) * NS;
        // software pipeline: the tensor-memory store of one sub-block completes (and is
        // announced on cvt_full, once per warp: 128 arrivals on one barrier serialise)
        // while the next one is decoded
        int pend = -1;
        for (long long cit = g; cit < total_sub; cit += 2) {
            const long long it = cit / NS;
            const int sb = (int)(cit % NS), s = (int)(it % RS), t = (int)(cit % CS);
            // every thread waits itself; the result is made warp-uniform (tcgen05.st is warp-wide)
            const bool got = mbar_wait_bounded(&raw_full[s], (uint32_t)(it / RS) & 1u, &s_abort) &&
                             mbar_wait_bounded(&cvt_empty[t], ((uint32_t)(cit / CS) & 1u) ^ 1u, &s_abort);
            if (!__all_sync(0xffffffffu, got)) break;
            uint32_t v[32];
            uint8_t *rawp = sRaw + s * C::kRawBytes;
            bool bad_scale = false;
            convert_row<FMT>(rawp, sb, r, v, bad_scale);
            if (bad_scale) set_error(p.err, DSPARK_ERR_BAD_INPUT);
            bf16_tile_to_f16<BN>(rawp + C::kDataBytes + C::kScaleBytes + sb * C::kBBytes, gthr, p.err);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (pend >= 0) {
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&cvt_full[pend]);
            }
            tc_fence_after();
            tmem_st32(tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(C::kACol0 + 32 * t), v);
            pend = t;
        }
        if (pend >= 0) {
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&cvt_full[pend]);
        }
    } else {
        pdl_wait();
        // epilogue: warps 2..5, TMEM lane quadrant = warp % 4
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const int et = threadIdx.x - 64;
        const int nch = p.paired ? 64 : 128;
        int seg = 0;
        long long u = u0;
        while (u < u1) {
            const int tile = (int)(u / p.KB);
            const long long tbeg = (long long)tile * p.KB, tend = tbeg + p.KB;
            const long long seg_end = min(u1, tend);
            const bool whole = (u == tbeg) && (seg_end == tend);
            const int a = seg & 1;
            const bool got = mbar_wait_bounded(&tfull[a], ((uint32_t)seg >> 1) & 1u, &s_abort);
            if (!named_bar_and(2, 128, got)) break;
            tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * BN);
            const int slot = (tile == (int)(u0 / p.KB)) ? 2 * cta : 2 * cta + 1;
            // output channel of this accumulator row and its scale
            const bool second = p.paired && row >= 64;
            const int n_row = p.paired ? tile * 64 + (row & 63) : tile * 128 + row;
            const bool scaled_here = whole || p.epi == EPI_PENDING;
            const float rs = (scaled_here && n_row < p.n_out) ? gemm_row_scale(p, n_row, second) : 1.f;
            for (int c0 = 0; c0 < BN; c0 += 16) {
                float v[16];
                tmem_ld16(taddr + (uint32_t)c0, v);
                if (p.epi == EPI_PENDING) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] *= rs;
                    gemm_pending_store<BN>(p, slot, row, c0, v);
                } else if (whole) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] *= rs;
                    if (p.paired) {
                        if (q >= 2) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) xchg[(row - 64) * 17 + j] = v[j];
                        }
                        named_bar_sync(1, 128);
                        const int n = tile * 64 + row;
                        if (q < 2 && n < p.n_out) {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (c0 + j < p.M) gemm_store_swiglu(p, n, c0 + j, v[j], xchg[row * 17 + j]);
                        }
                        named_bar_sync(1, 128);
                    } else {
                        const int n = tile * 128 + row;
                        if (n < p.n_out) {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (c0 + j < p.M) gemm_store(p, n, c0 + j, v[j]);
                        }
                    }
                } else {
                    float4 *dst = (float4 *)(p.partials + ((size_t)slot * 128 + row) * BN + c0);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[a]);
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
                    gemm_reduce_tile<BN, true, 2>(p, tile, c_lo, c_hi, et, nch);
                }
            }
            u = seg_end;
            ++seg;
        }
    }
    __syncthreads();
    if (s_abort) {
        if (threadIdx.x == 0) set_error(p.err, DSPARK_ERR_TIMEOUT);
        if (warp == 0 && lane == 0) {
            for (int s = 0; s < RS; ++s)
                if (armed & (1u << s)) mbar_drain(&raw_full[s], (armed_par >> s) & 1u);
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
