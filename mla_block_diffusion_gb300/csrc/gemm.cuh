// Skinny-M weight-streaming GEMM on the 5th-generation tensor core.
//
//   y[m, n] = sum_k W[n, k] * x[m, k]      (W bf16 [N, K] row-major, x bf16 [M, K], M = 7 * batch)
//
// Every linear map of the drafter has M = 7 * batch rows against a weight
// matrix of millions of entries, so the weights are read exactly once and the
// kernel is bound by HBM. The product is computed "swapped": the weight tile is
// the A operand (128 output channels x 64 k, M = 128 of tcgen05.mma) and the few
// activation rows are the B operand (N = BN, a multiple of 16). The accumulator
// lives in TMEM (two buffers of BN fp32 columns).
//
// Roles (one CTA per SM, 6 warps):
//   warp 0    TMA producer: streams W tiles (evict-first) and x tiles into a
//             ring of shared-memory stages, completing on "full" mbarriers;
//   warp 1    MMA issuer: one thread issues 4 x tcgen05.mma (K = 16 each) per
//             stage and frees the stage with tcgen05.commit on "empty";
//   warps 2-5 epilogue: tcgen05.ld the accumulator (TMEM lane = output channel),
//             apply the output functor or write a split partial.
//
// Work split (stream-K): the (tile, k-block) units are divided into equal
// contiguous ranges, one per CTA, so every SM streams the same number of
// weight bytes. A tile covered by one CTA is finished directly from TMEM. A
// tile split across CTAs is finished by whichever contributor arrives last
// (atomic counter, no waiting): it sums the partials of all contributors in
// increasing CTA order, so the result does not depend on arrival order.
#pragma once

#include "common.cuh"

namespace ds {

// EPI_PENDING: no reduction in the GEMM; every CTA leaves its rows in the
// partials (GemmPending layout) and the consuming kernel sums them.
enum GemmEpi { EPI_STORE = 0, EPI_ADD = 1, EPI_SWIGLU = 2, EPI_PENDING = 3 };

struct GemmParams {
    int n_out;          // output channels
    int K;              // reduction length
    int M;              // valid activation rows (<= BN)
    int KB;             // k-blocks of 64
    int tiles;          // output tiles (128 channels, or 64 when paired)
    long long units;    // tiles * KB
    int grid;           // CTAs
    int paired;         // SwiGLU: A rows 0-63 from gate, 64-127 from up
    int epi;            // GemmEpi
    float *out_f32;     // [M, ldo]
    __nv_bfloat16 *out_bf16;
    int ldo;
    float *partials;    // [2 * grid][128][BN]
    int *counters;      // [tiles], zero between launches
    int *err;
    // weight-only formats: the accumulator row of output channel n is multiplied by
    // qscale[n] (FP8 per-channel scales; qscale2 for the up rows of a paired tile) or
    // by gscale / gscale2 (NVFP4 per-tensor scales). Unused for bf16 weights.
    const float *qscale, *qscale2;
    float gscale, gscale2;
    L2Prefetch pf;      // weights of a later kernel, pulled into L2 by the producer
    const __nv_bfloat16 *act;  // the activations [M, K] (read directly by the FP8 kernel)
    // Several matrices in one launch (the layers' kv_a rows of the latent-cache
    // append): tiles [l tpl, (l + 1) tpl) belong to matrix l, whose activations are
    // rows l brows .. of the B map and whose output starts lay_stride floats after
    // matrix l - 1's. tpl = 0: one matrix.
    int tpl, brows;
    long long lay_stride;
    // Pairwise reduction (every CTA's range covers at least one tile, so a split
    // tile has two contributors): CTA c + 1 takes the tile's last k-blocks first
    // thing, writes them to its slot 2(c + 1) and raises counters[tile]; CTA c,
    // which reaches the tile's first k-blocks last, reads that partial ahead of
    // its own last MMA, adds it (fixed order: c's sum, then c + 1's) and runs the
    // epilogue, then lowers the flag. No atomic and no second pass.
    int pair_red;
};

// Per-row output multiplier of a weight-only quantised matrix.
__device__ inline float gemm_row_scale(const GemmParams &p, int n, bool second) {
    if (p.qscale) return second ? p.qscale2[n] : p.qscale[n];
    return second ? p.gscale2 : p.gscale;
}

constexpr int kGemmMaxSmem = 232448;

template <int BN>
struct GemmCfg {
    static constexpr int kABytes = 128 * 128;  // 128 rows x 64 bf16
    static constexpr int kBBytes = BN * 128;   // BN rows x 64 bf16
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kXchgFloats = 64 * 17;
    static constexpr int kFixed = 1024 + kXchgFloats * 4 + 512;
    static constexpr int kStagesFit = (kGemmMaxSmem - kFixed) / kStageBytes;
    // 11 stages leave about 23 KB of the SM's shared memory for the next
    // kernel's CTAs to become resident early beside this one
    static constexpr int kStages = kStagesFit > 11 ? 11 : kStagesFit;
    static constexpr int kSmemBytes = kFixed + kStages * kStageBytes;
    static constexpr int kTmemCols = (2 * BN <= 32)    ? 32
                                     : (2 * BN <= 64)  ? 64
                                     : (2 * BN <= 128) ? 128
                                     : (2 * BN <= 256) ? 256
                                                       : 512;
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "tcgen05 M=128 needs N in 16..256, step 16");
    static_assert(kStages >= 3, "pipeline too shallow");
};

__device__ inline float silu_f(float g) { return g / (1.0f + __expf(-g)); }

__device__ inline void gemm_store(const GemmParams &p, int n, int m, float v) {
    float *dst = p.out_f32 + (size_t)m * p.ldo + n;
    if (p.epi == EPI_ADD)
        *dst += v;
    else
        *dst = v;
}

__device__ inline void gemm_store_swiglu(const GemmParams &p, int n, int m, float g, float u) {
    p.out_bf16[(size_t)m * p.ldo + n] = __float2bfloat16(silu_f(g) * u);
}

// EPI_PENDING: 16 accumulator columns (activation rows c0 ..) of tile row `row`
// into the slot (only the valid rows; a warp writes 128 consecutive bytes per row).
template <int BN>
__device__ __forceinline__ void gemm_pending_store(const GemmParams &p, int slot, int row, int c0,
                                                   const float (&v)[16]) {
    float *dst = p.partials + ((size_t)slot * BN + c0) * 128 + row;
#pragma unroll
    for (int j = 0; j < 16; ++j)
        if (c0 + j < p.M) dst[(size_t)j * 128] = v[j];
}

// Sum of the split partials of one tile, contributors in increasing CTA order
// (fixed order: the result does not depend on which CTA arrived last). Thread
// et owns output channel et and takes the valid rows in chunks of 8: the two
// float4 of every contributor of a batch of U are loaded before any is added,
// so a tile split over up to U CTAs costs one L2 round trip per chunk.
template <int BN, bool SCALED, int U, bool PAIRED>
__device__ __forceinline__ void gemm_reduce_impl(const GemmParams &p, int tile, int c_lo, int c_hi, int et, int n) {
    for (int c0 = 0; c0 < p.M; c0 += 8) {
        float a1[8], a2[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) a1[j] = a2[j] = 0.f;
        for (int cc = c_lo; cc <= c_hi; cc += U) {
            float4 v1[U][2], v2[PAIRED ? U : 1][2];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (cc + u <= c_hi) {
                    const int first_t = (int)(gemm_unit_begin(cc + u, p.units, p.grid) / p.KB);
                    const int sl = (tile == first_t) ? 2 * (cc + u) : 2 * (cc + u) + 1;
                    const float4 *src = (const float4 *)(p.partials + ((size_t)sl * 128 + et) * BN + c0);
                    v1[u][0] = __ldcg(src);
                    v1[u][1] = __ldcg(src + 1);
                    if (PAIRED) {
                        const float4 *src2 = src + 64 * BN / 4;
                        v2[u][0] = __ldcg(src2);
                        v2[u][1] = __ldcg(src2 + 1);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (cc + u <= c_hi) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        a1[4 * j] += v1[u][j].x;
                        a1[4 * j + 1] += v1[u][j].y;
                        a1[4 * j + 2] += v1[u][j].z;
                        a1[4 * j + 3] += v1[u][j].w;
                        if (PAIRED) {
                            a2[4 * j] += v2[u][j].x;
                            a2[4 * j + 1] += v2[u][j].y;
                            a2[4 * j + 2] += v2[u][j].z;
                            a2[4 * j + 3] += v2[u][j].w;
                        }
                    }
                }
            }
        }
        if (SCALED) {
            const float f1 = gemm_row_scale(p, n, false), f2 = PAIRED ? gemm_row_scale(p, n, true) : 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                a1[j] *= f1;
                a2[j] *= f2;
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (c0 + j < p.M) {
                if (PAIRED)
                    gemm_store_swiglu(p, n, c0 + j, a1[j], a2[j]);
                else
                    gemm_store(p, n, c0 + j, a1[j]);
            }
        }
    }
}

template <int BN, bool SCALED = false, int U = 8>
__device__ __forceinline__ void gemm_reduce_tile(const GemmParams &p, int tile, int c_lo, int c_hi, int et, int nch) {
    const int n = tile * nch + et;
    if (et >= nch || n >= p.n_out) return;
    if (p.paired)
        gemm_reduce_impl<BN, SCALED, (U > 1 ? U / 2 : 1), true>(p, tile, c_lo, c_hi, et, n);
    else
        gemm_reduce_impl<BN, SCALED, U, false>(p, tile, c_lo, c_hi, et, n);
}

// The weight maps of a several-matrix launch.
struct GemmMaps {
    CUtensorMap m[DSPARK_MAX_LAYERS];
};

// The kernel body; MULTI: tiles of several matrices (GemmParams::tpl), the A
// maps from `maps`, no paired tiles and no pending output.
template <int BN, bool MULTI>
DS_DEVINL void gemm_swapab_body(const CUtensorMap *mA, const CUtensorMap *mA2, const CUtensorMap *mB,
                                const GemmParams &p, const GemmMaps *maps) {
    const CUtensorMap &tmA = *mA, &tmA2 = *mA2, &tmB = *mB;
    using C = GemmCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;
    uint8_t *sB = smem + C::kStages * C::kABytes;
    float *xchg = (float *)(sB + C::kStages * C::kBBytes);
    uint64_t *full = (uint64_t *)(xchg + C::kXchgFloats);
    uint64_t *empty = full + C::kStages;
    uint64_t *tfull = empty + C::kStages;  // [2]
    uint64_t *tempty = tfull + 2;          // [2]
    uint64_t *done = tempty + 2;           // [1]
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    __shared__ int s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const long long u0 = gemm_unit_begin(cta, p.units, p.grid);
    const long long u1 = gemm_unit_begin(cta + 1, p.units, p.grid);

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
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
        if (!MULTI) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmA2);
        }
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) tmem_alloc(&s_tmem, C::kTmemCols);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    // producer bookkeeping for the drain after an abort
    uint32_t armed = 0, armed_par = 0;

    pdl_trigger();
    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            // Weights do not depend on the previous kernel: the first ring
            // stages get their weight tiles before the dependency wait.
            const long long pre = min((long long)C::kStages, u1 - u0);
            for (long long it = 0; it < pre; ++it) {
                const long long u = u0 + it;
                const int s = (int)it;
                const int tile = (int)(u / p.KB), kb = (int)(u % p.KB);
                mbar_arrive_expect_tx(&full[s], C::kStageBytes);
                armed |= 1u << s;
                uint8_t *a = sA + s * C::kABytes;
                if (MULTI) {
                    const CUtensorMap *ml = &maps->m[tile / p.tpl];
                    tma_load_2d_hint(a, ml, kb * 64, (tile % p.tpl) * 128, &full[s], pol);
                    tma_load_2d_hint(a + 8192, ml, kb * 64, (tile % p.tpl) * 128 + 64, &full[s], pol);
                } else if (p.paired) {
                    tma_load_2d_hint(a, &tmA, kb * 64, tile * 64, &full[s], pol);
                    tma_load_2d_hint(a + 8192, &tmA2, kb * 64, tile * 64, &full[s], pol);
                } else {
                    tma_load_2d_hint(a, &tmA, kb * 64, tile * 128, &full[s], pol);
                    tma_load_2d_hint(a + 8192, &tmA, kb * 64, tile * 128 + 64, &full[s], pol);
                }
            }
            l2_prefetch_share(p.pf, (unsigned int)cta, (unsigned int)p.grid);
            pdl_wait();
            for (long long it = 0; it < pre; ++it)
                tma_load_2d(sB + (int)it * C::kBBytes, &tmB, (int)((u0 + it) % p.KB) * 64,
                            MULTI ? (int)((u0 + it) / p.KB / p.tpl) * p.brows : 0, &full[(int)it]);
            long long it = pre;
            for (long long u = u0 + pre; u < u1; ++u, ++it) {
                const int s = (int)(it % C::kStages);
                const uint32_t round = (uint32_t)(it / C::kStages);
                if (!mbar_wait_bounded(&empty[s], (round & 1u) ^ 1u, &s_abort)) break;
                const int tile = (int)(u / p.KB), kb = (int)(u % p.KB);
                mbar_arrive_expect_tx(&full[s], C::kStageBytes);
                armed |= 1u << s;
                armed_par = (armed_par & ~(1u << s)) | ((round & 1u) << s);
                uint8_t *a = sA + s * C::kABytes;
                if (MULTI) {
                    const CUtensorMap *ml = &maps->m[tile / p.tpl];
                    tma_load_2d_hint(a, ml, kb * 64, (tile % p.tpl) * 128, &full[s], pol);
                    tma_load_2d_hint(a + 8192, ml, kb * 64, (tile % p.tpl) * 128 + 64, &full[s], pol);
                } else if (p.paired) {
                    tma_load_2d_hint(a, &tmA, kb * 64, tile * 64, &full[s], pol);
                    tma_load_2d_hint(a + 8192, &tmA2, kb * 64, tile * 64, &full[s], pol);
                } else {
                    tma_load_2d_hint(a, &tmA, kb * 64, tile * 128, &full[s], pol);
                    tma_load_2d_hint(a + 8192, &tmA, kb * 64, tile * 128 + 64, &full[s], pol);
                }
                tma_load_2d(sB + s * C::kBBytes, &tmB, kb * 64, MULTI ? (tile / p.tpl) * p.brows : 0, &full[s]);
            }
        } else {
            pdl_wait();
        }
    } else if (warp == 1) {
        pdl_wait();
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, BN);
            long long it = 0, u = u0;
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
                for (; u < seg_end; ++u, ++it) {
                    const int s = (int)(it % C::kStages);
                    const uint32_t round = (uint32_t)(it / C::kStages);
                    if (!mbar_wait_bounded(&full[s], round & 1u, &s_abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sdesc_k_sw128(smem_u32(sA + s * C::kABytes));
                    const uint64_t bd = sdesc_k_sw128(smem_u32(sB + s * C::kBBytes));
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_bf16(d, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), idesc,
                                 (first && k == 0) ? 0u : 1u);
                    first = false;
                    mma_commit(&empty[s]);
                }
                if (!ok) break;
                mma_commit(&tfull[a]);
                ++seg;
            }
            // every MMA this thread issued has completed once "done" flips
            mma_commit(done);
            mbar_drain(done, 0);
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
        constexpr int kPairMax = BN <= 32 ? BN : 1;  // pairwise reduction for BN <= 32
        while (u < u1) {
            const int tile = (int)(u / p.KB);
            const long long tbeg = (long long)tile * p.KB, tend = tbeg + p.KB;
            const long long seg_end = min(u1, tend);
            const bool whole = (u == tbeg) && (seg_end == tend);
            const bool pair_head = p.pair_red && !whole && seg_end == u1 && u1 < tend;  // this CTA reduces
            const bool pair_tail = p.pair_red && !whole && u == u0 && u0 > tbeg;        // CTA c - 1 reduces
            const int a = seg & 1;
            float pv[kPairMax];
            bool got = true;
            if (pair_head && BN <= 32) {
                // CTA c + 1's partial of this tile, read before this CTA's own last MMA completes
                if (et == 0) {
                    const unsigned long long t0 = globaltimer();
                    while (ld_volatile_i32(&p.counters[tile]) == 0) {
                        if (s_abort || globaltimer() - t0 > kWaitLimitNs) {
                            s_abort = 1;
                            break;
                        }
                    }
                    __threadfence();
                }
                named_bar_sync(1, 128);
                const float4 *src = (const float4 *)(p.partials + ((size_t)(2 * (cta + 1)) * 128 + row) * BN);
#pragma unroll
                for (int j = 0; j < kPairMax / 4; ++j) {
                    const float4 t = __ldcg(src + j);
                    pv[4 * j] = t.x;
                    pv[4 * j + 1] = t.y;
                    pv[4 * j + 2] = t.z;
                    pv[4 * j + 3] = t.w;
                }
                got = !s_abort;
            }
            got = got && mbar_wait_bounded(&tfull[a], ((uint32_t)seg >> 1) & 1u, &s_abort);
            if (!named_bar_and(2, 128, got)) break;  // uniform exit keeps the named barriers matched
            tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * BN);
            const int slot = (tile == (int)(u0 / p.KB)) ? 2 * cta : 2 * cta + 1;
            const bool final = whole || (pair_head && BN <= 32);
            // the tile's own matrix (several-matrix launches): its output base and tile index
            GemmParams pl = p;
            const int tl = MULTI ? tile % p.tpl : tile;
            if (MULTI) pl.out_f32 = p.out_f32 + (long long)(tile / p.tpl) * p.lay_stride;
#pragma unroll
            for (int c0 = 0; c0 < BN; c0 += 16) {
                float v[16];
                tmem_ld16(taddr + (uint32_t)c0, v);
                if (pair_head && BN <= 32) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] += pv[(c0 + j) % kPairMax];
                }
                if (p.epi == EPI_PENDING) {
                    gemm_pending_store<BN>(p, slot, row, c0, v);
                } else if (final) {
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
                        const int n = tl * 128 + row;
                        if (n < p.n_out) {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (c0 + j < p.M) gemm_store(pl, n, c0 + j, v[j]);
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
            if (pair_head && BN <= 32) {
                named_bar_sync(1, 128);
                if (et == 0) p.counters[tile] = 0;  // the flag is consumed
            } else if (pair_tail && BN <= 32) {
                __threadfence();
                named_bar_sync(1, 128);
                if (et == 0) st_volatile_i32(&p.counters[tile], 1);
            } else if (!whole && p.epi != EPI_PENDING) {
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
                    if (MULTI) {
                        const int n = tl * 128 + et;
                        if (n < p.n_out) gemm_reduce_impl<BN, false, 4, false>(pl, tile, c_lo, c_hi, et, n);
                    } else {
                        gemm_reduce_tile<BN, false, 4>(p, tile, c_lo, c_hi, et, nch);
                    }
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
            for (int s = 0; s < C::kStages; ++s)
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

// Shared memory keeps one CTA per SM; the launch bound of two caps the
// registers at 170 so that the next (small) kernel's warps fit in the register
// files of the SM sub-partitions beside this CTA's and start early.
template <int BN>
__global__ void __launch_bounds__(192, 2)
    gemm_swapab_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                       const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
    gemm_swapab_body<BN, false>(&tmA, &tmA2, &tmB, p, nullptr);
}

// Several matrices of the same shape against their own activation rows in one
// launch (the layers of the latent-cache append).
template <int BN>
__global__ void __launch_bounds__(192, 2)
    gemm_layers_kernel(const __grid_constant__ CUtensorMap tmB, const GemmParams p, const __grid_constant__ GemmMaps maps) {
    gemm_swapab_body<BN, true>(&tmB, &tmB, &tmB, p, &maps);
}

}  // namespace ds
