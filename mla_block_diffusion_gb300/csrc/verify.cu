// Lossless verification of a drafted block against the target's logits.
//
// Model cards: the target verifies the 7 drafted tokens in one pass and the
// output distribution equals the target's ("kimi-k3-dspark-gguf", intro);
// greedy verification is an argmax match, probabilistic verification samples
// at temperature T with top-p, and "rejection_sample_method": "block" verifies
// the drafted block as a unit ("Kimi-K3-DSpark-NVFP4", Quick Start / Sampling
// options). Block verification follows the published block verification
// method (Sun et al. 2024).
//
// Greedy: the argmax of every target row (lowest id on ties), then the first
// mismatch.
//
// Probabilistic (token by token) and block: every row's exact top-p nucleus
// first. For a row l at temperature T the spec's weights are
// E_v = floor(2^32 exp^(l_v / T - m)) with keys K_v = (E_v << 18) | (2^18-1-v);
// the nucleus is every key >= K*, where K* is the key at which the running
// weight of the keys in descending order first reaches
// tau = max(1, floor(S * P32 / 2^32)), S = sum E. One cluster of 8 CTAs holds
// one row in shared memory and finds K* exactly:
//   1. a histogram of E over 33 x 64 bins (E's binary exponent and the next 6
//      bits: every bin holds a contiguous range of E, so whole bins lie above
//      or below the crossing), merged over the cluster and copied to every
//      CTA through distributed shared memory; its total is S;
//   2. the crossing bin (the suffix weight from the top reaches tau);
//   3. the keys of that bin (a few hundred for flat rows) gathered into one
//      CTA, which ranks them exactly.
// When the crossing bin holds more keys than that CTA takes (ties, flat rows
// of huge vocabularies), refinement levels over 10-bit digits of the key
// narrow it down instead. No grid-wide barrier and no global atomics. Then one
// cluster per sequence makes the accept decisions (one lane per position) and
// the one draw of the step (a weighted pick in id order).
#include "exact_div.cuh"
#include "sampling_spec.cuh"

#include <algorithm>

namespace ds {

// ---------------------------------------------------------------------------
// Distributed shared memory: loads, stores and an atomic add on the same
// shared-memory location of another CTA of the cluster. Stores become visible
// to that CTA after the next cluster barrier both pass.
// ---------------------------------------------------------------------------
DS_DEVINL uint32_t peer_addr(const void *local, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
    return a;
}
DS_DEVINL unsigned long long ld_peer_u64(const void *local, uint32_t rank) {
    unsigned long long v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(peer_addr(local, rank)) : "memory");
    return v;
}
DS_DEVINL uint32_t ld_peer_u32(const void *local, uint32_t rank) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(peer_addr(local, rank)) : "memory");
    return v;
}
DS_DEVINL void st_peer_u64(void *local, uint32_t rank, unsigned long long v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(peer_addr(local, rank)), "l"(v) : "memory");
}
DS_DEVINL void st_peer_u32(void *local, uint32_t rank, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_addr(local, rank)), "r"(v) : "memory");
}
DS_DEVINL uint32_t atom_add_peer_u32(void *local, uint32_t rank, uint32_t v) {
    uint32_t old;
    asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(peer_addr(local, rank)), "r"(v)
                 : "memory");
    return old;
}

// 1D bulk copy global -> shared, completing on an mbarrier (16-byte aligned
// addresses, size a multiple of 16).
DS_DEVINL void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

constexpr int kVCl = 8;          // CTAs per cluster
constexpr int kVThreads = 1024;
constexpr int kVWarps = kVThreads / 32;
constexpr int kSub = 32;         // bins per group
constexpr int kMant0 = 6;        // level 0: binary exponent of E (0..32) x 6 mantissa bits
constexpr int kBins0 = 33 << kMant0;
constexpr int kGroups0 = kBins0 / kSub;
constexpr int kDigitBits = 10;   // refinement levels: 10-bit digits of the key
constexpr int kBinsK = 1 << kDigitBits;
constexpr int kGroupsK = kBinsK / kSub;
constexpr int kHistBins = kBinsK > kBins0 ? kBinsK : kBins0;
constexpr int kMaxGroups = kHistBins / kSub;
constexpr int kCandCap = kVThreads;  // keys of the crossing bin ranked in one CTA
static_assert(kHistBins >= kCandCap, "a CTA lists its crossing-bin keys in the merged-histogram space");
constexpr int kMaxLevels = 8;        // level 0 + at most 5 refinements of the 44-bit residual key
constexpr int kMassSlices = 64;      // CTAs per block-verification row for the residual masses (2 per lane of a warp)
constexpr size_t kStageMax = 200 * 1024;  // largest staging of the draw rows in shared memory
constexpr int kStatWords = 4;
constexpr int kNucBatch = 5;         // float4 loads in flight per thread in the row pass

// Part [lo, hi) of cluster rank c over ids [r0, r1): whole quads from r0, the
// last CTA to r1.
DS_DEVINL void cl_part(int r0, int r1, int c, int &lo, int &hi) {
    const int nq = (r1 - r0) / 4;
    lo = r0 + 4 * (int)((long long)c * nq / kVCl);
    hi = c == kVCl - 1 ? r1 : r0 + 4 * (int)((long long)(c + 1) * nq / kVCl);
}
__host__ __device__ inline int max_part(int V) { return 4 * ((V / 4 + kVCl - 1) / kVCl) + 4; }

// Level-0 bin of a weight E >= 1: 64 * msb(E) + the 6 bits below the msb.
DS_DEVINL int coarse_bin(unsigned long long E) {
    const int msb = 63 - __clzll((long long)E);
    const unsigned frac = msb >= kMant0 ? (unsigned)(E >> (msb - kMant0)) & 63u : (unsigned)(E << (kMant0 - msb)) & 63u;
    return (msb << kMant0) + (int)frac;
}
// The same from the bits of e (E = weight_bits(e) >= 1): msb(E) = exponent(e) - 95,
// and for msb >= 6 the 6 bits below it are e's top mantissa bits.
DS_DEVINL int coarse_bin_bits(float e) {
    const uint32_t u = __float_as_uint(e);
    const int ex = (int)(u >> 23);
    if (ex >= 95 + kMant0) return ((ex - 95) << kMant0) + (int)((u >> (23 - kMant0)) & 63u);
    return coarse_bin(weight_bits(e));
}
// The smallest E of level-0 bin b and the number of low bits of E that vary inside it.
DS_DEVINL void coarse_range(int b, unsigned long long &lo, int &wbits) {
    const int msb = b >> kMant0, frac = b & 63;
    if (msb >= kMant0) {
        lo = (unsigned long long)(64 + frac) << (msb - kMant0);
        wbits = msb - kMant0;
    } else {
        lo = (unsigned long long)(64 + frac) >> (kMant0 - msb);
        wbits = 0;
    }
}

// First group merged by cluster rank r (groups [gstart(r), gstart(r + 1))).
DS_DEVINL int gstart(int ngroups, int r) { return r * ngroups / kVCl; }

// Shared memory of the nucleus kernel (dynamic): the row part, this CTA's
// histogram of the current level (a bin's weight as two 32-bit sums, of E's
// low 16 bits and of E >> 16: 32-bit shared-memory atomics; a CTA's bin holds
// fewer than 2^15 elements of E <= 2^32), the merged histogram (every CTA holds
// all of it), and the gathered keys of the crossing bin (rank 0).
struct NucLayout {
    size_t row, h2, hc, mw, mc, gtot, cand, total;
    __host__ __device__ explicit NucLayout(int V) {
        size_t o = 0;
        row = o;
        o += (size_t)max_part(V) * 4;
        o = (o + 15) & ~(size_t)15;
        h2 = o;  // per bin {sum of E & 0xFFFF, sum of E >> 16}
        o += (size_t)kHistBins * 8;
        hc = o;
        o += (size_t)kHistBins * 4;
        o = (o + 15) & ~(size_t)15;
        mw = o;
        o += (size_t)kHistBins * 8;
        mc = o;
        o += (size_t)kHistBins * 4;
        o = (o + 15) & ~(size_t)15;
        gtot = o;
        o += (size_t)kMaxGroups * 8;
        cand = o;
        o += (size_t)kCandCap * 8;
        total = o;
    }
};

// Per-row refinement state, identical in every CTA of the row's cluster.
struct NucState {
    float m;                        // max of l / T
    int b0, sh, done, d;
    unsigned long long S, tau, above, lo, pre, Sn, kstar;
    float elo, ehi;                 // the level-0 crossing bin as a range of e = E / 2^32
    // crossing of the last level
    int fbin;
    unsigned fcount;
    unsigned long long fw, fabove;
};

// Warp 0: the crossing of the merged histogram (local copies): the largest bin
// whose suffix weight (itself and every bin above it) reaches `need`. Fills
// st.fbin / fw / fcount / fabove (weight of the bins above it). At level 0
// (need == 0) the row's total S and tau = max(1, floor(S * P32 / 2^32)) come
// from the same group totals first. Lane l holds groups 4l .. 4l + 3. Returns
// false when the whole histogram weighs less than need.
DS_DEVINL bool find_crossing(int ngroups, unsigned long long need, unsigned long long P32,
                             const unsigned long long *gtot, const unsigned long long *mw, const uint32_t *mc,
                             NucState &st) {
    const int lane = threadIdx.x & 31;
    unsigned long long gv[4], tot = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int g = 4 * lane + q;
        gv[q] = g < ngroups ? gtot[g] : 0ull;
        tot += gv[q];
    }
    const unsigned long long suf = warp_suffix_u64(tot);
    if (need == 0) {  // level 0: the row's total weight sets tau
        const unsigned long long S = __shfl_sync(0xffffffffu, suf, 0);
        const unsigned long long tau = (unsigned long long)(((unsigned __int128)S * P32) >> 32);
        need = tau < 1 ? 1 : tau;
        if (lane == 0) {
            st.S = S;
            st.tau = need;
        }
    }
    const unsigned mask = __ballot_sync(0xffffffffu, suf >= need);
    if (!mask) return false;
    const int L = 31 - __clz((int)mask);
    // inside lane L: the highest of its groups whose suffix reaches need
    int g = 0;
    unsigned long long above_g = 0;
    if (lane == L) {
        unsigned long long acc = suf - tot;
        for (int q = 3; q >= 0; --q) {
            if (acc + gv[q] >= need) {
                g = 4 * lane + q;
                break;
            }
            acc += gv[q];
        }
        above_g = acc;
    }
    g = __shfl_sync(0xffffffffu, g, L);
    above_g = __shfl_sync(0xffffffffu, above_g, L);
    const unsigned long long w = mw[g * kSub + lane];
    const uint32_t c = mc[g * kSub + lane];
    const unsigned long long suf2 = warp_suffix_u64(w);
    const unsigned long long need2 = need - above_g;
    const unsigned mask2 = __ballot_sync(0xffffffffu, suf2 >= need2);
    if (!mask2) return false;
    const int j = 31 - __clz((int)mask2);
    const unsigned long long ex = __shfl_sync(0xffffffffu, suf2 - w, j);
    const unsigned long long wj = __shfl_sync(0xffffffffu, w, j);
    const uint32_t cj = __shfl_sync(0xffffffffu, c, j);
    if (lane == 0) {
        st.fbin = g * kSub + j;
        st.fw = wj;
        st.fcount = cj;
        st.fabove = above_g + ex;
    }
    return true;
}

// Row gr of the verification: target rows 0..B of every sequence, then (with a
// sampled draft) its draft rows 0..B-1.
__host__ __device__ inline int ver_rows_per_seq(const VerifyParams &p) { return p.draft_greedy ? p.B + 1 : 2 * p.B + 1; }
DS_DEVINL const float *ver_row(const VerifyParams &p, int gr) {
    const int R = ver_rows_per_seq(p), b = gr / R, j = gr % R;
    if (j <= p.B) return p.P + ((size_t)b * (p.B + 1) + j) * p.V;
    return p.ell + ((size_t)b * p.B + (j - p.B - 1)) * p.V;
}
// The drafted token scored by row gr (-1 for the bonus row).
DS_DEVINL int ver_row_token(const VerifyParams &p, int gr) {
    const int R = ver_rows_per_seq(p), b = gr / R, j = gr % R;
    const int pos = j < p.B ? j : (j == p.B ? -1 : j - p.B - 1);
    return pos < 0 ? -1 : p.tokens[b * p.B + pos];
}

// Per-row statistics, 4 words per row: the ordered max of l / T, K*, S_n (weight
// of the nucleus), and e_t (the nucleus weight of the row's drafted token: E_t if
// its key is in the nucleus, else 0; 0 for the bonus row).
struct RowStats {
    float m;
    unsigned long long kstar, Sn, et;
};
DS_DEVINL RowStats row_stats(const VerifyParams &p, int gr) {
    const unsigned long long *s = p.scratch + kStatWords * (size_t)gr;
    RowStats r;
    r.m = ord2f((uint32_t)s[0]);
    r.kstar = s[1];
    r.Sn = s[2];
    r.et = s[3];
    return r;
}

// Whether element (e, key) lies in the current refinement range: the level-0
// crossing bin (e in [elo, ehi)) and the known top bits of its residual key.
DS_DEVINL bool in_range(float e, unsigned long long key, const NucState &st) {
    if (!(e >= st.elo && e < st.ehi)) return false;
    return ((key - (st.lo << 18)) >> st.sh) == st.pre;
}

// Rank 0: the row's statistics (the drafted token's nucleus weight from its logit).
DS_DEVINL void write_stats(const VerifyParams &p, int gr, int tok, float lt, float T, const NucState &st,
                           unsigned long long kstar) {
    unsigned long long et = 0;
    if (tok >= 0) {
        const unsigned long long E = weight_of(lt, T, st.m);
        et = key_of(E, tok) >= kstar ? E : 0ull;
    }
    unsigned long long *o = p.scratch + kStatWords * (size_t)gr;
    o[0] = f2ord(st.m);
    o[1] = kstar;
    o[2] = st.Sn;
    o[3] = et;
}

// Rank 0 (the whole CTA): K* among the N <= kCandCap gathered keys of the
// level-0 crossing bin, by histogram refinement over 10-bit digits of their
// residual keys (key - (lo << 18), st.sh bits): the crossing digit of each round
// narrows the active keys until one is left. hw / hc are 1024-bin scratch.
DS_DEVINL void cta_select(const unsigned long long *cand, uint32_t N, NucState &st, unsigned long long *hw,
                          uint32_t *hc, unsigned long long *gt) {
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const unsigned long long key = t < (int)N ? cand[t] : 0ull, E = key >> 18;
    const unsigned long long R = key - (st.lo << 18);
    bool active = t < (int)N;
    for (int round = 0; round < 6; ++round) {
        const int sh = st.sh, d = sh < kDigitBits ? sh : kDigitBits;
        hw[t] = 0;
        hc[t] = 0;
        __syncthreads();
        const int digit = (int)((R >> (sh - d)) & ((1ull << d) - 1));
        if (active) {
            atomicAdd(&hw[digit], E);
            atomicAdd(&hc[digit], 1u);
        }
        __syncthreads();
        {
            const unsigned long long gs = warp_sum_u64(hw[t]);
            if (lane == 0) gt[warp] = gs;
        }
        __syncthreads();
        if (warp == 0) {
            const unsigned long long need = st.tau - st.above;
            const unsigned long long tot = gt[lane], suf = warp_suffix_u64(tot);
            const unsigned mask = __ballot_sync(0xffffffffu, suf >= need);
            const int g = mask ? 31 - __clz((int)mask) : 0;
            const unsigned long long above_g = __shfl_sync(0xffffffffu, suf - tot, g);
            const unsigned long long w = hw[g * kSub + lane];
            const uint32_t c = hc[g * kSub + lane];
            const unsigned long long suf2 = warp_suffix_u64(w);
            const unsigned mask2 = __ballot_sync(0xffffffffu, suf2 >= need - above_g);
            const int j = mask2 ? 31 - __clz((int)mask2) : 0;
            const unsigned long long ex = __shfl_sync(0xffffffffu, suf2 - w, j);
            const unsigned long long wj = __shfl_sync(0xffffffffu, w, j);
            const uint32_t cj = __shfl_sync(0xffffffffu, c, j);
            if (lane == 0) {
                if (!mask || !mask2) {
                    st.done = 2;  // unreachable with exact weights
                } else {
                    st.fbin = g * kSub + j;
                    st.fw = wj;
                    st.fcount = cj;
                    st.above += above_g + ex;
                    st.pre = (st.pre << d) | (unsigned long long)st.fbin;
                    st.sh = sh - d;
                    if (cj == 1 || st.sh == 0) {
                        st.Sn = st.above + wj;
                        st.done = 1;
                    }
                }
            }
        }
        __syncthreads();
        active = active && digit == st.fbin;
        if (st.done) {
            if (st.done == 1 && active) st.kstar = key;
            __syncthreads();
            return;
        }
    }
}

// ---------------------------------------------------------------------------
// Exact top-p nucleus of every row: grid (8, rows), clusters of 8 along x.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kVThreads, 1) nucleus_rows_kernel(VerifyParams p) {
    extern __shared__ __align__(16) uint8_t vsm[];
    __shared__ NucState st;
    __shared__ unsigned long long red[33];
    __shared__ unsigned long long s_cmax, s_key;
    __shared__ uint32_t s_cnt, s_lcnt, s_base, s_counts[kVCl];
    __shared__ float s_lt;
    pdl_trigger();
    const NucLayout NL(p.V);
    float *yv = (float *)(vsm + NL.row);
    uint32_t *h2 = (uint32_t *)(vsm + NL.h2), *hc = (uint32_t *)(vsm + NL.hc);
    unsigned long long *mw = (unsigned long long *)(vsm + NL.mw);
    uint32_t *mc = (uint32_t *)(vsm + NL.mc);
    unsigned long long *gtot = (unsigned long long *)(vsm + NL.gtot);
    unsigned long long *cand = (unsigned long long *)(vsm + NL.cand);
    const uint32_t rank = cluster_rank();
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int gr = blockIdx.y;
    int lo, hi;
    cl_part(0, p.V, (int)rank, lo, hi);
    const int n = hi - lo;
    const float T = p.T;
    for (int i = t; i < kHistBins; i += kVThreads) {
        *(uint2 *)(h2 + 2 * i) = make_uint2(0u, 0u);
        hc[i] = 0;
    }
    if (t == 0) s_cnt = 0;
    pdl_wait();
    const float *row = ver_row(p, gr);
    int tok = -1;
    if (rank == 0 && t == 0) {  // the drafted token's logit, read early
        tok = ver_row_token(p, gr);
        if (tok >= p.V || tok < -1) {
            set_error(p.err, DSPARK_ERR_OOB);
            tok = 0;
        }
        s_lt = tok >= 0 ? row[tok] : 0.f;
    }
    // 1. y = l / T into shared memory, this CTA's max (the thread's float4 loads
    // issued kNucBatch at a time, so the part costs one or two HBM round trips)
    const float *rp = row + lo;
    unsigned long long mx = 0;
    bool bad = false;
    for (int j0 = 4 * t; j0 < n; j0 += 4 * kVThreads * kNucBatch) {
        float4 l[kNucBatch];
#pragma unroll
        for (int u = 0; u < kNucBatch; ++u) {
            const int j = j0 + 4 * kVThreads * u;
            l[u] = j < n ? __ldg((const float4 *)(rp + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kNucBatch; ++u) {
            const int j = j0 + 4 * kVThreads * u;
            if (j >= n) break;
            const float y0 = div_T(l[u].x, T), y1 = div_T(l[u].y, T), y2 = div_T(l[u].z, T), y3 = div_T(l[u].w, T);
            if (!isfinite(y0) || !isfinite(y1) || !isfinite(y2) || !isfinite(y3)) bad = true;
            *(float4 *)(yv + j) = make_float4(y0, y1, y2, y3);
            mx = max(mx, (unsigned long long)max(max(f2ord(y0), f2ord(y1)), max(f2ord(y2), f2ord(y3))));
        }
    }
    if (bad) set_error(p.err, DSPARK_ERR_BAD_INPUT);
    mx = block_max_u64(mx, red);
    if (t == 0) s_cmax = mx;
    cluster_sync();
    if (warp == 0) {
        // lane r reads CTA r's maximum
        const unsigned long long m = warp_max_u64(lane < kVCl ? ld_peer_u64(&s_cmax, (uint32_t)lane) : 0ull);
        if (lane == 0) st.m = ord2f((uint32_t)m);
    }
    if (t == 0) {
        st.above = 0;
        st.done = 0;
        st.Sn = 0;
        st.kstar = ~0ull;
        st.b0 = 0;
        st.sh = 0;
        st.lo = 0;
        st.pre = 0;
        st.d = 0;
        st.elo = 0.f;
        st.ehi = 0.f;
    }
    __syncthreads();
    // 2. e = exp^(y - m) in place and the level-0 histogram (its total is S)
    const float m = st.m;
    for (int j = t; j < n; j += kVThreads) {
        const float e = exp_hat(__fsub_rn(yv[j], m));
        yv[j] = e;
        const unsigned long long E = weight_bits(e);
        if (E) {
            const int bin = coarse_bin_bits(e);
            atomicAdd(&h2[2 * bin], (uint32_t)(E & 0xFFFFu));
            atomicAdd(&h2[2 * bin + 1], (uint32_t)(E >> 16));
        }
    }
    const unsigned long long P32 = top_p_q32(p.top_p);
    // 3. merge and copy to every CTA, find the crossing; rank the crossing
    // bin's keys, or refine further when there are too many of them
    for (int level = 0; level < kMaxLevels; ++level) {
        const int ngroups = level ? kGroupsK : kGroups0;
        if (level > 0) {
            const int sh = st.sh, d = st.d;
            for (int j = t; j < n; j += kVThreads) {
                const float e = yv[j];
                if (!(e >= st.elo && e < st.ehi)) continue;
                const unsigned long long E = weight_bits(e);
                const unsigned long long R = key_of(E, lo + j) - (st.lo << 18);
                if ((R >> sh) != st.pre) continue;
                const int bin = (int)((R >> (sh - d)) & ((1ull << d) - 1));
                atomicAdd(&h2[2 * bin], (uint32_t)(E & 0xFFFFu));
                atomicAdd(&h2[2 * bin + 1], (uint32_t)(E >> 16));
                atomicAdd(&hc[bin], 1u);
            }
        }
        cluster_sync();  // A: every CTA's histogram of this level is complete
        {
            const int g0 = gstart(ngroups, (int)rank), g1 = gstart(ngroups, (int)rank + 1);
            if (warp < g1 - g0) {
                const int bin = (g0 + warp) * kSub + lane;
                unsigned long long w = 0;
                uint32_t c = 0;
#pragma unroll
                for (int r = 0; r < kVCl; ++r) {
                    const unsigned long long v = ld_peer_u64(h2 + 2 * bin, (uint32_t)r);
                    w += (v & 0xFFFFFFFFull) + ((v >> 32) << 16);
                    if (level > 0) c += ld_peer_u32(hc + bin, (uint32_t)r);
                }
                const unsigned long long gsum = warp_sum_u64(w);
#pragma unroll
                for (int r = 0; r < kVCl; ++r) {
                    st_peer_u64(mw + bin, (uint32_t)r, w);
                    st_peer_u32(mc + bin, (uint32_t)r, c);
                    if (lane == 0) st_peer_u64(gtot + g0 + warp, (uint32_t)r, gsum);
                }
            }
        }
        cluster_sync();  // B: every CTA holds the merged histogram; peers are done with this one
        for (int i = t; i < kHistBins; i += kVThreads) {
            *(uint2 *)(h2 + 2 * i) = make_uint2(0u, 0u);
            hc[i] = 0;
        }
        if (warp == 0) {
            const bool found = find_crossing(ngroups, level ? st.tau - st.above : 0ull, P32, gtot, mw, mc, st);
            if (lane == 0) {
                if (!found) {  // the weights never reach tau (non-finite input): an empty nucleus
                    set_error(p.err, DSPARK_ERR_BAD_INPUT);
                    st.done = 2;
                } else {
                    st.above += st.fabove;
                    if (level == 0) {
                        st.b0 = st.fbin;
                        int wb;
                        coarse_range(st.b0, st.lo, wb);
                        st.sh = wb + 18;
                        st.pre = 0;
                        // E in [lo, lo + 2^wb) <=> e in [lo, lo + 2^wb) / 2^32 (exact in fp32)
                        st.elo = __uint_as_float(0x2F800000u) * (float)st.lo;  // 2^-32 * lo
                        st.ehi = __uint_as_float(0x2F800000u) * (float)(st.lo + (1ull << wb));
                    } else {
                        st.pre = (st.pre << st.d) | (unsigned long long)st.fbin;
                        st.sh -= st.d;
                    }
                    st.d = st.sh < kDigitBits ? st.sh : kDigitBits;
                    if (level > 0 && (st.fcount == 1 || st.sh == 0)) {
                        st.Sn = st.above + st.fw;
                        st.done = 1;
                    }
                }
            }
        }
        __syncthreads();
        if (st.done) break;
        if (level == 0) {
            // gather the crossing bin's keys into rank 0: list them here (in the
            // merged-histogram space, free until the ranking), reserve a range of
            // rank 0's slots with one atomic, tell every CTA the count, copy the list
            if (t == 0) s_lcnt = 0;
            __syncthreads();
            unsigned long long *lst = mw;
            for (int j = t; j < n; j += kVThreads) {
                const float e = yv[j];
                if (!(e >= st.elo && e < st.ehi)) continue;
                const uint32_t slot = atomicAdd(&s_lcnt, 1u);
                if (slot < (uint32_t)kCandCap) lst[slot] = key_of(weight_bits(e), lo + j);
            }
            __syncthreads();
            if (t == 0) {
                s_base = atom_add_peer_u32(&s_cnt, 0u, s_lcnt);
                for (int r = 0; r < kVCl; ++r) st_peer_u32(&s_counts[rank], (uint32_t)r, s_lcnt);
            }
            __syncthreads();
            {
                const uint32_t nl = min(s_lcnt, (uint32_t)kCandCap);
                for (uint32_t i = t; i < nl; i += kVThreads) {
                    const uint32_t slot = s_base + i;
                    if (slot < (uint32_t)kCandCap) st_peer_u64(cand + slot, 0u, lst[i]);
                }
            }
            cluster_sync();  // G: every key is in rank 0, every count in every CTA
            uint32_t N = 0;
            for (int r = 0; r < kVCl; ++r) N += s_counts[r];
            if (N <= (uint32_t)kCandCap) {
                if (rank == 0) {
                    cta_select(cand, N, st, mw, mc, red);
                    if (t == 0) {
                        if (st.done != 1) set_error(p.err, DSPARK_ERR_BAD_INPUT);
                        write_stats(p, gr, tok, s_lt, T, st, st.done == 1 ? st.kstar : ~0ull);
                    }
                }
                return;
            }
        }
    }
    if (!st.done && t == 0) set_error(p.err, DSPARK_ERR_BAD_INPUT);
    // the one key of the final bin: its CTA stores it in rank 0's shared memory
    if (st.done == 1) {
        for (int j = t; j < n; j += kVThreads) {
            const float e = yv[j];
            if (!(e >= st.elo && e < st.ehi)) continue;
            const unsigned long long key = key_of(weight_bits(e), lo + j);
            if (in_range(e, key, st)) st_peer_u64(&s_key, 0u, key);
        }
    }
    cluster_sync();  // the key is in rank 0; no CTA leaves while a peer may still read its shared memory
    if (rank == 0 && t == 0) write_stats(p, gr, tok, s_lt, T, st, st.done == 1 ? s_key : ~0ull);
}

// ---------------------------------------------------------------------------
// One weighted pick by the CTAs of a cluster over ids [r0, r1): the smallest v
// whose running weight base + sum_{r0 <= u <= v} weight(u) exceeds the target.
// With W24 >= 0 the range is the whole draw (base 0) and the target is
// floor(total * W24 / 2^24) of the range's total; otherwise `target` is given.
// Every warp sums a contiguous segment of the CTA's part (lanes strided, so
// the reads are coalesced), the cluster learns each CTA's total through
// distributed shared memory, and the one warp whose segment holds the target
// walks it lane-contiguously. Writes v to *out (nothing when no weight
// reaches the target).
// ---------------------------------------------------------------------------
struct DrawScan {
    unsigned long long wlo[kVWarps], whi[kVWarps];  // warp totals, then their exclusive prefixes
    unsigned long long tlo, thi;   // this CTA's total
    unsigned long long blo, bhi;   // weight before this CTA (plus base)
    unsigned long long glo, ghi;   // the target
};

DS_DEVINL void u128_split(unsigned __int128 v, unsigned long long &lo, unsigned long long &hi) {
    lo = (unsigned long long)v;
    hi = (unsigned long long)(v >> 64);
}
DS_DEVINL unsigned __int128 u128_join(unsigned long long lo, unsigned long long hi) {
    return ((unsigned __int128)hi << 64) | lo;
}
DS_DEVINL unsigned __int128 shfl_u128(unsigned __int128 v, int src) {
    unsigned long long lo, hi;
    u128_split(v, lo, hi);
    return u128_join(__shfl_sync(0xffffffffu, lo, src), __shfl_sync(0xffffffffu, hi, src));
}
DS_DEVINL unsigned __int128 warp_sum_u128(unsigned __int128 v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        unsigned long long lo, hi;
        u128_split(v, lo, hi);
        v += u128_join(__shfl_xor_sync(0xffffffffu, lo, o), __shfl_xor_sync(0xffffffffu, hi, o));
    }
    return v;
}
// Inclusive prefix over the lanes (lane order).
DS_DEVINL unsigned __int128 warp_incl_u128(unsigned __int128 v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        unsigned long long lo, hi;
        u128_split(v, lo, hi);
        const unsigned __int128 w = u128_join(__shfl_up_sync(0xffffffffu, lo, o), __shfl_up_sync(0xffffffffu, hi, o));
        if (lane >= o) v += w;
    }
    return v;
}

template <class WF>
DS_DEVINL void cluster_pick(WF weight, int r0, int r1, long long W24, unsigned __int128 base, unsigned __int128 target,
                            int32_t *out, DrawScan &ds_) {
    const uint32_t rank = cluster_rank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int lo, hi;
    cl_part(r0, r1, (int)rank, lo, hi);
    const int n = hi - lo;
    const int segw = 32 * ((n + 32 * kVWarps - 1) / (32 * kVWarps));
    const int s0 = lo + warp * segw, s1 = min(hi, s0 + segw);
    unsigned __int128 mine = 0;
    for (int v = s0 + lane; v < s1; v += 32) mine += weight(v);
    mine = warp_sum_u128(mine);
    if (lane == 0) u128_split(mine, ds_.wlo[warp], ds_.whi[warp]);
    __syncthreads();
    static_assert(kVWarps == 32, "one warp total per lane");
    if (warp == 0) {  // the warps' exclusive prefixes and the CTA's total
        const unsigned __int128 x = u128_join(ds_.wlo[lane], ds_.whi[lane]);
        const unsigned __int128 inc = warp_incl_u128(x);
        u128_split(inc - x, ds_.wlo[lane], ds_.whi[lane]);
        if (lane == 31) u128_split(inc, ds_.tlo, ds_.thi);
    }
    cluster_sync();  // every CTA's total is in its shared memory
    if (warp == 0) {  // lane r reads CTA r's total
        const unsigned __int128 x =
            lane < kVCl ? u128_join(ld_peer_u64(&ds_.tlo, (uint32_t)lane), ld_peer_u64(&ds_.thi, (uint32_t)lane))
                        : (unsigned __int128)0;
        const unsigned __int128 inc = warp_incl_u128(x);
        const unsigned __int128 before = shfl_u128(inc - x, (int)rank), total = shfl_u128(inc, 31);
        if (lane == 0) {
            const unsigned __int128 tg = W24 >= 0 ? (total * (unsigned __int128)(W24 & 0xFFFFFF)) >> 24 : target;
            u128_split(base + before, ds_.blo, ds_.bhi);
            u128_split(tg, ds_.glo, ds_.ghi);
        }
    }
    cluster_sync();  // peers have read this CTA's total
    const unsigned __int128 tg = u128_join(ds_.glo, ds_.ghi);
    const unsigned __int128 start = u128_join(ds_.blo, ds_.bhi) + u128_join(ds_.wlo[warp], ds_.whi[warp]);
    if (s0 < s1 && start <= tg && tg < start + mine) {
        // this warp's segment holds the target: lanes take contiguous runs
        const int per = (s1 - s0 + 31) / 32;
        const int v0 = s0 + lane * per, v1 = min(s1, v0 + per);
        unsigned __int128 run = 0;
        for (int v = v0; v < v1; ++v) run += weight(v);
        const unsigned __int128 incl = warp_incl_u128(run);
        const unsigned __int128 st0 = start + incl - run;
        if (v0 < v1 && st0 <= tg && tg < st0 + run) {
            unsigned __int128 cum = st0;
            for (int v = v0; v < v1; ++v) {
                cum += weight(v);
                if (cum > tg) {
                    *out = v;
                    break;
                }
            }
        }
    }
}

// A draw over a whole vocabulary of V ids.
template <class WF>
DS_DEVINL void cluster_draw(WF weight, int V, uint32_t W24, int32_t *out, DrawScan &ds_) {
    cluster_pick(weight, 0, V, (long long)(W24 & 0xFFFFFFu), 0, 0, out, ds_);
}

// Stage this CTA's part of up to two rows (cl_part of [0, V)) into shared
// memory with bulk copies; returns false if the copies did not land in time.
DS_DEVINL bool stage_rows(float *dst0, const float *row0, float *dst1, const float *row1, int V, uint64_t *bar,
                          volatile int *s_fail) {
    int lo, hi;
    cl_part(0, V, (int)cluster_rank(), lo, hi);
    const uint32_t bytes = (uint32_t)(hi - lo) * 4u;
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar, bytes * (row1 ? 2u : 1u));
        constexpr uint32_t kPiece = 32768;
        for (uint32_t o = 0; o < bytes; o += kPiece) {
            const uint32_t b = bytes - o < kPiece ? bytes - o : kPiece;
            bulk_g2s((uint8_t *)dst0 + o, (const uint8_t *)(row0 + lo) + o, b, bar);
            if (row1) bulk_g2s((uint8_t *)dst1 + o, (const uint8_t *)(row1 + lo) + o, b, bar);
        }
    }
    __syncthreads();
    bool ok = mbar_wait_bounded(bar, 0, s_fail);
    __syncthreads();
    ok = ok && !*s_fail;
    if (!ok && threadIdx.x == 0) mbar_drain(bar, 0);  // copies in flight land before the buffer is abandoned
    __syncthreads();
    return ok;
}

// ---------------------------------------------------------------------------
// Token-by-token probabilistic verification. Accept t_i iff
// U * Eq_t * Sp < 2^32 * Ep_t * Sq (U 32-bit, purpose 2); on the first reject
// draw from max(0, Ep_v Sq - Eq_v Sp) (purpose 3), after 7 accepts draw the
// bonus from the last target row (purpose 4). With a greedy draft q is one-hot
// on the drafted token (Eq = Sq = 1). The accept test of every position uses
// only its rows' statistics, so the B tests run at once (one lane each) and
// the first failing one ends the run. The draw: kDrawSlices CTAs per sequence
// sum the weights of their vocabulary slices (every SM takes part), then one
// CTA per sequence picks inside the slice that holds the target.
// ---------------------------------------------------------------------------
constexpr int kDrawSlices = 128;
constexpr int kDrawThreads = 1024;  // a run of one or two ids per thread at V = 163,840

// The draw's weight of id v after `a` accepts: the bonus row's nucleus weight
// (a == B) or the residual max(0, Ep_v Sq - Eq_v Sp) at position a.
struct TokenDraw {
    const float *prow, *qrow;
    float T, mp, mq;
    unsigned long long ksp, Sp, ksq, Sq;
    int bonus, dg, t;
    // from id v's target logit lp and draft logit lq (lq unused for the bonus
    // row and a greedy draft)
    DS_DEVINL unsigned __int128 of(float lp, float lq, int v) const {
        const unsigned long long Ep = weight_of(lp, T, mp);
        const unsigned long long ep = key_of(Ep, v) >= ksp ? Ep : 0ull;
        if (bonus) return ep;
        unsigned long long eq;
        if (dg) {
            eq = (v == t) ? 1ull : 0ull;
        } else {
            const unsigned long long Eq = weight_of(lq, T, mq);
            eq = key_of(Eq, v) >= ksq ? Eq : 0ull;
        }
        const unsigned __int128 x = (unsigned __int128)ep * Sq, y = (unsigned __int128)eq * Sp;
        return x > y ? x - y : (unsigned __int128)0;
    }
};

// The weights of the contiguous run of ids [v0, v1), their logits loaded eight
// ids at a time (a run costs one L2 round trip per eight ids, not one per id).
// With `out`, stops at the first id whose running total (from `base`) exceeds
// `target` and writes it there.
constexpr int kRunBatch = 8;
DS_DEVINL unsigned __int128 run_weights(const TokenDraw &d, int v0, int v1, unsigned __int128 base,
                                        unsigned __int128 target, int32_t *out) {
    unsigned __int128 cum = base;
    const bool q = !d.bonus && !d.dg;
    for (int g = v0; g < v1; g += kRunBatch) {
        float lp[kRunBatch], lq[kRunBatch];
#pragma unroll
        for (int j = 0; j < kRunBatch; ++j) {
            lp[j] = g + j < v1 ? __ldg(d.prow + g + j) : 0.f;
            lq[j] = (q && g + j < v1) ? __ldg(d.qrow + g + j) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < kRunBatch; ++j) {
            if (g + j >= v1) break;
            cum += d.of(lp[j], lq[j], g + j);
            if (out && cum > target) {
                *out = g + j;
                return cum;
            }
        }
    }
    return cum;
}

// Slice x of kDrawSlices over [0, V).
DS_DEVINL void draw_slice(int V, int x, int &lo, int &hi) {
    lo = (int)((long long)V * x / kDrawSlices);
    hi = (int)((long long)V * (x + 1) / kDrawSlices);
}
// Partial sums of the draws: [b][slice] * 2 words, after the row statistics and the block masses.
DS_DEVINL unsigned long long *draw_parts(const VerifyParams &p) {
    return p.scratch + kStatWords * (size_t)p.bs * (2 * p.B + 1) + (size_t)p.bs * p.B * kMassSlices * 2;
}

// grid (kDrawSlices, bs): every CTA sums the draw weights of its slice; the
// last CTA of a sequence to finish (a counter in the workspace, returned to
// zero by that CTA) makes the decisions, writes the outputs, finds the slice
// that holds the draw's target floor(total * W24 / 2^24) and picks inside it.
// No CTA waits for another.
__global__ void __launch_bounds__(kDrawThreads, 1) verify_token_draw_kernel(VerifyParams p) {
    __shared__ DrawScan dsm;
    __shared__ TokenDraw s_d;
    __shared__ int s_a, s_last, s_slice;
    __shared__ uint32_t s_W;
    __shared__ unsigned long long s_blo, s_bhi, s_tlo, s_thi;
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.y, B = p.B, V = p.V, R = ver_rows_per_seq(p);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Warp 0, lane j = position j: the accept test of every position and the
    // draw's parameters in one round of loads (target row j's statistics for
    // j <= B, the draft row's for j < B); the first reject (or B) picks the lane
    // whose statistics the draw takes.
    int tj = 0, a = 0;
    if (warp == 0) {
        RowStats sp{}, sq{};
        int raw = 0;
        if (lane <= B) sp = row_stats(p, b * R + lane);
        if (lane < B) {
            raw = p.tokens[b * B + lane];
            tj = raw;
            if (raw < 0 || raw >= V) {
                set_error(p.err, DSPARK_ERR_OOB);
                tj = 0;
            }
            if (!p.draft_greedy) sq = row_stats(p, b * R + B + 1 + lane);
        }
        bool acc = false;
        if (lane < B) {
            const unsigned long long eq = p.draft_greedy ? 1ull : sq.et, Sq = p.draft_greedy ? 1ull : sq.Sn;
            const uint32_t U = philox_word(p.seed, (uint32_t)b, p.step, (uint32_t)lane, 2u);
            const unsigned __int128 lhs = (unsigned __int128)U * eq * sp.Sn;
            const unsigned __int128 rhs = ((unsigned __int128)sp.et << 32) * Sq;
            acc = lhs < rhs;
        }
        const unsigned rej = __ballot_sync(0xffffffffu, lane < B && !acc);
        a = rej ? __ffs((int)rej) - 1 : B;
        if (lane == a) {
            TokenDraw d;
            d.bonus = a == B;
            d.dg = p.draft_greedy;
            d.T = p.T;
            d.prow = p.P + ((size_t)b * (B + 1) + a) * V;
            d.mp = sp.m;
            d.ksp = sp.kstar;
            d.Sp = sp.Sn;
            d.qrow = p.ell + ((size_t)b * B + (d.bonus ? 0 : a)) * V;
            d.t = d.bonus ? 0 : min(max(raw, 0), V - 1);
            const bool q = !d.bonus && !d.dg;
            d.mq = q ? sq.m : 0.f;
            d.ksq = q ? sq.kstar : 0ull;
            d.Sq = q ? sq.Sn : 1ull;
            s_d = d;
            s_a = a;
            // the draw's uniform, needed only by the last CTA: formed here, off its path
            s_W = philox_word(p.seed, (uint32_t)b, p.step, (uint32_t)a, a == B ? 4u : 3u) >> 8;
        }
    }
    __syncthreads();
    const TokenDraw d = s_d;
    a = s_a;
    // this CTA's slice of the vocabulary as one contiguous run per thread
    int lo, hi;
    draw_slice(V, blockIdx.x, lo, hi);
    const int per = (hi - lo + (int)blockDim.x - 1) / (int)blockDim.x;
    int v0 = min(hi, lo + (int)threadIdx.x * per), v1 = min(hi, v0 + per);
    unsigned __int128 run = run_weights(d, v0, v1, 0, 0, nullptr);
    {
        const unsigned __int128 ws = warp_sum_u128(run);
        if (lane == 0) u128_split(ws, dsm.wlo[warp], dsm.whi[warp]);
    }
    __syncthreads();
    unsigned long long *parts = draw_parts(p) + (size_t)b * kDrawSlices * 2;
    if (warp == 0) {  // the CTA's total from the warp totals, then the count
        const int nw = (int)(blockDim.x >> 5);
        const unsigned __int128 tot =
            warp_sum_u128(lane < nw ? u128_join(dsm.wlo[lane], dsm.whi[lane]) : (unsigned __int128)0);
        if (lane == 0) {
            parts[2 * blockIdx.x] = (unsigned long long)tot;
            parts[2 * blockIdx.x + 1] = (unsigned long long)(tot >> 64);
            __threadfence();
            const unsigned old = atomicAdd(p.draw_count + b, 1u);
            s_last = old == (unsigned)(kDrawSlices - 1);
        }
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (warp == 0) {
        if (lane == 0) p.draw_count[b] = 0u;
        // the outputs
        if (lane < a) p.out_tokens[b * (B + 1) + lane] = tj;
        if (lane > a && lane <= B) p.out_tokens[b * (B + 1) + lane] = -1;
        if (lane == 0) p.accept_len[b] = a;
        // the target and its slice: lane l holds slices 4l .. 4l + 3
        static_assert(kDrawSlices == 128, "four slices per lane");
        unsigned __int128 x[4], sum = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int c = 4 * lane + k;
            x[k] = u128_join(ldcg_u64(parts + 2 * c), ldcg_u64(parts + 2 * c + 1));
            sum += x[k];
        }
        const unsigned __int128 incl = warp_incl_u128(sum);
        const unsigned __int128 total = shfl_u128(incl, 31);
        const unsigned __int128 tg = (total * (unsigned __int128)(s_W & 0xFFFFFFu)) >> 24;
        unsigned __int128 ex = incl - sum;
        int cand = -1;
        unsigned __int128 before = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (cand < 0 && x[k] > 0 && ex <= tg && tg < ex + x[k]) {
                cand = 4 * lane + k;
                before = ex;
            }
            ex += x[k];
        }
        const unsigned hit = __ballot_sync(0xffffffffu, cand >= 0);
        const int src = hit ? __ffs((int)hit) - 1 : 0;
        const int c = __shfl_sync(0xffffffffu, cand, src);
        const unsigned __int128 bf = shfl_u128(before, src);
        if (lane == 0) {
            s_slice = hit ? c : -1;  // no slice when the total weight is zero
            u128_split(bf, s_blo, s_bhi);
            u128_split(tg, s_tlo, s_thi);
        }
    }
    __syncthreads();
    if (s_slice < 0) return;
    const unsigned __int128 tg = u128_join(s_tlo, s_thi);
    // the target's slice again as runs: the thread whose run holds the target walks it
    draw_slice(V, s_slice, lo, hi);
    const int per2 = (hi - lo + (int)blockDim.x - 1) / (int)blockDim.x;
    v0 = min(hi, lo + (int)threadIdx.x * per2);
    v1 = min(hi, v0 + per2);
    run = run_weights(d, v0, v1, 0, 0, nullptr);
    const unsigned __int128 rinc = warp_incl_u128(run);
    if (lane == 31) u128_split(rinc, dsm.wlo[warp], dsm.whi[warp]);
    __syncthreads();
    // every warp forms its own exclusive prefix from the warp totals
    const int nw = (int)(blockDim.x >> 5);
    const unsigned __int128 wt = lane < nw ? u128_join(dsm.wlo[lane], dsm.whi[lane]) : (unsigned __int128)0;
    const unsigned __int128 winc = warp_incl_u128(wt);
    const unsigned __int128 wex = shfl_u128(winc - wt, warp);
    const unsigned __int128 start = u128_join(s_blo, s_bhi) + wex + rinc - run;
    if (v0 < v1 && run > 0 && start <= tg && tg < start + run)
        run_weights(d, v0, v1, start, tg, p.out_tokens + b * (B + 1) + a);
}

// ---------------------------------------------------------------------------
// Block verification (rejection_sample_method "block"; the published block
// verification method). Probabilities are the spec's in-nucleus rationals
// rounded once to double; every residual-mass term is a double (multiply,
// then subtract) truncated to a multiple of 2^-80, and the masses are exact
// 128-bit sums, so the decisions do not depend on the order of summation.
// ---------------------------------------------------------------------------
DS_DEVINL unsigned __int128 fx80(double x) {
    if (!(x > 0.0)) return 0;
    const unsigned long long bits = (unsigned long long)__double_as_longlong(x);
    const int e = (int)((bits >> 52) & 0x7FF);
    if (e == 0) return 0;
    const unsigned long long mnt = (bits & ((1ull << 52) - 1)) | (1ull << 52);
    const int sh = e - 995;  // x * 2^80 = mnt * 2^(e - 1075 + 80)
    if (sh >= 0) return (unsigned __int128)mnt << sh;
    if (sh <= -53) return 0;
    return (unsigned __int128)(mnt >> (-sh));
}

DS_DEVINL double fx80_to_double(unsigned __int128 s) {
    if (s == 0) return 0.0;
    const unsigned long long hi = (unsigned long long)(s >> 64), lo = (unsigned long long)s;
    const int n = hi ? 128 - __clzll((long long)hi) : 64 - __clzll((long long)lo);
    if (n <= 53) return ldexp((double)lo, -80);
    return ldexp((double)(unsigned long long)(s >> (n - 53)), n - 53 - 80);
}

// One row of the spec as in-nucleus probabilities (one-hot for a greedy draft):
// the rational e / S rounded once to double (exact_div: the IEEE quotient in
// integer arithmetic).
struct BlockRow {
    const float *row;
    float m;
    unsigned long long kstar, S;
    ExactDivisor div;
    int onehot;  // -1: a spec row; else the one token of a greedy draft
    DS_DEVINL double prob(int v, float T) const { return onehot >= 0 ? (v == onehot ? 1.0 : 0.0) : prob_l(row[v], v, T); }
    // from id v's logit l, already loaded
    DS_DEVINL double prob_l(float l, int v, float T) const {
        if (onehot >= 0) return v == onehot ? 1.0 : 0.0;
        const unsigned long long E = weight_of(l, T, m);
        const unsigned long long e = key_of(E, v) >= kstar ? E : 0ull;
        return e ? exact_div(e, div) : 0.0;
    }
};

// fx80(RN(RN(pi p(v)) - q(v))); the double operations that cannot change the
// value are skipped (p = 0 gives no term, pi = 1 and q = 0 are exact).
DS_DEVINL unsigned __int128 block_term(const BlockRow &rp, const BlockRow &rq, double pi, float T, int v) {
    const double a = rp.prob(v, T);
    if (a == 0.0) return 0;
    const double x = pi == 1.0 ? a : __dmul_rn(pi, a);
    const double c = rq.prob(v, T);
    return fx80(c == 0.0 ? x : __dsub_rn(x, c));
}
// The same from the logits of id v in the two rows, already loaded.
DS_DEVINL unsigned __int128 block_term_l(const BlockRow &rp, const BlockRow &rq, double pi, float T, int v, float lp,
                                         float lq) {
    const double a = rp.prob_l(lp, v, T);
    if (a == 0.0) return 0;
    const double x = pi == 1.0 ? a : __dmul_rn(pi, a);
    const double c = rq.prob_l(lq, v, T);
    return fx80(c == 0.0 ? x : __dsub_rn(x, c));
}

DS_DEVINL int block_token(const VerifyParams &p, int b, int i) {
    const int t = p.tokens[b * p.B + i];
    return (t < 0 || t >= p.V) ? 0 : t;
}
DS_DEVINL BlockRow block_rowp(const VerifyParams &p, int b, int i) {
    BlockRow r;
    r.row = p.P + ((size_t)b * (p.B + 1) + i) * p.V;
    const RowStats s = row_stats(p, b * ver_rows_per_seq(p) + i);
    r.m = s.m;
    r.kstar = s.kstar;
    r.S = s.Sn;
    r.div = exact_divisor(s.Sn ? s.Sn : 1ull);
    r.onehot = -1;
    return r;
}
DS_DEVINL BlockRow block_rowq(const VerifyParams &p, int b, int i) {
    BlockRow r;
    if (p.draft_greedy) {
        r.row = nullptr;
        r.m = 0.f;
        r.kstar = r.S = 0;
        r.div = exact_divisor(1ull);
        r.onehot = block_token(p, b, i);
        return r;
    }
    r.row = p.ell + ((size_t)b * p.B + i) * p.V;
    const RowStats s = row_stats(p, b * ver_rows_per_seq(p) + p.B + 1 + i);
    r.m = s.m;
    r.kstar = s.kstar;
    r.S = s.Sn;
    r.div = exact_divisor(s.Sn ? s.Sn : 1ull);
    r.onehot = -1;
    return r;
}
constexpr int kMaxBlockRows = 17;  // block <= 16, plus the bonus row
constexpr int kMassBatch = 5;      // pairs of ids whose logits a thread loads at once
constexpr int kMassThreads = 512;

// Warp 0: pi_0..pi_B of sequence b into pis[] (pi_0 = 1,
// pi_k = min(pi_{k-1} p_{k-1}(t_k) / q_{k-1}(t_k), 1)); the per-position ratios
// come from the rows' statistics (one lane each), the chain from lane 0.
DS_DEVINL void block_pis(const VerifyParams &p, int b, double *pis) {
    const int lane = threadIdx.x & 31, B = p.B, R = ver_rows_per_seq(p);
    double a = 0.0, c = 1.0, ratio = 0.0;
    if (lane < B) {
        const RowStats sp = row_stats(p, b * R + lane);
        a = sp.et ? __ddiv_rn((double)sp.et, (double)sp.Sn) : 0.0;
        if (!p.draft_greedy) {
            const RowStats sq = row_stats(p, b * R + B + 1 + lane);
            c = sq.et ? __ddiv_rn((double)sq.et, (double)sq.Sn) : 0.0;
        }
        // p_k(t_k) / q_k(t_k) does not depend on the chain: every lane divides at once
        if (c != 0.0) ratio = __ddiv_rn(a, c);
    }
    double pi = 1.0;
    if (lane == 0) pis[0] = 1.0;
    for (int k = 1; k <= B; ++k) {
        const double ak = __shfl_sync(0xffffffffu, a, k - 1), ck = __shfl_sync(0xffffffffu, c, k - 1);
        const double rk = __shfl_sync(0xffffffffu, ratio, k - 1);
        if (ck == 0.0) {
            pi = (ak > 0.0 && pi > 0.0) ? 1.0 : 0.0;
        } else {
            const double x = __dmul_rn(pi, rk);
            pi = x < 1.0 ? x : 1.0;
        }
        if (lane == 0) pis[k] = pi;
    }
}
// Partial residual masses: [(b * B + i) * kMassSlices + slice] * 2 words, after the row statistics.
DS_DEVINL unsigned long long *block_masses(const VerifyParams &p) {
    return p.scratch + kStatWords * (size_t)p.bs * ver_rows_per_seq(p);
}
// pi_0..pi_B of every sequence as double bits ([b * kMaxBlockRows + k]), after the draw's slice totals.
DS_DEVINL unsigned long long *block_pi_words(const VerifyParams &p) {
    return p.scratch + kStatWords * (size_t)p.bs * (2 * p.B + 1) + (size_t)p.bs * p.B * kMassSlices * 2 +
           (size_t)p.bs * kDrawSlices * 2;
}

// Residual masses S_i = sum_x max(pi_i p_i(x) - q_i(x), 0) for i < B: grid
// (kMassSlices, bs * B), one vocabulary slice per CTA.
__global__ void __launch_bounds__(kMassThreads) verify_block_mass_kernel(VerifyParams p) {
    __shared__ double s_pis[kMaxBlockRows];
    __shared__ unsigned long long rlo[kMassThreads / 32], rhi[kMassThreads / 32];
    __shared__ BlockRow s_rows[2];
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.y / p.B, i = blockIdx.y % p.B;
    if (threadIdx.x < 32) {
        if (blockIdx.x == 0 && i == 0 && threadIdx.x < p.B) {
            const int t0 = p.tokens[b * p.B + threadIdx.x];
            if (t0 < 0 || t0 >= p.V) set_error(p.err, DSPARK_ERR_OOB);
        }
        block_pis(p, b, s_pis);
        __syncwarp();
        // one CTA per sequence keeps the chain for the decisions
        if (blockIdx.x == 0 && i == 0 && (int)threadIdx.x <= p.B)
            block_pi_words(p)[(size_t)b * kMaxBlockRows + threadIdx.x] =
                (unsigned long long)__double_as_longlong(s_pis[threadIdx.x]);
    } else if (threadIdx.x == 32) {  // the rows' divisors, beside the pi chain
        s_rows[0] = block_rowp(p, b, i);
    } else if (threadIdx.x == 64) {
        s_rows[1] = block_rowq(p, b, i);
    }
    __syncthreads();
    const double pi = s_pis[i];
    const BlockRow rp = s_rows[0], rq = s_rows[1];
    const int np = p.V / 2;
    const int lo = (int)((long long)blockIdx.x * np / gridDim.x), hi = (int)((long long)(blockIdx.x + 1) * np / gridDim.x);
    // the thread's pairs of ids, their logits loaded kMassBatch pairs at a time
    unsigned __int128 acc = 0;
    const bool lq_ = rq.onehot < 0;
    for (int p0 = lo + (int)threadIdx.x; p0 < hi; p0 += (int)blockDim.x * kMassBatch) {
        float lp[2 * kMassBatch], lq[2 * kMassBatch];
#pragma unroll
        for (int u = 0; u < kMassBatch; ++u) {
            const int pp = p0 + (int)blockDim.x * u;
            const bool in = pp < hi;
            lp[2 * u] = in ? __ldg(rp.row + 2 * pp) : 0.f;
            lp[2 * u + 1] = in ? __ldg(rp.row + 2 * pp + 1) : 0.f;
            lq[2 * u] = (in && lq_) ? __ldg(rq.row + 2 * pp) : 0.f;
            lq[2 * u + 1] = (in && lq_) ? __ldg(rq.row + 2 * pp + 1) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kMassBatch; ++u) {
            const int pp = p0 + (int)blockDim.x * u;
            if (pp >= hi) break;
            acc += block_term_l(rp, rq, pi, p.T, 2 * pp, lp[2 * u], lq[2 * u]) +
                   block_term_l(rp, rq, pi, p.T, 2 * pp + 1, lp[2 * u + 1], lq[2 * u + 1]);
        }
    }
    acc = warp_sum_u128(acc);
    if ((threadIdx.x & 31) == 0) u128_split(acc, rlo[threadIdx.x >> 5], rhi[threadIdx.x >> 5]);
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned __int128 tot = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += u128_join(rlo[w], rhi[w]);
        unsigned long long *dst = block_masses(p) + ((size_t)blockIdx.y * gridDim.x + blockIdx.x) * 2;
        dst[0] = (unsigned long long)tot;
        dst[1] = (unsigned long long)(tot >> 64);
    }
}

// Decisions and the one draw of block verification: grid (8, bs), clusters of 8.
// eta_i = (U_i < h_i 2^32) with h_i = S_i / (S_i + 1 - pi_i) (i < B), h_B = pi_B;
// tau = the last accepted position; then a draw from max(pi_tau p_tau - q_tau, 0)
// (purpose 3), from target row tau when that residual is empty, or the bonus
// (purpose 4) when tau = B. The residual draw's total and its slice totals are
// the masses of position tau, so only the slice that holds the target is walked.
__global__ void __launch_bounds__(kVThreads, 1) verify_block_final_kernel(VerifyParams p) {
    extern __shared__ __align__(16) float tsm[];  // the staged target row (when p.stage)
    __shared__ DrawScan dsm;
    __shared__ double s_pis[kMaxBlockRows];
    __shared__ int s_tau, s_plain, s_slice;
    __shared__ unsigned long long s_rlo, s_rhi, s_tlo, s_thi;
    __shared__ unsigned long long s_mlo[kMaxBlockRows], s_mhi[kMaxBlockRows];
    __shared__ BlockRow s_rp[kMaxBlockRows], s_rq[kMaxBlockRows];
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ volatile int s_fail;
    pdl_trigger();
    if (threadIdx.x == 0) s_fail = 0;
    pdl_wait();
    const int b = blockIdx.y, B = p.B, V = p.V;
    const uint32_t rank = cluster_rank();
    const unsigned long long *ms = block_masses(p);
    {
        // warp 1 + i: the mass S_i of position i < B from its 64 slice partials
        // (two per lane, one round of loads), beside warp 0's pi chain
        const int w = (int)(threadIdx.x >> 5) - 1, lane = threadIdx.x & 31;
        static_assert(kMassSlices == 64, "two slices per lane");
        if (w >= 0 && w < B) {
            const unsigned long long *src = ms + ((size_t)(b * B + w) * kMassSlices) * 2;
            const unsigned __int128 x = u128_join(src[4 * lane], src[4 * lane + 1]) +
                                        u128_join(src[4 * lane + 2], src[4 * lane + 3]);
            const unsigned __int128 S = warp_sum_u128(x);
            if (lane == 0) u128_split(S, s_mlo[w], s_mhi[w]);
        }
        // warps B + 1 .. 31 (lane 0): the target rows 0..B and the draft rows
        // 0..B-1 with their divisors, whichever position the decisions pick
        if (w >= B && lane == 0) {
            for (int j = w - B; j < 2 * B + 1; j += 31 - B) {
                if (j <= B)
                    s_rp[j] = block_rowp(p, b, j);
                else
                    s_rq[j - B - 1] = block_rowq(p, b, j - B - 1);
            }
        }
    }
    // the pi chain as the residual-mass kernel formed it
    if ((int)threadIdx.x <= B)
        s_pis[threadIdx.x] = __longlong_as_double((long long)block_pi_words(p)[(size_t)b * kMaxBlockRows + threadIdx.x]);
    __syncthreads();
    if (threadIdx.x < 32) {
        // the decisions (one lane each)
        const int i = threadIdx.x;
        const unsigned __int128 Si = i < B ? u128_join(s_mlo[i], s_mhi[i]) : (unsigned __int128)0;
        bool eta = false;
        if (i >= 1 && i <= B) {
            const double pi_i = s_pis[i];
            double h;
            if (i < B) {
                const double S = fx80_to_double(Si);
                const double den = __dadd_rn(S, __dsub_rn(1.0, pi_i));
                h = den > 0.0 ? __ddiv_rn(S, den) : 0.0;
            } else {
                h = pi_i;
            }
            const uint32_t U = philox_word(p.seed, (uint32_t)b, p.step, (uint32_t)(i - 1), 2u);
            eta = (double)U < __dmul_rn(h, 4294967296.0);
        }
        const unsigned acc = __ballot_sync(0xffffffffu, eta);
        const int tau = acc ? 31 - __clz((int)acc) : 0;  // the last accepted position
        const unsigned __int128 St = shfl_u128(Si, tau);
        const bool plain = (tau == B || St == 0);
        if (i == 0) {
            s_tau = tau;
            s_plain = plain ? 1 : 0;
        }
        if (!plain) {  // warp-uniform
            // the residual draw's target and the mass slice that holds it: lane l
            // holds slices 2l and 2l + 1; an inclusive scan of the lane totals
            // finds the first slice whose running mass exceeds the target
            const uint32_t W = philox_word(p.seed, (uint32_t)b, p.step, (uint32_t)tau, 3u) >> 8;
            const unsigned __int128 tg = (St * (unsigned __int128)(W & 0xFFFFFFu)) >> 24;
            const unsigned long long *src = ms + ((size_t)(b * B + tau) * kMassSlices) * 2;
            const unsigned __int128 x0 = u128_join(src[4 * i], src[4 * i + 1]);
            const unsigned __int128 x1 = u128_join(src[4 * i + 2], src[4 * i + 3]);
            unsigned __int128 incl = x0 + x1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                unsigned long long lo, hi;
                u128_split(incl, lo, hi);
                const unsigned __int128 up = u128_join(__shfl_up_sync(0xffffffffu, lo, o), __shfl_up_sync(0xffffffffu, hi, o));
                if (i >= o) incl += up;
            }
            const unsigned __int128 ex = incl - x0 - x1;
            int cand = -1;
            unsigned __int128 before = 0;
            if (ex + x0 > tg) {
                cand = 2 * i;
                before = ex;
            } else if (ex + x0 + x1 > tg) {
                cand = 2 * i + 1;
                before = ex + x0;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, cand >= 0);
            // the target lies below the total, so a slice holds it; the last slice otherwise
            const int src_lane = hit ? __ffs((int)hit) - 1 : 31;
            if (!hit && i == 31) {
                cand = kMassSlices - 1;
                before = ex + x0;
            }
            const int c = __shfl_sync(0xffffffffu, cand, src_lane);
            const unsigned __int128 bf = shfl_u128(before, src_lane);
            if (i == 0) {
                s_slice = c;
                u128_split(bf, s_rlo, s_rhi);
                u128_split(tg, s_tlo, s_thi);
            }
        }
        if (rank == 0) {
            if (i == 0) p.accept_len[b] = tau;
            if (i <= B) p.out_tokens[b * (B + 1) + i] = i < tau ? block_token(p, b, i) : -1;
        }
    }
    __syncthreads();
    const int tau = s_tau;
    int32_t *dst = p.out_tokens + b * (B + 1) + tau;
    const BlockRow rp = s_rp[tau];
    const float T = p.T;
    if (s_plain) {
        const uint32_t W = philox_word(p.seed, (uint32_t)b, p.step, (uint32_t)tau, tau == B ? 4u : 3u) >> 8;
        const float *pb = rp.row;
        int off = 0;
        if (p.stage) {
            if (stage_rows(tsm, rp.row, nullptr, nullptr, V, &s_bar, &s_fail)) {
                int hi;
                cl_part(0, V, (int)rank, off, hi);
                pb = tsm;
            } else {
                set_error(p.err, DSPARK_ERR_TIMEOUT);
            }
        }
        auto wf = [&](int v) -> unsigned __int128 {
            const unsigned long long E = weight_of(pb[v - off], T, rp.m);
            return key_of(E, v) >= rp.kstar ? (unsigned __int128)E : (unsigned __int128)0;
        };
        cluster_draw(wf, V, W, dst, dsm);
    } else {
        const BlockRow rq = s_rq[tau];
        const double pi = s_pis[tau];
        auto wf = [&](int v) -> unsigned __int128 { return block_term(rp, rq, pi, T, v); };
        const int np = V / 2, c = s_slice;
        const int r0 = 2 * (int)((long long)c * np / kMassSlices), r1 = 2 * (int)((long long)(c + 1) * np / kMassSlices);
        cluster_pick(wf, r0, r1, -1, u128_join(s_rlo, s_rhi), u128_join(s_tlo, s_thi), dst, dsm);
    }
}

// ---------------------------------------------------------------------------
// Greedy: row argmax keys (zero between launches) then a finalize kernel that
// also returns the keys to zero.
// ---------------------------------------------------------------------------
__global__ void verify_argmax_kernel(const float *__restrict__ P, int rows, int V, unsigned long long *keys, int *err) {
    pdl_trigger();
    pdl_wait();
    __shared__ unsigned long long red[33];
    const int row = blockIdx.y;
    const int nslices = gridDim.x;
    const int npairs = V / 2;
    const int lo = (int)((long long)blockIdx.x * npairs / nslices);
    const int hi = (int)((long long)(blockIdx.x + 1) * npairs / nslices);
    unsigned long long best = 0;
    bool bad = false;
    const float *pr = P + (size_t)row * V;
    // four independent pair loads in flight per thread
    for (int pp0 = lo + threadIdx.x; pp0 < hi; pp0 += 4 * blockDim.x) {
        float2 l[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int pp = pp0 + u * blockDim.x;
            l[u] = pp < hi ? __ldcs((const float2 *)(pr + 2 * pp)) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int pp = pp0 + u * blockDim.x;
            if (pp < hi) {
                if (!isfinite(l[u].x) || !isfinite(l[u].y)) bad = true;
                best = max(best, max(argmax_key(l[u].x, 2 * pp), argmax_key(l[u].y, 2 * pp + 1)));
            }
        }
    }
    if (bad) set_error(err, DSPARK_ERR_BAD_INPUT);
    best = block_max_u64(best, red);
    if (threadIdx.x == 0) atomicMax(&keys[row], best);
}

__global__ void verify_greedy_finalize(const int32_t *__restrict__ tokens, int bs, int B, int V,
                                       unsigned long long *keys, int32_t *accept_len, int32_t *out_tokens, int *err) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= bs) return;
    unsigned long long *k = keys + (size_t)b * (B + 1);
    int a = 0;
    for (; a < B; ++a) {
        const int t = tokens[b * B + a];
        if (t < 0 || t >= V) {
            set_error(err, DSPARK_ERR_OOB);
            break;
        }
        if (argmax_token(k[a]) != t) break;
        out_tokens[b * (B + 1) + a] = t;
    }
    out_tokens[b * (B + 1) + a] = argmax_token(k[a]);
    for (int j = a + 1; j <= B; ++j) out_tokens[b * (B + 1) + j] = -1;
    accept_len[b] = a;
    for (int j = 0; j <= B; ++j) k[j] = 0;
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
size_t verify_scratch_words(int bs, int B, int grid) {
    (void)grid;
    return kStatWords * (size_t)bs * (2 * B + 1) + (size_t)bs * B * kMassSlices * 2 + (size_t)bs * kDrawSlices * 2 +
           (size_t)bs * kMaxBlockRows;
}

bool verify_setup(int V) {
    const size_t smem = NucLayout(V).total;
    const size_t stage2 = (size_t)2 * max_part(V) * 4;
    if (cudaFuncSetAttribute(nucleus_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess ||
        (stage2 <= kStageMax && cudaFuncSetAttribute(verify_block_final_kernel,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     (int)(stage2 / 2)) != cudaSuccess)) {
        (void)cudaGetLastError();
        return false;
    }
    return true;
}

cudaError_t launch_verify(VerifyParams p, int grid, cudaStream_t st) {
    if (p.verify_mode == DSPARK_GREEDY) {
        const int rows = p.bs * (p.B + 1);
        // about two CTAs per SM over all rows
        const int slices = std::max(1, std::min(64, (2 * grid + rows - 1) / rows));
        cudaError_t e = launch_pdl(verify_argmax_kernel, dim3(slices, rows), dim3(256), 0, st, p.P, rows, p.V,
                                   p.scratch, p.err);
        if (e != cudaSuccess) return e;
        return launch_pdl(verify_greedy_finalize, dim3((p.bs + 127) / 128), dim3(128), 0, st, p.tokens, p.bs, p.B, p.V,
                          p.scratch, p.accept_len, p.out_tokens, p.err);
    }
    const int nrows = p.bs * ver_rows_per_seq(p);
    cudaError_t e = launch_pdl_cluster(nucleus_rows_kernel, dim3(kVCl, nrows), dim3(kVThreads), NucLayout(p.V).total,
                                       st, kVCl, p);
    if (e != cudaSuccess) return e;
    const size_t stage2 = (size_t)2 * max_part(p.V) * 4;
    p.stage = stage2 <= kStageMax ? 1 : 0;
    if (p.verify_mode == DSPARK_BLOCK) {
        e = launch_pdl(verify_block_mass_kernel, dim3(kMassSlices, p.bs * p.B), dim3(kMassThreads), 0, st, p);
        if (e != cudaSuccess) return e;
        return launch_pdl_cluster(verify_block_final_kernel, dim3(kVCl, p.bs), dim3(kVThreads),
                                  p.stage ? stage2 / 2 : 0, st, kVCl, p);
    }
    return launch_pdl(verify_token_draw_kernel, dim3(kDrawSlices, p.bs), dim3(kDrawThreads), 0, st, p);
}

}  // namespace ds
