// Markov rollout of the DSpark step (verification is in verify.cu).
//
// Model cards: a low-rank sequential Markov head drafts the 7 tokens of a
// block ("Kimi-K3-DSpark-NVFP4", Original model card / Model Overview; Markov
// rank 256, "Kimi K3 DSpark Q8_0 GGUF", Architecture metadata); greedy or
// probabilistic draft sampling ("Kimi-K3-DSpark-NVFP4", Sampling options).
//
// Every decision is made in exact integers on 2^32-scaled weights so that it
// is reproducible bit for bit: for a logit row l at temperature T,
//   y_v = l_v / T, m = max y, E_v = floor(2^32 * exp^(y_v - m)),
// where exp^ is this library's own fp32 exp (Cody-Waite reduction by ln 2 with
// a 16-bit head, the degree-7 Taylor polynomial in Horner form with fused
// multiply-adds, then scaling by 2^n). The top-p nucleus is the shortest run of
// keys (E_v << 18 | (2^18 - 1 - v)) in descending order whose weight reaches
// tau = max(1, floor(S * P32 / 2^32)); the rollout finds it over the grid by
// histogram levels (grid_nucleus below). Draws use 24-bit uniforms from Philox4x32-10 (Salmon et
// al., SC'11) keyed by the seed with counter (step, seq, pos, purpose) and pick
// the smallest id whose running weight (ascending ids) exceeds
// floor(total * W / 2^24).
//
// The rollout runs cooperatively (all CTAs resident) and synchronises through a
// bounded grid barrier in the workspace.
#include "sampling_spec.cuh"

#include <algorithm>

namespace ds {

constexpr int kRowsPerGroup = 8;    // rows whose histograms share one grid barrier per level

// Limit of the inter-CTA waits: the workspace's wait_ns when set, else kWaitLimitNs.
DS_DEVINL unsigned long long grid_wait_limit(const SampleCtl *ctl) {
    const unsigned long long w = *(const volatile unsigned long long *)&ctl->wait_ns;
    return w ? w : kWaitLimitNs;
}

// ---------------------------------------------------------------------------
// Bounded grid barrier (all CTAs resident: cooperative launch). On expiry the
// error word gets DSPARK_ERR_TIMEOUT and every later barrier returns false.
// ---------------------------------------------------------------------------
__device__ bool grid_barrier(SampleCtl *ctl, volatile int *s_fail, int *err) {
    __syncthreads();
    if (threadIdx.x == 0 && !*s_fail) {
        volatile unsigned int *genp = &ctl->bar_gen;
        const unsigned int gen = *genp;
        __threadfence();
        const unsigned int arrived = atomicAdd(&ctl->bar_count, 1u) + 1u;
        if (arrived == gridDim.x) {
            atomicExch(&ctl->bar_count, 0u);
            __threadfence();
            atomicAdd(&ctl->bar_gen, 1u);
        } else {
            const unsigned long long t0 = globaltimer(), limit = grid_wait_limit(ctl);
            while (*genp == gen) {
                if (globaltimer() - t0 > limit) {
                    set_error(err, DSPARK_ERR_TIMEOUT);
                    *s_fail = 1;
                    break;
                }
                __nanosleep(64);
            }
        }
        __threadfence();
    }
    __syncthreads();
    return !*s_fail;
}

// Pair slice [lo, hi) of this CTA over npairs pairs of vocabulary ids.
DS_DEVINL void pair_slice(int npairs, int &lo, int &hi) {
    lo = (int)((long long)blockIdx.x * npairs / gridDim.x);
    hi = (int)((long long)(blockIdx.x + 1) * npairs / gridDim.x);
}

// ---------------------------------------------------------------------------
// Exact nucleus of up to kRowsPerGroup rows over the grid (each CTA owns a
// slice of every row), for the probabilistic draft. Level 0 histograms the
// binary exponent (octave) of E; the crossing octave (the suffix weight from
// the top reaches tau) holds K*. Every later level histograms the next 10 bits
// of the residual key R = K - (2^octave << 18) inside the crossing range, until
// the crossing bin holds one key (its largest key is K*). A CTA adds only its
// non-empty bins to the row's global level buffer (one atomic each), so each
// level costs one grid barrier and few global atomics.
// ---------------------------------------------------------------------------
constexpr int kGBins = 1024;   // bins of a refinement level (10-bit digits); the octave level uses 33
constexpr int kGDigit = 10;
constexpr int kGLevels = 6;    // the octave + at most 5 digits of the <= 50-bit residual key

// Global histogram of one row and level: weights, counts, largest keys and the
// totals of groups of 32 bins (zero on entry).
struct GLevel {
    unsigned long long w[kGBins];
    unsigned int c[kGBins];
    unsigned long long k[kGBins];
    unsigned long long g[kGBins / 32];
};

struct NucleusSmem {
    unsigned long long hw[kGBins];  // this CTA's histogram of one row and level
    unsigned int hc[kGBins];
    unsigned long long hk[kGBins];
    // per-row state (identical in every CTA)
    unsigned long long tau[kRowsPerGroup], above[kRowsPerGroup], pre[kRowsPerGroup];
    unsigned long long kstar[kRowsPerGroup], Sn[kRowsPerGroup];
    int oct[kRowsPerGroup], sh[kRowsPerGroup], done[kRowsPerGroup];
    float ymax[kRowsPerGroup];
    unsigned long long red[33];
};

DS_DEVINL int octave_of(unsigned long long E) { return 63 - __clzll((long long)E); }

__device__ bool grid_nucleus(const float *const *rowp, int nrows, int V, float T, float top_p, NucleusSmem &sm,
                             GLevel *gl, SampleCtl *ctl, volatile int *s_fail, int *err) {
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    int lo, hi;
    pair_slice(V / 2, lo, hi);
    const unsigned long long P32 = top_p_q32(top_p);
    if (t < nrows) {
        sm.done[t] = 0;
        sm.above[t] = 0;
        sm.pre[t] = 0;
        sm.oct[t] = 0;
        sm.sh[t] = 0;
        sm.kstar[t] = ~0ull;
        sm.Sn[t] = 0;
    }
    __syncthreads();
    for (int level = 0; level < kGLevels; ++level) {
        const int nb = level ? kGBins : 33;
        for (int r = 0; r < nrows; ++r) {
            if (sm.done[r]) continue;
            for (int i = t; i < nb; i += blockDim.x) {
                sm.hw[i] = 0;
                sm.hc[i] = 0;
                sm.hk[i] = 0;
            }
            __syncthreads();
            const float ym = sm.ymax[r];
            const int oct = sm.oct[r], sh = sm.sh[r], d = sh < kGDigit ? sh : kGDigit;
            const unsigned long long pre = sm.pre[r], base = (1ull << oct) << 18;
            const float *row = rowp[r];
            for (int pp = lo + t; pp < hi; pp += blockDim.x) {
                const float2 l = *(const float2 *)(row + 2 * pp);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int v = 2 * pp + e;
                    const unsigned long long E = weight_of(e ? l.y : l.x, T, ym);
                    if (!E) continue;
                    const unsigned long long K = key_of(E, v);
                    int bin;
                    if (level == 0) {
                        bin = octave_of(E);
                    } else {
                        if (octave_of(E) != oct) continue;
                        const unsigned long long R = K - base;
                        if ((R >> sh) != pre) continue;
                        bin = (int)((R >> (sh - d)) & ((1ull << d) - 1));
                    }
                    atomicAdd(&sm.hw[bin], E);
                    atomicAdd(&sm.hc[bin], 1u);
                    atomicMax(&sm.hk[bin], K);
                }
            }
            __syncthreads();
            GLevel &G = gl[level * nrows + r];
            for (int i = t; i < nb; i += blockDim.x) {
                if (sm.hc[i]) {
                    atomicAdd(&G.w[i], sm.hw[i]);
                    atomicAdd(&G.c[i], sm.hc[i]);
                    atomicMax(&G.k[i], sm.hk[i]);
                }
            }
            for (int g = warp; 32 * g < nb; g += blockDim.x >> 5) {
                const unsigned long long gs = warp_sum_u64(32 * g + lane < nb ? sm.hw[32 * g + lane] : 0ull);
                if (lane == 0 && gs) atomicAdd(&G.g[g], gs);
            }
            __syncthreads();
        }
        if (!grid_barrier(ctl, s_fail, err)) return false;
        // every CTA finds every row's crossing the same way (warp r: row r)
        if (warp < nrows && !sm.done[warp]) {
            const int r = warp;
            const GLevel &G = gl[level * nrows + r];
            const int ngroups = (nb + 31) / 32;
            const unsigned long long tot = lane < ngroups ? ldcg_u64(&G.g[lane]) : 0ull;
            const unsigned long long suf = warp_suffix_u64(tot);
            unsigned long long need;
            if (level == 0) {
                const unsigned long long S = __shfl_sync(0xffffffffu, suf, 0);
                const unsigned long long tau = (unsigned long long)(((unsigned __int128)S * P32) >> 32);
                need = tau < 1 ? 1 : tau;
                if (lane == 0) sm.tau[r] = need;
            } else {
                need = sm.tau[r] - sm.above[r];
            }
            const unsigned mask = __ballot_sync(0xffffffffu, suf >= need);
            const int g = mask ? 31 - __clz((int)mask) : 0;
            const unsigned long long above_g = __shfl_sync(0xffffffffu, suf - tot, g);
            const int bi = 32 * g + lane;
            const unsigned long long w = bi < nb ? ldcg_u64(&G.w[bi]) : 0ull;
            const unsigned c = bi < nb ? __ldcg(&G.c[bi]) : 0u;
            const unsigned long long k = bi < nb ? ldcg_u64(&G.k[bi]) : 0ull;
            const unsigned long long suf2 = warp_suffix_u64(w);
            const unsigned mask2 = __ballot_sync(0xffffffffu, suf2 >= need - above_g);
            const int j = mask2 ? 31 - __clz((int)mask2) : 0;
            const unsigned long long ex = __shfl_sync(0xffffffffu, suf2 - w, j);
            const unsigned long long wj = __shfl_sync(0xffffffffu, w, j);
            const unsigned cj = __shfl_sync(0xffffffffu, c, j);
            const unsigned long long kj = __shfl_sync(0xffffffffu, k, j);
            if (lane == 0) {
                if (!mask || !mask2) {  // the weights never reach tau (non-finite input)
                    set_error(err, DSPARK_ERR_BAD_INPUT);
                    sm.done[r] = 2;
                } else {
                    const int bin = 32 * g + j;
                    sm.above[r] += above_g + ex;
                    if (level == 0) {
                        sm.oct[r] = bin;
                        sm.sh[r] = bin + 18;
                        sm.pre[r] = 0;
                    } else {
                        const int sh = sm.sh[r], d = sh < kGDigit ? sh : kGDigit;
                        sm.pre[r] = (sm.pre[r] << d) | (unsigned long long)(bin);
                        sm.sh[r] = sh - d;
                    }
                    if (cj == 1 || (level > 0 && sm.sh[r] == 0)) {
                        sm.kstar[r] = kj;
                        sm.Sn[r] = sm.above[r] + wj;
                        sm.done[r] = 1;
                    }
                }
            }
        }
        __syncthreads();
        bool all = true;
        for (int r = 0; r < nrows; ++r) all = all && sm.done[r] != 0;
        if (all) return true;
    }
    if (t == 0) set_error(err, DSPARK_ERR_BAD_INPUT);
    return true;
}

// Weighted draws of nrows rows at once over vocabulary ids in ascending order:
// for row r the smallest v whose running weight exceeds floor(total_r * W24_r / 2^24),
// with weight = E_v inside the row's nucleus (key >= kstar[r]), else 0; total_r = Sn[r].
// gParts: [nrows][gridDim.x][2] words (overwritten). One grid barrier. The CTA
// holding row r's target writes the id to outs[r].
struct DrawSmem {
    unsigned long long lo[kSampThreads], hi[kSampThreads];
    unsigned long long tot[4];
};

__device__ bool grid_draw_rows(const float *const *rowp, int nrows, int V, float T, NucleusSmem &sm,
                               const uint32_t *W24, unsigned long long *gParts, int32_t *const *outs, DrawSmem &ds_,
                               SampleCtl *ctl, volatile int *s_fail, int *err) {
    int lo, hi;
    pair_slice(V / 2, lo, hi);
    const int t = threadIdx.x;
    for (int r = 0; r < nrows; ++r) {
        const float *row = rowp[r];
        const float ym = sm.ymax[r];
        const unsigned long long ks = sm.kstar[r];
        unsigned long long s = 0;
        for (int pp = lo + t; pp < hi; pp += blockDim.x) {
            const float2 l = *(const float2 *)(row + 2 * pp);
            const unsigned long long E0 = weight_of(l.x, T, ym), E1 = weight_of(l.y, T, ym);
            s += (key_of(E0, 2 * pp) >= ks ? E0 : 0ull) + (key_of(E1, 2 * pp + 1) >= ks ? E1 : 0ull);
        }
        s = block_sum_u64(s, sm.red);  // a CTA's slice weighs < 2^50
        if (t == 0) gParts[((size_t)r * gridDim.x + blockIdx.x) * 2] = s;
    }
    if (!grid_barrier(ctl, s_fail, err)) return false;
    for (int r = 0; r < nrows; ++r) {
        // the slice totals' prefix up to this CTA (threads c: CTA c)
        unsigned long long before = 0, total = 0;
        for (int c = t; c < (int)gridDim.x; c += blockDim.x) {
            const unsigned long long x = ldcg_u64(&gParts[((size_t)r * gridDim.x + c) * 2]);
            total += x;
            if (c < (int)blockIdx.x) before += x;
        }
        before = block_sum_u64(before, sm.red);
        total = block_sum_u64(total, sm.red);
        const unsigned long long mine = ldcg_u64(&gParts[((size_t)r * gridDim.x + blockIdx.x) * 2]);
        const unsigned long long target = (unsigned long long)(((unsigned __int128)total * (W24[r] & 0xFFFFFFu)) >> 24);
        if (!(mine > 0 && before <= target && target < before + mine)) continue;  // uniform over the CTA
        // this CTA holds the target: contiguous pairs per thread, then a scan
        const float *row = rowp[r];
        const float ym = sm.ymax[r];
        const unsigned long long ks = sm.kstar[r];
        auto wf = [&](int v) -> unsigned long long {
            const unsigned long long E = weight_of(row[v], T, ym);
            return key_of(E, v) >= ks ? E : 0ull;
        };
        const int n = hi - lo;
        const int per = (n + blockDim.x - 1) / blockDim.x;
        const int t0 = lo + t * per, t1 = min(hi, t0 + per);
        unsigned long long my = 0;
        for (int pp = t0; pp < t1; ++pp) my += wf(2 * pp) + wf(2 * pp + 1);
        ds_.lo[t] = my;
        __syncthreads();
        if (t == 0) {
            unsigned long long acc = before;
            for (int u = 0; u < (int)blockDim.x; ++u) {
                const unsigned long long x = ds_.lo[u];
                ds_.lo[u] = acc;
                acc += x;
            }
        }
        __syncthreads();
        const unsigned long long ex = ds_.lo[t];
        if (t0 < t1 && ex <= target && target < ex + my) {
            unsigned long long cum = ex;
            for (int v = 2 * t0; v < 2 * t1; ++v) {
                cum += wf(v);
                if (cum > target) {
                    *outs[r] = v;
                    break;
                }
            }
        }
        __syncthreads();
    }
    return true;
}

// ---------------------------------------------------------------------------
// Markov rollout
// ---------------------------------------------------------------------------
constexpr int kRollChunk = 8;  // sequences per pass over w2

// scratch layout (words):
//   amax [B][bs] | pick [B][bs] | parts [B][bs][grid][2] | levels [B][bs][kGLevels] GLevel
// (the level buffers of step i, group g: [kGLevels][rows of g], rows from g * kRowsPerGroup)
struct RollLayout {
    size_t amax, pick, parts, levels, total;
    __host__ __device__ RollLayout(int bs, int B, int grid) {
        amax = 0;
        pick = amax + (size_t)B * bs;
        parts = pick + (size_t)B * bs;
        levels = parts + (size_t)B * bs * grid * 2;
        total = levels + (size_t)B * bs * kGLevels * (sizeof(GLevel) / 8);
    }
};

size_t rollout_scratch_words(int bs, int B, int grid) { return RollLayout(bs, B, grid).total; }

DS_DEVINL uint64_t policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// w2 storage of the rollout. The CTA owns the vocabulary pairs [lo, hi) (whole
// 16-byte quads); thread t owns pair lo + t ("primary") and, when the slice is
// wider than the CTA, pair lo + t + blockDim ("secondary").
//  - Rows [0, Kt) of the primary pairs live in tensor memory for the whole
//    kernel (Kt = min(r, 128): 128 columns per thread, all 512 columns of the
//    SM), rows [0, Kt) of the secondary pairs in shared memory; both are read
//    from global memory once at kernel start.
//  - Rows [Kt, r) stream every pass through a ring of kRollStages shared-memory
//    stages of kRollKC rows, filled by 2D tensor copies issued by thread 0
//    (L2 evict-last: w2 is re-read every step) and completing on "full"
//    mbarriers; every warp releases a stage on its "empty" mbarrier. w2 does
//    not depend on the drafted tokens, so the ring runs ahead of the compute
//    across steps and grid barriers.
// The tensor-memory part is used when the secondary pairs fit kRollSec slots.
constexpr int kRollKC = 16;
constexpr int kRollStages = 4;
constexpr int kRollTmemRows = 128;
constexpr int kRollSec = 32;
constexpr int kRollWarps = kSampThreads / 32;

// A stage holds nbox tensor boxes of kRollKC rows x box_w pairs (w2 seen as a
// uint32 matrix [r, V / 2]); the CTA's slice starts at pair lo of every box row.
struct RollRing {
    uint8_t *stage;           // [kRollStages][nbox][kRollKC][box_w] uint32
    uint64_t *full, *empty;   // [kRollStages] each
    int box_w, nbox;          // pairs per box row, boxes per stage
    uint32_t stage_bytes;
    int kt;                   // rows held on chip (tensor memory / secondary smem)
    int nchunks;              // streamed chunks per pass over w2 (rows kt .. r-1)
    long long issued;         // chunks issued (thread 0's count)
    long long consumed;       // chunks read by this thread
    long long total;
};

// Box width and count of the w2 tiles of a rollout over V with grid CTAs: the
// largest slice (pairs) in as few boxes of <= 256 pairs as possible, the width
// a multiple of 4 pairs (16 bytes).
__host__ __device__ void rollout_box(int V, int grid, int *box_w, int *nbox) {
    const int nq = V / 8;
    const int max_pairs = 4 * ((nq + grid - 1) / grid);
    const int n = (max_pairs + 255) / 256;
    *nbox = n < 1 ? 1 : n;
    *box_w = ((max_pairs + *nbox - 1) / *nbox + 3) / 4 * 4;
    if (*box_w < 4) *box_w = 4;
}

// Thread 0: issue the next chunk into its stage once every warp has released
// the stage's previous chunk. False on a timeout or an abort.
DS_DEVINL bool ring_issue(RollRing &rg, const CUtensorMap *tm, int lo, uint64_t pol, volatile int *abort) {
    if (rg.issued >= rg.total) return true;
    const long long c = rg.issued;
    const int s = (int)(c % kRollStages);
    if (c >= kRollStages &&
        !mbar_wait_bounded(&rg.empty[s], (uint32_t)((c / kRollStages - 1) & 1), abort))
        return false;
    const int k0 = rg.kt + (int)(c % rg.nchunks) * kRollKC;
    mbar_arrive_expect_tx(&rg.full[s], rg.stage_bytes);
    uint8_t *dst = rg.stage + (size_t)s * rg.stage_bytes;
    for (int j = 0; j < rg.nbox; ++j)
        tma_load_2d_hint(dst + (size_t)j * kRollKC * rg.box_w * 4, tm, lo + j * rg.box_w, k0, &rg.full[s], pol);
    rg.issued = c + 1;
    return true;
}

// Every chunk issued lands before the kernel exits (bounded waits).
DS_DEVINL void ring_drain(RollRing &rg) {
    if (threadIdx.x != 0) return;
    for (long long c = rg.consumed; c < rg.issued; ++c)
        mbar_drain(&rg.full[c % kRollStages], (uint32_t)((c / kRollStages) & 1));
}

// Two fp32 chains of bf16 products: lo += u * w.lo, hi += u * w.hi, where u is
// the low (HI = false) or high half of u2. The bf16 operands widen exactly, so
// each step is one IEEE fp32 FMA with a single rounding (identical to fmaf on
// the widened values).
template <bool HI>
DS_DEVINL void fma_bf16x2(float &lo, float &hi, uint32_t u2, uint32_t w) {
    if (HI)
        asm("{\n\t.reg .b16 wl, wh, ul, uh;\n\tmov.b32 {wl, wh}, %2;\n\tmov.b32 {ul, uh}, %3;\n\t"
            "fma.rn.f32.bf16 %0, uh, wl, %0;\n\tfma.rn.f32.bf16 %1, uh, wh, %1;\n\t}"
            : "+f"(lo), "+f"(hi)
            : "r"(w), "r"(u2));
    else
        asm("{\n\t.reg .b16 wl, wh, ul, uh;\n\tmov.b32 {wl, wh}, %2;\n\tmov.b32 {ul, uh}, %3;\n\t"
            "fma.rn.f32.bf16 %0, ul, wl, %0;\n\tfma.rn.f32.bf16 %1, ul, wh, %1;\n\t}"
            : "+f"(lo), "+f"(hi)
            : "r"(w), "r"(u2));
}

// The chains: acc_v = fmaf(u_k, w2[k][v], acc_v) for k in order, per sequence
// and vocabulary id (each an IEEE fp32 FMA of bf16 operands, bit-identical to the
// oracle's fmaf chain on the widened values). u (w1[t_{i-1}], bf16, the same for
// every thread) comes from shared memory eight k at a time (one 16-byte load per
// sequence); w2 stays in its bf16 pairs.
// A thread owns its primary pair for all NB sequences of the pass (p0, p1)
// and, by EX: 0 nothing more; 1 one extra chain, a leftover pair of the CTA for
// one sequence (s0[0], s1[0]: the leftover pairs' chains are spread one per
// thread so that no warp does twice the work); 2 a leftover pair for all NB
// sequences (s0, s1), when the leftovers are too many to spread.
template <int NB>
struct RollAcc {
    float p0[NB], p1[NB], s0[NB], s1[NB];
};

// rows k0 .. k0 + 7 of the chains (k0 a multiple of 8); wv0 / wv1: the w2 pairs
template <int NB, int EX>
DS_DEVINL void roll_rows8(const uint32_t (&wv0)[8], const uint32_t (&wv1)[8], int k0, const uint16_t (*s_ub)[256],
                          int ex_seq, RollAcc<NB> &a) {
    uint4 uq[NB];
#pragma unroll
    for (int bb = 0; bb < NB; ++bb) uq[bb] = *(const uint4 *)&s_ub[bb][k0];
    uint4 ue = make_uint4(0u, 0u, 0u, 0u);
    if (EX == 1) ue = *(const uint4 *)&s_ub[ex_seq][k0];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int bb = 0; bb < NB; ++bb) {
            const uint32_t u2 = (j >> 1) == 0 ? uq[bb].x : (j >> 1) == 1 ? uq[bb].y : (j >> 1) == 2 ? uq[bb].z : uq[bb].w;
            if (j & 1) {
                fma_bf16x2<true>(a.p0[bb], a.p1[bb], u2, wv0[j]);
                if (EX == 2) fma_bf16x2<true>(a.s0[bb], a.s1[bb], u2, wv1[j]);
            } else {
                fma_bf16x2<false>(a.p0[bb], a.p1[bb], u2, wv0[j]);
                if (EX == 2) fma_bf16x2<false>(a.s0[bb], a.s1[bb], u2, wv1[j]);
            }
        }
        if (EX == 1) {
            const uint32_t u2 = (j >> 1) == 0 ? ue.x : (j >> 1) == 1 ? ue.y : (j >> 1) == 2 ? ue.z : ue.w;
            if (j & 1)
                fma_bf16x2<true>(a.s0[0], a.s1[0], u2, wv1[j]);
            else
                fma_bf16x2<false>(a.s0[0], a.s1[0], u2, wv1[j]);
        }
    }
}
// one row k of the chains (tails whose length is not a multiple of 8)
template <int NB, int EX>
DS_DEVINL void roll_row1(uint32_t wv0, uint32_t wv1, int k, const uint16_t (*s_ub)[256], int ex_seq, RollAcc<NB> &a) {
#pragma unroll
    for (int bb = 0; bb < NB; ++bb) {
        const uint32_t u2 = s_ub[bb][k];
        fma_bf16x2<false>(a.p0[bb], a.p1[bb], u2, wv0);
        if (EX == 2) fma_bf16x2<false>(a.s0[bb], a.s1[bb], u2, wv1);
    }
    if (EX == 1) fma_bf16x2<false>(a.s0[0], a.s1[0], (uint32_t)s_ub[ex_seq][k], wv1);
}

// One streamed chunk of rows k0 .. k0 + rows - 1.
template <int NB, int EX>
DS_DEVINL void roll_chunk(const uint32_t *w, int wpr, int rows, int k0, int o0, int o1, bool has0, bool has1,
                          const uint16_t (*s_ub)[256], int ex_seq, RollAcc<NB> &a) {
    int kk = 0;
    if ((k0 & 7) == 0) {
        for (; kk + 8 <= rows; kk += 8) {
            uint32_t wv0[8], wv1[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                wv0[j] = has0 ? w[(kk + j) * wpr + o0] : 0u;
                wv1[j] = (EX != 0 && has1) ? w[(kk + j) * wpr + o1] : 0u;
            }
            roll_rows8<NB, EX>(wv0, wv1, k0 + kk, s_ub, ex_seq, a);
        }
    }
    for (; kk < rows; ++kk)
        roll_row1<NB, EX>(has0 ? w[kk * wpr + o0] : 0u, (EX != 0 && has1) ? w[kk * wpr + o1] : 0u, k0 + kk, s_ub,
                          ex_seq, a);
}

// Rows [0, kt) of the chains from tensor memory (primary pairs: this thread's
// lane and columns) and the leftover pairs' rows in shared memory (column sp).
// Warp-collective.
template <int NB, int EX>
DS_DEVINL void roll_tmem16(const uint32_t (&v)[16], int k16, int kt, const uint32_t (*s_sec)[kRollSec], int sp,
                           bool has1, const uint16_t (*s_ub)[256], int ex_seq, RollAcc<NB> &a) {
    if (k16 + 16 <= kt) {
#pragma unroll
        for (int j8 = 0; j8 < 16; j8 += 8) {
            uint32_t wv0[8], wv1[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                wv0[j] = v[j8 + j];
                wv1[j] = (EX != 0 && has1) ? s_sec[k16 + j8 + j][sp] : 0u;
            }
            roll_rows8<NB, EX>(wv0, wv1, k16 + j8, s_ub, ex_seq, a);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (k16 + j < kt)
                roll_row1<NB, EX>(v[j], (EX != 0 && has1) ? s_sec[k16 + j][sp] : 0u, k16 + j, s_ub, ex_seq, a);
    }
}
template <int NB, int EX>
DS_DEVINL void roll_tmem_rows(uint32_t taddr, int kt, const uint32_t (*s_sec)[kRollSec], int sp, bool has1,
                              const uint16_t (*s_ub)[256], int ex_seq, RollAcc<NB> &a) {
    for (int k16 = 0; k16 < kt; k16 += 16) {
        uint32_t v[16];
        tmem_ld16u(taddr + (uint32_t)k16, v);
        roll_tmem16<NB, EX>(v, k16, kt, s_sec, sp, has1, s_ub, ex_seq, a);
    }
}

// The chains of one pass in a given EX mode.
template <int NB, int EX>
DS_DEVINL bool roll_pass(const RolloutParams &p, const CUtensorMap *tm, int lo, RollRing &rg, uint32_t taddr,
                         const uint32_t (*s_sec)[kRollSec], const uint16_t (*s_ub)[256], int sp, int ex_seq, bool has0,
                         bool has1, int o0, int o1, uint64_t pol, volatile int *s_fail, RollAcc<NB> &acc) {
    const int r = p.r, lane = threadIdx.x & 31;
    if (rg.kt > 0) roll_tmem_rows<NB, EX>(taddr, rg.kt, s_sec, sp, has1, s_ub, ex_seq, acc);
    bool failed = false;
    for (int ch = 0; ch < rg.nchunks; ++ch) {
        const long long c = rg.consumed;
        const int s = (int)(c % kRollStages);
        if (!failed && !mbar_wait_bounded(&rg.full[s], (uint32_t)((c / kRollStages) & 1), s_fail)) {
            set_error(p.err, DSPARK_ERR_TIMEOUT);
            failed = true;
        }
        if (!failed) {
            const uint32_t *w = (const uint32_t *)(rg.stage + (size_t)s * rg.stage_bytes);
            const int k0 = rg.kt + ch * kRollKC, rows = min(kRollKC, r - k0);
            roll_chunk<NB, EX>(w, rg.box_w, rows, k0, o0, o1, has0, has1, s_ub, ex_seq, acc);
            rg.consumed = c + 1;
        }
        __syncwarp();
        if (lane == 0 && !failed) mbar_arrive(&rg.empty[s]);
        // thread 0 refills after its own chunk: the stage it refills was released by
        // every warp one chunk earlier, so the wait rarely holds this warp
        if (!failed && threadIdx.x == 0 && !ring_issue(rg, tm, lo, pol, s_fail)) {
            set_error(p.err, DSPARK_ERR_TIMEOUT);
            *s_fail = 1;
        }
    }
    return !failed;
}

template <int NB>
__device__ void rollout_logits(const RolloutParams &p, const CUtensorMap *tm, int i, int b0, int nb, int lo, int hi,
                               RollRing &rg, uint32_t taddr, const uint32_t (*s_sec)[kRollSec],
                               const uint16_t (*s_ub)[256], unsigned long long *amax,
                               unsigned long long (*red8)[kRollWarps], uint64_t pol, volatile int *s_fail) {
    const int V = p.V;
    RollAcc<NB> acc;
#pragma unroll
    for (int bb = 0; bb < NB; ++bb) acc.p0[bb] = acc.p1[bb] = acc.s0[bb] = acc.s1[bb] = 0.f;
    const int nt = (int)blockDim.x;
    const int q0 = threadIdx.x;
    const bool has0 = lo + q0 < hi;
    // the CTA's leftover pairs lo + nt + sp (sp < nsec): one chain per thread
    // (pair sp = t / NB, sequence t % NB) when they fit, else pair t for all NB
    const int nsec = max(0, hi - lo - nt);
    const bool spread = NB > 1 && nsec * NB <= nt;
    const int sp = spread ? (int)threadIdx.x / NB : (int)threadIdx.x;
    const int ex_seq = spread ? (int)threadIdx.x % NB : 0;
    const bool has1 = spread ? (int)threadIdx.x < nsec * NB : (int)threadIdx.x < nsec;
    const int q1 = nt + sp;
    const bool two = __any_sync(0xffffffffu, has1);  // warp-uniform
    // word offsets of the thread's pairs in a stage (row 0)
    const int o0 = (q0 / rg.box_w) * kRollKC * rg.box_w + q0 % rg.box_w;
    const int o1 = (q1 / rg.box_w) * kRollKC * rg.box_w + q1 % rg.box_w;
    bool ok;
    if (!two)
        ok = roll_pass<NB, 0>(p, tm, lo, rg, taddr, s_sec, s_ub, sp, ex_seq, has0, has1, o0, o1, pol, s_fail, acc);
    else if (spread)
        ok = roll_pass<NB, 1>(p, tm, lo, rg, taddr, s_sec, s_ub, sp, ex_seq, has0, has1, o0, o1, pol, s_fail, acc);
    else
        ok = roll_pass<NB, 2>(p, tm, lo, rg, taddr, s_sec, s_ub, sp, ex_seq, has0, has1, o0, o1, pol, s_fail, acc);
    if (!ok) *s_fail = 1;
    unsigned long long best[NB];
#pragma unroll
    for (int bb = 0; bb < NB; ++bb) best[bb] = 0;
    bool bad = false;
    // one output pair pp for sequence bb with chain values d0, d1
    auto emit = [&](int pp, int bb, float d0, float d1) -> unsigned long long {
        const size_t off = ((size_t)(b0 + bb) * p.B + i) * V + 2 * pp;
        const float2 z = *(const float2 *)(p.z + off);
        const float l0 = __fadd_rn(z.x, d0), l1 = __fadd_rn(z.y, d1);
        *(float2 *)(p.ell + off) = make_float2(l0, l1);
        if (!isfinite(l0) || !isfinite(l1)) bad = true;
        unsigned long long k0, k1;
        if (p.draft_mode == DSPARK_GREEDY) {
            k0 = argmax_key(l0, 2 * pp);
            k1 = argmax_key(l1, 2 * pp + 1);
        } else {
            k0 = f2ord(__fdiv_rn(l0, p.T));
            k1 = f2ord(__fdiv_rn(l1, p.T));
        }
        return max(k0, k1);
    };
    if (has0) {
#pragma unroll
        for (int bb = 0; bb < NB; ++bb)
            if (bb < nb) best[bb] = max(best[bb], emit(lo + q0, bb, acc.p0[bb], acc.p1[bb]));
    }
    if (has1) {
        if (spread) {
            if (ex_seq < nb) {
                const unsigned long long k = emit(lo + q1, ex_seq, acc.s0[0], acc.s1[0]);
#pragma unroll
                for (int bb = 0; bb < NB; ++bb)
                    if (bb == ex_seq) best[bb] = max(best[bb], k);
            }
        } else {
#pragma unroll
            for (int bb = 0; bb < NB; ++bb)
                if (bb < nb) best[bb] = max(best[bb], emit(lo + q1, bb, acc.s0[bb], acc.s1[bb]));
        }
    }
    if (bad) set_error(p.err, DSPARK_ERR_BAD_INPUT);
    // every sequence's maximum over the CTA in one round: warp maxima, one barrier,
    // then one thread per sequence (the caller's next barrier frees red8)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int bb = 0; bb < NB; ++bb) {
        best[bb] = warp_max_u64(best[bb]);
        if (lane == 0) red8[bb][warp] = best[bb];
    }
    __syncthreads();
    if ((int)threadIdx.x < nb) {
        unsigned long long m = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = max(m, red8[threadIdx.x][w]);
        atomicMax(&amax[b0 + threadIdx.x], m);
    }
}

// Vocabulary pairs of this CTA for the rollout: quads of 4 pairs (16 bytes of
// a w2 row) so every bulk copy is 16-byte aligned.
DS_DEVINL void quad_slice(int V, int &lo, int &hi) {
    const int nq = V / 8;
    lo = 4 * (int)((long long)blockIdx.x * nq / gridDim.x);
    hi = 4 * (int)((long long)(blockIdx.x + 1) * nq / gridDim.x);
}

__global__ void __launch_bounds__(kSampThreads, 1)
    rollout_kernel(const __grid_constant__ CUtensorMap tmW2, RolloutParams p) {
    __shared__ NucleusSmem sm;
    __shared__ DrawSmem dsm;
    __shared__ __align__(16) uint16_t s_ub[kRollChunk][256];  // w1[t_{i-1}] (bf16 bits), per sequence of the pass
    __shared__ unsigned long long s_red8[kRollChunk][kRollWarps];
    __shared__ __align__(8) uint64_t s_full[kRollStages], s_empty[kRollStages];
    __shared__ int s_prev[kMaxSampBs];
    __shared__ volatile int s_fail;
    __shared__ const float *s_rows[kRowsPerGroup];
    __shared__ uint32_t s_w24[kRowsPerGroup];
    __shared__ int32_t *s_outs[kRowsPerGroup];
    __shared__ uint32_t s_tmem_base;
    __shared__ uint32_t s_sec[kRollTmemRows][kRollSec];  // secondary pairs, rows [0, kt)
    extern __shared__ __align__(128) uint8_t ring_smem[];
    static_assert(kSampThreads == 512, "tensor-memory layout: 4 warps per lane quadrant, 128 columns each");
    const RollLayout L(p.bs, p.B, gridDim.x);
    unsigned long long *sc = p.scratch;
    const int V = p.V, r = p.r;
    int lo, hi;
    quad_slice(V, lo, hi);
    RollRing rg;
    rg.stage = ring_smem;
    rg.full = s_full;
    rg.empty = s_empty;
    rollout_box(V, gridDim.x, &rg.box_w, &rg.nbox);
    rg.stage_bytes = (uint32_t)(rg.nbox * kRollKC * rg.box_w * 4);
    // on-chip rows when every CTA's secondary pairs fit the kRollSec slots
    const int max_pairs = 4 * ((V / 8 + (int)gridDim.x - 1) / (int)gridDim.x);
    rg.kt = (max_pairs <= kSampThreads + kRollSec) ? min(r, kRollTmemRows) : 0;
    rg.nchunks = (r - rg.kt + kRollKC - 1) / kRollKC;
    rg.issued = rg.consumed = 0;
    rg.total = (long long)p.B * ((p.bs + kRollChunk - 1) / kRollChunk) * rg.nchunks;
    const uint64_t pol = policy_evict_last();
    if (hi <= lo) rg.total = 0;
    if (threadIdx.x == 0) {
        s_fail = 0;
        for (int st = 0; st < kRollStages; ++st) {
            mbar_init(&s_full[st], 1);
            mbar_init(&s_empty[st], kRollWarps);
        }
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&tmW2);
        for (int st = 0; st < kRollStages - 1; ++st) ring_issue(rg, &tmW2, lo, pol, &s_fail);
    }
    // rows [0, kt) of w2 into tensor memory (primary pairs) and shared memory (secondary)
    const int warp = threadIdx.x >> 5;
    if (rg.kt > 0 && warp == 0) tmem_alloc(&s_tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = s_tmem_base + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(128 * (warp >> 2));
    if (rg.kt > 0) {
        const uint32_t *w2w = (const uint32_t *)p.w2;
        const size_t rowp = (size_t)V / 2;
        const bool has0 = lo + (int)threadIdx.x < hi;
        for (int k32 = 0; k32 < rg.kt; k32 += 32) {
            uint32_t v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j)
                v[j] = (has0 && k32 + j < rg.kt) ? __ldg(w2w + (size_t)(k32 + j) * rowp + lo + threadIdx.x) : 0u;
            tmem_st32(taddr + (uint32_t)k32, v);
        }
        tmem_st_wait();
        if (threadIdx.x < kRollSec) {
            const int q1 = lo + (int)threadIdx.x + (int)blockDim.x;
            for (int k = 0; k < rg.kt; ++k) s_sec[k][threadIdx.x] = q1 < hi ? __ldg(w2w + (size_t)k * rowp + q1) : 0u;
        }
    }
    // the level buffers of the nucleus are needed (and zeroed) only for a probabilistic draft
    const size_t zero_words = p.draft_mode == DSPARK_GREEDY ? L.levels : L.total;
    for (size_t w = (size_t)blockIdx.x * blockDim.x + threadIdx.x; w < zero_words; w += (size_t)gridDim.x * blockDim.x)
        sc[w] = 0;
    for (int b = threadIdx.x; b < p.bs; b += blockDim.x) {
        int a = p.anchor[b];
        if (a < 0 || a >= V) {
            set_error(p.err, DSPARK_ERR_OOB);
            a = 0;
        }
        s_prev[b] = a;
    }
    __threadfence();
    bool ok = grid_barrier(p.ctl, &s_fail, p.err);

    for (int i = 0; i < p.B && ok; ++i) {
        // ell_i = z_i + fp32 FMA chain of w1[t_{i-1}] against w2 (k in order)
        for (int b0 = 0; b0 < p.bs && ok; b0 += kRollChunk) {
            const int nb = min(kRollChunk, p.bs - b0);
            for (int idx = threadIdx.x; idx < kRollChunk * r; idx += blockDim.x) {
                const int bb = idx / r, k = idx % r;
                s_ub[bb][k] = bb < nb ? __bfloat16_as_ushort(p.w1[(size_t)s_prev[b0 + bb] * r + k]) : (uint16_t)0;
            }
            __syncthreads();
            if (hi > lo) {
                if (nb == 1)
                    rollout_logits<1>(p, &tmW2, i, b0, 1, lo, hi, rg, taddr, s_sec, s_ub,
                                      sc + L.amax + (size_t)i * p.bs, s_red8, pol, &s_fail);
                else
                    rollout_logits<kRollChunk>(p, &tmW2, i, b0, nb, lo, hi, rg, taddr, s_sec, s_ub,
                                               sc + L.amax + (size_t)i * p.bs, s_red8, pol, &s_fail);
            }
            __syncthreads();
            ok = !s_fail;
        }
        if (!ok || !grid_barrier(p.ctl, &s_fail, p.err)) {
            ok = false;
            break;
        }
        if (p.draft_mode == DSPARK_GREEDY) {
            for (int b = threadIdx.x; b < p.bs; b += blockDim.x) {
                const int t = argmax_token(ldcg_u64(&sc[L.amax + (size_t)i * p.bs + b]));
                s_prev[b] = t;
                if (blockIdx.x == 0) p.tokens[b * p.B + i] = t;
            }
            __syncthreads();
            continue;
        }
        // probabilistic: nucleus of ell_i / T per sequence, then a draw
        for (int g0 = 0; g0 < p.bs && ok; g0 += kRowsPerGroup) {
            const int nr = min(kRowsPerGroup, p.bs - g0);
            if (threadIdx.x < nr) {
                s_rows[threadIdx.x] = p.ell + ((size_t)(g0 + threadIdx.x) * p.B + i) * V;
                sm.ymax[threadIdx.x] = ord2f((uint32_t)ldcg_u64(&sc[L.amax + (size_t)i * p.bs + g0 + threadIdx.x]));
            }
            __syncthreads();
            GLevel *gl = (GLevel *)(sc + L.levels) + ((size_t)i * p.bs + g0) * kGLevels;
            if (!grid_nucleus(s_rows, nr, V, p.T, p.top_p, sm, gl, p.ctl, &s_fail, p.err)) {
                ok = false;
                break;
            }
            if (threadIdx.x < nr) {
                const int b = g0 + threadIdx.x;
                s_w24[threadIdx.x] = philox_word(p.seed, (uint32_t)b, p.step, (uint32_t)i, 1u) >> 8;
                s_outs[threadIdx.x] = (int32_t *)&sc[L.pick + (size_t)i * p.bs + b];
            }
            __syncthreads();
            if (!grid_draw_rows(s_rows, nr, V, p.T, sm, s_w24, sc + L.parts + ((size_t)i * p.bs + g0) * gridDim.x * 2,
                                s_outs, dsm, p.ctl, &s_fail, p.err)) {
                ok = false;
                break;
            }
        }
        if (!ok || !grid_barrier(p.ctl, &s_fail, p.err)) {
            ok = false;
            break;
        }
        for (int b = threadIdx.x; b < p.bs; b += blockDim.x) {
            const int t = (int)(uint32_t)ldcg_u64(&sc[L.pick + (size_t)i * p.bs + b]);
            s_prev[b] = t;
            if (blockIdx.x == 0) p.tokens[b * p.B + i] = t;
        }
        __syncthreads();
    }
    ring_drain(rg);
    tc_fence_before();
    __syncthreads();
    if (rg.kt > 0 && warp == 0) {
        tc_fence_after();
        tmem_dealloc(s_tmem_base, 512);
    }
}

// ---------------------------------------------------------------------------
// Greedy rollout of one sequence with the CTA's w2 slice held on chip.
//
// The slice (pairs [lo, hi), all r rows) is read from HBM once per launch:
//  - rows [0, 128) of the primary pairs (thread t: pair lo + t) live in
//    tensor memory, laid out as in the streaming kernel;
//  - rows [128, 160) of the primary pairs live in 32 registers of their thread;
//  - rows [0, 160) of the secondary pairs (lo + 512 + t, lanes of warp 0) live
//    in shared memory;
//  - rows [160, r) of every pair stay in shared memory: 16-row blocks in six
//    slots, the same slots that first stage the load (block j in slot j % 6).
// Between steps the CTAs do not meet at a barrier: each one publishes its best
// greedy key for step i in a word of its own and reads every CTA's word. The
// winner's w1 row is prefetched into L2 by the CTA that found it.
// ---------------------------------------------------------------------------
constexpr int kResSlots = 6;
constexpr int kResTmemRows = 128;
constexpr int kResRegRows = 32;
constexpr int kResOnRows = kResTmemRows + kResRegRows;
constexpr int kResSec = 32;
constexpr int kResMaxRank = kResOnRows + kRollKC * kResSlots;
constexpr int kResGatherPerLane = 8;  // key words read by each lane of the gathering warp

struct ResLayout {  // dynamic shared memory, bytes
    uint32_t stage_bytes, slots, sec, u, red, bars, total;
    __host__ __device__ ResLayout(int V, int grid) {
        int box_w, nbox;
        rollout_box(V, grid, &box_w, &nbox);
        stage_bytes = (uint32_t)(nbox * kRollKC * box_w * 4);
        slots = 0;
        sec = slots + kResSlots * stage_bytes;
        u = sec + kResOnRows * kResSec * 4;
        red = u + kResMaxRank * 2;
        bars = red + 32 * 8;
        total = bars + kResSlots * 8;
    }
};

// Chains of this thread's pairs (four fp32 accumulators: primary lo/hi, secondary lo/hi).
struct ResAcc {
    float p0, p1, s0, s1;
};

// Eight rows k0 .. k0 + 7 (k0 a multiple of 8): u from s_u (bf16), the primary
// pair's words in v, the secondary pair's (TWO) in column t of s_sec.
template <bool TWO>
DS_DEVINL void res_rows8(const uint32_t (&v)[8], int k0, const uint32_t (*s_sec)[kResSec], int t,
                         const uint16_t *s_u, ResAcc &a) {
    const uint4 uq = *(const uint4 *)(s_u + k0);
    const uint32_t u2[4] = {uq.x, uq.y, uq.z, uq.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (j & 1)
            fma_bf16x2<true>(a.p0, a.p1, u2[j >> 1], v[j]);
        else
            fma_bf16x2<false>(a.p0, a.p1, u2[j >> 1], v[j]);
        if (TWO) {
            const uint32_t w = s_sec[k0 + j][t];
            if (j & 1)
                fma_bf16x2<true>(a.s0, a.s1, u2[j >> 1], w);
            else
                fma_bf16x2<false>(a.s0, a.s1, u2[j >> 1], w);
        }
    }
}

// One step's chains of this thread's pairs, k in order.
template <bool TWO>
DS_DEVINL void res_chain(uint32_t taddr, int r, const uint32_t (&wr)[kResRegRows], const uint8_t *slots,
                         uint32_t stage_bytes, int box_w, int o0, int o1, const uint32_t (*s_sec)[kResSec], int t,
                         const uint16_t *s_u, ResAcc &a) {
    // rows [0, min(r, 128)) from tensor memory, 8 columns per load, two loads in flight
    const int nck = min(r, kResTmemRows) / 8;
    uint32_t va[8], vb[8];
    tmem_ld8_issue(taddr, va);
    for (int c = 0; c < nck; c += 2) {
        tmem_ld_wait_tied(va);
        if (c + 1 < nck) tmem_ld8_issue(taddr + 8u * (uint32_t)(c + 1), vb);
        res_rows8<TWO>(va, 8 * c, s_sec, t, s_u, a);
        if (c + 1 < nck) {
            tmem_ld_wait_tied(vb);
            if (c + 2 < nck) tmem_ld8_issue(taddr + 8u * (uint32_t)(c + 2), va);
            res_rows8<TWO>(vb, 8 * (c + 1), s_sec, t, s_u, a);
        }
    }
    // rows [128, min(r, 160)) from registers
    if (r > kResTmemRows) {
#pragma unroll
        for (int j8 = 0; j8 < kResRegRows; j8 += 8) {
            if (kResTmemRows + j8 < r) {
                const uint32_t v[8] = {wr[j8], wr[j8 + 1], wr[j8 + 2], wr[j8 + 3],
                                       wr[j8 + 4], wr[j8 + 5], wr[j8 + 6], wr[j8 + 7]};
                res_rows8<TWO>(v, kResTmemRows + j8, s_sec, t, s_u, a);
            }
        }
    }
    // rows [160, r) from the shared-memory blocks
    for (int j = kResOnRows / kRollKC; j < r / kRollKC; ++j) {
        const uint32_t *w = (const uint32_t *)(slots + (size_t)(j % kResSlots) * stage_bytes);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 uq = *(const uint4 *)(s_u + kRollKC * j + 8 * h);
            const uint32_t u2[4] = {uq.x, uq.y, uq.z, uq.w};
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int row = 8 * h + kk;
                if (kk & 1)
                    fma_bf16x2<true>(a.p0, a.p1, u2[kk >> 1], w[row * box_w + o0]);
                else
                    fma_bf16x2<false>(a.p0, a.p1, u2[kk >> 1], w[row * box_w + o0]);
                if (TWO) {
                    if (kk & 1)
                        fma_bf16x2<true>(a.s0, a.s1, u2[kk >> 1], w[row * box_w + o1]);
                    else
                        fma_bf16x2<false>(a.s0, a.s1, u2[kk >> 1], w[row * box_w + o1]);
                }
            }
        }
    }
}

// ell and the greedy key of one pair.
DS_DEVINL unsigned long long res_pair_out(float d0, float d1, float2 z, int pp, float *ell, bool &bad) {
    const float l0 = __fadd_rn(z.x, d0), l1 = __fadd_rn(z.y, d1);
    *(float2 *)(ell + 2 * pp) = make_float2(l0, l1);
    if (!isfinite(l0) || !isfinite(l1)) bad = true;
    return max(argmax_key(l0, 2 * pp), argmax_key(l1, 2 * pp + 1));
}

// Split grid barrier (one thread): arrive once this CTA's earlier writes are
// done, wait later. The generation read before arriving is the one to wait past.
DS_DEVINL unsigned int grid_arrive(SampleCtl *ctl) {
    volatile unsigned int *genp = &ctl->bar_gen;
    const unsigned int gen = *genp;
    __threadfence();
    if (atomicAdd(&ctl->bar_count, 1u) + 1u == gridDim.x) {
        atomicExch(&ctl->bar_count, 0u);
        __threadfence();
        atomicAdd(&ctl->bar_gen, 1u);
    }
    return gen;
}
DS_DEVINL bool grid_wait(SampleCtl *ctl, unsigned int gen, int *err) {
    volatile unsigned int *genp = &ctl->bar_gen;
    const unsigned long long t0 = globaltimer(), limit = grid_wait_limit(ctl);
    while (*genp == gen) {
        if (globaltimer() - t0 > limit) {
            set_error(err, DSPARK_ERR_TIMEOUT);
            return false;
        }
        __nanosleep(32);
    }
    __threadfence();
    return true;
}

__global__ void __launch_bounds__(kSampThreads, 1)
    rollout_greedy_resident_kernel(const __grid_constant__ CUtensorMap tmW2, RolloutParams p) {
    extern __shared__ __align__(128) uint8_t rsm[];
    __shared__ volatile int s_fail;
    __shared__ uint32_t s_tmem_base;
    __shared__ unsigned int s_gen;
    __shared__ int s_tok;
    const ResLayout RL(p.V, gridDim.x);
    uint8_t *slots = rsm + RL.slots;
    uint32_t(*s_sec)[kResSec] = (uint32_t(*)[kResSec])(rsm + RL.sec);
    uint16_t *s_u = (uint16_t *)(rsm + RL.u);  // bf16 bits of w1[t_{i-1}]
    unsigned long long *red = (unsigned long long *)(rsm + RL.red);
    uint64_t *full = (uint64_t *)(rsm + RL.bars);

    const int V = p.V, r = p.r, B = p.B;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int grid = gridDim.x;
    unsigned long long *keys = p.scratch;  // [B][grid]: best greedy key of every CTA per step
    const uint16_t *w1 = (const uint16_t *)p.w1;
    int lo, hi;
    quad_slice(V, lo, hi);
    const bool any = hi > lo;
    int box_w, nbox;
    rollout_box(V, grid, &box_w, &nbox);
    const int nblk = r / kRollKC;
    const int nstage = min(nblk, kResOnRows / kRollKC);
    const uint64_t pol = policy_evict_first();  // w2 is read once per launch
    int issued = 0, waited = 0;                 // thread 0's counts of w2 blocks

    if (t == 0) {
        s_fail = 0;
        for (int s = 0; s < kResSlots; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&s_tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    auto issue = [&](int j) {
        const int s = j % kResSlots;
        mbar_arrive_expect_tx(&full[s], RL.stage_bytes);
        uint8_t *dst = slots + (size_t)s * RL.stage_bytes;
        for (int b = 0; b < nbox; ++b)
            tma_load_2d_hint(dst + (size_t)b * kRollKC * box_w * 4, &tmW2, lo + b * box_w, kRollKC * j, &full[s], pol);
    };
    if (t == 0 && any) {
        tma_prefetch_desc(&tmW2);
        for (int j = 0; j < min(nblk, kResSlots); ++j) issue(j);
        issued = min(nblk, kResSlots);
    }
    // The key words start at zero (a published key never is); every CTA's
    // zeroing is done before any CTA publishes (split grid barrier below).
    for (int w = blockIdx.x * blockDim.x + t; w < B * grid; w += grid * blockDim.x) keys[w] = 0ull;
    int a = p.anchor[0];
    if (a < 0 || a >= V) {
        set_error(p.err, DSPARK_ERR_OOB);
        a = 0;
    }
    for (int k = t; k < r; k += blockDim.x) s_u[k] = w1[(size_t)a * r + k];
    __syncthreads();
    if (t == 32) s_gen = grid_arrive(p.ctl);

    // load: blocks 0 .. nstage-1 go to tensor memory / registers / s_sec
    const uint32_t taddr = s_tmem_base + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(128 * (warp >> 2));
    const int q0 = t, q1 = t + kSampThreads;
    const bool has0 = lo + q0 < hi, has1 = lo + q1 < hi;
    // word offsets of the pairs in a slot (row 0); lanes without a pair read word 0
    const int o0 = has0 ? (q0 / box_w) * kRollKC * box_w + q0 % box_w : 0;
    const int o1 = has1 ? (q1 / box_w) * kRollKC * box_w + q1 % box_w : 0;
    uint32_t wr[kResRegRows];
#pragma unroll
    for (int j = 0; j < kResRegRows; ++j) wr[j] = 0u;
    bool ok = true;
    for (int j = 0; j < nstage; ++j) {
        const int s = j % kResSlots;
        bool got = ok && any && mbar_wait_bounded(&full[s], (uint32_t)((j / kResSlots) & 1), &s_fail);
        got = __all_sync(0xffffffffu, got);
        if (got) {
            const uint32_t *w = (const uint32_t *)(slots + (size_t)s * RL.stage_bytes);
            if (j < kResTmemRows / kRollKC) {
                uint32_t v[16];
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) v[kk] = has0 ? w[kk * box_w + o0] : 0u;
                tmem_st16(taddr + 16u * (uint32_t)j, v);
            } else if (j == kResTmemRows / kRollKC) {
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) wr[kk] = has0 ? w[kk * box_w + o0] : 0u;
            } else {
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) wr[16 + kk] = has0 ? w[kk * box_w + o0] : 0u;
            }
            if (t < kResSec)
                for (int kk = 0; kk < 16; ++kk) s_sec[kRollKC * j + kk][t] = has1 ? w[kk * box_w + o1] : 0u;
            if (t == 0) waited = j + 1;
        }
        __syncthreads();
        ok = !s_fail;
        if (t == 0 && ok && any && j + kResSlots < nblk) {
            issue(j + kResSlots);
            issued = j + kResSlots + 1;
        }
    }
    tmem_st_wait();
    for (int j = nstage; j < nblk && ok && any; ++j) {
        if (!mbar_wait_bounded(&full[j % kResSlots], (uint32_t)((j / kResSlots) & 1), &s_fail)) break;
        if (t == 0) waited = j + 1;
    }
    if (t == 32 && !grid_wait(p.ctl, s_gen, p.err)) s_fail = 1;
    __syncthreads();
    ok = !s_fail;
    tc_fence_after();

    const bool two = __any_sync(0xffffffffu, has1);
    for (int i = 0; i < B && ok; ++i) {
        const float *zi = p.z + (size_t)i * V;
        float *elli = p.ell + (size_t)i * V;
        const float2 z0 = has0 ? *(const float2 *)(zi + 2 * (lo + q0)) : make_float2(0.f, 0.f);
        const float2 z1 = has1 ? *(const float2 *)(zi + 2 * (lo + q1)) : make_float2(0.f, 0.f);
        ResAcc acc = {0.f, 0.f, 0.f, 0.f};
        if (two)
            res_chain<true>(taddr, r, wr, slots, RL.stage_bytes, box_w, o0, o1, s_sec, t, s_u, acc);
        else
            res_chain<false>(taddr, r, wr, slots, RL.stage_bytes, box_w, o0, o1, s_sec, t, s_u, acc);
        unsigned long long best = 0ull;
        bool bad = false;
        if (has0) best = res_pair_out(acc.p0, acc.p1, z0, lo + q0, elli, bad);
        if (has1) best = max(best, res_pair_out(acc.s0, acc.s1, z1, lo + q1, elli, bad));
        if (bad) set_error(p.err, DSPARK_ERR_BAD_INPUT);
        best = warp_max_u64(best);
        if (lane == 0) red[warp] = best;
        __syncthreads();  // every warp's best is in red; s_u is no longer read this step
        if (warp == 0) {
            unsigned long long m = lane < kSampThreads / 32 ? red[lane] : 0ull;
            m = warp_max_u64(m);
            if (lane == 0) {
                st_relaxed_u64(&keys[(size_t)i * grid + blockIdx.x], m ? m : 1ull);
                if (m && i + 1 < B) prefetch_l2_bulk(w1 + (size_t)argmax_token(m) * r, (uint32_t)r * 2u);
            }
            // every CTA's key of step i: lane l reads CTAs l, l + 32, ... (keys are
            // never zero once published); short sleeps between rounds
            const unsigned long long *kp = keys + (size_t)i * grid;
            unsigned long long g = 0ull;
            uint32_t pending = 0u;
            for (int c = 0; lane + 32 * c < grid; ++c) pending |= 1u << c;
            const unsigned long long t0 = globaltimer(), limit = grid_wait_limit(p.ctl);
            while (__any_sync(0xffffffffu, pending != 0u)) {
                unsigned long long kv[kResGatherPerLane];
#pragma unroll
                for (int c = 0; c < kResGatherPerLane; ++c)
                    kv[c] = (pending >> c) & 1u ? ld_relaxed_u64(kp + lane + 32 * c) : 0ull;
#pragma unroll
                for (int c = 0; c < kResGatherPerLane; ++c)
                    if (kv[c]) {
                        g = max(g, kv[c]);
                        pending &= ~(1u << c);
                    }
                if (pending) {
                    if (s_fail || globaltimer() - t0 > limit) {
                        set_error(p.err, DSPARK_ERR_TIMEOUT);
                        s_fail = 1;
                        pending = 0u;
                    } else {
                        __nanosleep(20);
                    }
                }
            }
            g = warp_max_u64(g);
            if (lane == 0) {
                const int tok = argmax_token(g);
                s_tok = tok;
                if (blockIdx.x == 0) p.tokens[i] = tok;
            }
        }
        __syncthreads();  // the token of step i is in s_tok
        ok = !s_fail;
        if (ok && i + 1 < B) {
            const int tok = s_tok;
            for (int k4 = t; 4 * k4 < r; k4 += blockDim.x)
                *(uint2 *)(s_u + 4 * k4) = *(const uint2 *)(w1 + (size_t)tok * r + 4 * k4);
        }
        __syncthreads();  // s_u holds w1[t_i]
    }
    if (t == 0)
        for (int j = waited; j < issued; ++j) mbar_drain(&full[j % kResSlots], (uint32_t)((j / kResSlots) & 1));
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(s_tmem_base, 512);
    }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
// Dynamic shared memory of the rollout's w2 ring for a vocabulary and grid.
size_t rollout_ring_bytes(int V, int grid) {
    int box_w, nbox;
    rollout_box(V, grid, &box_w, &nbox);
    return (size_t)kRollStages * nbox * kRollKC * box_w * 4;
}

int sampling_max_grid(int num_sms, int V) {
    int a = 0;
    // the rollout gives each thread at most two vocabulary pairs of its CTA's slice
    if (4 * ((V / 8 + num_sms - 1) / num_sms) > 2 * kSampThreads) return 0;
    const size_t ring = rollout_ring_bytes(V, num_sms);
    if (cudaFuncSetAttribute(rollout_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ring) != cudaSuccess)
        return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, rollout_kernel, kSampThreads, ring) != cudaSuccess) return 0;
    return a >= 1 ? num_sms : 0;
}

// The resident greedy rollout needs r a multiple of 16 up to 256, at most
// kResSec secondary pairs per CTA, a key word per CTA read by one thread each,
// and its shared memory.
bool rollout_resident_setup(int V, int r, int grid) {
    if (r <= 0 || r % kRollKC != 0 || r > kResMaxRank || grid <= 0 || grid > 32 * kResGatherPerLane) return false;
    if (4 * ((V / 8 + grid - 1) / grid) > kSampThreads + kResSec) return false;
    const ResLayout RL(V, grid);
    int a = 0;
    if (cudaFuncSetAttribute(rollout_greedy_resident_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)RL.total) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, rollout_greedy_resident_kernel, kSampThreads, RL.total) !=
            cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return a >= 1;
}

cudaError_t launch_rollout(const CUtensorMap &w2_map, RolloutParams p, int grid, bool resident, cudaStream_t st) {
    carveout_max((const void *)rollout_greedy_resident_kernel);
    carveout_max((const void *)rollout_kernel);
    CUtensorMap tm = w2_map;
    void *args[] = {&tm, &p};
    if (resident && p.bs == 1 && p.draft_mode == DSPARK_GREEDY && ((uintptr_t)p.w1 & 15u) == 0)
        return cudaLaunchCooperativeKernel((void *)rollout_greedy_resident_kernel, dim3(grid), dim3(kSampThreads),
                                           args, ResLayout(p.V, grid).total, st);
    return cudaLaunchCooperativeKernel((void *)rollout_kernel, dim3(grid), dim3(kSampThreads), args,
                                       rollout_ring_bytes(p.V, grid), st);
}

}  // namespace ds
