// MLA attention of the draft block on the 5th-generation tensor core.
//
// Every query row of a sequence (block tokens x heads) attends to the same
// latent keys K_j = [c_kv,j || k_r,j] and values V_j = c_kv,j: the cache tokens
// 0..ctx-1 from the paged latent pool plus the block's own latents, with no
// mask (non-causal block) ("Kimi-K3-DSpark-NVFP4", Model Overview; the MLA
// absorbed form, "kimi-k3-dspark-gguf", Runtime status).
//
// A CTA owns 128 query rows, one range of 64-token chunks of the KV sequence
// (a split) and one 256-column half of the latent output (2 CTAs share a row
// tile and both compute its scores: tensor memory holds 256 output columns
// beside S and P, not 512). The Q tile is the A operand of S = Q K^T in two
// pieces: its first 320 dimensions stay in shared memory (five 128 x 64 boxes
// in the 128-byte swizzle), the last 256 in tensor memory. Tensor memory:
//   [0, 128)         Q dimensions 320..575, bf16 pairs
//   64 columns       S, fp32 (128 rows x 64 keys)
//   32 columns       P = exp2(S - m), bf16 pairs (A operand of O += P V)
//   DVP columns      O, fp32 (128 rows x the CTA's output columns)
// A chunk is one page of the pool (64 rows of DQK bf16), brought by TMA as
// DQK/64 boxes of 64 x 64 in the 128-byte swizzle: K-major for S, and the same
// bytes read MN-major give V for O. The softmax keeps a per-row reference max
// and rescales O only when a new maximum exceeds it by more than 2^8 (the
// result is the same: O and the row sum carry the same reference).
//
// The Q tile (128 rows x DQK) arrives by TMA: its shared-memory piece in its
// own region, its tensor-memory piece in the space of KV stage 1 (the first
// chunk goes to stage 0); the softmax warps move that piece to tensor memory,
// after which stage 1 takes KV chunks again. A stage's
// boxes outside the CTA's value columns are refilled as soon as the scores
// that read them are done, the value boxes once P V has read them.
//
// Roles (6 warps): warp 0 TMA producer; warp 1 MMA issuer and tensor-memory
// owner; warps 2-5 move Q, run the softmax (one thread per row) and write the
// split partial. All waits are bounded; a timeout raises DSPARK_ERR_TIMEOUT.
#include "internal.h"

namespace ds {

constexpr int kTcRows = 128;     // query rows per CTA (tcgen05 M)
constexpr int kTcKeys = 64;      // keys per chunk (one page)
constexpr int kTcStages = 2;     // KV chunk stages in shared memory
constexpr int kTcPgAhead = 8;    // page numbers the producer reads ahead of their chunks
constexpr float kTcRescaleLog2 = 8.f;
constexpr int kTcMaxChunks = 48;  // chunks per CTA at most when the grid fills the GPU anyway

template <int DQK, int DV>
struct TcCfg {
    static constexpr int kBoxes = (DQK + 63) / 64;         // 64-column boxes per key row
    static constexpr int kDQKP = kBoxes * 64;              // padded score width
    static constexpr int kDVP = DV < 256 ? DV : 256;       // output columns per CTA
    static constexpr int kParts = DV / kDVP;
    static constexpr int kBoxBytes = kTcKeys * 128;        // 64 rows x 128 B
    static constexpr int kTileBytes = kBoxes * kBoxBytes;
    static constexpr int kQBoxBytes = kTcRows * 128;       // 128 rows x 64 bf16
    static constexpr int kQsBoxes = 5;                     // Q boxes kept in shared memory (A from a descriptor)
    static constexpr int kQtBoxes = kBoxes - kQsBoxes;     // Q boxes in tensor memory
    static constexpr int kQsBytes = kQsBoxes * kQBoxBytes;
    static constexpr int kQtBytes = kQtBoxes * kQBoxBytes;
    static constexpr int kQCol = 0;
    static constexpr int kSCol = kQtBoxes * 32;
    static constexpr int kPCol = kSCol + 64;
    static constexpr int kOCol = kPCol + 32;
    static constexpr int kSmem = 1024 + kQsBytes + kTcStages * kTileBytes + 256;
    static_assert(kQtBytes <= (kTcStages - 1) * kTileBytes, "the tensor-memory piece of Q fits KV stage 1");
    static_assert(kOCol + kDVP <= 512, "tensor memory");
    static_assert(DV % kDVP == 0 && kDVP % 64 == 0, "output part: whole 64-column atoms");
    static_assert(kSmem <= 232448, "shared memory");
};

bool attention_tc_supported(int dqk, int dv) { return dqk == 576 && dv == 512; }

struct TcAttnParams {
    const __nv_bfloat16 *qt;      // [bs, R, DQK]
    int R;                        // rows per sequence
    int n_pages;
    const int32_t *page_table;    // [bs, max_pages]
    int max_pages;
    const int32_t *ctx_len;       // [bs]
    int max_ctx;
    int block;                    // the block's own latents: rows b * block .. of blk_kv
    int splits, cps;              // splits and chunks per split (chunk index space: ctx pages, then the block)
    float scale_log2;
    float *o_lat;                 // [bs, R, DV] (splits == 1)
    float *part_o;                // [bs, splits, R, DV]
    float *part_ml;               // [bs, splits, R, 2]
    int *err;
};

// 16 columns of the warp's lane quadrant without the completion wait (several
// loads share one tcgen05.wait::ld).
DS_DEVINL void tmem_ld16_nw(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
DS_DEVINL void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 2^x by the MUFU instruction (relative error about 2^-22, flushes denormals).
DS_DEVINL float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

DS_DEVINL uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// Warp-uniform bounded wait (every lane takes the same branch after it).
DS_DEVINL bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, abort));
}

// Shared memory keeps one CTA per SM; the launch bound of two only caps the
// registers, so the next kernel's CTAs can become resident beside this one.
template <int DQK, int DV>
__global__ void __launch_bounds__(192, 2)
    mla_attention_tc_kernel(const __grid_constant__ CUtensorMap tmPool, const __grid_constant__ CUtensorMap tmBlk,
                            const __grid_constant__ CUtensorMap tmQ, const TcAttnParams p) {
    using C = TcCfg<DQK, DV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sQs = smem;                   // Q dimensions 0 .. 64 * kQsBoxes - 1 (A operand from shared memory)
    uint8_t *sKV = smem + C::kQsBytes;
    uint64_t *bars = (uint64_t *)(sKV + kTcStages * C::kTileBytes);
    uint64_t *kv_full = bars, *kv_empty = bars + kTcStages;
    uint64_t *s_full = bars + 2 * kTcStages, *s_free = s_full + 1, *p_ready = s_full + 2, *pv_done = s_full + 3;
    uint64_t *q_ready = s_full + 4, *mma_done = s_full + 5, *q_full = s_full + 6;
    uint64_t *kv_kfree = s_full + 7;  // [kTcStages]: a stage's score-only boxes are free
    uint8_t *sQ = sKV + C::kTileBytes;  // Q's tensor-memory piece, in KV stage 1 until it is moved
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    __shared__ int s_pg[kTcPgAhead];  // page ring of the producer

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x / C::kParts, part = blockIdx.x % C::kParts;
    const int split = blockIdx.y, b = blockIdx.z;
    const int r0 = tile * kTcRows;

    pdl_trigger();
    {
        // a split past the end of this sequence's chunks: only its (max, sum) words
        // (empty), for the split combine; nothing else is set up
        int cx = p.ctx_len[b];
        if (cx < 0 || cx > p.max_ctx) cx = 0;
        if (split * p.cps > (cx + kTcKeys - 1) / kTcKeys) {
            if (p.splits > 1 && part == 0 && threadIdx.x >= 64) {
                pdl_wait();
                const int rr = r0 + (int)threadIdx.x - 64;
                if (rr < p.R)
                    *(float2 *)(p.part_ml + (((size_t)b * p.splits + split) * p.R + rr) * 2) = make_float2(-INFINITY, 0.f);
            }
            return;
        }
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < kTcStages; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
            mbar_init(&kv_kfree[i], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_free, 4);
        mbar_init(p_ready, 4);
        mbar_init(pv_done, 1);
        mbar_init(q_ready, 4);
        mbar_init(mma_done, 1);
        mbar_init(q_full, 1);
        s_abort = 0;
        fence_mbar_init();
    }
    if (threadIdx.x == 32) {
        tma_prefetch_desc(&tmPool);
        tma_prefetch_desc(&tmBlk);
        tma_prefetch_desc(&tmQ);
    }
    if (warp == 1) tmem_alloc(&s_tmem, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    // ctx_len, the page table and the page pool are inputs of the step: read
    // before the dependency wait (the queries and the block latents are not)
    int ctx = p.ctx_len[b];
    if (ctx < 0 || ctx > p.max_ctx) {
        if (threadIdx.x == 0) set_error(p.err, DSPARK_ERR_OOB);
        ctx = 0;
    }
    const int npages = (ctx + kTcKeys - 1) / kTcKeys;  // chunks [0, npages): pages; chunk npages: the block
    const int c_begin = split * p.cps;
    const int c_end = min(npages + 1, c_begin + p.cps);
    const int nch = c_end > c_begin ? c_end - c_begin : 0;
    int issued = 0;
    bool q_issued = false;

    if (warp != 0 || lane != 0) pdl_wait();
    if (warp == 0) {
        if (lane == 0) {
            // Boxes of KV chunk i into stage i % kTcStages: the value boxes of this
            // CTA's output part (vals) or all the others. Every chunk's expected
            // bytes are set with its first boxes.
            constexpr int kVb = C::kDVP / 64;  // value boxes of the part
            const int vb0 = part * kVb;
            auto load_boxes = [&](int i, int pg, bool vals) {
                const int st = i % kTcStages;
                if (!vals) mbar_arrive_expect_tx(&kv_full[st], (uint32_t)C::kTileBytes);
                uint8_t *dst = sKV + st * C::kTileBytes;
#pragma unroll 1
                for (int j = 0; j < C::kBoxes; ++j) {
                    if ((j >= vb0 && j < vb0 + kVb) != vals) continue;
                    if (pg >= 0)
                        tma_load_2d(dst + j * C::kBoxBytes, &tmPool, j * 64, pg * kTcKeys, &kv_full[st]);
                    else
                        tma_load_2d(dst + j * C::kBoxBytes, &tmBlk, j * 64, b * p.block, &kv_full[st]);
                }
            };
            // The first kTcPgAhead page numbers (inputs of the step) are requested in one
            // round of loads before the dependency wait; the Q tile goes first after it,
            // then chunk 0. A ring of page numbers keeps the loop free of waits on
            // page-table loads. (No bulk L2 prefetch of pages: it occupies the same copy
            // engine as the chunk loads and delays them.)
            int raw[kTcPgAhead];
#pragma unroll
            for (int i = 0; i < kTcPgAhead; ++i)
                raw[i] = (i < nch && c_begin + i < npages) ? __ldg(p.page_table + (size_t)b * p.max_pages + c_begin + i) : 0;
            pdl_wait();
            mbar_arrive_expect_tx(q_full, (uint32_t)(C::kQsBytes + C::kQtBytes));
#pragma unroll 1
            for (int j = 0; j < C::kBoxes; ++j) {
                uint8_t *dst = j < C::kQsBoxes ? sQs + j * C::kQBoxBytes : sQ + (j - C::kQsBoxes) * C::kQBoxBytes;
                tma_load_3d(dst, &tmQ, j * 64, r0, b, q_full);
            }
            q_issued = true;
#pragma unroll
            for (int i = 0; i < kTcPgAhead; ++i) {
                const bool is_page = i < nch && c_begin + i < npages;
                int pg = raw[i];
                if (is_page && (pg < 0 || pg >= p.n_pages)) {
                    set_error(p.err, DSPARK_ERR_OOB);
                    pg = 0;
                }
                s_pg[i] = is_page ? pg : -1;
            }
            if (nch > 0) {
                load_boxes(0, s_pg[0], false);
                load_boxes(0, s_pg[0], true);
                issued = 1;
            }
            // Stages 1.. hold the Q tile until the softmax warps have moved it. A stage's
            // boxes other than this part's values are free once the scores of the chunk
            // before have been computed, the value boxes once its P V has been; a chunk
            // whose first boxes are out always gets the rest, so it lands even after an abort.
            if (nch > 1 && mbar_wait_bounded(q_ready, 0, &s_abort)) {
                for (int i = 1; i < nch; ++i) {
                    const int st = i % kTcStages;
                    const uint32_t par = (uint32_t)((i / kTcStages - 1) & 1);
                    if (i >= kTcStages && !mbar_wait_bounded(&kv_kfree[st], par, &s_abort)) break;
                    const int pg = s_pg[i % kTcPgAhead];
                    load_boxes(i, pg, false);
                    if (i >= kTcStages) mbar_wait_bounded(&kv_empty[st], par, &s_abort);
                    load_boxes(i, pg, true);
                    issued = i + 1;
                    if (s_abort) break;
                    if (i + kTcPgAhead < nch) {
                        const int c = c_begin + i + kTcPgAhead;
                        int pn = -1;
                        if (c < npages) {
                            pn = p.page_table[(size_t)b * p.max_pages + c];
                            if (pn < 0 || pn >= p.n_pages) {
                                set_error(p.err, DSPARK_ERR_OOB);
                                pn = 0;
                            }
                        }
                        s_pg[i % kTcPgAhead] = pn;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(kTcRows, kTcKeys);
            constexpr uint32_t idPV = idesc_bf16_f32(kTcRows, C::kDVP) | kIdescBMajorMN;
            // S(i) = Q K_i^T once K_i has landed and the softmax has read S(i-1)
            auto issue_s = [&](int i) -> bool {
                const int st = i % kTcStages;
                if (!mbar_wait_bounded(&kv_full[st], (uint32_t)((i / kTcStages) & 1), &s_abort)) return false;
                if (i > 0 && !mbar_wait_bounded(s_free, (uint32_t)((i - 1) & 1), &s_abort)) return false;
                tc_fence_after();
                // Descriptors as one base plus immediates: the 14-bit start-address field
                // of box j, slice k is (base + 8 KB j + 32 B k) >> 4, never past 256 KB.
                // A short issue sequence keeps this thread ahead of the tensor pipe even
                // when a softmax warp shares its scheduler.
                const uint64_t bd0 = sdesc_k_sw128(smem_u32(sKV + st * C::kTileBytes));
                const uint64_t ad0 = sdesc_k_sw128(smem_u32(sQs));
#pragma unroll
                for (int kk = 0; kk < 4 * C::kQsBoxes; ++kk)
                    mma_bf16(tmem + C::kSCol, ad0 + (uint64_t)((kk >> 2) * (C::kQBoxBytes >> 4) + 2 * (kk & 3)),
                             bd0 + (uint64_t)((kk >> 2) * (C::kBoxBytes >> 4) + 2 * (kk & 3)), idS, kk > 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 4 * C::kQsBoxes; kk < C::kDQKP / 16; ++kk)
                    mma_bf16_tmem_a(tmem + C::kSCol, tmem + C::kQCol + 8 * (kk - 4 * C::kQsBoxes),
                                    bd0 + (uint64_t)((kk >> 2) * (C::kBoxBytes >> 4) + 2 * (kk & 3)), idS, 1u);
                mma_commit(s_full);
                mma_commit(&kv_kfree[st]);
                return true;
            };
            bool ok = nch == 0 || (mbar_wait_bounded(q_ready, 0, &s_abort) && issue_s(0));
            for (int i = 0; i < nch && ok; ++i) {
                const int st = i % kTcStages;
                // the next chunk's scores overlap this chunk's softmax
                if (i + 1 < nch && !issue_s(i + 1)) break;
                if (!mbar_wait_bounded(p_ready, (uint32_t)(i & 1), &s_abort)) break;
                tc_fence_after();
                const uint32_t base = smem_u32(sKV + st * C::kTileBytes);
                const uint32_t vbase = base + (part * C::kDVP / 64) * C::kBoxBytes;
#pragma unroll
                for (int kk = 0; kk < kTcKeys / 16; ++kk) {
                    const uint64_t vd = sdesc_mn_sw128(vbase + kk * 16 * 128, C::kBoxBytes, 1024);
                    mma_bf16_tmem_a(tmem + C::kOCol, tmem + C::kPCol + 8 * kk, vd, idPV, (i > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(pv_done);
                mma_commit(&kv_empty[st]);
            }
            mma_commit(mma_done);
            mbar_drain(mma_done, 0);
        }
        __syncwarp();
    } else {
        // warps 2..5: one query row per thread (TMEM lane quadrant = warp % 4)
        const int q4 = warp & 3;
        const int row = 32 * q4 + lane, r = r0 + row;
        const bool rv = r < p.R;
        const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
        // Q row's tensor-memory piece from the TMA tile (128-byte swizzle: 16-byte
        // piece j of row r sits at piece j ^ (r & 7)) into tensor memory as bf16
        // pairs; rows past R are zero
        bool ok = warp_wait(q_full, 0, &s_abort);
        if (ok) {
            const uint8_t *qrow = sQ + row * 128;
#pragma unroll 1
            for (int bq = 0; bq < C::kQtBoxes; ++bq) {
                uint32_t v[32];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint4 u = *(const uint4 *)(qrow + bq * C::kQBoxBytes + ((j ^ (row & 7)) << 4));
                    v[4 * j] = u.x;
                    v[4 * j + 1] = u.y;
                    v[4 * j + 2] = u.z;
                    v[4 * j + 3] = u.w;
                }
                tmem_st32(tl + C::kQCol + 32 * bq, v);
            }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && ok) mbar_arrive(q_ready);

        float m_ref = -INFINITY, lsum = 0.f;
        int done = 0;
        for (int i = 0; i < nch && ok; ++i) {
            const int c = c_begin + i;
            const int nvalid = c < npages ? min(kTcKeys, ctx - c * kTcKeys) : p.block;
            if (!warp_wait(s_full, (uint32_t)(i & 1), &s_abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[4][16];
#pragma unroll
            for (int t = 0; t < 4; ++t) tmem_ld16_nw(tl + C::kSCol + 16 * t, sr[t]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free);
            // the maximum of the raw scores, then scaled (the scale is positive and
            // rounding monotone, so this is the maximum of the scaled scores)
            const bool full = nvalid >= kTcKeys;
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int j = 0; j < 64; ++j)
                if (full || j < nvalid) mx4[j & 3] = fmaxf(mx4[j & 3], __uint_as_float(sr[j >> 4][j & 15]));
            const float mx = __fmul_rn(fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])), p.scale_log2);
            const float m_new = fmaxf(m_ref, mx);
            const bool rescale = (m_ref == -INFINITY) ? (m_new != -INFINITY) : (m_new > m_ref + kTcRescaleLog2);
            float corr = 1.f;
            if (rescale) {
                corr = (m_ref == -INFINITY) ? 0.f : exp2f(m_ref - m_new);
                m_ref = m_new;
            }
            uint32_t pk[32];
            float ls4[4] = {0.f, 0.f, 0.f, 0.f};
            const bool live = m_ref != -INFINITY;
            const float nm = live ? -m_ref : 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                // p = 2^(s * scale_log2 - m): one FMA and one MUFU ex2 per score
                float p0 = ex2_approx(__fmaf_rn(__uint_as_float(sr[(2 * j) >> 4][(2 * j) & 15]), p.scale_log2, nm));
                float p1 = ex2_approx(__fmaf_rn(__uint_as_float(sr[(2 * j + 1) >> 4][(2 * j + 1) & 15]), p.scale_log2, nm));
                if (!live || (!full && 2 * j >= nvalid)) p0 = 0.f;
                if (!live || (!full && 2 * j + 1 >= nvalid)) p1 = 0.f;
                ls4[j & 3] += p0 + p1;
                pk[j] = pack_bf16x2(p0, p1);
            }
            lsum = lsum * corr + ((ls4[0] + ls4[1]) + (ls4[2] + ls4[3]));
            // P and O are free once the previous chunk's P V has completed
            if (i > 0 && !warp_wait(pv_done, (uint32_t)((i - 1) & 1), &s_abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (i > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll 1
                for (int t = 0; t < C::kDVP / 16; ++t) {
                    float v[16];
                    uint32_t u[16];
                    tmem_ld16(tl + C::kOCol + 16 * t, v);
#pragma unroll
                    for (int j = 0; j < 16; ++j) u[j] = __float_as_uint(v[j] * corr);
                    tmem_st16(tl + C::kOCol + 16 * t, u);
                }
            }
            if (nvalid < kTcKeys) {
                // keys past the valid range: zero their value rows (this CTA's columns) so that
                // P = 0 meets finite values in P V
                uint8_t *tileb = sKV + (i % kTcStages) * C::kTileBytes + (part * C::kDVP / 64) * C::kBoxBytes;
                const int nrow = kTcKeys - nvalid, per_box = nrow * 8;  // 16-byte pieces per box
                for (int idx = threadIdx.x - 64; idx < per_box * (C::kDVP / 64); idx += 128) {
                    const int bx = idx / per_box, rem = idx % per_box;
                    *(uint4 *)(tileb + bx * C::kBoxBytes + (nvalid + rem / 8) * 128 + (rem % 8) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            tmem_st32(tl + C::kPCol, pk);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_ready);
            done = i + 1;
        }
        if (ok && done > 0 && !warp_wait(pv_done, (uint32_t)((done - 1) & 1), &s_abort)) ok = false;
        tc_fence_after();
        if (ok) {
            const size_t pr = ((size_t)b * p.splits + split) * p.R + (rv ? r : 0);
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            float *dst = p.splits == 1 ? p.o_lat + ((size_t)b * p.R + (rv ? r : 0)) * DV + part * C::kDVP
                                       : p.part_o + pr * DV + part * C::kDVP;
            // 64 columns per tensor-memory round trip
#pragma unroll
            for (int t = 0; t < C::kDVP / 64; ++t) {
                uint32_t u[4][16];
                if (done > 0) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) tmem_ld16_nw(tl + C::kOCol + 64 * t + 16 * k, u[k]);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
#pragma unroll
                        for (int j = 0; j < 16; ++j) u[k][j] = 0u;
                }
                if (rv) {
#pragma unroll
                    for (int j = 0; j < 64; j += 4) {
                        float4 o = make_float4(__uint_as_float(u[j >> 4][j & 15]), __uint_as_float(u[j >> 4][(j & 15) + 1]),
                                               __uint_as_float(u[j >> 4][(j & 15) + 2]),
                                               __uint_as_float(u[j >> 4][(j & 15) + 3]));
                        if (p.splits == 1) o = make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
                        *(float4 *)(dst + 64 * t + j) = o;
                    }
                }
            }
            if (rv && p.splits > 1 && part == 0) *(float2 *)(p.part_ml + pr * 2) = make_float2(m_ref, lsum);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (s_abort) {
        if (threadIdx.x == 0) set_error(p.err, DSPARK_ERR_TIMEOUT);
        if (warp == 0 && lane == 0) {
            // the last chunk issued to each stage lands before shared memory is released
            for (int i = issued - 1; i >= 0 && i >= issued - kTcStages; --i)
                mbar_drain(&kv_full[i % kTcStages], (uint32_t)((i / kTcStages) & 1));
            if (q_issued) mbar_drain(q_full, 0);
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Split plan of the tensor-core attention: about one wave of CTAs
// (row tiles x output parts x splits x sequences), whole chunks per split.
int attention_tc_splits(int R, int dv, int bs, int max_ctx, int num_sms, int *cps) {
    const int tiles = (R + kTcRows - 1) / kTcRows;
    const int parts = dv / (dv < 256 ? dv : 256);
    const int chunks = (max_ctx + kTcKeys - 1) / kTcKeys + 1;
    int s = num_sms / (tiles * parts * bs);
    if (s < 1) s = 1;
    // When the unsplit grid already fills the GPU (many sequences), the contexts
    // differ and each CTA would walk its own sequence's whole context: split so
    // that no CTA takes more than kTcMaxChunks chunks (short sequences leave
    // their upper splits empty; those CTAs exit at once).
    if (tiles * parts * bs >= num_sms) s = max(s, (chunks + kTcMaxChunks - 1) / kTcMaxChunks);
    if (s > chunks) s = chunks;
    if (s > 20) s = 20;  // the fused split combine takes up to 20 splits
    *cps = (chunks + s - 1) / s;
    return (chunks + *cps - 1) / *cps;
}

cudaError_t launch_attention_tc(const CUtensorMap &pool_map, const CUtensorMap &blk_map, const CUtensorMap &q_map,
                                const AttnParams &a,
                                int cps, int bs, int dqk, int dv, cudaStream_t st, bool combine) {
    if (!attention_tc_supported(dqk, dv)) return cudaErrorInvalidValue;
    using C = TcCfg<576, 512>;
    static bool attr = false;
    if (!attr) {
        const cudaError_t e = cudaFuncSetAttribute(mla_attention_tc_kernel<576, 512>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    TcAttnParams p;
    memset(&p, 0, sizeof(p));
    p.qt = a.qt;
    p.R = a.R;
    p.n_pages = a.n_pages;
    p.page_table = a.page_table;
    p.max_pages = a.max_pages;
    p.ctx_len = a.ctx_len;
    p.max_ctx = a.max_ctx;
    p.block = a.block;
    p.splits = a.splits;
    p.cps = cps;
    p.scale_log2 = a.scale_log2;
    p.o_lat = a.o_lat;
    p.part_o = a.part_o;
    p.part_ml = a.part_ml;
    p.err = a.err;
    const int tiles = (a.R + kTcRows - 1) / kTcRows;
    dim3 grid(tiles * C::kParts, a.splits, bs);
    cudaError_t e = launch_pdl(mla_attention_tc_kernel<576, 512>, grid, dim3(192), (size_t)C::kSmem, st, pool_map,
                               blk_map, q_map, p);
    if (e != cudaSuccess || a.splits == 1 || !combine) return e;
    return launch_attn_combine(a, bs, dv, st);
}

}  // namespace ds
