// Host side of libdspark: argument checks, workspace layout, TMA descriptors
// and the launch sequence of each entry point declared in include/dspark.h.
//
// Workspace layout: a 64 KB control block at offset 0 (error word, grid-barrier
// words, greedy-verify argmax keys, GEMM tile counters; all of it must be zero
// before the first call and the kernels return it to zero), then the GEMM split
// partials, the per-step activations and the sampling scratch.
#include <math.h>
#include <string.h>

#include <new>

#include "gemm.cuh"
#include "gemm_q.cuh"
#include "gemm_f8.cuh"
#include "internal.h"

using namespace ds;

namespace {

constexpr int kMaxBs = 32;
constexpr size_t kCtlBytes = 64 * 1024;
constexpr size_t kCtlErr = 0, kCtlSample = 64, kCtlKeys = 128, kCtlDraw = 8192, kCtlCounters = 16896;
constexpr int kMaxCounters = (int)((kCtlBytes - kCtlCounters) / sizeof(int));

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    }
    return fn;
}

// bf16 matrix [rows, cols] row-major, boxes of 64 columns x box_rows rows, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || !base) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 tensor [outer, rows, cols] read in boxes of 64 columns x box_rows rows of
// one outer index, 128-byte swizzle; rows past `rows` read as zero.
bool make_map_3d(CUtensorMap *m, const void *base, uint64_t outer, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || !base) return false;
    cuuint64_t dims[3] = {cols, rows, outer};
    cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// uint8 matrix [rows, cols_bytes] (quantised weights or their group scales).
bool encode_map_u32(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_inner,
                    uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || !base) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 4};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_u8(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols_bytes, uint32_t box_inner,
                 uint32_t box_rows, bool swizzle128) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || !base) return false;
    cuuint64_t dims[2] = {cols_bytes, rows};
    cuuint64_t strides[1] = {cols_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same bytes seen as 16-bit elements (cols_bytes / 2 of them per row): a
// 128-byte box row is 64 elements instead of 128, and the tensor-memory-access
// unit moves the tile in half the element steps. The shared-memory image of a
// tile is identical to the byte view's (the swizzle acts on 16-byte chunks).
bool make_map_u16view(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols_bytes, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || !base || (cols_bytes & 1u)) return false;
    cuuint64_t dims[2] = {cols_bytes / 2, rows};
    cuuint64_t strides[1] = {cols_bytes};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// A weight-only quantised matrix: raw-code and group-scale descriptors plus its
// output scales.
struct QMat {
    CUtensorMap data;    // raw codes as 16-bit elements, boxes of 128 bytes x 64 rows
    CUtensorMap scales;
    const float *rowscale;  // FP8 per-channel
    float gscale;           // NVFP4 per-tensor
};

bool make_qmat(QMat *q, const dspark_mat_t &m, int fmt, uint64_t rows, uint64_t cols) {
    if (fmt == DSPARK_FMT_FP8) {
        q->rowscale = (const float *)m.scale;
        q->gscale = 1.f;
        return make_map_u16view(&q->data, m.data, rows, cols, 64) &&
               make_map_u8(&q->scales, m.data, rows, cols, 128, 64, true);
    }
    q->rowscale = nullptr;
    if (fmt == DSPARK_FMT_MXFP4) {
        q->gscale = 1.f;
        return make_map_u16view(&q->data, m.data, rows, cols / 2, 64) &&
               make_map_u8(&q->scales, m.scale, rows, cols / 32, 16, 64, false);
    }
    q->gscale = m.global_scale;
    return make_map_u16view(&q->data, m.data, rows, cols / 2, 64) &&
           make_map_u8(&q->scales, m.scale, rows, cols / 16, 16, 64, false);
}

int bn_for(int M) {
    if (M <= 16) return 16;
    if (M <= 32) return 32;
    if (M <= 64) return 64;
    if (M <= 128) return 128;
    return 224;
}

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

struct Layout {
    size_t partials, hn, qkv, cq, q, qt, blk, olat, part_o, part_ml, ov, act, hout, scratch, app_hn, app_kv, total;
    int splits, tok_per_split;
    int tc, cps;                 // tensor-core attention and its chunks per split
};

}  // namespace

struct dspark_handle {
    dspark_geom_t g;
    dspark_weights_t w;
    int num_sms;
    int samp_grid;
    bool roll_resident;         // greedy one-sequence rollout with w2 on chip
    RopeTable rope;
    float scale_log2;
    CUtensorMap fc, lm_head;
    CUtensorMap w2;             // Markov w2 as uint32 pairs [rank, vocab / 2], rollout boxes
    CUtensorMap qkv_a[DSPARK_MAX_LAYERS], q_b[DSPARK_MAX_LAYERS], o[DSPARK_MAX_LAYERS], gate[DSPARK_MAX_LAYERS],
        up[DSPARK_MAX_LAYERS], down[DSPARK_MAX_LAYERS];
    // weight-only formats: the quantised matrices
    QMat qfc, qq_b[DSPARK_MAX_LAYERS], qo[DSPARK_MAX_LAYERS], qgate[DSPARK_MAX_LAYERS], qup[DSPARK_MAX_LAYERS],
        qdown[DSPARK_MAX_LAYERS];
    // activation descriptors, cached per (workspace, bs)
    const void *c_ws = nullptr;
    int c_bs = -1;
    CUtensorMap b_hn, b_cq, b_ov, b_act, b_hout;
    CUtensorMap b_blk;                       // block latents, tensor-core attention
    CUtensorMap b_qt;                        // absorbed queries [bs, block * heads, kvd], tensor-core attention
    CUtensorMap kva[DSPARK_MAX_LAYERS];      // kv_a rows of the fused q_a || kv_a weights
    const void *c_app_ws = nullptr;
    int c_app_rows = -1;
    CUtensorMap b_app;                       // normed context features of appended tokens
    const void *c_pool[DSPARK_MAX_LAYERS] = {};
    int c_npages[DSPARK_MAX_LAYERS] = {};
    CUtensorMap pool_map[DSPARK_MAX_LAYERS]; // per-layer page pools, tensor-core attention
    const void *c_aux = nullptr;
    int c_aux_bs = -1;
    CUtensorMap b_aux;
};

namespace {

// Split of the KV sequence for attention: enough CTAs to cover the SMs, at
// least 4 chunks of 64 tokens per split.
int attn_splits(const dspark_handle *h, int bs, int max_ctx, int *tok_per_split) {
    const dspark_geom_t &g = h->g;
    const int R = g.block * g.n_heads;
    const int qtiles = (R + 63) / 64;
    const int chunks = (max_ctx + g.block + 63) / 64;
    const int want = (h->num_sms + qtiles * bs - 1) / (qtiles * bs);
    const int cap = (chunks + 3) / 4;
    int s = want < cap ? want : cap;
    if (s < 1) s = 1;
    if (s > 64) s = 64;
    const int cps = (chunks + s - 1) / s;
    *tok_per_split = cps * 64;
    return (chunks + cps - 1) / cps;
}

Layout layout_for(const dspark_handle *h, int bs, int max_ctx) {
    const dspark_geom_t &g = h->g;
    Layout L;
    const size_t M = (size_t)g.block * bs;
    const size_t kvd = g.kv_lora + g.d_rope;
    const size_t R = (size_t)g.block * g.n_heads;
    L.tc = attention_tc_supported((int)kvd, g.kv_lora) ? 1 : 0;
    L.cps = 0;
    L.tok_per_split = 0;
    L.splits = L.tc ? attention_tc_splits((int)R, g.kv_lora, bs, max_ctx, h->num_sms, &L.cps)
                    : attn_splits(h, bs, max_ctx, &L.tok_per_split);
    size_t off = kCtlBytes;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = up256(off + bytes);
        return o;
    };
    L.partials = take((size_t)2 * h->num_sms * 128 * bn_for((int)M) * 4);
    L.hn = take(M * g.hidden * 2);
    L.qkv = take(M * (g.q_lora + kvd) * 4);
    L.cq = take(M * g.q_lora * 2);
    L.q = take(M * g.n_heads * (g.d_nope + g.d_rope) * 4);
    L.qt = take(M * g.n_heads * kvd * 2);
    L.blk = take(M * kvd * 2);
    L.olat = take(M * g.n_heads * g.kv_lora * 4);
    const size_t np = L.splits > 1 ? (size_t)bs * L.splits * R : 0;
    L.part_o = take(np * g.kv_lora * 4);
    L.part_ml = take(np * 2 * 4);
    L.ov = take(M * g.n_heads * g.d_v * 2);
    L.act = take(M * g.inter * 2);
    L.hout = take(M * g.hidden * 2);
    const size_t sw1 = rollout_scratch_words(bs, g.block, h->num_sms);
    const size_t sw2 = verify_scratch_words(bs, g.block, h->num_sms);
    L.scratch = take((sw1 > sw2 ? sw1 : sw2) * 8);
    // latent-cache append: up to block + 1 new tokens per sequence
    const size_t A = (size_t)(g.block + 1) * bs;
    L.app_hn = take((size_t)g.n_layers * A * g.hidden * 2);
    L.app_kv = take((size_t)g.n_layers * A * kvd * 4);
    L.total = off;
    return L;
}

// Grid of a weight GEMM: about `per` units per CTA, at most one CTA per SM. A
// pending output (the consumer sums the split partials) needs every CTA's range
// within one tile (grid >= tiles) and few CTAs per tile; otherwise, or when no
// pending output is asked for, the GEMM reduces in place (pend->part = nullptr).
void gemm_grid(GemmParams &p, int per, int num_sms, int BN, GemmPending *pend) {
    long long grid = p.units / per;
    if (grid > num_sms) grid = num_sms;
    if (grid < 1) grid = 1;
    if (pend) {
        memset(pend, 0, sizeof(*pend));
        const long long g2 = grid < p.tiles ? p.tiles : grid;
        if (!p.paired && p.tiles <= num_sms && g2 <= p.units && p.units * g2 < (1ll << 31)) {
            grid = g2;
            p.epi = EPI_PENDING;
            pend->part = p.partials;
            pend->units = (int)p.units;
            pend->grid = (int)grid;
            pend->KB = p.KB;
            pend->BN = BN;
        }
    }
    p.grid = (int)grid;
    // pairwise reduction: every CTA's range covers at least one tile
    p.pair_red = (p.epi != EPI_PENDING && BN <= 32 && p.units / p.grid >= p.KB) ? 1 : 0;
}

template <int BN>
cudaError_t gemm_t(const CUtensorMap &A, const CUtensorMap &A2, const CUtensorMap &B, GemmParams p, int num_sms,
                   cudaStream_t st, GemmPending *pend) {
    using C = GemmCfg<BN>;
    static bool attr = false;
    if (!attr) {
        const cudaError_t e = cudaFuncSetAttribute(gemm_swapab_kernel<BN>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    gemm_grid(p, 4, num_sms, BN, pend);
    return launch_pdl(gemm_swapab_kernel<BN>, dim3(p.grid), dim3(192), (size_t)C::kSmemBytes, st, A, A2, B, p);
}

cudaError_t gemm(const dspark_handle *h, const CUtensorMap &A, const CUtensorMap *A2, const CUtensorMap &B, int n_out,
                 int K, int M, int epi, float *out_f32, __nv_bfloat16 *out_bf16, int ldo, void *ws, cudaStream_t st,
                 const L2Prefetch *pf = nullptr, GemmPending *pend = nullptr) {
    GemmParams p;
    memset(&p, 0, sizeof(p));
    if (pf) p.pf = *pf;
    p.n_out = n_out;
    p.K = K;
    p.M = M;
    p.paired = A2 != nullptr;
    p.epi = epi;
    p.out_f32 = out_f32;
    p.out_bf16 = out_bf16;
    p.ldo = ldo;
    p.KB = (K + 63) / 64;
    p.tiles = p.paired ? (n_out + 63) / 64 : (n_out + 127) / 128;
    p.units = (long long)p.tiles * p.KB;
    if (p.tiles > kMaxCounters) return cudaErrorInvalidValue;
    p.counters = (int *)((char *)ws + kCtlCounters);
    p.err = (int *)((char *)ws + kCtlErr);
    p.partials = (float *)((char *)ws + kCtlBytes);  // first region after the control block
    const CUtensorMap &a2 = A2 ? *A2 : A;
    switch (bn_for(M)) {
        case 16: return gemm_t<16>(A, a2, B, p, h->num_sms, st, pend);
        case 32: return gemm_t<32>(A, a2, B, p, h->num_sms, st, pend);
        case 64: return gemm_t<64>(A, a2, B, p, h->num_sms, st, pend);
        case 128: return gemm_t<128>(A, a2, B, p, h->num_sms, st, pend);
        default: return gemm_t<224>(A, a2, B, p, h->num_sms, st, pend);
    }
}

template <int BN>
cudaError_t gemm_layers_t(const GemmMaps &maps, const CUtensorMap &B, GemmParams p, int num_sms, cudaStream_t st) {
    using C = GemmCfg<BN>;
    static bool attr = false;
    if (!attr) {
        const cudaError_t e =
            cudaFuncSetAttribute(gemm_layers_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    gemm_grid(p, 4, num_sms, BN, nullptr);
    p.pair_red = 0;
    return launch_pdl(gemm_layers_kernel<BN>, dim3(p.grid), dim3(192), (size_t)C::kSmemBytes, st, B, p, maps);
}

// L matrices of n_out x K (maps.m[0..L)) against activation rows l * M .. of B:
// out[l] = W_l x_l, [M][n_out] fp32 each, one after another.
cudaError_t gemm_layers(const dspark_handle *h, const GemmMaps &maps, int L, const CUtensorMap &B, int n_out, int K,
                        int M, float *out, void *ws, cudaStream_t st) {
    GemmParams p;
    memset(&p, 0, sizeof(p));
    p.n_out = n_out;
    p.K = K;
    p.M = M;
    p.epi = EPI_STORE;
    p.out_f32 = out;
    p.ldo = n_out;
    p.KB = (K + 63) / 64;
    p.tpl = (n_out + 127) / 128;
    p.brows = M;
    p.lay_stride = (long long)M * n_out;
    p.tiles = L * p.tpl;
    p.units = (long long)p.tiles * p.KB;
    if (p.tiles > kMaxCounters) return cudaErrorInvalidValue;
    p.counters = (int *)((char *)ws + kCtlCounters);
    p.err = (int *)((char *)ws + kCtlErr);
    p.partials = (float *)((char *)ws + kCtlBytes);
    switch (bn_for(M)) {
        case 16: return gemm_layers_t<16>(maps, B, p, h->num_sms, st);
        case 32: return gemm_layers_t<32>(maps, B, p, h->num_sms, st);
        case 64: return gemm_layers_t<64>(maps, B, p, h->num_sms, st);
        case 128: return gemm_layers_t<128>(maps, B, p, h->num_sms, st);
        default: return gemm_layers_t<224>(maps, B, p, h->num_sms, st);
    }
}

template <int BN, int FMT>
cudaError_t gemm_q_t(const QMat &A, const QMat *A2, const CUtensorMap &B, GemmParams p, int num_sms,
                     cudaStream_t st, GemmPending *pend) {
    using C = GemmQCfg<BN, FMT>;
    static bool attr = false;
    if (!attr) {
        const cudaError_t e =
            cudaFuncSetAttribute(gemm_q_kernel<BN, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    p.KB = (p.K + C::kKR - 1) / C::kKR;
    p.units = (long long)p.tiles * p.KB;
    gemm_grid(p, 2, num_sms, BN, pend);
    p.qscale = A.rowscale;
    p.qscale2 = A2 ? A2->rowscale : nullptr;
    p.gscale = A.gscale;
    p.gscale2 = A2 ? A2->gscale : 1.f;
    const QMat &a2 = A2 ? *A2 : A;
    return launch_pdl(gemm_q_kernel<BN, FMT>, dim3(p.grid), dim3(C::kThreads), (size_t)C::kSmemBytes, st, A.data,
                      a2.data, A.scales, a2.scales, B, p);
}

template <int MR>
cudaError_t gemm_f8_t(const QMat &A, const QMat *A2, GemmParams p, int num_sms, cudaStream_t st, GemmPending *pend) {
    using C = GemmF8Cfg<MR>;
    static bool attr = false;
    if (!attr) {
        const cudaError_t e =
            cudaFuncSetAttribute(gemm_f8_kernel<MR>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    p.KB = (p.K + 127) / 128;
    p.units = (long long)p.tiles * p.KB;
    gemm_grid(p, 2, num_sms, MR, pend);
    p.pair_red = 0;
    p.qscale = A.rowscale;
    p.qscale2 = A2 ? A2->rowscale : nullptr;
    const QMat &a2 = A2 ? *A2 : A;
    return launch_pdl(gemm_f8_kernel<MR>, dim3(p.grid), dim3(C::kThreads), (size_t)C::kSmemBytes, st, A.data, a2.data,
                      p);
}

cudaError_t gemm_q(const dspark_handle *h, const QMat &A, const QMat *A2, const CUtensorMap &B, const void *xact,
                   int n_out, int K, int M,
                   int epi, float *out_f32, __nv_bfloat16 *out_bf16, int ldo, void *ws, cudaStream_t st,
                   GemmPending *pend = nullptr, const L2Prefetch *pf = nullptr) {
    GemmParams p;
    memset(&p, 0, sizeof(p));
    if (pf) p.pf = *pf;
    p.n_out = n_out;
    p.K = K;
    p.M = M;
    p.paired = A2 != nullptr;
    p.epi = epi;
    p.out_f32 = out_f32;
    p.out_bf16 = out_bf16;
    p.ldo = ldo;
    p.tiles = p.paired ? (n_out + 63) / 64 : (n_out + 127) / 128;
    if (p.tiles > kMaxCounters) return cudaErrorInvalidValue;
    p.counters = (int *)((char *)ws + kCtlCounters);
    p.err = (int *)((char *)ws + kCtlErr);
    p.partials = (float *)((char *)ws + kCtlBytes);
    p.act = (const __nv_bfloat16 *)xact;
    const int bn = bn_for(M);
    if (h->g.weight_format == DSPARK_FMT_FP8) {
        // up to 32 activation rows: E4M3 weights straight into the tensor core
        if (M <= 8) return gemm_f8_t<8>(A, A2, p, h->num_sms, st, pend);
        if (bn == 16) return gemm_f8_t<16>(A, A2, p, h->num_sms, st, pend);
        if (bn == 32) return gemm_f8_t<32>(A, A2, p, h->num_sms, st, pend);
        if (bn == 64) return gemm_q_t<64, DSPARK_FMT_FP8>(A, A2, B, p, h->num_sms, st, pend);
    } else if (h->g.weight_format == DSPARK_FMT_NVFP4) {
        if (bn == 16) return gemm_q_t<16, DSPARK_FMT_NVFP4>(A, A2, B, p, h->num_sms, st, pend);
        if (bn == 32) return gemm_q_t<32, DSPARK_FMT_NVFP4>(A, A2, B, p, h->num_sms, st, pend);
        if (bn == 64) return gemm_q_t<64, DSPARK_FMT_NVFP4>(A, A2, B, p, h->num_sms, st, pend);
    } else {
        if (bn == 16) return gemm_q_t<16, DSPARK_FMT_MXFP4>(A, A2, B, p, h->num_sms, st, pend);
        if (bn == 32) return gemm_q_t<32, DSPARK_FMT_MXFP4>(A, A2, B, p, h->num_sms, st, pend);
        if (bn == 64) return gemm_q_t<64, DSPARK_FMT_MXFP4>(A, A2, B, p, h->num_sms, st, pend);
    }
    return cudaErrorInvalidValue;
}

// The bytes of a (possibly quantised) weight matrix of rows x cols, as L2
// prefetch ranges: data, then the scales of the weight-only formats.
L2Prefetch mat_prefetch(const dspark_mat_t &m, int fmt, uint64_t rows, uint64_t cols) {
    L2Prefetch pf;
    memset(&pf, 0, sizeof(pf));
    uint64_t db = rows * cols * 2, sb = 0;
    if (fmt == DSPARK_FMT_FP8) {
        db = rows * cols;
        sb = rows * 4;
    } else if (fmt == DSPARK_FMT_NVFP4) {
        db = rows * cols / 2;
        sb = rows * cols / 16;
    } else if (fmt == DSPARK_FMT_MXFP4) {
        db = rows * cols / 2;
        sb = rows * cols / 32;
    }
    if (m.data && aligned16(m.data)) {
        pf.ptr[0] = (const uint8_t *)m.data;
        pf.bytes[0] = db & ~15ull;
    }
    if (sb && m.scale && aligned16(m.scale)) {
        pf.ptr[1] = (const uint8_t *)m.scale;
        pf.bytes[1] = sb & ~15ull;
    }
    return pf;
}

dspark_status check_geom(const dspark_geom_t *g) {
    if (g->hidden <= 0 || g->n_aux <= 0 || g->n_layers <= 0 || g->n_layers > DSPARK_MAX_LAYERS || g->n_heads <= 0 ||
        g->q_lora <= 0 || g->kv_lora <= 0 || g->d_nope <= 0 || g->d_rope <= 0 || g->d_v <= 0 || g->inter <= 0 ||
        g->vocab <= 0 || g->rank <= 0 || g->block <= 0)
        return DSPARK_ERR_SHAPE;
    if (g->hidden % 64 || g->q_lora % 64 || g->kv_lora % 64 || g->inter % 64 || (g->n_heads * g->d_v) % 64 ||
        g->d_rope % 4 || g->d_rope > 128 || g->vocab % 8 || g->vocab >= (1 << 18) || g->rank > 256 ||
        g->block > 16 || g->page_size != 64 || g->d_nope > 256 || g->d_nope % 16 || g->d_v % 16 ||
        g->kv_lora > 512 || g->q_lora + g->kv_lora > 8192)
        return DSPARK_ERR_UNSUPPORTED;
    if (!attention_supported(g->kv_lora + g->d_rope, g->kv_lora)) return DSPARK_ERR_UNSUPPORTED;
    if (g->weight_format != DSPARK_FMT_BF16 && g->weight_format != DSPARK_FMT_FP8 &&
        g->weight_format != DSPARK_FMT_NVFP4 && g->weight_format != DSPARK_FMT_MXFP4)
        return DSPARK_ERR_UNSUPPORTED;
    // MXFP4 stages cover 512 inputs (16 scale bytes per row: whole 16-byte TMA boxes)
    if (g->weight_format == DSPARK_FMT_MXFP4 &&
        ((g->n_aux * g->hidden) % 512 || g->q_lora % 512 || (g->n_heads * g->d_v) % 512 || g->hidden % 512 ||
         g->inter % 512))
        return DSPARK_ERR_UNSUPPORTED;
    // NVFP4 group-scale rows (in / 16 bytes) must be whole 16-byte TMA strides
    if (g->weight_format == DSPARK_FMT_NVFP4 &&
        ((g->n_aux * g->hidden) % 256 || g->q_lora % 256 || (g->n_heads * g->d_v) % 256 || g->hidden % 256 ||
         g->inter % 256))
        return DSPARK_ERR_UNSUPPORTED;
    if (!(g->eps >= 0.f) || !(g->rope_theta > 0.f)) return DSPARK_ERR_SHAPE;
    if ((g->vocab + 127) / 128 > kMaxCounters) return DSPARK_ERR_UNSUPPORTED;
    return DSPARK_OK;
}

#define REQ(p)                                      \
    do {                                            \
        if (!(p)) return DSPARK_ERR_NULL;           \
        if (!aligned16(p)) return DSPARK_ERR_ALIGN; \
    } while (0)

dspark_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA; }

bool bad_sampling(float T, float top_p) { return !(T > 0.f) || !isfinite(T) || !(top_p > 0.f) || !(top_p <= 1.f); }

dspark_status check_ws(const dspark_handle_t *h, void *ws, size_t ws_bytes, int bs, int max_ctx) {
    if (h->g.weight_format != DSPARK_FMT_BF16 && h->g.block * bs > 64) return DSPARK_ERR_UNSUPPORTED;
    if (!ws) return DSPARK_ERR_WORKSPACE;
    if (!aligned16(ws)) return DSPARK_ERR_ALIGN;
    if (ws_bytes < layout_for(h, bs, max_ctx).total) return DSPARK_ERR_WORKSPACE;
    return DSPARK_OK;
}

}  // namespace

namespace ds {
const dspark_geom_t *handle_geom(const dspark_handle_t *h) { return &h->g; }
int handle_num_sms(const dspark_handle_t *h) { return h->num_sms; }
const CUtensorMap *handle_fc_map(const dspark_handle_t *h) { return &h->fc; }
bool encode_bf16_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    return make_map(m, base, rows, cols, box_rows);
}
}  // namespace ds

extern "C" {

const char *dspark_status_str(dspark_status s) {
    switch (s) {
        case DSPARK_OK: return "ok";
        case DSPARK_ERR_NULL: return "null pointer";
        case DSPARK_ERR_ALIGN: return "pointer not 16-byte aligned";
        case DSPARK_ERR_SHAPE: return "size or sampling control out of range";
        case DSPARK_ERR_UNSUPPORTED: return "unsupported geometry or format";
        case DSPARK_ERR_CUDA: return "CUDA call failed";
        case DSPARK_ERR_WORKSPACE: return "workspace missing or too small";
        case DSPARK_ERR_TIMEOUT: return "bounded device wait expired";
        case DSPARK_ERR_BAD_INPUT: return "non-finite value in the input";
        case DSPARK_ERR_OOB: return "page id, token id or context length out of range";
    }
    return "unknown status";
}

dspark_status dspark_create(const dspark_geom_t *geom, const dspark_weights_t *wts, dspark_handle_t **out) {
    if (!geom || !wts || !out) return DSPARK_ERR_NULL;
    *out = nullptr;
    const dspark_status st = check_geom(geom);
    if (st != DSPARK_OK) return st;
    const dspark_geom_t &g = *geom;
    REQ(wts->w_fc.data);
    REQ(wts->final_norm);
    REQ(wts->w_lm);
    REQ(wts->markov_w1);
    REQ(wts->markov_w2);
    REQ(wts->w_conf);
    for (int l = 0; l < g.n_layers; ++l) {
        const dspark_layer_weights_t &L = wts->layers[l];
        REQ(L.attn_norm);
        REQ(L.w_qkv_a);
        REQ(L.q_a_norm);
        REQ(L.kv_a_norm);
        REQ(L.w_q_b.data);
        REQ(L.w_kv_b);
        REQ(L.w_o.data);
        REQ(L.mlp_norm);
        REQ(L.w_gate.data);
        REQ(L.w_up.data);
        REQ(L.w_down.data);
    }
    if (g.weight_format != DSPARK_FMT_BF16) {
        auto req_mat = [&](const dspark_mat_t &m) -> dspark_status {
            if (!m.scale) return DSPARK_ERR_NULL;
            if (!aligned16(m.scale)) return DSPARK_ERR_ALIGN;
            if (g.weight_format == DSPARK_FMT_NVFP4 && !(m.global_scale > 0.f)) return DSPARK_ERR_SHAPE;
            return DSPARK_OK;
        };
        dspark_status q = req_mat(wts->w_fc);
        for (int l = 0; l < g.n_layers && q == DSPARK_OK; ++l) {
            const dspark_layer_weights_t &L = wts->layers[l];
            for (const dspark_mat_t *m : {&L.w_q_b, &L.w_o, &L.w_gate, &L.w_up, &L.w_down})
                if (q == DSPARK_OK) q = req_mat(*m);
        }
        if (q != DSPARK_OK) return q;
    }
    if (!encode_fn()) return DSPARK_ERR_CUDA;
    dspark_handle *h = new (std::nothrow) dspark_handle();
    if (!h) return DSPARK_ERR_CUDA;
    h->g = g;
    h->w = *wts;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        delete h;
        return DSPARK_ERR_CUDA;
    }
    h->samp_grid = sampling_max_grid(h->num_sms, g.vocab);
    if (h->samp_grid <= 0) {
        delete h;
        return DSPARK_ERR_CUDA;
    }
    h->roll_resident = rollout_resident_setup(g.vocab, g.rank, h->samp_grid);
    if (!verify_setup(g.vocab)) {
        delete h;
        return DSPARK_ERR_CUDA;
    }
    // RoPE frequencies; YaRN "NTK-by-parts" ramp when yarn_factor > 1
    memset(&h->rope, 0, sizeof(h->rope));
    for (int j = 0; j < g.d_rope / 2; ++j) {
        double inv = pow((double)g.rope_theta, -2.0 * j / g.d_rope);
        if (g.yarn_factor > 1.f) {
            const double rot = (double)g.yarn_orig_ctx * inv / (2.0 * M_PI);
            double gamma = (rot - g.yarn_alpha) / ((double)g.yarn_beta - g.yarn_alpha);
            gamma = gamma < 0 ? 0 : (gamma > 1 ? 1 : gamma);
            inv = (1.0 - gamma) * inv / g.yarn_factor + gamma * inv;
        }
        h->rope.inv_freq[j] = inv;
    }
    double mscale2 = 1.0;
    if (g.yarn_factor > 1.f) {
        const double m = 0.1 * log((double)g.yarn_factor) + 1.0;
        mscale2 = m * m;
    }
    h->scale_log2 = (float)(mscale2 / sqrt((double)(g.d_nope + g.d_rope)) * 1.4426950408889634);
    const bool bf16w = g.weight_format == DSPARK_FMT_BF16;
    int roll_box_w = 0, roll_nbox = 0;
    rollout_box(g.vocab, h->samp_grid, &roll_box_w, &roll_nbox);
    bool ok = encode_map_u32(&h->w2, wts->markov_w2, g.rank, (uint64_t)g.vocab / 2, (uint32_t)roll_box_w, 16) &&
              make_map(&h->lm_head, wts->w_lm, g.vocab, g.hidden, 64) &&
              (!bf16w || make_map(&h->fc, wts->w_fc.data, g.hidden, (uint64_t)g.n_aux * g.hidden, 64));
    const int kvd = g.kv_lora + g.d_rope;
    for (int l = 0; l < g.n_layers && ok; ++l) {
        const dspark_layer_weights_t &L = wts->layers[l];
        ok = make_map(&h->qkv_a[l], L.w_qkv_a, g.q_lora + kvd, g.hidden, 64) &&
             make_map(&h->kva[l], (const char *)L.w_qkv_a + (size_t)g.q_lora * g.hidden * 2, kvd, g.hidden, 64);
        if (ok && bf16w)
            ok = make_map(&h->q_b[l], L.w_q_b.data, (uint64_t)g.n_heads * (g.d_nope + g.d_rope), g.q_lora, 64) &&
                 make_map(&h->o[l], L.w_o.data, g.hidden, (uint64_t)g.n_heads * g.d_v, 64) &&
                 make_map(&h->gate[l], L.w_gate.data, g.inter, g.hidden, 64) &&
                 make_map(&h->up[l], L.w_up.data, g.inter, g.hidden, 64) &&
                 make_map(&h->down[l], L.w_down.data, g.hidden, g.inter, 64);
    }
    const int fmt = g.weight_format;
    if (ok && fmt != DSPARK_FMT_BF16) {
        ok = make_qmat(&h->qfc, wts->w_fc, fmt, g.hidden, (uint64_t)g.n_aux * g.hidden);
        for (int l = 0; l < g.n_layers && ok; ++l) {
            const dspark_layer_weights_t &L = wts->layers[l];
            ok = make_qmat(&h->qq_b[l], L.w_q_b, fmt, (uint64_t)g.n_heads * (g.d_nope + g.d_rope), g.q_lora) &&
                 make_qmat(&h->qo[l], L.w_o, fmt, g.hidden, (uint64_t)g.n_heads * g.d_v) &&
                 make_qmat(&h->qgate[l], L.w_gate, fmt, g.inter, g.hidden) &&
                 make_qmat(&h->qup[l], L.w_up, fmt, g.inter, g.hidden) &&
                 make_qmat(&h->qdown[l], L.w_down, fmt, g.hidden, g.inter);
        }
    }
    if (!ok) {
        delete h;
        return DSPARK_ERR_CUDA;
    }
    *out = h;
    return DSPARK_OK;
}

void dspark_destroy(dspark_handle_t *h) { delete h; }

size_t dspark_workspace_bytes(const dspark_handle_t *h, int max_bs, int max_ctx) {
    if (!h || max_bs <= 0 || max_bs > kMaxBs || max_ctx < 0) return 0;
    return layout_for(h, max_bs, max_ctx).total;
}

dspark_status dspark_fuse_ctx(dspark_handle_t *h, const void *aux, float *x, int bs, void *ws, size_t ws_bytes,
                              void *stream) {
    if (!h) return DSPARK_ERR_NULL;
    if (bs <= 0 || bs > kMaxBs) return DSPARK_ERR_SHAPE;
    REQ(aux);
    REQ(x);
    const dspark_status st = check_ws(h, ws, ws_bytes, bs, 0);
    if (st) return st;
    const dspark_geom_t &g = h->g;
    const int M = g.block * bs;
    if (h->c_aux != aux || h->c_aux_bs != bs) {
        if (!make_map(&h->b_aux, aux, M, (uint64_t)g.n_aux * g.hidden, bn_for(M))) return DSPARK_ERR_CUDA;
        h->c_aux = aux;
        h->c_aux_bs = bs;
    }
    if (g.weight_format != DSPARK_FMT_BF16)
        return cuda_status(gemm_q(h, h->qfc, nullptr, h->b_aux, aux, g.hidden, g.n_aux * g.hidden, M, EPI_STORE, x, nullptr,
                                  g.hidden, ws, (cudaStream_t)stream));
    return cuda_status(gemm(h, h->fc, nullptr, h->b_aux, g.hidden, g.n_aux * g.hidden, M, EPI_STORE, x, nullptr,
                            g.hidden, ws, (cudaStream_t)stream));
}

dspark_status dspark_draft_block(dspark_handle_t *h, float *x, const dspark_kv_t *kv, float *h_out, float *z, int bs,
                                 void *ws, size_t ws_bytes, void *stream) {
    if (!h || !kv) return DSPARK_ERR_NULL;
    if (bs <= 0 || bs > kMaxBs || kv->max_ctx < 0 || kv->n_pages <= 0 || kv->max_pages <= 0) return DSPARK_ERR_SHAPE;
    if ((long long)kv->max_pages * h->g.page_size < kv->max_ctx) return DSPARK_ERR_SHAPE;
    REQ(x);
    REQ(h_out);
    REQ(z);
    REQ(kv->page_table);
    REQ(kv->ctx_len);
    const dspark_geom_t &g = h->g;
    for (int l = 0; l < g.n_layers; ++l) REQ(kv->pools[l]);
    const dspark_status st = check_ws(h, ws, ws_bytes, bs, kv->max_ctx);
    if (st) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const Layout L = layout_for(h, bs, kv->max_ctx);
    char *w = (char *)ws;
    int *err = (int *)(w + kCtlErr);
    const int M = g.block * bs;
    const int kvd = g.kv_lora + g.d_rope, qhd = g.d_nope + g.d_rope;
    __nv_bfloat16 *hn = (__nv_bfloat16 *)(w + L.hn), *cq = (__nv_bfloat16 *)(w + L.cq);
    __nv_bfloat16 *qt = (__nv_bfloat16 *)(w + L.qt), *blk = (__nv_bfloat16 *)(w + L.blk);
    __nv_bfloat16 *ov = (__nv_bfloat16 *)(w + L.ov), *act = (__nv_bfloat16 *)(w + L.act);
    __nv_bfloat16 *hout = (__nv_bfloat16 *)(w + L.hout);
    float *qkv = (float *)(w + L.qkv), *q = (float *)(w + L.q), *olat = (float *)(w + L.olat);
    if (h->c_ws != ws || h->c_bs != bs) {
        const uint32_t bn = bn_for(M);
        if (!make_map(&h->b_hn, hn, M, g.hidden, bn) || !make_map(&h->b_cq, cq, M, g.q_lora, bn) ||
            !make_map(&h->b_ov, ov, M, (uint64_t)g.n_heads * g.d_v, bn) ||
            !make_map(&h->b_act, act, M, g.inter, bn) || !make_map(&h->b_hout, hout, M, g.hidden, bn) ||
            (L.tc && (!make_map(&h->b_blk, blk, M, kvd, 64) ||
                      !make_map_3d(&h->b_qt, qt, bs, (uint64_t)g.block * g.n_heads, kvd, 128))))
            return DSPARK_ERR_CUDA;
        h->c_ws = ws;
        h->c_bs = bs;
    }
    AttnParams ap;
    memset(&ap, 0, sizeof(ap));
    ap.qt = qt;
    ap.R = g.block * g.n_heads;
    ap.n_pages = kv->n_pages;
    ap.page = g.page_size;
    ap.page_table = kv->page_table;
    ap.max_pages = kv->max_pages;
    ap.ctx_len = kv->ctx_len;
    ap.max_ctx = kv->max_ctx;
    ap.blk_kv = blk;
    ap.block = g.block;
    ap.splits = L.splits;
    ap.tok_per_split = L.tok_per_split;
    ap.cps = L.cps;
    ap.scale_log2 = h->scale_log2;
    ap.o_lat = olat;
    ap.part_o = (float *)(w + L.part_o);
    ap.part_ml = (float *)(w + L.part_ml);
    ap.err = err;
#define RUN(call)                                      \
    do {                                               \
        if ((call) != cudaSuccess) return DSPARK_ERR_CUDA; \
    } while (0)
    const bool quant = g.weight_format != DSPARK_FMT_BF16;
    // The q_a || kv_a, q_b, o_proj and down GEMMs leave their split partials
    // pending; the next kernel (latent norms, q absorption, RMSNorm with the
    // residual add) sums them while reading its input. Off when the row kernels
    // on clusters do not fit the geometry.
    const bool defer = row_cluster_fits(g.hidden) && row_cluster_fits(g.q_lora + kvd);
    GemmPending pend_x, pend_qkv, pend_q, pend_o;  // part == nullptr: the output was reduced in place
    memset(&pend_x, 0, sizeof(pend_x));
    GemmPending *const want_qkv = defer ? &pend_qkv : nullptr, *const want_q = defer ? &pend_q : nullptr;
    GemmPending *const want_o = defer ? &pend_o : nullptr, *const want_x = defer ? &pend_x : nullptr;
    for (int l = 0; l < g.n_layers; ++l) {
        const dspark_layer_weights_t &W = h->w.layers[l];
        // The block's first kernel releases the rest only after its dependency wait:
        // the latent norms, q absorption, attention and combine read ctx_len, the page
        // table and the pool before their own waits, and a cache append launched
        // earlier may still be writing them until then.
        const bool first = l == 0;
        if (defer)
            RUN(launch_rmsnorm_cluster(x, g.hidden, &pend_x, true, W.attn_norm, g.hidden, g.eps, hn, g.hidden, nullptr,
                                       0, M, err, s, first));
        else
            RUN(launch_rmsnorm(x, g.hidden, W.attn_norm, g.hidden, g.eps, hn, g.hidden, nullptr, 0, M, err, s, first));
        // q_b's weights stream into L2 while the latency-bound q_a || kv_a GEMM runs
        const L2Prefetch pf_qb = mat_prefetch(W.w_q_b, g.weight_format, (uint64_t)g.n_heads * qhd, g.q_lora);
        RUN(gemm(h, h->qkv_a[l], nullptr, h->b_hn, g.q_lora + kvd, g.hidden, M, EPI_STORE, qkv, nullptr,
                 g.q_lora + kvd, ws, s, &pf_qb, want_qkv));
        if (defer)
            RUN(launch_latent_cluster(qkv, g.q_lora + kvd, &pend_qkv, g.q_lora, g.kv_lora, g.d_rope, W.q_a_norm,
                                      W.kv_a_norm, g.eps, kv->ctx_len, g.block, kv->max_ctx, h->rope, cq, blk, M, err,
                                      s));
        else
            RUN(launch_latent(qkv, g.q_lora + kvd, g.q_lora, g.kv_lora, g.d_rope, W.q_a_norm, W.kv_a_norm, g.eps,
                              kv->ctx_len, g.block, kv->max_ctx, h->rope, cq, blk, M, err, s));
        // kv_b (k_b for the q absorption next, v_b for the v absorption) streams
        // into L2 while the q_b GEMM runs
        L2Prefetch pf_kvb;
        memset(&pf_kvb, 0, sizeof(pf_kvb));
        if (aligned16(W.w_kv_b)) {
            pf_kvb.ptr[0] = (const uint8_t *)W.w_kv_b;
            pf_kvb.bytes[0] = ((uint64_t)g.n_heads * (g.d_nope + g.d_v) * g.kv_lora * 2) & ~15ull;
        }
        RUN(quant ? gemm_q(h, h->qq_b[l], nullptr, h->b_cq, cq, g.n_heads * qhd, g.q_lora, M, EPI_STORE, q, nullptr,
                           g.n_heads * qhd, ws, s, want_q, &pf_kvb)
                  : gemm(h, h->q_b[l], nullptr, h->b_cq, g.n_heads * qhd, g.q_lora, M, EPI_STORE, q, nullptr,
                         g.n_heads * qhd, ws, s, &pf_kvb, want_q));
        RUN(launch_q_absorb(q, M, g.n_heads, g.d_nope, g.d_rope, g.kv_lora, g.d_v, (const __nv_bfloat16 *)W.w_kv_b,
                            kv->ctx_len, g.block, kv->max_ctx, h->rope, qt, s, want_q));
        ap.pool = (const __nv_bfloat16 *)kv->pools[l];
        if (L.tc) {
            if (h->c_pool[l] != kv->pools[l] || h->c_npages[l] != kv->n_pages) {
                if (!make_map(&h->pool_map[l], kv->pools[l], (uint64_t)kv->n_pages * g.page_size, kvd, 64))
                    return DSPARK_ERR_CUDA;
                h->c_pool[l] = kv->pools[l];
                h->c_npages[l] = kv->n_pages;
            }
            // the split combine is fused with the v absorption when it fits
            const bool fused = attn_combine_vabsorb_fits(g.d_v, g.kv_lora, L.splits);
            RUN(launch_attention_tc(h->pool_map[l], h->b_blk, h->b_qt, ap, L.cps, bs, kvd, g.kv_lora, s, !fused));
            if (fused)
                RUN(launch_attn_combine_vabsorb(ap, M, g.n_heads, g.d_nope, g.d_v, g.kv_lora,
                                                (const __nv_bfloat16 *)W.w_kv_b, ov, s));
            else
                RUN(launch_v_absorb(olat, M, g.n_heads, g.d_nope, g.d_v, g.kv_lora, (const __nv_bfloat16 *)W.w_kv_b,
                                    ov, s));
        } else {
            RUN(launch_attention(ap, bs, kvd, g.kv_lora, s));
            RUN(launch_v_absorb(olat, M, g.n_heads, g.d_nope, g.d_v, g.kv_lora, (const __nv_bfloat16 *)W.w_kv_b, ov, s));
        }
        RUN(quant ? gemm_q(h, h->qo[l], nullptr, h->b_ov, ov, g.hidden, g.n_heads * g.d_v, M, EPI_ADD, x, nullptr, g.hidden,
                           ws, s, want_o)
                  : gemm(h, h->o[l], nullptr, h->b_ov, g.hidden, g.n_heads * g.d_v, M, EPI_ADD, x, nullptr, g.hidden, ws,
                         s, nullptr, want_o));
        if (defer)
            RUN(launch_rmsnorm_cluster(x, g.hidden, &pend_o, true, W.mlp_norm, g.hidden, g.eps, hn, g.hidden, nullptr, 0,
                                       M, err, s));
        else
            RUN(launch_rmsnorm(x, g.hidden, W.mlp_norm, g.hidden, g.eps, hn, g.hidden, nullptr, 0, M, err, s));
        RUN(quant ? gemm_q(h, h->qgate[l], &h->qup[l], h->b_hn, hn, g.inter, g.hidden, M, EPI_SWIGLU, nullptr, act, g.inter,
                           ws, s)
                  : gemm(h, h->gate[l], &h->up[l], h->b_hn, g.inter, g.hidden, M, EPI_SWIGLU, nullptr, act, g.inter, ws,
                         s));
        RUN(quant ? gemm_q(h, h->qdown[l], nullptr, h->b_act, act, g.hidden, g.inter, M, EPI_ADD, x, nullptr, g.hidden, ws, s,
                           want_x)
                  : gemm(h, h->down[l], nullptr, h->b_act, g.hidden, g.inter, M, EPI_ADD, x, nullptr, g.hidden, ws, s,
                         nullptr, want_x));
    }
    if (defer)
        RUN(launch_rmsnorm_cluster(x, g.hidden, &pend_x, true, h->w.final_norm, g.hidden, g.eps, hout, g.hidden, h_out,
                                   g.hidden, M, err, s));
    else
        RUN(launch_rmsnorm(x, g.hidden, h->w.final_norm, g.hidden, g.eps, hout, g.hidden, h_out, g.hidden, M, err, s));
    RUN(gemm(h, h->lm_head, nullptr, h->b_hout, g.vocab, g.hidden, M, EPI_STORE, z, nullptr, g.vocab, ws, s));
    return DSPARK_OK;
}

dspark_status dspark_markov_rollout(dspark_handle_t *h, const float *z, const int32_t *anchor,
                                    const dspark_sample_t *sample, int32_t *tokens, float *ell, int bs, void *ws,
                                    size_t ws_bytes, void *stream) {
    if (!h || !sample) return DSPARK_ERR_NULL;
    if (bs <= 0 || bs > kMaxBs) return DSPARK_ERR_SHAPE;
    REQ(z);
    REQ(anchor);
    REQ(tokens);
    REQ(ell);
    if (sample->draft_mode != DSPARK_GREEDY && sample->draft_mode != DSPARK_PROBABILISTIC) return DSPARK_ERR_SHAPE;
    if (sample->draft_mode == DSPARK_PROBABILISTIC && bad_sampling(sample->temperature, sample->top_p))
        return DSPARK_ERR_SHAPE;
    const dspark_status st = check_ws(h, ws, ws_bytes, bs, 0);
    if (st) return st;
    const dspark_geom_t &g = h->g;
    const Layout L = layout_for(h, bs, 0);
    RolloutParams p;
    memset(&p, 0, sizeof(p));
    p.z = z;
    p.anchor = anchor;
    p.w1 = (const __nv_bfloat16 *)h->w.markov_w1;
    p.w2 = (const __nv_bfloat16 *)h->w.markov_w2;
    p.tokens = tokens;
    p.ell = ell;
    p.bs = bs;
    p.B = g.block;
    p.V = g.vocab;
    p.r = g.rank;
    p.draft_mode = sample->draft_mode;
    p.T = sample->temperature;
    p.top_p = sample->top_p;
    p.seed = sample->seed;
    p.step = sample->step;
    p.scratch = (unsigned long long *)((char *)ws + L.scratch);
    p.ctl = (SampleCtl *)((char *)ws + kCtlSample);
    p.err = (int *)((char *)ws + kCtlErr);
    return cuda_status(launch_rollout(h->w2, p, h->samp_grid, h->roll_resident, (cudaStream_t)stream));
}

dspark_status dspark_kv_append(dspark_handle_t *h, const float *x_new, int n_max, const int32_t *n_new,
                               const dspark_kv_t *kv, int bs, void *ws, size_t ws_bytes, void *stream) {
    if (!h || !kv) return DSPARK_ERR_NULL;
    const dspark_geom_t &g = h->g;
    if (bs <= 0 || bs > kMaxBs || n_max <= 0 || n_max > g.block + 1 || kv->max_ctx < 0 || kv->n_pages <= 0 ||
        kv->max_pages <= 0)
        return DSPARK_ERR_SHAPE;
    if (n_max * bs > 224) return DSPARK_ERR_UNSUPPORTED;
    REQ(x_new);
    REQ(n_new);
    REQ(kv->page_table);
    REQ(kv->ctx_len);
    for (int l = 0; l < g.n_layers; ++l) REQ(kv->pools[l]);
    if (!ws) return DSPARK_ERR_WORKSPACE;
    if (!aligned16(ws)) return DSPARK_ERR_ALIGN;
    const Layout L = layout_for(h, bs, kv->max_ctx);
    if (ws_bytes < L.total) return DSPARK_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    char *w = (char *)ws;
    int *err = (int *)(w + kCtlErr);
    const int A = n_max * bs;
    const int kvd = g.kv_lora + g.d_rope;
    __nv_bfloat16 *hn = (__nv_bfloat16 *)(w + L.app_hn);
    float *kvo = (float *)(w + L.app_kv);
    const int nl = g.n_layers;
    if (h->c_app_ws != ws || h->c_app_rows != A) {
        if (!make_map(&h->b_app, hn, (uint64_t)nl * A, g.hidden, bn_for(A))) return DSPARK_ERR_CUDA;
        h->c_app_ws = ws;
        h->c_app_rows = A;
    }
    const int cap = kv->max_pages * g.page_size;
    // The layers' entries do not depend on each other: every layer's pre-norm in
    // one launch, every layer's kv_a rows in one GEMM launch, one scatter.
    AppendLayers al;
    memset(&al, 0, sizeof(al));
    for (int l = 0; l < nl; ++l) {
        al.g_attn[l] = h->w.layers[l].attn_norm;
        al.g_kv[l] = h->w.layers[l].kv_a_norm;
        al.pool[l] = (__nv_bfloat16 *)kv->pools[l];
    }
    RUN(launch_append_norm(x_new, g.hidden, al, nl, g.hidden, g.eps, hn, A, err, s));
    static_assert(sizeof(GemmMaps) == sizeof(h->kva), "one map per layer");
    RUN(gemm_layers(h, *reinterpret_cast<const GemmMaps *>(h->kva), nl, h->b_app, kvd, g.hidden, A, kvo, ws, s));
    RUN(launch_kv_scatter_layers(kvo, (size_t)A * kvd, nl, al, g.kv_lora, g.d_rope, g.eps, h->rope, n_new, n_max,
                                 kv->ctx_len, kv->page_table, kv->max_pages, g.page_size, kv->n_pages, cap, bs, err,
                                 s));
    // the append is the one call that advances ctx_len (documented in the header)
    RUN(launch_ctx_advance(const_cast<int32_t *>(kv->ctx_len), n_new, n_max, cap, bs, err, s));
    return DSPARK_OK;
}

dspark_status dspark_confidence(dspark_handle_t *h, const float *h_out, float *conf, int bs, void *stream) {
    if (!h) return DSPARK_ERR_NULL;
    if (bs <= 0 || bs > kMaxBs) return DSPARK_ERR_SHAPE;
    REQ(h_out);
    REQ(conf);
    return cuda_status(launch_confidence(h_out, h->g.hidden, h->w.w_conf, h->w.b_conf, conf, h->g.block * bs,
                                         (cudaStream_t)stream));
}

dspark_status dspark_verify(dspark_handle_t *h, const float *target_logits, const float *ell, const int32_t *tokens,
                            const dspark_sample_t *sample, int32_t *accept_len, int32_t *out_tokens, int bs, void *ws,
                            size_t ws_bytes, void *stream) {
    if (!h || !sample) return DSPARK_ERR_NULL;
    if (bs <= 0 || bs > kMaxBs) return DSPARK_ERR_SHAPE;
    REQ(target_logits);
    REQ(tokens);
    REQ(accept_len);
    REQ(out_tokens);
    if (sample->verify_mode != DSPARK_GREEDY && sample->verify_mode != DSPARK_PROBABILISTIC &&
        sample->verify_mode != DSPARK_BLOCK)
        return DSPARK_ERR_SHAPE;
    if (sample->draft_mode != DSPARK_GREEDY && sample->draft_mode != DSPARK_PROBABILISTIC) return DSPARK_ERR_SHAPE;
    const bool prob = sample->verify_mode != DSPARK_GREEDY;  // token-by-token or block
    if (prob && bad_sampling(sample->temperature, sample->top_p)) return DSPARK_ERR_SHAPE;
    if (prob && sample->draft_mode != DSPARK_GREEDY) REQ(ell);
    const dspark_status st = check_ws(h, ws, ws_bytes, bs, 0);
    if (st) return st;
    const dspark_geom_t &g = h->g;
    const Layout L = layout_for(h, bs, 0);
    VerifyParams p;
    memset(&p, 0, sizeof(p));
    p.P = target_logits;
    p.ell = ell;
    p.tokens = tokens;
    p.accept_len = accept_len;
    p.out_tokens = out_tokens;
    p.bs = bs;
    p.B = g.block;
    p.V = g.vocab;
    p.verify_mode = sample->verify_mode;
    p.draft_greedy = sample->draft_mode == DSPARK_GREEDY;
    p.T = sample->temperature;
    p.top_p = sample->top_p;
    p.seed = sample->seed;
    p.step = sample->step;
    p.scratch =
        prob ? (unsigned long long *)((char *)ws + L.scratch) : (unsigned long long *)((char *)ws + kCtlKeys);
    p.ctl = (SampleCtl *)((char *)ws + kCtlSample);
    p.err = (int *)((char *)ws + kCtlErr);
    p.draw_count = (unsigned int *)((char *)ws + kCtlDraw);
    return cuda_status(launch_verify(p, h->samp_grid, (cudaStream_t)stream));
}

dspark_status dspark_check(dspark_handle_t *h, void *ws, void *stream) {
    if (!h) return DSPARK_ERR_NULL;
    if (!ws) return noalloc_check(stream);  // the allocation-free fusion's own error word
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return DSPARK_ERR_CUDA;
    int err = 0;
    if (cudaMemcpy(&err, (char *)ws + kCtlErr, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return DSPARK_ERR_CUDA;
    if (err) {
        const int zero = 0;
        if (cudaMemcpy((char *)ws + kCtlErr, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
            return DSPARK_ERR_CUDA;
    }
    return (dspark_status)err;
}

}  // extern "C"
