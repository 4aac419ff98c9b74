// Internal declarations shared by the translation units of libdspark.
#pragma once

#include "common.cuh"

namespace ds {

// Per-pair RoPE angular frequencies (YaRN-adjusted when enabled), fp64.
struct RopeTable {
    double inv_freq[64];
};

struct AttnParams {
    const __nv_bfloat16 *qt;        // [bs, R, DQK] absorbed, roped queries
    int R;                          // block * n_heads rows per sequence
    const __nv_bfloat16 *pool;      // [n_pages, page, DQK]
    int n_pages, page;
    const int32_t *page_table;      // [bs, max_pages]
    int max_pages;
    const int32_t *ctx_len;         // [bs]
    int max_ctx;
    const __nv_bfloat16 *blk_kv;    // [bs * block, DQK]
    int block;
    int splits, tok_per_split;      // KV split plan (tok_per_split a multiple of 64)
    int cps;                        // tensor-core path: 64-token chunks per split (split s: chunks s cps ..)
    float scale_log2;               // softmax scale * log2(e)
    float *o_lat;                   // [bs, R, DV]
    float *part_o;                  // [bs, splits, R, DV]
    float *part_ml;                 // [bs, splits, R, 2]
    int *err;
};

// late: release the dependent kernels only after this kernel's own dependency
// wait (the first kernel of a draft block)
cudaError_t launch_rmsnorm(const float *x, int ldx, const float *g, int H, float eps, __nv_bfloat16 *y, int ldy,
                           float *y32, int ldy32, int M, int *err, cudaStream_t st, bool late = false);
cudaError_t launch_latent(const float *qkv, int ld, int q_lora, int kv_lora, int d_rope, const float *g_q,
                          const float *g_kv, float eps, const int32_t *ctx_len, int block, int max_ctx,
                          const RopeTable &rt, __nv_bfloat16 *cq, __nv_bfloat16 *blk_kv, int M, int *err,
                          cudaStream_t st);
// q read from q, or (pend->part set) formed from the q_b GEMM's pending partials.
cudaError_t launch_q_absorb(const float *q, int M, int n_h, int d_nope, int d_rope, int kv_lora, int d_v,
                            const __nv_bfloat16 *w_kvb, const int32_t *ctx_len, int block, int max_ctx,
                            const RopeTable &rt, __nv_bfloat16 *qt, cudaStream_t st,
                            const GemmPending *pend = nullptr);
// Row kernels on clusters of CTAs (one cluster per row). With a pending input
// the row is the sum of a GEMM's split partials: the RMSNorm adds it to x
// (add) or stores it in x, then normalises; the latent kernel normalises it.
bool row_cluster_fits(int H);
cudaError_t launch_rmsnorm_cluster(float *x, int ldx, const GemmPending *pend, bool add, const float *g, int H,
                                   float eps, __nv_bfloat16 *y, int ldy, float *y32, int ldy32, int M, int *err,
                                   cudaStream_t st, bool late = false);
cudaError_t launch_latent_cluster(const float *qkv, int ld, const GemmPending *pend, int q_lora, int kv_lora,
                                  int d_rope, const float *g_q, const float *g_kv, float eps, const int32_t *ctx_len,
                                  int block, int max_ctx, const RopeTable &rt, __nv_bfloat16 *cq,
                                  __nv_bfloat16 *blk_kv, int M, int *err, cudaStream_t st);
// The attention's split combine fused with the v absorption (the split
// partials, or o_lat when there is one split, -> bf16 [M, n_h * d_v]).
bool attn_combine_vabsorb_fits(int d_v, int kv_lora, int splits);
cudaError_t launch_attn_combine_vabsorb(const AttnParams &p, int M, int n_h, int d_nope, int d_v, int kv_lora,
                                        const __nv_bfloat16 *w_kvb, __nv_bfloat16 *out, cudaStream_t st);
cudaError_t launch_v_absorb(const float *o_lat, int M, int n_h, int d_nope, int d_v, int kv_lora,
                            const __nv_bfloat16 *w_kvb, __nv_bfloat16 *out, cudaStream_t st);
bool attention_supported(int dqk, int dv);
cudaError_t launch_attention(const AttnParams &p, int bs, int dqk, int dv, cudaStream_t st);
cudaError_t launch_attn_combine(const AttnParams &p, int bs, int dv, cudaStream_t st);
// Per-layer pointers of the latent-cache append (first n used).
struct AppendLayers {
    const float *g_attn[DSPARK_MAX_LAYERS];  // attention pre-norm gains
    const float *g_kv[DSPARK_MAX_LAYERS];    // kv_a norm gains
    __nv_bfloat16 *pool[DSPARK_MAX_LAYERS];  // page pools
};
// y[l][m] = RMSNorm(x[m]) * g_attn[l] (bf16, [L][M][H]) for every layer at once.
cudaError_t launch_append_norm(const float *x, int ldx, const AppendLayers &al, int L, int H, float eps,
                               __nv_bfloat16 *y, int M, int *err, cudaStream_t st);
// Latent-cache append, every layer at once: rows b * n_max + j (j < n_new[b]) of
// layer l's kv [*, kv_lora + d_rope] (at kv + l * kv_stride) become
// [RMSNorm(c_kv) * g_kv[l] || RoPE(k_r, ctx_len[b] + j)] bf16 in pool[l].
// Positions at or beyond cap, invalid pages and n_new outside [0, n_max] are
// reported (DSPARK_ERR_OOB) and not written.
cudaError_t launch_kv_scatter_layers(const float *kv, size_t kv_stride, int L, const AppendLayers &al, int kv_lora,
                                     int d_rope, float eps, const RopeTable &rt, const int32_t *n_new, int n_max,
                                     const int32_t *ctx_len, const int32_t *page_table, int max_pages, int page,
                                     int n_pages, int cap, int bs, int *err, cudaStream_t st);
cudaError_t launch_ctx_advance(int32_t *ctx_len, const int32_t *n_new, int n_max, int cap, int bs, int *err,
                               cudaStream_t st);
// Tensor-core attention (latent 512 + rope 64): pool_map views one layer's page
// pool as bf16 [n_pages * 64, dqk], blk_map the block latents [bs * block, dqk],
// both with 64 x 64 boxes in the 128-byte swizzle.
bool attention_tc_supported(int dqk, int dv);
int attention_tc_splits(int R, int dv, int bs, int max_ctx, int num_sms, int *cps);
// combine = false: the caller combines the splits (launch_attn_combine_vabsorb).
cudaError_t launch_attention_tc(const CUtensorMap &pool_map, const CUtensorMap &blk_map, const CUtensorMap &q_map,
                                const AttnParams &a, int cps, int bs, int dqk, int dv, cudaStream_t st, bool combine = true);
cudaError_t launch_confidence(const float *h_out, int H, const float *w, float bias, float *conf, int M,
                              cudaStream_t st);

// Grid-barrier words inside the workspace (zero before the first launch), and
// the limit of the sampling kernels' inter-CTA waits in nanoseconds (0: the
// default kWaitLimitNs; a caller may set a shorter one).
struct SampleCtl {
    unsigned int bar_count;
    unsigned int bar_gen;
    unsigned long long wait_ns;
};

struct RolloutParams {
    const float *z;                 // [bs, B, V]
    const int32_t *anchor;          // [bs]
    const __nv_bfloat16 *w1;        // [V, r]
    const __nv_bfloat16 *w2;        // [r, V]
    int32_t *tokens;                // [bs, B]
    float *ell;                     // [bs, B, V]
    int bs, B, V, r;
    int draft_mode;
    float T, top_p;
    unsigned long long seed;
    unsigned int step;
    unsigned long long *scratch;    // zeroed by the kernel itself at start
    SampleCtl *ctl;
    int *err;
};

struct VerifyParams {
    const float *P;                 // [bs, B + 1, V] target logits
    const float *ell;               // [bs, B, V]
    const int32_t *tokens;          // [bs, B]
    int32_t *accept_len;            // [bs]
    int32_t *out_tokens;            // [bs, B + 1]
    int bs, B, V;
    int verify_mode, draft_greedy;
    int stage;                      // the draws stage their rows in shared memory (set by the launcher)
    unsigned int *draw_count;       // [bs] CTAs done per sequence (zero between launches)
    float T, top_p;
    unsigned long long seed;
    unsigned int step;
    unsigned long long *scratch;    // greedy: argmax keys, zero between launches; else row statistics and masses
    SampleCtl *ctl;
    int *err;
};

// Read-only views of a handle and the tensor-map encoder (defined with the handle).
const dspark_geom_t *handle_geom(const dspark_handle_t *h);
int handle_num_sms(const dspark_handle_t *h);
const CUtensorMap *handle_fc_map(const dspark_handle_t *h);
bool encode_bf16_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows);

// Error word of the allocation-free fusion's fixed scratch on the current
// device (synchronises the stream; reads and clears the word).
dspark_status noalloc_check(void *stream);

size_t rollout_scratch_words(int bs, int B, int grid);
size_t verify_scratch_words(int bs, int B, int grid);
cudaError_t launch_rollout(const CUtensorMap &w2_map, RolloutParams p, int grid, bool resident, cudaStream_t st);
// Whether the greedy one-sequence rollout can hold w2 on chip for this
// vocabulary, rank and grid (sets the kernel's shared-memory limit).
bool rollout_resident_setup(int V, int r, int grid);
// w2 tile geometry of the rollout (pairs per box row, boxes per stage); its
// tensor map views w2 as uint32 pairs [r, V / 2] with boxes {box_w, 16}.
__host__ __device__ void rollout_box(int V, int grid, int *box_w, int *nbox);
cudaError_t launch_verify(VerifyParams p, int grid, cudaStream_t st);
// Shared-memory limit of the verification's nucleus kernel for this vocabulary.
bool verify_setup(int V);
int sampling_max_grid(int num_sms, int V);

}  // namespace ds
