/*
 * dspark.h -- C ABI of the DSpark draft-and-verify step on one GB300 (sm_103a).
 *
 * The step drafts a 7-token block with an MLA-native speculative drafter and
 * verifies it losslessly against target logits. It is defined by three model
 * cards for the Kimi-K3 DSpark drafter:
 *   [P1] "kimi-k3-dspark-gguf" (alphaneural.io)
 *   [P2] "Kimi K3 DSpark Q8_0 GGUF" (graysoft.dev)
 *   [P3] "Kimi-K3-DSpark-NVFP4" (huggingface.co), including its embedded
 *        "Original model card".
 *
 * Conventions for every entry point:
 *  - Device pointers are CUDA device addresses owned by the caller; the library
 *    never frees them. Matrices are row-major [out, in]; bf16 is IEEE
 *    bfloat16 bits in uint16 storage.
 *  - All compute calls are asynchronous on the given stream (a cudaStream_t
 *    passed as void*) and never block. Host-detectable errors (null or
 *    misaligned pointers, sizes, unsupported geometry) return immediately with
 *    nothing launched. Errors the kernels detect (a non-finite logit, an
 *    out-of-range page or token id, an expired bounded wait) are recorded in an
 *    error word inside the workspace; read it with dspark_check().
 *  - Every pointer passed to a kernel must be 16-byte aligned.
 *  - A handle is used by one stream at a time; calls that share a workspace
 *    must be ordered on one stream. Stream order is all the ordering needed:
 *    the kernels overlap their neighbours' tails (programmatic dependent
 *    launch), but each reads what an earlier call wrote (the cache append's
 *    pages and ctx_len included) only after that call has completed.
 *  - The workspace is caller-allocated (dspark_workspace_bytes) and must be
 *    zero-filled once before its first use; the kernels keep its counters at
 *    zero afterwards. After dspark_check() reports DSPARK_ERR_TIMEOUT the
 *    workspace must be zero-filled again. Bytes 72..79 of the workspace hold
 *    an optional limit, in nanoseconds (uint64), on the waits of the rollout's
 *    and verification's CTAs for one another; 0 (the zero fill) means 2 s.
 *  - Batch size bs is 1..32 for every call.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DSPARK_OK = 0,
    DSPARK_ERR_NULL = 1,          /* a required pointer is null */
    DSPARK_ERR_ALIGN = 2,         /* a pointer is not 16-byte aligned */
    DSPARK_ERR_SHAPE = 3,         /* a size or sampling control is out of range */
    DSPARK_ERR_UNSUPPORTED = 4,   /* geometry or weight format the kernels do not cover */
    DSPARK_ERR_CUDA = 5,          /* a CUDA runtime or driver call failed */
    DSPARK_ERR_WORKSPACE = 6,     /* workspace pointer null or smaller than required */
    DSPARK_ERR_TIMEOUT = 16,      /* device: a bounded inter-CTA wait expired */
    DSPARK_ERR_BAD_INPUT = 17,    /* device: a logit or intermediate was not finite, an
                                     activation entering an NVFP4/MXFP4 GEMM (or an FP8 GEMM
                                     of more than 32 rows) exceeded 65504, or an MXFP4 scale
                                     lies outside 2^-22 .. 2^13 */
    DSPARK_ERR_OOB = 18           /* device: page id, token id or ctx_len out of range */
} dspark_status;

enum { DSPARK_FMT_BF16 = 0, DSPARK_FMT_FP8 = 1, DSPARK_FMT_NVFP4 = 2, DSPARK_FMT_MXFP4 = 3 };
enum { DSPARK_GREEDY = 0, DSPARK_PROBABILISTIC = 1, DSPARK_BLOCK = 2 /* verify_mode only */ };

/*
 * Drafter geometry. Full Kimi-K3 DSpark: hidden 7168, 5 captured states, 5
 * layers, 64 heads, q_lora 1536, kv_lora 512, nope 128, rope 64, v 128, SwiGLU
 * 14336, vocab 163840, Markov rank 256, block 7 ([P1] "GGUF metadata", "How it
 * works"; [P2] "Architecture metadata"; [P3] "Model Overview").
 * Supported by the kernels: hidden, q_lora, kv_lora, inter, n_heads*d_v
 * multiples of 64; (kv_lora + d_rope, kv_lora) one of (576, 512), (288, 256),
 * (160, 128), (80, 64); q_lora + kv_lora <= 8192; d_nope <= 256; d_rope a
 * multiple of 4 and <= 128; block <= 16;
 * rank <= 256; vocab even and < 2^18; page_size 64; weight_format BF16, FP8
 * (E4M3 per output row), NVFP4 (E2M1, E4M3 group-16 scales, global scale;
 * then hidden, q_lora, n_heads*d_v and inter multiples of 256) or MXFP4 (E2M1,
 * E8M0 power-of-two scales per 32 inputs; then those sizes multiples of 512).
 * With FP8, NVFP4 or MXFP4, block * bs <= 64 per call. FP8 GEMMs of up to 32 rows take
 * the bf16 activations exactly (as two E4M3 terms per row and 128-k chunk); NVFP4,
 * MXFP4 and FP8 above 32 rows take them in f16, so they must stay within +-65504
 * (see DSPARK_ERR_BAD_INPUT).
 */
typedef struct {
    int hidden, n_aux, n_layers, n_heads;
    int q_lora, kv_lora, d_nope, d_rope, d_v;
    int inter, vocab, rank, block;
    float rope_theta;     /* RoPE base (10000) */
    float eps;            /* RMSNorm epsilon, inside the root */
    float yarn_factor;    /* YaRN scale s; <= 1 means plain RoPE ([P2]: YaRN-16 from 65,536) */
    int yarn_orig_ctx;    /* original context of YaRN */
    float yarn_alpha, yarn_beta;  /* YaRN ramp bounds in rotations (1, 32) */
    int page_size;        /* tokens per latent-KV page */
    int weight_format;    /* DSPARK_FMT_*: format of fc, q_b, o, gate, up, down */
} dspark_geom_t;

/* One quantisable matrix: bf16 data, or FP8 E4M3 data [out,in] + fp32 scale
 * [out], or NVFP4 packed E2M1 data [out,in/2] + E4M3 scales [out,in/16] + a
 * global fp32 scale ([P3] "What is quantized to what": MLP, o_proj, q_b_proj,
 * context_proj; group 16 with E4M3 scales), or MXFP4 packed E2M1 data
 * [out,in/2] + E8M0 scale bytes [out,in/32] (2^(byte - 127); the global scale
 * is ignored). Packed codes: the even input in the low nibble. */
typedef struct {
    const void *data;
    const void *scale;
    float global_scale;
} dspark_mat_t;

/* Per-layer weights (device pointers, non-owning). Norm gains fp32. */
typedef struct {
    const float *attn_norm;   /* [hidden] */
    const void *w_qkv_a;      /* bf16 [q_lora + kv_lora + d_rope, hidden]: fused q_a || kv_a_with_mqa ([P3]) */
    const float *q_a_norm;    /* [q_lora] */
    const float *kv_a_norm;   /* [kv_lora] */
    dspark_mat_t w_q_b;       /* [n_heads * (d_nope + d_rope), q_lora] */
    const void *w_kv_b;       /* bf16 [n_heads * (d_nope + d_v), kv_lora]: per head d_nope rows of k_b, then d_v rows of v_b */
    dspark_mat_t w_o;         /* [hidden, n_heads * d_v] */
    const float *mlp_norm;    /* [hidden] */
    dspark_mat_t w_gate;      /* [inter, hidden] */
    dspark_mat_t w_up;        /* [inter, hidden] */
    dspark_mat_t w_down;      /* [hidden, inter] */
} dspark_layer_weights_t;

#define DSPARK_MAX_LAYERS 16

typedef struct {
    dspark_mat_t w_fc;                                   /* [hidden, n_aux * hidden] ([P2] fc.weight; [P3] context_proj) */
    dspark_layer_weights_t layers[DSPARK_MAX_LAYERS];    /* first n_layers used */
    const float *final_norm;                             /* [hidden] */
    const void *w_lm;                                    /* bf16 [vocab, hidden]: the target's lm_head ([P3] "Measurement") */
    const void *markov_w1;                               /* bf16 [vocab, rank] */
    const void *markov_w2;                               /* bf16 [rank, vocab] ([P2] Markov rank 256, two low-rank matrices) */
    const float *w_conf;                                 /* fp32 [hidden] confidence head */
    float b_conf;
} dspark_weights_t;

/* Paged latent KV cache: per layer a pool [n_pages, page_size, kv_lora + d_rope]
 * bf16 of normalised latents || roped keys, shared with the target's layout
 * ([P3] "Model Overview": the draft's pages unify with the target's cache).
 * Token j of sequence b lives at pool[page_table[b*max_pages + j/page_size]][j % page_size].
 * Read-only during a draft. */
typedef struct {
    const void *pools[DSPARK_MAX_LAYERS];  /* device */
    int n_pages;
    const int32_t *page_table;  /* device int32 [bs, max_pages] */
    int max_pages;
    const int32_t *ctx_len;     /* device int32 [bs] */
    int max_ctx;                /* host bound on every ctx_len (sets the split of the KV loop) */
} dspark_kv_t;

/* Sampling controls ([P3] "Quick Start / Sampling options": draft_sample_method
 * greedy | probabilistic; temperature 1.0, top_p 0.95 in production). The
 * uniforms are Philox4x32-10 words keyed by seed with counter (step, seq, pos,
 * purpose); purposes 1 draft, 2 accept, 3 residual, 4 bonus. */
typedef struct {
    int draft_mode;     /* DSPARK_GREEDY or DSPARK_PROBABILISTIC */
    int verify_mode;    /* DSPARK_GREEDY, DSPARK_PROBABILISTIC or DSPARK_BLOCK */
    float temperature;  /* > 0 for probabilistic modes */
    float top_p;        /* (0, 1] */
    uint64_t seed;
    uint32_t step;
} dspark_sample_t;

typedef struct dspark_handle dspark_handle_t;

/* Create a handle for one geometry and weight set on the current CUDA device.
 * Copies the geometry and the weight pointers (not the weights) and encodes the
 * TMA descriptors of the weight matrices. Allocates no device memory.
 * Errors: NULL, ALIGN, SHAPE, UNSUPPORTED, CUDA. */
dspark_status dspark_create(const dspark_geom_t *geom, const dspark_weights_t *weights, dspark_handle_t **out);
void dspark_destroy(dspark_handle_t *h);

/* Bytes of workspace the compute calls need for up to max_bs sequences and
 * contexts up to max_ctx tokens (split partials, activations, counters,
 * error word); 0 if an argument is out of range. */
size_t dspark_workspace_bytes(const dspark_handle_t *h, int max_bs, int max_ctx);

/* (1) fc context fusion ([P2] "Architecture metadata": fc.weight consumes
 * five captured hidden states; [P3] context_proj):
 *   x[b,i,:] = W_fc [aux[b,i,0,:] || ... || aux[b,i,n_aux-1,:]]
 * aux bf16 [bs, block, n_aux, hidden]; x fp32 [bs, block, hidden] (overwritten). */
dspark_status dspark_fuse_ctx(dspark_handle_t *h, const void *aux, float *x, int bs,
                              void *ws, size_t ws_bytes, void *stream);

/* (2) The block-diffusion layers, final norm and lm_head ([P3] "Model
 * Overview": 5 dense layers, non-causal attention, 7 tokens in one pass; [P1]
 * "Runtime status": MLA q_a / kv_a_mqa / k_b / v_b with split RoPE dims).
 * Per layer: RMSNorm; fused q_a||kv_a; latent norms; RoPE on the rope parts at
 * positions ctx_len[b] + i; q_b; k_b absorbed into q; non-causal attention over
 * the cached latents and the block's own latents; v_b absorbed into the
 * output; o_proj + residual; RMSNorm; SwiGLU MLP + residual. Then
 * h_out = RMSNorm(x) and z = W_lm h_out.
 * x fp32 [bs, block, hidden] is the residual stream and is updated in place.
 * h_out fp32 [bs, block, hidden]; z fp32 [bs, block, vocab]. */
dspark_status dspark_draft_block(dspark_handle_t *h, float *x, const dspark_kv_t *kv, float *h_out, float *z,
                                 int bs, void *ws, size_t ws_bytes, void *stream);

/* (3) Low-rank Markov rollout ([P3] "Model Overview": a low-rank sequential
 * Markov head supplies the intra-block dependency; [P1] "How it works"):
 *   t_0 = anchor[b]; for i = 1..block:
 *     ell_i[v] = z_i[v] + fp32 FMA chain over k = 0..rank-1 of w1[t_{i-1},k] * w2[k,v]
 *     t_i = argmax ell_i (lowest id on ties), or a draw by the sampling spec.
 * z fp32 [bs, block, vocab]; anchor int32 [bs]; tokens int32 [bs, block];
 * ell fp32 [bs, block, vocab]. */
dspark_status dspark_markov_rollout(dspark_handle_t *h, const float *z, const int32_t *anchor,
                                    const dspark_sample_t *sample, int32_t *tokens, float *ell, int bs,
                                    void *ws, size_t ws_bytes, void *stream);

/* (4) Confidence head ([P1] "How it works": decides when to draft and when to
 * fall back): conf[b,i] = sigmoid(w_conf . h_out[b,i,:] + b_conf).
 * h_out fp32 [bs, block, hidden]; conf fp32 [bs, block]. */
dspark_status dspark_confidence(dspark_handle_t *h, const float *h_out, float *conf, int bs, void *stream);

/* (5) Lossless verification ([P1] intro: the output distribution equals the
 * target's; [P3] "Sampling options": at temperature 0 an argmax match).
 * target_logits fp32 [bs, block+1, vocab] (row i scores block position i, row
 * block is the bonus position); ell fp32 [bs, block, vocab] (unused with a
 * greedy draft); tokens int32 [bs, block].
 * Greedy: accept the leading drafts equal to argmax of the target rows, then
 * emit the target's argmax. Probabilistic: accept t_i with probability
 * min(1, p_i(t_i)/q_i(t_i)); on the first reject draw from norm(max(0, p - q));
 * if all are accepted draw a bonus from p_{block+1}. Exact integer arithmetic
 * on 2^32-scaled weights; with a greedy draft q_i is one-hot on t_i.
 * Block (DSPARK_BLOCK, [P3] "Sampling options": rejection_sample_method block
 * verifies the drafted block as a unit; the published block verification
 * method): pi_0 = 1, pi_i = min(pi_{i-1} p_{i-1}(t_i)/q_{i-1}(t_i), 1),
 * h_i = S_i / (S_i + 1 - pi_i) with S_i = sum_x max(pi_i p_i(x) - q_i(x), 0),
 * h_block = pi_block; independent decisions U_i < h_i * 2^32; the last accepted
 * position tau; then a draw from max(pi_tau p_tau - q_tau, 0) (tau < block) or
 * the bonus. Probabilities are the spec's rationals rounded once to double;
 * residual terms are doubles truncated to 2^-80 and summed exactly in 128 bits.
 * accept_len int32 [bs] in 0..block; out_tokens int32 [bs, block+1] (accepted
 * drafts, then the correction or bonus token, then -1). */
dspark_status dspark_verify(dspark_handle_t *h, const float *target_logits, const float *ell, const int32_t *tokens,
                            const dspark_sample_t *sample, int32_t *accept_len, int32_t *out_tokens, int bs,
                            void *ws, size_t ws_bytes, void *stream);

/* (6) Latent-cache append of newly verified tokens ("Kimi-K3-DSpark-NVFP4",
 * Model Overview: draft and target share one 576-element latent layout, so the
 * draft's pages unify with the target's cache). For every layer l and every
 * sequence b, token j < n_new[b] with context features x_new[b, j, :] gets the
 * entry [RMSNorm(c_kv) * kv_a_norm || RoPE(k_r, pos)] (kv = the kv_a rows of
 * w_qkv_a applied to RMSNorm(x_new) * attn_norm) written to
 * kv->pools[l][page_table[b, pos / 64], pos % 64] with pos = ctx_len[b] + j;
 * afterwards ctx_len[b] += n_new[b] (device, in place).
 * x_new fp32 [bs, n_max, hidden], every row finite (rows j >= n_new[b] are read
 * and ignored); n_new int32 [bs] on the device; 1 <= n_max <= block + 1 and
 * n_max * bs <= 224. The workspace is the one of dspark_draft_block for the same
 * bs and kv->max_ctx. Device errors (DSPARK_ERR_OOB): n_new outside [0, n_max],
 * a position at or beyond max_pages * 64, a page id outside [0, n_pages); such
 * entries are not written and that sequence's ctx_len is not advanced. */
dspark_status dspark_kv_append(dspark_handle_t *h, const float *x_new, int n_max, const int32_t *n_new,
                               const dspark_kv_t *kv, int bs, void *ws, size_t ws_bytes, void *stream);

/* fc context fusion without a workspace: the same product as dspark_fuse_ctx,
 * for callers that cannot allocate device memory for a workspace (a serving
 * process whose device memory another allocator has already reserved, a
 * latency-critical path that may not call cudaMalloc, a plugin host that does
 * not let libraries own device buffers). The model cards have no counterpart:
 * this is a deployment convenience of this library.
 * Scratch (split partials, tile counters, an error word) lives in one
 * ~2.5 MiB array inside the library, resident on every device that loads it
 * until the process exits. Limits: bs <= 2, hidden <= 131072; larger sizes
 * return DSPARK_ERR_SHAPE. Only bf16 fc weights: a handle with another
 * weight_format gets DSPARK_ERR_UNSUPPORTED before anything is launched. The
 * first call on a device resolves the array's device address and sets the
 * kernel's shared-memory limit (host threads making that first call at once
 * are serialised); make that first call before any stream capture. Each call
 * clears the tile counters it needs on its stream. All calls share the one
 * array: calls that overlap on the GPU (different streams, or several handles
 * at once) race and must be serialised by the caller. Device-side errors of
 * this call (an expired bounded wait) stay in the array's own error word until
 * dspark_check(h, NULL, stream) reads and clears it. Allocates nothing.
 * aux bf16 [bs, block, n_aux, hidden]; x fp32 [bs, block, hidden] (overwritten). */
dspark_status dspark_fuse_ctx_noalloc(dspark_handle_t *h, const void *aux, float *x, int bs, void *stream);

/* Synchronise the stream, return and clear the device error word
 * (DSPARK_OK if no kernel recorded an error since the last check). With
 * ws == NULL the word read is the one of dspark_fuse_ctx_noalloc's fixed
 * scratch on the current device. */
dspark_status dspark_check(dspark_handle_t *h, void *ws, void *stream);

const char *dspark_status_str(dspark_status s);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
