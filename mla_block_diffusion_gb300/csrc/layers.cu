// Per-layer kernels of the DSpark draft pass other than the weight GEMMs:
// RMSNorm, latent norms + RoPE, k_b / v_b absorption, paged latent-KV MLA
// attention (split over the KV sequence, fixed-order combine), confidence.
//
// Model cards: 5 dense block-diffusion layers with non-causal attention over a
// 7-token block, MLA with a 576-element latent per token shared with the target
// ("Kimi-K3-DSpark-NVFP4", Original model card / Model Overview); MLA tensors
// q_a, kv_a_mqa, k_b, v_b and split RoPE dims ("kimi-k3-dspark-gguf", Runtime
// status); kv_b absorbed, norms high precision ("Kimi-K3-DSpark-NVFP4", What is
// quantized to what).
#include <cstring>

#include "internal.h"

namespace ds {

// cos/sin of pos * inv_freq: the angle is reduced modulo 2 pi in fp64 (a few
// fp64 operations, exact enough at positions ~10^5), then evaluated in fp32.
DS_DEVINL void rope_cs(double pos, double inv_freq, float &c, float &s) {
    const double two_pi = 6.283185307179586476925286766559;
    const double inv_two_pi = 0.15915494309189533576888376337251;
    const double a = pos * inv_freq;
    const double r = fma(-two_pi, rint(a * inv_two_pi), a);  // a reduced to about [-pi, pi]
    sincosf((float)r, &s, &c);
}

__device__ float block_sum(float v, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float r = (threadIdx.x < nw) ? red[threadIdx.x] : 0.f;
    if (warp == 0) r = warp_sum(r);
    if (threadIdx.x == 0) red[32] = r;
    __syncthreads();
    return red[32];
}

// ---------------------------------------------------------------------------
// RMSNorm: y = x / sqrt(mean(x^2) + eps) * g, written as bf16 (GEMM operand)
// and optionally fp32. One CTA per row; H a multiple of 4. The gains are read
// before the wait on the producing kernel; the first 4 * blockDim float4 of the
// row stay in registers between the two passes. With `late` (the first kernel
// of a draft block) the kernel releases its dependents only after its own
// dependency wait: the block's later kernels read the context lengths, page
// table and latent pool before their waits, and an earlier cache append may
// still be writing them until that wait returns.
// ---------------------------------------------------------------------------
constexpr int kNormThreads = 512;

__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const float *__restrict__ x, int ldx,
                                                               const float *__restrict__ g, int H, float eps,
                                                               __nv_bfloat16 *__restrict__ y, int ldy,
                                                               float *__restrict__ y32, int ldy32, int *err, int late) {
    if (!late) pdl_trigger();
    __shared__ float red[33];
    const int m = blockIdx.x, n4 = H / 4;
    const float4 *xr = (const float4 *)(x + (size_t)m * ldx);
    const float4 *g4 = (const float4 *)g;
    float4 gr[4], v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = threadIdx.x + u * blockDim.x;
        gr[u] = i < n4 ? __ldg(g4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    pdl_wait();
    if (late) pdl_trigger();
    float ss = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = threadIdx.x + u * blockDim.x;
        v[u] = i < n4 ? xr[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) ss += v[u].x * v[u].x + v[u].y * v[u].y + v[u].z * v[u].z + v[u].w * v[u].w;
    for (int i = threadIdx.x + 4 * blockDim.x; i < n4; i += blockDim.x) {
        const float4 t = xr[i];
        ss += t.x * t.x + t.y * t.y + t.z * t.z + t.w * t.w;
    }
    ss = block_sum(ss, red);
    if (!isfinite(ss) && threadIdx.x == 0) set_error(err, DSPARK_ERR_BAD_INPUT);
    const float r = rsqrtf(ss / (float)H + eps);
    auto emit = [&](int i, float4 t, float4 gg) {
        const float4 o = make_float4(t.x * r * gg.x, t.y * r * gg.y, t.z * r * gg.z, t.w * r * gg.w);
        __nv_bfloat162 *yb = (__nv_bfloat162 *)(y + (size_t)m * ldy + 4 * i);
        yb[0] = __floats2bfloat162_rn(o.x, o.y);
        yb[1] = __floats2bfloat162_rn(o.z, o.w);
        if (y32) ((float4 *)(y32 + (size_t)m * ldy32))[i] = o;
    };
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = threadIdx.x + u * blockDim.x;
        if (i < n4) emit(i, v[u], gr[u]);
    }
    for (int i = threadIdx.x + 4 * blockDim.x; i < n4; i += blockDim.x) emit(i, xr[i], g4[i]);
}

// ---------------------------------------------------------------------------
// Latent norms and RoPE of the fused q_a || kv_a output (one CTA per row):
//   c_q = RMSNorm(qa) * g_q -> bf16 (operand of q_b)
//   c_kv = RMSNorm(kv[:kv_lora]) * g_kv, k_r = RoPE(kv[kv_lora:], ctx_len + i)
//   -> the block's own latent KV entries [c_kv || k_r] bf16.
// Angles are formed in fp64 (positions reach ~10^5).
// ---------------------------------------------------------------------------
__device__ float2 block_sum2(float2 v, float2 *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    v.x = warp_sum(v.x);
    v.y = warp_sum(v.y);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float2 r = (threadIdx.x < nw) ? red[threadIdx.x] : make_float2(0.f, 0.f);
    if (warp == 0) {
        r.x = warp_sum(r.x);
        r.y = warp_sum(r.y);
    }
    if (threadIdx.x == 0) red[32] = r;
    __syncthreads();
    return red[32];
}

constexpr int kLatentThreads = 512;

// One CTA per row; q_lora and kv_lora multiples of 4. Each thread keeps its
// float4 pieces of the row (at most 4: the row holds up to 2048 + 512 values).
__global__ void __launch_bounds__(kLatentThreads) latent_kernel(
    const float *__restrict__ qkv, int ld, int q_lora, int kv_lora, int d_rope, const float *__restrict__ g_q,
    const float *__restrict__ g_kv, float eps, const int32_t *__restrict__ ctx_len, int block, int max_ctx,
    RopeTable rt, __nv_bfloat16 *__restrict__ cq, __nv_bfloat16 *__restrict__ blk_kv, int *err) {
    pdl_trigger();
    __shared__ float2 red[33];
    const int m = blockIdx.x;
    const int b = m / block, i = m % block;
    const int nq4 = q_lora / 4, nk4 = kv_lora / 4, n4 = nq4 + nk4;
    const float4 *row = (const float4 *)(qkv + (size_t)m * ld);
    // gains first (inputs of the step), then the row
    float4 gr[4], v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int t = threadIdx.x + u * blockDim.x;
        gr[u] = t < nq4 ? __ldg((const float4 *)g_q + t)
                        : (t < n4 ? __ldg((const float4 *)g_kv + (t - nq4)) : make_float4(0.f, 0.f, 0.f, 0.f));
    }
    int c = ctx_len[b];
    pdl_wait();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int t = threadIdx.x + u * blockDim.x;
        v[u] = t < n4 ? row[t] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float2 ss = make_float2(0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int t = threadIdx.x + u * blockDim.x;
        const float sq = v[u].x * v[u].x + v[u].y * v[u].y + v[u].z * v[u].z + v[u].w * v[u].w;
        if (t < nq4)
            ss.x += sq;
        else
            ss.y += sq;
    }
    ss = block_sum2(ss, red);
    if ((!isfinite(ss.x) || !isfinite(ss.y)) && threadIdx.x == 0) set_error(err, DSPARK_ERR_BAD_INPUT);
    const float rq = rsqrtf(ss.x / (float)q_lora + eps), rk = rsqrtf(ss.y / (float)kv_lora + eps);
    const int kvd = kv_lora + d_rope;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int t = threadIdx.x + u * blockDim.x;
        if (t < n4) {
            const float r = t < nq4 ? rq : rk;
            __nv_bfloat16 *dst = t < nq4 ? cq + (size_t)m * q_lora + 4 * t : blk_kv + (size_t)m * kvd + 4 * (t - nq4);
            __nv_bfloat162 *d2 = (__nv_bfloat162 *)dst;
            d2[0] = __floats2bfloat162_rn(v[u].x * r * gr[u].x, v[u].y * r * gr[u].y);
            d2[1] = __floats2bfloat162_rn(v[u].z * r * gr[u].z, v[u].w * r * gr[u].w);
        }
    }
    if (c < 0 || c > max_ctx) {
        if (threadIdx.x == 0) set_error(err, DSPARK_ERR_OOB);
        c = 0;
    }
    const double pos = (double)(c + i);
    const float *rp = qkv + (size_t)m * ld + q_lora + kv_lora;
    for (int p = threadIdx.x; p < d_rope / 2; p += blockDim.x) {
        float fc, fs;
        rope_cs(pos, rt.inv_freq[p], fc, fs);
        const float x0 = rp[2 * p], x1 = rp[2 * p + 1];
        blk_kv[(size_t)m * kvd + kv_lora + 2 * p] = __float2bfloat16(x0 * fc - x1 * fs);
        blk_kv[(size_t)m * kvd + kv_lora + 2 * p + 1] = __float2bfloat16(x0 * fs + x1 * fc);
    }
}

// ---------------------------------------------------------------------------
// Row kernels of a cluster of kRowCl CTAs per row. Each CTA owns a slice of
// whole float4 of the row (at most kRowVals per thread, kept in registers);
// the slices' sums of squares meet in distributed shared memory and are added
// in rank order, so every CTA forms the same scale. The row is either read
// (pend.part == nullptr) or formed from the split partials a GEMM left pending
// (plus the row itself when `add`). Little shared memory, so the CTAs become
// resident beside a running weight GEMM and wait there.
// ---------------------------------------------------------------------------
constexpr int kRowCl = 8;
constexpr int kRowClThreads = 256;
constexpr int kRowVals = 2;      // float4 per thread
constexpr int kRowClTiles = 16;  // channel tiles a CTA's slice may touch

// The tiles [t0, t0 + nt) of a pending output into shared memory.
DS_DEVINL void row_tiles(const GemmPending &pend, int t0, int nt, PendTile *tiles) {
    if (pend.part && (int)threadIdx.x < nt) tiles[threadIdx.x] = pend_tile(pend, t0 + threadIdx.x);
}

// This CTA's slice [i0, i1) (float4 units) of a row of n4 float4.
DS_DEVINL void row_slice(int n4, int &i0, int &i1) {
    const uint32_t k = cluster_rank();
    i0 = (int)((long long)k * n4 / kRowCl);
    i1 = (int)((long long)(k + 1) * n4 / kRowCl);
}

// The cluster's exchange of (a, b) sums. Before the dependency wait each CTA
// sets up a local mbarrier that expects one 8-byte value from every CTA of the
// cluster (cluster_sum_setup, then a cluster barrier so that no value arrives
// before its barrier exists). cluster_sum2: thread k sends this CTA's sum to
// slot `rank` of CTA k (st.async, counted on CTA k's mbarrier), every thread
// arrives on a relaxed cluster barrier (waited at exit: a CTA stays a valid
// target until every peer has sent), the CTA waits for its own eight values and
// adds them in rank order. Every thread of every CTA calls both.
DS_DEVINL void cluster_sum_setup(uint64_t *bar) {
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar, (uint32_t)(kRowCl * sizeof(float2)));
    }
    cluster_sync();
}
DS_DEVINL float2 cluster_sum2(float2 v, float2 *red, float2 *parts, uint64_t *bar, volatile int *fail) {
    v = block_sum2(v, red);
    if (threadIdx.x < (unsigned)kRowCl) st_async_peer_f2(parts + cluster_rank(), bar, threadIdx.x, v);
    cluster_arrive_relaxed();
    if (!mbar_wait_bounded(bar, 0, fail)) *fail = 1;
    float2 t = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kRowCl; ++k) {
        t.x += parts[k].x;
        t.y += parts[k].y;
    }
    return t;
}

// Row value at float4 index i (pending or read).
DS_DEVINL float4 row_value(const float4 *row, const GemmPending &pend, const PendTile *tiles, int t0, int m, int i) {
    if (!pend.part) return row[i];
    const int n = 4 * i;
    return pending_sum4(pend, tiles[(n >> 7) - t0], m, n & 127);
}

// RMSNorm: x <- (add ? x : 0) + pending (written back: x is the residual
// stream), y = x / sqrt(mean(x^2) + eps) * g as bf16, y32 as fp32 when given.
// Grid (kRowCl, M); H a multiple of 4.
__global__ void __launch_bounds__(kRowClThreads) rmsnorm_cluster_kernel(
    float *__restrict__ x, int ldx, GemmPending pend, int add, const float *__restrict__ g, int H, float eps,
    __nv_bfloat16 *__restrict__ y, int ldy, float *__restrict__ y32, int ldy32, int *err, int late) {
    if (!late) pdl_trigger();  // (late: as in rmsnorm_kernel)
    __shared__ float2 red[33];
    __shared__ float2 s_parts[kRowCl];
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ volatile int s_fail;
    __shared__ PendTile s_tiles[kRowClTiles];
    const int m = blockIdx.y;
    int i0, i1;
    row_slice(H / 4, i0, i1);
    const int t0 = (4 * i0) >> 7, nt = i1 > i0 ? ((4 * (i1 - 1)) >> 7) - t0 + 1 : 0;
    row_tiles(pend, t0, nt, s_tiles);  // depends only on the GEMM's shape
    const float4 *g4 = (const float4 *)g;
    float4 gv[kRowVals];
#pragma unroll
    for (int k = 0; k < kRowVals; ++k) {
        const int i = i0 + threadIdx.x + k * kRowClThreads;
        gv[k] = i < i1 ? __ldg(g4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (threadIdx.x == 0) s_fail = 0;
    cluster_sum_setup(&s_bar);
    pdl_wait();
    if (late) pdl_trigger();
    float4 *xr = (float4 *)(x + (size_t)m * ldx);
    float4 v[kRowVals];
    float ss = 0.f;
    // the row itself first (the residual, or the plain input), then the partials
#pragma unroll
    for (int k = 0; k < kRowVals; ++k) {
        const int i = i0 + threadIdx.x + k * kRowClThreads;
        v[k] = (i < i1 && (!pend.part || add)) ? xr[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < kRowVals; ++k) {
        const int i = i0 + threadIdx.x + k * kRowClThreads;
        if (i < i1 && pend.part) {
            const int n = 4 * i;
            const float4 p = pending_sum4(pend, s_tiles[(n >> 7) - t0], m, n & 127);
            v[k] = make_float4(v[k].x + p.x, v[k].y + p.y, v[k].z + p.z, v[k].w + p.w);
            xr[i] = v[k];
        }
        ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
    }
    const float tot = cluster_sum2(make_float2(ss, 0.f), red, s_parts, &s_bar, &s_fail).x;
    if (threadIdx.x == 0 && s_fail) set_error(err, DSPARK_ERR_TIMEOUT);
    if (!isfinite(tot) && threadIdx.x == 0 && cluster_rank() == 0) set_error(err, DSPARK_ERR_BAD_INPUT);
    const float r = rsqrtf(tot / (float)H + eps);
#pragma unroll
    for (int k = 0; k < kRowVals; ++k) {
        const int i = i0 + threadIdx.x + k * kRowClThreads;
        if (i < i1) {
            const float4 t = v[k], gg = gv[k];
            const float4 o = make_float4(t.x * r * gg.x, t.y * r * gg.y, t.z * r * gg.z, t.w * r * gg.w);
            __nv_bfloat162 *yb = (__nv_bfloat162 *)(y + (size_t)m * ldy + 4 * i);
            yb[0] = __floats2bfloat162_rn(o.x, o.y);
            yb[1] = __floats2bfloat162_rn(o.z, o.w);
            if (y32) ((float4 *)(y32 + (size_t)m * ldy32))[i] = o;
        }
    }
    cluster_wait();
}

// Latent norms and RoPE of the q_a || kv_a output (see latent_kernel), the row
// read or formed from pending partials. Grid (kRowCl, M).
__global__ void __launch_bounds__(kRowClThreads) latent_cluster_kernel(
    const float *__restrict__ qkv, int ld, GemmPending pend, int q_lora, int kv_lora, int d_rope,
    const float *__restrict__ g_q, const float *__restrict__ g_kv, float eps, const int32_t *__restrict__ ctx_len,
    int block, int max_ctx, RopeTable rt, __nv_bfloat16 *__restrict__ cq, __nv_bfloat16 *__restrict__ blk_kv,
    int *err) {
    pdl_trigger();
    __shared__ float2 red[33];
    __shared__ float2 s_parts[kRowCl];
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ volatile int s_fail;
    __shared__ PendTile s_tiles[kRowClTiles];
    const int m = blockIdx.y, b = m / block, pos_i = m % block;
    const int nq4 = q_lora / 4, nk4 = kv_lora / 4, n4 = nq4 + nk4 + d_rope / 4;
    int i0, i1;
    row_slice(n4, i0, i1);
    const int t0 = (4 * i0) >> 7, nt = i1 > i0 ? ((4 * (i1 - 1)) >> 7) - t0 + 1 : 0;
    row_tiles(pend, t0, nt, s_tiles);
    float4 gv[kRowVals];
#pragma unroll
    for (int k = 0; k < kRowVals; ++k) {
        const int i = i0 + threadIdx.x + k * kRowClThreads;
        gv[k] = i < nq4 ? __ldg((const float4 *)g_q + i)
                        : (i < nq4 + nk4 && i < i1 ? __ldg((const float4 *)g_kv + (i - nq4))
                                                   : make_float4(0.f, 0.f, 0.f, 0.f));
    }
    int c = ctx_len[b];
    if (threadIdx.x == 0) s_fail = 0;
    cluster_sum_setup(&s_bar);
    pdl_wait();
    const float4 *row = (const float4 *)(qkv + (size_t)m * ld);
    float4 v[kRowVals];
    float2 ss = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kRowVals; ++k) {
        const int i = i0 + threadIdx.x + k * kRowClThreads;
        v[k] = i < i1 ? row_value(row, pend, s_tiles, t0, m, i) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float sq = v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
        if (i < nq4)
            ss.x += sq;
        else if (i < nq4 + nk4)
            ss.y += sq;
    }
    ss = cluster_sum2(ss, red, s_parts, &s_bar, &s_fail);
    if (threadIdx.x == 0 && s_fail) set_error(err, DSPARK_ERR_TIMEOUT);
    if ((!isfinite(ss.x) || !isfinite(ss.y)) && threadIdx.x == 0 && cluster_rank() == 0)
        set_error(err, DSPARK_ERR_BAD_INPUT);
    const float rq = rsqrtf(ss.x / (float)q_lora + eps), rk = rsqrtf(ss.y / (float)kv_lora + eps);
    if (c < 0 || c > max_ctx) {
        if (threadIdx.x == 0 && cluster_rank() == 0) set_error(err, DSPARK_ERR_OOB);
        c = 0;
    }
    const int kvd = kv_lora + d_rope;
#pragma unroll
    for (int k = 0; k < kRowVals; ++k) {
        const int i = i0 + threadIdx.x + k * kRowClThreads;
        if (i >= i1) continue;
        const float4 t = v[k];
        if (i < nq4 + nk4) {
            const bool isq = i < nq4;
            const float r = isq ? rq : rk;
            const float4 gg = gv[k];
            __nv_bfloat162 *d2 = (__nv_bfloat162 *)(isq ? cq + (size_t)m * q_lora + 4 * i
                                                        : blk_kv + (size_t)m * kvd + 4 * (i - nq4));
            d2[0] = __floats2bfloat162_rn(t.x * r * gg.x, t.y * r * gg.y);
            d2[1] = __floats2bfloat162_rn(t.z * r * gg.z, t.w * r * gg.w);
        } else {
            // two RoPE pairs (2p, 2p + 1), p = 2 (i - nq4 - nk4) and the next
            const int p = 2 * (i - nq4 - nk4);
            const double pos = (double)(c + pos_i);
            float c0, s0, c1, s1;
            rope_cs(pos, rt.inv_freq[p], c0, s0);
            rope_cs(pos, rt.inv_freq[p + 1], c1, s1);
            __nv_bfloat16 *dst = blk_kv + (size_t)m * kvd + kv_lora + 2 * p;
            dst[0] = __float2bfloat16(t.x * c0 - t.y * s0);
            dst[1] = __float2bfloat16(t.x * s0 + t.y * c0);
            dst[2] = __float2bfloat16(t.z * c1 - t.w * s1);
            dst[3] = __float2bfloat16(t.z * s1 + t.w * c1);
        }
    }
    cluster_wait();
}

// ---------------------------------------------------------------------------
// q absorption: Q_h = [W_kb,h^T q_nope,h || RoPE(q_rope,h)] per row and head,
// bf16 [M, n_h, kv_lora + d_rope]. Grid (n_h, kv_lora / 64), 128 threads: a CTA
// owns one head and 64 latent columns; warp w takes the quarter w of d_nope and
// lane l the column pair 2l, so every d row of W_kb is one coalesced 128-byte
// read. The thread's W_kb slice (<= 64 bf16 pairs) is loaded once into
// registers; the rows sweep in chunks of 8 from shared memory and the four
// quarter sums are added in quarter order.
// ---------------------------------------------------------------------------
constexpr int kQAbsRows = 8;
constexpr int kQAbsTiles = 4;  // channel tiles of one head's q (d_nope + d_rope <= 384)
constexpr int kQAbsCols = 64;

template <int MAXDQ>
__global__ void __launch_bounds__(128) q_absorb_kernel(const float *__restrict__ q, int M, int n_h, int d_nope,
                                                       int d_rope, int kv_lora, int d_v,
                                                       const __nv_bfloat16 *__restrict__ w_kvb,
                                                       const int32_t *__restrict__ ctx_len, int block, int max_ctx,
                                                       RopeTable rt, __nv_bfloat16 *__restrict__ qt,
                                                       GemmPending pend) {
    pdl_trigger();
    extern __shared__ float sm[];
    __shared__ PendTile s_tiles[kQAbsTiles];
    float *sq = sm;                             // [kQAbsRows][d_nope]
    float *red = sm + kQAbsRows * d_nope;       // [4][kQAbsRows][kQAbsCols]
    const int h = blockIdx.x, c0 = blockIdx.y * kQAbsCols;
    const int lane = threadIdx.x & 31, qd = threadIdx.x >> 5;
    const int dq = d_nope / 4;  // <= 64
    const int qhd = d_nope + d_rope, kvd = kv_lora + d_rope;
    // q may be pending (the q_b GEMM's split partials): the slots of the head's channel tiles
    const int qt0 = (h * qhd) >> 7, qnt = ((h * qhd + qhd - 1) >> 7) - qt0 + 1;
    if (pend.part && (int)threadIdx.x < qnt) s_tiles[threadIdx.x] = pend_tile(pend, qt0 + threadIdx.x);
    __syncthreads();
    auto qval = [&](int m, int d) -> float {
        if (!pend.part) return q[((size_t)m * n_h + h) * qhd + d];
        const int n = h * qhd + d;
        return pending_sum1(pend, s_tiles[(n >> 7) - qt0], m, n & 127);
    };
    // the weights do not depend on the previous kernel: load them before the wait
    const __nv_bfloat16 *W = w_kvb + ((size_t)h * (d_nope + d_v) + qd * dq) * kv_lora + c0 + 2 * lane;
    uint32_t w[MAXDQ];
#pragma unroll
    for (int i = 0; i < MAXDQ; ++i) w[i] = i < dq ? __ldg((const unsigned int *)(W + (size_t)i * kv_lora)) : 0u;
    pdl_wait();
    for (int m0 = 0; m0 < M; m0 += kQAbsRows) {
        // one round of independent loads: thread t takes d = t, t + 128 of every row
#pragma unroll
        for (int dd = 0; dd < 2; ++dd) {
            const int d = threadIdx.x + dd * 128;
            float v[kQAbsRows];
#pragma unroll
            for (int mm = 0; mm < kQAbsRows; ++mm)
                v[mm] = (d < d_nope && m0 + mm < M) ? qval(m0 + mm, d) : 0.f;
            if (d < d_nope) {
#pragma unroll
                for (int mm = 0; mm < kQAbsRows; ++mm) sq[mm * d_nope + d] = v[mm];
            }
        }
        __syncthreads();
        float a0[kQAbsRows], a1[kQAbsRows];
#pragma unroll
        for (int mm = 0; mm < kQAbsRows; ++mm) a0[mm] = a1[mm] = 0.f;
#pragma unroll
        for (int i = 0; i < MAXDQ; ++i) {
            if (i < dq) {
                const float2 wf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
#pragma unroll
                for (int mm = 0; mm < kQAbsRows; ++mm) {
                    const float x = sq[mm * d_nope + qd * dq + i];
                    a0[mm] = fmaf(wf.x, x, a0[mm]);
                    a1[mm] = fmaf(wf.y, x, a1[mm]);
                }
            }
        }
#pragma unroll
        for (int mm = 0; mm < kQAbsRows; ++mm)
            *(float2 *)(red + ((size_t)qd * kQAbsRows + mm) * kQAbsCols + 2 * lane) = make_float2(a0[mm], a1[mm]);
        __syncthreads();
        for (int idx = threadIdx.x; idx < kQAbsRows * kQAbsCols / 2; idx += blockDim.x) {
            const int mm = idx / (kQAbsCols / 2), c2 = 2 * (idx % (kQAbsCols / 2)), m = m0 + mm;
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const float2 v = *(const float2 *)(red + ((size_t)g * kQAbsRows + mm) * kQAbsCols + c2);
                s0 += v.x;
                s1 += v.y;
            }
            if (m < M) *(__nv_bfloat162 *)(qt + ((size_t)m * n_h + h) * kvd + c0 + c2) = __floats2bfloat162_rn(s0, s1);
        }
        __syncthreads();
    }
    {
        // RoPE of q_rope, the rows spread over the head's column blocks
        const int np = d_rope / 2;
        for (int idx = blockIdx.y * blockDim.x + threadIdx.x; idx < M * np; idx += gridDim.y * blockDim.x) {
            const int m = idx / np, p = idx % np;
            int c = ctx_len[m / block];
            if (c < 0 || c > max_ctx) c = 0;
            float fc, fs;
            rope_cs((double)(c + m % block), rt.inv_freq[p], fc, fs);
            const float x0 = qval(m, d_nope + 2 * p), x1 = qval(m, d_nope + 2 * p + 1);
            __nv_bfloat16 *dst = qt + ((size_t)m * n_h + h) * kvd + kv_lora;
            dst[2 * p] = __float2bfloat16(x0 * fc - x1 * fs);
            dst[2 * p + 1] = __float2bfloat16(x0 * fs + x1 * fc);
        }
    }
}

// ---------------------------------------------------------------------------
// q absorption on 256-column chunks (the form the draft step uses): grid
// (n_h, ceil(kv_lora / 256)), 256 threads, one CTA per head and chunk, so the
// whole grid is one wave (its k_b slices come from L2: the q_b GEMM pulls
// kv_b there while it runs). Warp w takes
// columns [64 (w % 4), +64) of the chunk (lane l the pair 2l) and the half
// w / 4 of d_nope; the thread's slice (d_nope / 2 rows of one column pair)
// stays in registers. The 8 staged rows are swept at once from shared memory; the two
// halves' sums are added in half order.
// ---------------------------------------------------------------------------
constexpr int kQAbs2Cols = 256;
constexpr int kQAbs2Threads = 256;
constexpr int kQAbs2Rows = 8;
constexpr int kQAbs2MaxRope = 128;

template <int MAXDH>
__global__ void __launch_bounds__(kQAbs2Threads, 1) q_absorb2_kernel(
    const float *__restrict__ q, int M, int n_h, int d_nope, int d_rope, int kv_lora, int d_v,
    const __nv_bfloat16 *__restrict__ w_kvb, const int32_t *__restrict__ ctx_len, int block, int max_ctx,
    RopeTable rt, __nv_bfloat16 *__restrict__ qt, GemmPending pend) {
    pdl_trigger();
    // the head's q rows of a chunk of 8: nope and rope parts, staged in one batch of loads
    constexpr int LD = 2 * MAXDH + kQAbs2MaxRope;
    constexpr int kPer4 = kQAbsRows * LD / 4 / kQAbs2Threads;  // staged float4 per thread
    static_assert(kQAbsRows * LD % (4 * kQAbs2Threads) == 0, "whole float4 per thread");
    __shared__ __align__(16) float sq[kQAbsRows][LD];
    __shared__ float2 red[kQAbs2Rows][kQAbs2Cols / 2];  // the second half's sums
    __shared__ PendTile s_tiles[kQAbsTiles];
    const int h = blockIdx.x, c0 = blockIdx.y * kQAbs2Cols;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cg = warp & 3, half = warp >> 2;
    const int dh = d_nope / 2;
    const int cp = 32 * cg + lane;  // column pair within the chunk
    const int col = c0 + 2 * cp;
    const bool colv = col < kv_lora;
    const int qhd = d_nope + d_rope, kvd = kv_lora + d_rope;
    const int qt0 = (h * qhd) >> 7, qnt = ((h * qhd + qhd - 1) >> 7) - qt0 + 1;
    if (pend.part && (int)threadIdx.x < qnt) s_tiles[threadIdx.x] = pend_tile(pend, qt0 + threadIdx.x);
    // the k_b slice does not depend on the previous kernel: load it before the wait
    const __nv_bfloat16 *W = w_kvb + ((size_t)h * (d_nope + d_v) + half * dh) * kv_lora + col;
    uint32_t w[MAXDH];
#pragma unroll
    for (int i = 0; i < MAXDH; ++i)
        w[i] = (i < dh && colv) ? __ldg((const unsigned int *)(W + (size_t)i * kv_lora)) : 0u;
    const int np = d_rope / 2;
    __syncthreads();
    for (int m0 = 0; m0 < M; m0 += kQAbsRows) {
        // this thread's RoPE pair of the chunk (CTA column chunk 0 rotates): the angle
        // depends only on the inputs, so it is formed before the dependency wait
        const int rp = threadIdx.x, rmm = rp / (np > 0 ? np : 1), rpp = rp % (np > 0 ? np : 1);
        const bool rope_here = blockIdx.y == 0 && np > 0 && rp < kQAbsRows * np && m0 + rmm < M;
        float fc = 1.f, fs = 0.f;
        if (rope_here) {
            const int m = m0 + rmm;
            int c = ctx_len[m / block];
            if (c < 0 || c > max_ctx) c = 0;
            rope_cs((double)(c + m % block), rt.inv_freq[rpp], fc, fs);
        }
        if (m0 == 0) pdl_wait();
        // every position of the staged rows is written: the sweep multiplies the
        // ones past d_nope by zero weights, and stale bits there could be Inf or NaN.
        // Four positions per load; a pending q_b output is summed for all of the
        // thread's positions in one round trip.
        float4 v[kPer4];
        {
            PendTile tl[kPer4];
            int mr[kPer4], rr[kPer4];
            bool live[kPer4];
#pragma unroll
            for (int k = 0; k < kPer4; ++k) {
                const int idx = threadIdx.x + k * kQAbs2Threads, mm = idx / (LD / 4), pos = 4 * (idx % (LD / 4));
                const int m = m0 + mm;
                const int d = pos < d_nope ? pos
                                           : (pos >= 2 * MAXDH && pos < 2 * MAXDH + d_rope ? d_nope + pos - 2 * MAXDH : -1);
                live[k] = m < M && d >= 0;
                const int n = h * qhd + (live[k] ? d : 0);
                mr[k] = live[k] ? m : 0;
                rr[k] = n & 127;
                v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (!pend.part) {
                    if (live[k]) v[k] = __ldg((const float4 *)(q + ((size_t)m * n_h + h) * qhd + d));
                } else {
                    tl[k] = s_tiles[(n >> 7) - qt0];
                }
            }
            if (pend.part) pending_sum4_multi<kPer4, 4>(pend, tl, mr, rr, live, v);
        }
#pragma unroll
        for (int k = 0; k < kPer4; ++k) {
            const int idx = threadIdx.x + k * kQAbs2Threads;
            *(float4 *)&sq[idx / (LD / 4)][4 * (idx % (LD / 4))] = v[k];
        }
        __syncthreads();
        if (rope_here) {
            const int m = m0 + rmm;
            const float x0 = sq[rmm][2 * MAXDH + 2 * rpp], x1 = sq[rmm][2 * MAXDH + 2 * rpp + 1];
            __nv_bfloat16 *dst = qt + ((size_t)m * n_h + h) * kvd + kv_lora;
            dst[2 * rpp] = __float2bfloat16(x0 * fc - x1 * fs);
            dst[2 * rpp + 1] = __float2bfloat16(x0 * fs + x1 * fc);
        }
        for (int r0 = 0; r0 < kQAbsRows; r0 += kQAbs2Rows) {
            float a0[kQAbs2Rows], a1[kQAbs2Rows];
#pragma unroll
            for (int mm = 0; mm < kQAbs2Rows; ++mm) a0[mm] = a1[mm] = 0.f;
            const float *sqh = &sq[r0][0] + half * dh;
#pragma unroll
            for (int i = 0; i < MAXDH; i += 4) {
                float2 wf[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) wf[j] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i + j]));
#pragma unroll
                for (int mm = 0; mm < kQAbs2Rows; ++mm) {
                    const float4 x = *(const float4 *)(sqh + mm * LD + i);
                    a0[mm] = fmaf(wf[0].x, x.x, a0[mm]);
                    a1[mm] = fmaf(wf[0].y, x.x, a1[mm]);
                    a0[mm] = fmaf(wf[1].x, x.y, a0[mm]);
                    a1[mm] = fmaf(wf[1].y, x.y, a1[mm]);
                    a0[mm] = fmaf(wf[2].x, x.z, a0[mm]);
                    a1[mm] = fmaf(wf[2].y, x.z, a1[mm]);
                    a0[mm] = fmaf(wf[3].x, x.w, a0[mm]);
                    a1[mm] = fmaf(wf[3].y, x.w, a1[mm]);
                }
            }
            if (half == 1) {
#pragma unroll
                for (int mm = 0; mm < kQAbs2Rows; ++mm) red[mm][cp] = make_float2(a0[mm], a1[mm]);
            }
            __syncthreads();
            if (half == 0 && colv) {
#pragma unroll
                for (int mm = 0; mm < kQAbs2Rows; ++mm) {
                    const int m = m0 + r0 + mm;
                    if (m < M) {
                        const float2 o = red[mm][cp];
                        *(__nv_bfloat162 *)(qt + ((size_t)m * n_h + h) * kvd + col) =
                            __floats2bfloat162_rn(a0[mm] + o.x, a1[mm] + o.y);
                    }
                }
            }
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------------------
// Split combine fused with the v absorption (after the tensor-core attention):
// grid (n_h, ceil(M / 4)), 512 threads, one CTA per head and 4 rows. The CTA
// copies the head's v_b rows (d_v x kv_lora bf16; in L2: the q_b GEMM pulls
// kv_b in) into shared memory with asynchronous copies issued before the
// dependency wait, rows padded by 16 bytes (the rows a warp reads at once fall
// in different banks); forms its rows of o_lat from the attention's split
// partials (sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s over the non-empty
// splits, in split order; o_lat is read as is when there is one split), each
// thread loading its row's (m_s, l_s) with its partials in one round trip;
// then thread t forms the dot products of the channel pair (t % 64, 64 + t % 64)
// over the eighth t / 64 of the latent for the 4 rows, and the eighths are
// added in order through shared memory.
// ---------------------------------------------------------------------------
constexpr int kCVRows = 4;
constexpr int kCVThreads = 512;
constexpr int kCVMaxSplit = 20;
DS_DEVINL void cp_async16(void *smem_dst, const void *gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}

constexpr int kCVPairs = 64;                     // channel pairs per pass
constexpr int kCVParts = kCVThreads / kCVPairs;  // latent parts (8)

__global__ void __launch_bounds__(kCVThreads) attn_combine_vabsorb_kernel(
    const float *__restrict__ part_o, const float *__restrict__ part_ml, int splits, int R,
    const float *__restrict__ o_lat, int M, int n_h, int block, int d_nope, int d_v, int kv_lora,
    const __nv_bfloat16 *__restrict__ w_kvb, __nv_bfloat16 *__restrict__ out, const int32_t *__restrict__ ctx_len,
    int max_ctx, int cps) {
    pdl_trigger();
    extern __shared__ __align__(16) uint8_t smc[];
    const int wstride = kv_lora * 2 + 16;                              // bytes per staged v_b row
    uint8_t *sw = smc;                                                 // [d_v][wstride]
    float *so = (float *)(smc + (size_t)d_v * wstride);                // [kCVRows][kv_lora]
    float *sred = so + kCVRows * kv_lora;                              // [kCVParts][kCVRows][2 kCVPairs]
    const int h = blockIdx.x, m0 = blockIdx.y * kCVRows;
    const int mr = min(kCVRows, M - m0);
    const int c4n = kv_lora / 4;
    // the head's v_b rows: weights of the step, copied before the dependency wait
    const int c8n = kv_lora / 8;
    const uint4 *W4 = (const uint4 *)(w_kvb + ((size_t)h * (d_nope + d_v) + d_nope) * kv_lora);
    for (int i = threadIdx.x; i < d_v * c8n; i += blockDim.x)
        cp_async16(sw + (size_t)(i / c8n) * wstride + (i % c8n) * 16, W4 + i);
    asm volatile("cp.async.commit_group;" ::: "memory");
    pdl_wait();
    if (splits > 1) {
        // each thread loads its row's (max, sum) pairs with its partials (one round
        // trip) and forms the weights itself
        for (int i = threadIdx.x; i < kCVRows * c4n; i += blockDim.x) {
            const int mm = i / c4n, c4 = i % c4n;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            if (mm < mr) {
                const int m = m0 + mm, b = m / block, r = (m % block) * n_h + h;
                // the splits that hold chunks of this sequence (the others wrote only
                // an empty (max, sum) pair and no partial)
                int cx = ctx_len[b];
                if (cx < 0 || cx > max_ctx) cx = 0;
                const int nsv = min(splits, ((cx + 63) / 64 + 1 + cps - 1) / cps);
                const float *ml = part_ml + ((size_t)b * splits * R + r) * 2;
                const float4 *src = (const float4 *)(part_o + ((size_t)b * splits * R + r) * kv_lora) + c4;
                const size_t sstep = (size_t)R * kv_lora / 4;
                float2 w[kCVMaxSplit];
                float4 v[kCVMaxSplit];
#pragma unroll
                for (int s = 0; s < kCVMaxSplit; ++s) {
                    w[s] = s < nsv ? __ldcg((const float2 *)(ml + (size_t)s * R * 2)) : make_float2(0.f, 0.f);
                    v[s] = s < nsv ? __ldcg(src + s * sstep) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                float mx = -INFINITY;
#pragma unroll
                for (int s = 0; s < kCVMaxSplit; ++s)
                    if (s < nsv && w[s].y > 0.f) mx = fmaxf(mx, w[s].x);
                float den = 0.f;
#pragma unroll
                for (int s = 0; s < kCVMaxSplit; ++s) {
                    if (s < nsv && w[s].y > 0.f) {
                        const float e = exp2f(w[s].x - mx);
                        den += e * w[s].y;
                        acc.x += e * v[s].x;
                        acc.y += e * v[s].y;
                        acc.z += e * v[s].z;
                        acc.w += e * v[s].w;
                    }
                }
                const float inv = den > 0.f ? 1.f / den : 0.f;
                acc = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            }
            ((float4 *)so)[mm * c4n + c4] = acc;
        }
    } else {
        for (int i = threadIdx.x; i < kCVRows * c4n; i += blockDim.x) {
            const int mm = i / c4n, c4 = i % c4n;
            ((float4 *)so)[i] = mm < mr ? __ldcg((const float4 *)(o_lat + ((size_t)(m0 + mm) * n_h + h) * kv_lora) + c4)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    // v absorption: thread t takes the channel pair (e0 + t % 64, e0 + 64 + t % 64)
    // over the latent eighth t / 64 for the 4 rows (one read of a row of o serves
    // both channels); the eighths are added in order through shared memory
    const int part = threadIdx.x / kCVPairs, pr = threadIdx.x % kCVPairs, cp = kv_lora / kCVParts;
    for (int e0 = 0; e0 < d_v; e0 += 2 * kCVPairs) {
        const int ea = e0 + pr, eb = e0 + kCVPairs + pr;
        float a[2][kCVRows];
#pragma unroll
        for (int mm = 0; mm < kCVRows; ++mm) a[0][mm] = a[1][mm] = 0.f;
        if (ea < d_v) {
            const bool hb = eb < d_v;
            const uint8_t *wa = sw + (size_t)ea * wstride + part * cp * 2;
            const uint8_t *wb = sw + (size_t)(hb ? eb : ea) * wstride + part * cp * 2;
            const float *orow = so + part * cp;
            for (int c = 0; c < cp; c += 8) {
                float wf[2][8];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const uint4 wq = *(const uint4 *)((k ? wb : wa) + c * 2);
                    const uint32_t wu[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wu[j]));
                        wf[k][2 * j] = f.x;
                        wf[k][2 * j + 1] = f.y;
                    }
                }
#pragma unroll
                for (int mm = 0; mm < kCVRows; ++mm) {
                    const float4 x0 = *(const float4 *)(orow + mm * kv_lora + c);
                    const float4 x1 = *(const float4 *)(orow + mm * kv_lora + c + 4);
                    const float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                    for (int k = 0; k < 2; ++k)
#pragma unroll
                        for (int j = 0; j < 8; ++j) a[k][mm] = fmaf(wf[k][j], x[j], a[k][mm]);
                }
            }
        }
#pragma unroll
        for (int mm = 0; mm < kCVRows; ++mm) {
            sred[(part * kCVRows + mm) * (2 * kCVPairs) + pr] = a[0][mm];
            sred[(part * kCVRows + mm) * (2 * kCVPairs) + kCVPairs + pr] = a[1][mm];
        }
        __syncthreads();
        if ((int)threadIdx.x < kCVRows * 2 * kCVPairs) {
            const int mm = threadIdx.x / (2 * kCVPairs), ee = threadIdx.x % (2 * kCVPairs), e2 = e0 + ee;
            if (mm < mr && e2 < d_v) {
                float t = 0.f;
#pragma unroll
                for (int pp = 0; pp < kCVParts; ++pp) t += sred[(pp * kCVRows + mm) * (2 * kCVPairs) + ee];
                out[(size_t)(m0 + mm) * n_h * d_v + (size_t)h * d_v + e2] = __float2bfloat16(t);
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// v absorption: o_h = W_vb,h o_lat,h -> bf16 [M, n_h * d_v] (operand of o_proj).
// Grid (n_h, d_v / 16): a CTA owns 16 output channels of one head; 16 threads
// per channel each hold 4-element slices of the channel's W_vb row at
// interleaved float4 positions (so a half-warp reads 16 consecutive float4 of
// the latent: no bank conflicts), read once; the rows sweep in chunks of 16
// from shared memory; the 16 partial dots are reduced with shuffles.
// ---------------------------------------------------------------------------
constexpr int kVAbsRows = 8;

__global__ void __launch_bounds__(256, 4) v_absorb_kernel(const float *__restrict__ o_lat, int M, int n_h, int d_nope,
                                                       int d_v, int kv_lora, const __nv_bfloat16 *__restrict__ w_kvb,
                                                       __nv_bfloat16 *__restrict__ out) {
    pdl_trigger();
    extern __shared__ float so[];  // [kVAbsRows][kv_lora]
    const int h = blockIdx.x, e = blockIdx.y * 16 + (threadIdx.x >> 4), cg = threadIdx.x & 15;
    const __nv_bfloat16 *W = w_kvb + ((size_t)h * (d_nope + d_v) + d_nope + e) * kv_lora;
    const int nj = kv_lora / 64;  // float4 slices per thread (<= 8)
    // the weights do not depend on the previous kernel: read them before the wait
    float wv[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (j < nj) {
            const uint2 u = __ldg((const uint2 *)(W + 4 * (cg + 16 * j)));
            const float2 f0 = __bfloat1622float2(*(const __nv_bfloat162 *)&u.x);
            const float2 f1 = __bfloat1622float2(*(const __nv_bfloat162 *)&u.y);
            wv[j][0] = f0.x;
            wv[j][1] = f0.y;
            wv[j][2] = f1.x;
            wv[j][3] = f1.y;
        } else {
            wv[j][0] = wv[j][1] = wv[j][2] = wv[j][3] = 0.f;
        }
    }
    pdl_wait();
    const int c4n = kv_lora / 4;  // float4 per row (<= 128)
    for (int m0 = 0; m0 < M; m0 += kVAbsRows) {
        // one round of loads: thread t takes float4 column t % c4n of rows t / c4n + k * (256 / c4n)
        // kv_lora = 512: two rows per pass, four passes, all loads issued first
        float4 v[4];
        const int rstep = blockDim.x / c4n, c4 = threadIdx.x % c4n, rr0 = threadIdx.x / c4n;
        for (int k0 = 0; k0 * rstep < kVAbsRows; k0 += 4) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int mm = rr0 + (k0 + k) * rstep, m = m0 + mm;
                v[k] = (mm < kVAbsRows && m < M) ? ((const float4 *)(o_lat + ((size_t)m * n_h + h) * kv_lora))[c4]
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int mm = rr0 + (k0 + k) * rstep;
                if (mm < kVAbsRows) ((float4 *)so)[mm * c4n + c4] = v[k];
            }
        }
        __syncthreads();
        const int mmax = min(kVAbsRows, M - m0);
        for (int mm = 0; mm < mmax; ++mm) {
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (j < nj) {
                    const float4 x = *(const float4 *)(so + mm * kv_lora + 4 * (cg + 16 * j));
                    acc = fmaf(wv[j][0], x.x, acc);
                    acc = fmaf(wv[j][1], x.y, acc);
                    acc = fmaf(wv[j][2], x.z, acc);
                    acc = fmaf(wv[j][3], x.w, acc);
                }
            }
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (cg == 0) out[(size_t)(m0 + mm) * n_h * d_v + (size_t)h * d_v + e] = __float2bfloat16(acc);
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// MLA attention over the paged latent cache plus the block's own latents.
//
// All block * n_h query rows of a sequence share one latent key/value per token
// (K_j = [c_kv,j || k_r,j], V_j = c_kv,j), so every row of a CTA attends to the
// same 64-token chunks. A CTA owns 64 query rows and one contiguous range of
// tokens (split of the KV sequence); 8 warps: warp w computes the scores of
// rows 16*(w%4).. for the full key width and the output columns of half (w/4)
// of the latent. Scores and P.V use mma.sync m16n8k16 (bf16 in, fp32
// accumulate); the softmax is the online (running max) form in base 2.
// Tokens: j < ctx from the page pool, ctx <= j < ctx + block from the block
// latents; non-causal, so nothing is masked except past the range end.
// ---------------------------------------------------------------------------
DS_DEVINL void cp_async16(void *smem, const void *gmem, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem)), "l"(gmem), "r"(src_bytes)
                 : "memory");
}
DS_DEVINL void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
DS_DEVINL void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

DS_DEVINL void ldsm_x4(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
DS_DEVINL void ldsm_x4_t(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
DS_DEVINL void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, "
        "%2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
DS_DEVINL uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *(uint32_t *)&v;
}

template <int DQK, int DV>
struct AttnCfg {
    static constexpr int kRows = 64;
    static constexpr int kTok = 64;
    static constexpr int kPitch = DQK + 8;  // bf16 per smem row: +16 B keeps ldmatrix conflict-free
    static constexpr int kQBytes = kRows * kPitch * 2;
    static constexpr int kKVBytes = kTok * kPitch * 2;
    static constexpr int kSmem = kQBytes + 2 * kKVBytes;
    static constexpr int kNT = DV / 2 / 8;   // O n8-tiles per warp
    static constexpr int kChunks = DQK / 8;  // 16-byte pieces per row
    static_assert(DQK % 16 == 0 && DV % 32 == 0 && DV <= DQK, "latent dims");
};

template <int DQK, int DV>
__global__ void __launch_bounds__(256, 1) mla_attention_kernel(const AttnParams p) {
    pdl_trigger();
    pdl_wait();
    using C = AttnCfg<DQK, DV>;
    extern __shared__ __align__(16) uint8_t smem[];
    __nv_bfloat16 *sQ = (__nv_bfloat16 *)smem;
    __nv_bfloat16 *sKV = (__nv_bfloat16 *)(smem + C::kQBytes);

    const int b = blockIdx.z, split = blockIdx.y, r0 = blockIdx.x * C::kRows;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int ctx = p.ctx_len[b];
    if (ctx < 0 || ctx > p.max_ctx) {
        if (threadIdx.x == 0) set_error(p.err, DSPARK_ERR_OOB);
        ctx = 0;
    }
    const int ntok = ctx + p.block;
    const int j_begin = split * p.tok_per_split;
    const int j_end = min(ntok, j_begin + p.tok_per_split);
    const int nchunks = j_end > j_begin ? (j_end - j_begin + C::kTok - 1) / C::kTok : 0;

    const __nv_bfloat16 *qbase = p.qt + (size_t)b * p.R * DQK;
    for (int idx = threadIdx.x; idx < C::kRows * C::kChunks; idx += blockDim.x) {
        const int rr = idx / C::kChunks, ch = idx % C::kChunks, r = r0 + rr;
        const bool ok = r < p.R;
        cp_async16(sQ + rr * C::kPitch + ch * 8, qbase + (size_t)(ok ? r : 0) * DQK + ch * 8, ok ? 16 : 0);
    }
    auto load_chunk = [&](int ci, int buf) {
        __nv_bfloat16 *dst = sKV + buf * (C::kKVBytes / 2);
        const int j0 = j_begin + ci * C::kTok;
        for (int idx = threadIdx.x; idx < C::kTok * C::kChunks; idx += blockDim.x) {
            const int t = idx / C::kChunks, ch = idx % C::kChunks, j = j0 + t;
            const __nv_bfloat16 *src = p.blk_kv;
            int bytes = 0;
            if (j < j_end) {
                if (j < ctx) {
                    const int pg = p.page_table[(size_t)b * p.max_pages + j / p.page];
                    if (pg >= 0 && pg < p.n_pages) {
                        src = p.pool + ((size_t)pg * p.page + (j % p.page)) * DQK + ch * 8;
                        bytes = 16;
                    } else if (ch == 0) {
                        set_error(p.err, DSPARK_ERR_OOB);
                    }
                } else {
                    src = p.blk_kv + ((size_t)b * p.block + (j - ctx)) * DQK + ch * 8;
                    bytes = 16;
                }
            }
            cp_async16(dst + t * C::kPitch + ch * 8, src, bytes);
        }
    };
    if (nchunks > 0) load_chunk(0, 0);
    cp_async_commit();

    const int rg = warp & 3, vh = warp >> 2;
    const int g = lane >> 2, tq = lane & 3;
    float o[C::kNT][4];
#pragma unroll
    for (int i = 0; i < C::kNT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

    for (int ci = 0; ci < nchunks; ++ci) {
        if (ci + 1 < nchunks) load_chunk(ci + 1, (ci + 1) & 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const __nv_bfloat16 *kv = sKV + (ci & 1) * (C::kKVBytes / 2);
        float s[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll 4
        for (int kk = 0; kk < DQK / 16; ++kk) {
            uint32_t a[4];
            ldsm_x4(a, sQ + (rg * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * C::kPitch + kk * 16 + (lane >> 4) * 8);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bb[4];
                ldsm_x4(bb, kv + (np * 16 + (lane & 7) + ((lane >> 4) << 3)) * C::kPitch + kk * 16 +
                                ((lane >> 3) & 1) * 8);
                mma16816(s[2 * np], a, bb[0], bb[1]);
                mma16816(s[2 * np + 1], a, bb[2], bb[3]);
            }
        }
        const int j0 = j_begin + ci * C::kTok;
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = j0 + nt * 8 + 2 * tq + (e & 1);
                s[nt][e] = (j < j_end) ? s[nt][e] * p.scale_log2 : -INFINITY;
                mx[e >> 1] = fmaxf(mx[e >> 1], s[nt][e]);
            }
        }
        float corr[2], base[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            mx[h2] = fmaxf(mx[h2], __shfl_xor_sync(0xffffffffu, mx[h2], 1));
            mx[h2] = fmaxf(mx[h2], __shfl_xor_sync(0xffffffffu, mx[h2], 2));
            const float mn = fmaxf(mrow[h2], mx[h2]);
            base[h2] = (mn == -INFINITY) ? 0.f : mn;
            corr[h2] = exp2f(mrow[h2] - base[h2]);
            mrow[h2] = mn;
        }
        float ls[2] = {0.f, 0.f};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                s[nt][e] = exp2f(s[nt][e] - base[e >> 1]);
                ls[e >> 1] += s[nt][e];
            }
        }
        lrow[0] = lrow[0] * corr[0] + ls[0];
        lrow[1] = lrow[1] * corr[1] + ls[1];
#pragma unroll
        for (int nt = 0; nt < C::kNT; ++nt) {
            o[nt][0] *= corr[0];
            o[nt][1] *= corr[0];
            o[nt][2] *= corr[1];
            o[nt][3] *= corr[1];
        }
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
            uint32_t pa[4];
            pa[0] = pack_bf16(s[2 * kt][0], s[2 * kt][1]);
            pa[1] = pack_bf16(s[2 * kt][2], s[2 * kt][3]);
            pa[2] = pack_bf16(s[2 * kt + 1][0], s[2 * kt + 1][1]);
            pa[3] = pack_bf16(s[2 * kt + 1][2], s[2 * kt + 1][3]);
#pragma unroll
            for (int ntp = 0; ntp < C::kNT / 2; ++ntp) {
                uint32_t vb[4];
                ldsm_x4_t(vb, kv + (kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * C::kPitch + vh * (DV / 2) +
                                  ntp * 16 + (lane >> 4) * 8);
                mma16816(o[2 * ntp], pa, vb[0], vb[1]);
                mma16816(o[2 * ntp + 1], pa, vb[2], vb[3]);
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        lrow[h2] += __shfl_xor_sync(0xffffffffu, lrow[h2], 1);
        lrow[h2] += __shfl_xor_sync(0xffffffffu, lrow[h2], 2);
    }
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        const int r = r0 + rg * 16 + g + 8 * h2;
        if (r >= p.R) continue;
        if (p.splits == 1) {
            const float inv = lrow[h2] > 0.f ? 1.f / lrow[h2] : 0.f;
            float *dst = p.o_lat + ((size_t)b * p.R + r) * DV + vh * (DV / 2);
#pragma unroll
            for (int nt = 0; nt < C::kNT; ++nt)
                *(float2 *)(dst + nt * 8 + 2 * tq) = make_float2(o[nt][2 * h2] * inv, o[nt][2 * h2 + 1] * inv);
        } else {
            const size_t pr = ((size_t)b * p.splits + split) * p.R + r;
            float *dst = p.part_o + pr * DV + vh * (DV / 2);
#pragma unroll
            for (int nt = 0; nt < C::kNT; ++nt)
                *(float2 *)(dst + nt * 8 + 2 * tq) = make_float2(o[nt][2 * h2], o[nt][2 * h2 + 1]);
            if (vh == 0 && tq == 0) *(float2 *)(p.part_ml + pr * 2) = make_float2(mrow[h2], lrow[h2]);
        }
    }
}

// Fixed-order merge of the split partials: o = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s.
// The split weights are formed once in shared memory; each thread then reads
// its 4 columns of every split with independent loads.
__global__ void attn_combine_kernel(const float *__restrict__ part_o, const float *__restrict__ part_ml, int splits,
                                    int R, int DV, float *__restrict__ o_lat) {
    pdl_trigger();
    pdl_wait();
    __shared__ float sml[64][2];
    const int r = blockIdx.x, b = blockIdx.y;
    const size_t base = (size_t)b * splits * R + r;
    if (threadIdx.x < splits) {
        const float2 ml = *(const float2 *)(part_ml + (base + (size_t)threadIdx.x * R) * 2);
        sml[threadIdx.x][0] = ml.x;
        sml[threadIdx.x][1] = ml.y;
    }
    __syncthreads();
    // every thread forms the same weights from shared memory (fixed split order)
    float M = -INFINITY;
    for (int s = 0; s < splits; ++s)
        if (sml[s][1] > 0.f) M = fmaxf(M, sml[s][0]);
    float den = 0.f;
    for (int s = 0; s < splits; ++s)
        if (sml[s][1] > 0.f) den += exp2f(sml[s][0] - M) * sml[s][1];
    const float inv = den > 0.f ? 1.f / den : 0.f;
    for (int c = threadIdx.x * 4; c < DV; c += blockDim.x * 4) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int s = 0; s < splits; ++s) {
            if (!(sml[s][1] > 0.f)) continue;  // an empty split wrote no partial
            const float w = exp2f(sml[s][0] - M);
            const float4 v = __ldcg((const float4 *)(part_o + (base + (size_t)s * R) * DV + c));
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        }
        *(float4 *)(o_lat + ((size_t)b * R + r) * DV + c) =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
}

// Confidence head: c = sigmoid(w . h_out + b) per block row (H a multiple of 4;
// one CTA per row, the weight slice read before the wait, fixed-order sums).
__global__ void confidence_kernel(const float *__restrict__ h_out, int H, const float *__restrict__ w, float bias,
                                  float *__restrict__ conf) {
    pdl_trigger();
    __shared__ float red[33];
    const int m = blockIdx.x, n4 = H / 4;
    const float4 *w4 = (const float4 *)w;
    const float4 *x4 = (const float4 *)(h_out + (size_t)m * H);
    float4 wr[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = threadIdx.x + u * blockDim.x;
        wr[u] = i < n4 ? __ldg(w4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    pdl_wait();
    float acc = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = threadIdx.x + u * blockDim.x;
        if (i < n4) {
            const float4 x = x4[i];
            acc = fmaf(wr[u].x, x.x, fmaf(wr[u].y, x.y, fmaf(wr[u].z, x.z, fmaf(wr[u].w, x.w, acc))));
        }
    }
    for (int i = threadIdx.x + 4 * blockDim.x; i < n4; i += blockDim.x) {
        const float4 ww = w4[i], x = x4[i];
        acc = fmaf(ww.x, x.x, fmaf(ww.y, x.y, fmaf(ww.z, x.z, fmaf(ww.w, x.w, acc))));
    }
    acc = block_sum(acc, red);
    if (threadIdx.x == 0) conf[m] = 1.f / (1.f + expf(-(acc + bias)));
}

// ---------------------------------------------------------------------------
// Latent-cache append of newly verified tokens: per layer the kv_a projection of
// their context features (a GEMM before this kernel) becomes the cache entry
// [RMSNorm(c_kv) * g || RoPE(k_r, pos)] -- the layout the layer forms for its own
// block rows -- written at pos = ctx_len + j through the page table. One CTA per
// (token slot, sequence); slots j >= n_new[b] write nothing.
// ---------------------------------------------------------------------------
__global__ void kv_scatter_kernel(const float *__restrict__ kv_all, size_t kv_stride, AppendLayers al, int kv_lora,
                                  int d_rope, float eps, RopeTable rt,
                                  const int32_t *__restrict__ n_new, int n_max, const int32_t *__restrict__ ctx_len,
                                  const int32_t *__restrict__ page_table, int max_pages, int page, int n_pages, int cap,
                                  int *err) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[33];
    const int j = blockIdx.x, b = blockIdx.y, l = blockIdx.z;  // token slot, sequence, layer
    const float *kv = kv_all + (size_t)l * kv_stride;
    const float *g_kv = al.g_kv[l];
    __nv_bfloat16 *pool = al.pool[l];
    const int kvd = kv_lora + d_rope;
    const int n = n_new[b];
    if (n < 0 || n > n_max) {
        if (threadIdx.x == 0 && j == 0 && l == 0) set_error(err, DSPARK_ERR_OOB);
        return;
    }
    if (j >= n) return;
    const int c = ctx_len[b];
    const int pos = c + j;
    if (c < 0 || pos >= cap) {
        if (threadIdx.x == 0) set_error(err, DSPARK_ERR_OOB);
        return;
    }
    const int pg = page_table[(size_t)b * max_pages + pos / page];
    if (pg < 0 || pg >= n_pages) {
        if (threadIdx.x == 0) set_error(err, DSPARK_ERR_OOB);
        return;
    }
    const float *row = kv + ((size_t)b * n_max + j) * kvd;
    const float4 *row4 = (const float4 *)row;  // kv_lora a multiple of 64, rows 16-byte aligned
    float ss = 0.f;
    for (int i = threadIdx.x; i < kv_lora / 4; i += blockDim.x) {
        const float4 v = row4[i];
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    ss = block_sum(ss, red);
    if (!isfinite(ss) && threadIdx.x == 0) set_error(err, DSPARK_ERR_BAD_INPUT);
    const float r = rsqrtf(ss / (float)kv_lora + eps);
    __nv_bfloat16 *dst = pool + ((size_t)pg * page + pos % page) * kvd;
    const float4 *g4 = (const float4 *)g_kv;
    for (int i = threadIdx.x; i < kv_lora / 4; i += blockDim.x) {
        const float4 v = row4[i], g = __ldg(g4 + i);
        const __nv_bfloat162 a = __floats2bfloat162_rn(v.x * r * g.x, v.y * r * g.y);
        const __nv_bfloat162 c = __floats2bfloat162_rn(v.z * r * g.z, v.w * r * g.w);
        *(uint2 *)(dst + 4 * i) = make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&c));
    }
    for (int q = threadIdx.x; q < d_rope / 2; q += blockDim.x) {
        float fc, fs;
        rope_cs((double)pos, rt.inv_freq[q], fc, fs);
        const float x0 = row[kv_lora + 2 * q], x1 = row[kv_lora + 2 * q + 1];
        dst[kv_lora + 2 * q] = __float2bfloat16(x0 * fc - x1 * fs);
        dst[kv_lora + 2 * q + 1] = __float2bfloat16(x0 * fs + x1 * fc);
    }
}

// The append's pre-norms: row m of x normalised once and scaled by every
// layer's gain, y[l][m] = bf16(x[m] * rsqrt(mean x[m]^2 + eps) * g_attn[l]).
// Grid (M, L).
__global__ void __launch_bounds__(kNormThreads) append_norm_kernel(const float *__restrict__ x, int ldx,
                                                                   AppendLayers al, int H, float eps,
                                                                   __nv_bfloat16 *__restrict__ y, int M, int *err) {
    pdl_trigger();
    __shared__ float red[33];
    const int m = blockIdx.x, l = blockIdx.y, n4 = H / 4;
    const float4 *g4 = (const float4 *)al.g_attn[l];
    pdl_wait();
    const float4 *xr = (const float4 *)(x + (size_t)m * ldx);
    float ss = 0.f;
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 v = xr[i];
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    ss = block_sum(ss, red);
    if (!isfinite(ss) && threadIdx.x == 0 && l == 0) set_error(err, DSPARK_ERR_BAD_INPUT);
    const float r = rsqrtf(ss / (float)H + eps);
    uint2 *yr = (uint2 *)(y + ((size_t)l * M + m) * H);
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 v = xr[i], g = __ldg(g4 + i);
        const __nv_bfloat162 a = __floats2bfloat162_rn(v.x * r * g.x, v.y * r * g.y);
        const __nv_bfloat162 c = __floats2bfloat162_rn(v.z * r * g.z, v.w * r * g.w);
        yr[i] = make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&c));
    }
}

// ctx_len[b] += n_new[b] once every layer's entries are written (a sequence whose
// new length would pass the capacity keeps its length; the error is reported).
__global__ void ctx_advance_kernel(int32_t *__restrict__ ctx_len, const int32_t *__restrict__ n_new, int n_max,
                                   int cap, int bs, int *err) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= bs) return;
    const int n = n_new[b], c = ctx_len[b];
    if (n < 0 || n > n_max || c < 0 || c + n > cap) {
        set_error(err, DSPARK_ERR_OOB);
        return;
    }
    ctx_len[b] = c + n;
}

// ---------------------------------------------------------------------------
// Host-side launch wrappers
// ---------------------------------------------------------------------------
cudaError_t launch_rmsnorm(const float *x, int ldx, const float *g, int H, float eps, __nv_bfloat16 *y, int ldy,
                           float *y32, int ldy32, int M, int *err, cudaStream_t st, bool late) {
    return launch_pdl(rmsnorm_kernel, dim3(M), dim3(kNormThreads), 0, st, x, ldx, g, H, eps, y, ldy, y32, ldy32,
                      err, late ? 1 : 0);
}

cudaError_t launch_latent(const float *qkv, int ld, int q_lora, int kv_lora, int d_rope, const float *g_q,
                          const float *g_kv, float eps, const int32_t *ctx_len, int block, int max_ctx,
                          const RopeTable &rt, __nv_bfloat16 *cq, __nv_bfloat16 *blk_kv, int M, int *err,
                          cudaStream_t st) {
    return launch_pdl(latent_kernel, dim3(M), dim3(kLatentThreads), 0, st, qkv, ld, q_lora, kv_lora, d_rope, g_q, g_kv, eps,
                      ctx_len, block, max_ctx, rt, cq, blk_kv, err);
}

cudaError_t launch_q_absorb(const float *q, int M, int n_h, int d_nope, int d_rope, int kv_lora, int d_v,
                            const __nv_bfloat16 *w_kvb, const int32_t *ctx_len, int block, int max_ctx,
                            const RopeTable &rt, __nv_bfloat16 *qt, cudaStream_t st, const GemmPending *pend) {
    GemmPending pd;
    memset(&pd, 0, sizeof(pd));
    if (pend) pd = *pend;
    if (d_nope <= 128 && d_nope % 8 == 0 && d_rope % 4 == 0 && d_rope <= kQAbs2MaxRope &&
        d_rope / 2 * kQAbsRows <= kQAbs2Threads)
        return launch_pdl(q_absorb2_kernel<64>, dim3(n_h, (kv_lora + kQAbs2Cols - 1) / kQAbs2Cols),
                          dim3(kQAbs2Threads), 0, st, q, M, n_h, d_nope, d_rope, kv_lora, d_v, w_kvb, ctx_len, block,
                          max_ctx, rt, qt, pd);
    dim3 grid(n_h, kv_lora / kQAbsCols);
    const size_t smem = ((size_t)kQAbsRows * d_nope + (size_t)4 * kQAbsRows * kQAbsCols) * sizeof(float);
    // the thread's k_b slice (d_nope / 4 rows) in registers: 32 covers d_nope <= 128
    return launch_pdl(d_nope <= 128 ? q_absorb_kernel<32> : q_absorb_kernel<64>, grid, dim3(128), smem, st, q, M, n_h, d_nope, d_rope, kv_lora, d_v, w_kvb,
                      ctx_len, block, max_ctx, rt, qt, pd);
}

// Whether a row of H channels fits the cluster row kernels' tile bookkeeping.
bool row_cluster_fits(int H) {
    const int slice4 = (H / 4 + kRowCl - 1) / kRowCl;
    return H % 4 == 0 && slice4 <= kRowVals * kRowClThreads && slice4 * 4 / 128 + 2 <= kRowClTiles;
}

cudaError_t launch_rmsnorm_cluster(float *x, int ldx, const GemmPending *pend, bool add, const float *g, int H,
                                   float eps, __nv_bfloat16 *y, int ldy, float *y32, int ldy32, int M, int *err,
                                   cudaStream_t st, bool late) {
    if (!row_cluster_fits(H)) return cudaErrorInvalidValue;
    GemmPending pd;
    memset(&pd, 0, sizeof(pd));
    if (pend) pd = *pend;
    return launch_pdl_cluster(rmsnorm_cluster_kernel, dim3(kRowCl, M), dim3(kRowClThreads), 0, st, kRowCl, x, ldx,
                              pd, add ? 1 : 0, g, H, eps, y, ldy, y32, ldy32, err, late ? 1 : 0);
}

cudaError_t launch_latent_cluster(const float *qkv, int ld, const GemmPending *pend, int q_lora, int kv_lora,
                                  int d_rope, const float *g_q, const float *g_kv, float eps, const int32_t *ctx_len,
                                  int block, int max_ctx, const RopeTable &rt, __nv_bfloat16 *cq,
                                  __nv_bfloat16 *blk_kv, int M, int *err, cudaStream_t st) {
    const int H = q_lora + kv_lora + d_rope;
    if (!row_cluster_fits(H) || q_lora % 4 || kv_lora % 4 || d_rope % 4) return cudaErrorInvalidValue;
    GemmPending pd;
    memset(&pd, 0, sizeof(pd));
    if (pend) pd = *pend;
    return launch_pdl_cluster(latent_cluster_kernel, dim3(kRowCl, M), dim3(kRowClThreads), 0, st, kRowCl, qkv, ld,
                              pd, q_lora, kv_lora, d_rope, g_q, g_kv, eps, ctx_len, block, max_ctx, rt, cq, blk_kv,
                              err);
}

cudaError_t launch_v_absorb(const float *o_lat, int M, int n_h, int d_nope, int d_v, int kv_lora,
                            const __nv_bfloat16 *w_kvb, __nv_bfloat16 *out, cudaStream_t st) {
    dim3 grid(n_h, d_v / 16);
    const size_t smem = (size_t)kVAbsRows * kv_lora * sizeof(float);
    return launch_pdl(v_absorb_kernel, grid, dim3(256), smem, st, o_lat, M, n_h, d_nope, d_v, kv_lora, w_kvb, out);
}

template <int DQK, int DV>
static cudaError_t launch_attn_t(const AttnParams &p, int bs, int qtiles, cudaStream_t st) {
    using C = AttnCfg<DQK, DV>;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(mla_attention_kernel<DQK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::kSmem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    dim3 grid(qtiles, p.splits, bs);
    return launch_pdl(mla_attention_kernel<DQK, DV>, grid, dim3(256), (size_t)C::kSmem, st, p);
}

bool attention_supported(int dqk, int dv) {
    return (dqk == 576 && dv == 512) || (dqk == 80 && dv == 64) || (dqk == 160 && dv == 128) ||
           (dqk == 288 && dv == 256);
}

cudaError_t launch_attention(const AttnParams &p, int bs, int dqk, int dv, cudaStream_t st) {
    const int qtiles = (p.R + 63) / 64;
    cudaError_t e;
    if (dqk == 576 && dv == 512)
        e = launch_attn_t<576, 512>(p, bs, qtiles, st);
    else if (dqk == 80 && dv == 64)
        e = launch_attn_t<80, 64>(p, bs, qtiles, st);
    else if (dqk == 160 && dv == 128)
        e = launch_attn_t<160, 128>(p, bs, qtiles, st);
    else if (dqk == 288 && dv == 256)
        e = launch_attn_t<288, 256>(p, bs, qtiles, st);
    else
        return cudaErrorInvalidValue;
    if (e != cudaSuccess || p.splits == 1) return e;
    return launch_attn_combine(p, bs, dv, st);
}

// Shared memory of the fused combine + v absorption.
static size_t cvabs_smem(int d_v, int kv_lora) {
    return (size_t)d_v * (kv_lora * 2 + 16) + (size_t)kCVRows * kv_lora * 4 + (size_t)kCVParts * kCVRows * 2 * kCVPairs * 4;
}

bool attn_combine_vabsorb_fits(int d_v, int kv_lora, int splits) {
    return kv_lora % (8 * kCVParts) == 0 && splits <= kCVMaxSplit && cvabs_smem(d_v, kv_lora) <= 227u * 1024u;
}

cudaError_t launch_attn_combine_vabsorb(const AttnParams &p, int M, int n_h, int d_nope, int d_v, int kv_lora,
                                        const __nv_bfloat16 *w_kvb, __nv_bfloat16 *out, cudaStream_t st) {
    const size_t smem = cvabs_smem(d_v, kv_lora);
    static std::mutex mu;
    static size_t set_bytes = 0;  // the largest limit set so far (handles of several geometries)
    {
        std::lock_guard<std::mutex> lock(mu);
        if (smem > set_bytes) {
            const cudaError_t e = cudaFuncSetAttribute(attn_combine_vabsorb_kernel,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            set_bytes = smem;
        }
    }
    return launch_pdl(attn_combine_vabsorb_kernel, dim3(n_h, (M + kCVRows - 1) / kCVRows), dim3(kCVThreads), smem,
                      st, p.part_o, p.part_ml, p.splits, p.R, p.o_lat, M, n_h, p.block, d_nope, d_v, kv_lora, w_kvb,
                      out, p.ctx_len, p.max_ctx, p.cps > 0 ? p.cps : 1 << 20);
}

cudaError_t launch_attn_combine(const AttnParams &p, int bs, int dv, cudaStream_t st) {
    return launch_pdl(attn_combine_kernel, dim3(p.R, bs), dim3(128), 0, st, p.part_o, p.part_ml, p.splits, p.R, dv,
                      p.o_lat);
}

cudaError_t launch_kv_scatter_layers(const float *kv, size_t kv_stride, int L, const AppendLayers &al, int kv_lora,
                                     int d_rope, float eps, const RopeTable &rt, const int32_t *n_new, int n_max,
                                     const int32_t *ctx_len, const int32_t *page_table, int max_pages, int page,
                                     int n_pages, int cap, int bs, int *err, cudaStream_t st) {
    return launch_pdl(kv_scatter_kernel, dim3(n_max, bs, L), dim3(128), 0, st, kv, kv_stride, al, kv_lora, d_rope, eps,
                      rt, n_new, n_max, ctx_len, page_table, max_pages, page, n_pages, cap, err);
}

cudaError_t launch_append_norm(const float *x, int ldx, const AppendLayers &al, int L, int H, float eps,
                               __nv_bfloat16 *y, int M, int *err, cudaStream_t st) {
    return launch_pdl(append_norm_kernel, dim3(M, L), dim3(kNormThreads), 0, st, x, ldx, al, H, eps, y, M, err);
}

cudaError_t launch_ctx_advance(int32_t *ctx_len, const int32_t *n_new, int n_max, int cap, int bs, int *err,
                               cudaStream_t st) {
    return launch_pdl(ctx_advance_kernel, dim3((bs + 31) / 32), dim3(32), 0, st, ctx_len, n_new, n_max, cap, bs, err);
}

cudaError_t launch_confidence(const float *h_out, int H, const float *w, float bias, float *conf, int M,
                              cudaStream_t st) {
    return launch_pdl(confidence_kernel, dim3(M), dim3(512), 0, st, h_out, H, w, bias, conf);
}

}  // namespace ds
