/*
 * ORACLE -- test infrastructure only. Plain, slow, obviously correct CPU code
 * for the integer-exact parts of the DSpark draft-and-verify step: the
 * counter-based uniforms, the sampling spec (own exp, integer softmax weights,
 * top-p nucleus), the low-rank Markov rollout, and lossless verification.
 * Only tests, the smoke check and the benchmark's CPU-baseline leg may load
 * this library. It shares no code with the CUDA library.
 *
 * Pages (Kimi-K3-DSpark model cards):
 *  - "kimi-k3-dspark-gguf", intro: the target verifies the drafted tokens in
 *    one pass and the output distribution equals the target's alone.
 *  - "Kimi-K3-DSpark-NVFP4", "Original model card / Model Overview": a
 *    low-rank sequential Markov head supplies the intra-block dependency;
 *    "Quick Start / Sampling options": greedy vs probabilistic draft, and at
 *    temperature 0 verification is an argmax match.
 *  - "Kimi K3 DSpark Q8_0 GGUF", "Architecture metadata": Markov rank 256.
 * The pages give no sampler numerics; the fixed-point spec below is the
 * reading written down for this build (exact integers for every decision).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no fast-math).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef unsigned __int128 u128;

enum { OK = 0, ERR_BAD_INPUT = 17, ERR_OOB = 18, ERR_ALLOC = 19 };

/* ---------------------------------------------------------------------------
 * Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy
 * as 1, 2, 3", SC'11): 10 rounds of two 32x32->64 multiplies with the round
 * key bumped by the Weyl constants between rounds.
 * ------------------------------------------------------------------------- */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* One 32-bit uniform word for a decision: key = seed, counter = (step, seq, pos, purpose). */
uint32_t oracle_uniform_u32(uint64_t seed, uint32_t seq, uint32_t step, uint32_t pos, uint32_t purpose)
{
    uint32_t ctr[4] = {step, seq, pos, purpose};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    return out[0];
}

/* ---------------------------------------------------------------------------
 * Own fp32 exp for x <= 0 (Cody & Waite argument reduction, "Software Manual
 * for the Elementary Functions", 1980, then the degree-7 Taylor polynomial of
 * e^r in Horner form with explicit fused multiply-adds):
 *   n = rint(x * log2(e)),  r = x - n*ln2 (ln2 split into a 16-bit head and an
 *   fp32 tail so that n*head is exact),  e^x = 2^n * sum_{k<=7} r^k / k!.
 * Every step is one IEEE fp32 operation, so the result is bit-reproducible.
 * Below -23 the value is < 2^-32 and the spec's weight is 0 anyway.
 * ------------------------------------------------------------------------- */
static float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

float oracle_exp_hat(float x)
{
    if (!(x >= -23.0f)) return 0.0f;
    const float log2e = 1.44269502162933349609375f;          /* fp32(1/ln 2) */
    const float ln2_hi = 0.693145751953125f;                  /* 45426 / 2^16 */
    const float ln2_lo = 1.428606765330187045037746429443359375e-06f; /* fp32(ln2 - ln2_hi) */
    float t = x * log2e;
    float n = rintf(t);
    float r = fmaf(-n, ln2_hi, x);
    r = fmaf(-n, ln2_lo, r);
    /* 1/k! rounded to nearest fp32 */
    const float c7 = 1.98412701138295233249664306640625e-04f;
    const float c6 = 1.388888922519981861114501953125e-03f;
    const float c5 = 8.33333376795053482055664062500e-03f;
    const float c4 = 4.16666679084300994873046875e-02f;
    const float c3 = 1.66666671633720397949218750e-01f;
    float p = c7;
    p = fmaf(p, r, c6);
    p = fmaf(p, r, c5);
    p = fmaf(p, r, c4);
    p = fmaf(p, r, c3);
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    int ni = (int)n;
    float scale = f32_from_bits((uint32_t)(ni + 127) << 23);
    return p * scale;
}

/* ---------------------------------------------------------------------------
 * Sampling spec for one row of logits l[0..V) at temperature T > 0, top_p.
 *   y_v = l_v / T (fp32), m = max y, E_v = floor(2^32 * exp_hat(y_v - m)) (uint64)
 *   S = sum E;  tau = max(1, floor(S * P32 / 2^32)),  P32 = top_p * 2^32
 *   key_v = (E_v << 18) | (2^18 - 1 - v); nucleus = the shortest run of keys in
 *   descending order whose E-sum reaches tau; p_v = E_v / S_n inside it.
 * ------------------------------------------------------------------------- */
typedef struct {
    uint64_t S;       /* sum over the whole row */
    uint64_t kstar;   /* smallest key inside the nucleus */
    uint64_t Sn;      /* sum over the nucleus */
    int32_t size;     /* number of tokens in the nucleus */
} oracle_nucleus_t;

static int finite_row(const float *l, int V)
{
    for (int v = 0; v < V; ++v)
        if (!isfinite(l[v])) return 0;
    return 1;
}

uint64_t oracle_top_p_q32(float top_p)
{
    if (!(top_p > 0.0f)) return 0;
    if (top_p >= 1.0f) return (uint64_t)1 << 32;
    return (uint64_t)((double)top_p * 4294967296.0);  /* exact: top_p has 24 significant bits */
}

int oracle_row_weights(const float *l, int V, float T, uint64_t *E)
{
    if (!finite_row(l, V)) return ERR_BAD_INPUT;
    float m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        float y = l[v] / T;
        if (!isfinite(y)) return ERR_BAD_INPUT;
        if (y > m) m = y;
    }
    for (int v = 0; v < V; ++v) {
        float y = l[v] / T;
        float e = oracle_exp_hat(y - m);
        E[v] = (uint64_t)(e * 4294967296.0f);
    }
    return OK;
}

static uint64_t key_of(uint64_t E, int v) { return (E << 18) | (uint64_t)((1u << 18) - 1u - (uint32_t)v); }

static int cmp_desc_u64(const void *a, const void *b)
{
    uint64_t x = *(const uint64_t *)a, y = *(const uint64_t *)b;
    return (x < y) - (x > y);
}

int oracle_nucleus(const uint64_t *E, int V, float top_p, oracle_nucleus_t *out)
{
    uint64_t *keys = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)V);
    if (!keys) return ERR_ALLOC;
    uint64_t S = 0;
    for (int v = 0; v < V; ++v) {
        S += E[v];
        keys[v] = key_of(E[v], v);
    }
    qsort(keys, (size_t)V, sizeof(uint64_t), cmp_desc_u64);
    uint64_t tau = (uint64_t)(((u128)S * (u128)oracle_top_p_q32(top_p)) >> 32);
    if (tau < 1) tau = 1;
    uint64_t cum = 0;
    int k = 0;
    for (; k < V; ++k) {
        cum += keys[k] >> 18;
        if (cum >= tau) break;
    }
    if (k == V) k = V - 1;  /* unreachable: tau <= S */
    out->S = S;
    out->kstar = keys[k];
    out->Sn = cum;
    out->size = k + 1;
    free(keys);
    return OK;
}

/* Weight of token v inside the nucleus (0 outside). */
static uint64_t in_nucleus(const uint64_t *E, int v, uint64_t kstar)
{
    return key_of(E[v], v) >= kstar ? E[v] : 0;
}

/* Sample with a 24-bit uniform W: target = floor(S_n * W / 2^24); the token is the
 * smallest id whose running nucleus weight (ascending id) exceeds target. */
int32_t oracle_sample_nucleus(const uint64_t *E, int V, uint64_t kstar, uint64_t Sn, uint32_t W24)
{
    uint64_t target = (uint64_t)(((u128)Sn * (u128)(W24 & 0xFFFFFFu)) >> 24);
    uint64_t cum = 0;
    for (int v = 0; v < V; ++v) {
        cum += in_nucleus(E, v, kstar);
        if (cum > target) return v;
    }
    return -1;
}

/* Greedy pick: largest fp32 value, lowest id on ties. */
int oracle_argmax(const float *l, int V, int32_t *out)
{
    if (!finite_row(l, V)) return ERR_BAD_INPUT;
    int best = 0;
    for (int v = 1; v < V; ++v)
        if (l[v] > l[best]) best = v;
    *out = best;
    return OK;
}

/* One full draw from a logit row (used by the draft and by the bonus). */
static int draw_from_logits(const float *l, int V, float T, float top_p, uint32_t W24,
                            uint64_t *E, int32_t *tok)
{
    int st = oracle_row_weights(l, V, T, E);
    if (st) return st;
    oracle_nucleus_t nu;
    st = oracle_nucleus(E, V, top_p, &nu);
    if (st) return st;
    *tok = oracle_sample_nucleus(E, V, nu.kstar, nu.Sn, W24);
    return OK;
}

static float bf16_to_f32(uint16_t b) { return f32_from_bits((uint32_t)b << 16); }

/* ---------------------------------------------------------------------------
 * Markov rollout (one sequence). t_0 = anchor; for i = 1..B:
 *   delta_i[v] = fp32 fused-multiply-add chain over k = 0..r-1 of w1[t_{i-1},k] * w2[k,v]
 *   ell_i[v]   = z_i[v] + delta_i[v]   (fp32)
 *   t_i        = argmax ell_i (greedy) or a draw from the spec above (uniform
 *                purpose DRAFT, position i-1).
 * w1 bf16 [V, r], w2 bf16 [r, V], z fp32 [B, V], ell fp32 [B, V].
 * ------------------------------------------------------------------------- */
int oracle_markov_rollout(const float *z, int B, int V, int r, const uint16_t *w1, const uint16_t *w2,
                          int32_t anchor, int draft_mode, float T, float top_p, uint64_t seed,
                          uint32_t seq, uint32_t step, int32_t *tokens, float *ell)
{
    if (anchor < 0 || anchor >= V) return ERR_OOB;
    uint64_t *E = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)V);
    float *w1row = (float *)malloc(sizeof(float) * (size_t)r);
    if (!E || !w1row) { free(E); free(w1row); return ERR_ALLOC; }
    int32_t prev = anchor;
    int st = OK;
    for (int i = 0; i < B && st == OK; ++i) {
        for (int k = 0; k < r; ++k) w1row[k] = bf16_to_f32(w1[(size_t)prev * r + k]);
        float *row = ell + (size_t)i * V;
        for (int v = 0; v < V; ++v) {
            float acc = 0.0f;
            for (int k = 0; k < r; ++k) acc = fmaf(w1row[k], bf16_to_f32(w2[(size_t)k * V + v]), acc);
            row[v] = z[(size_t)i * V + v] + acc;
        }
        int32_t t;
        if (draft_mode == 0) {
            st = oracle_argmax(row, V, &t);
        } else {
            uint32_t W = oracle_uniform_u32(seed, seq, step, (uint32_t)i, 1u) >> 8;
            st = draw_from_logits(row, V, T, top_p, W, E, &t);
        }
        tokens[i] = t;
        prev = t;
    }
    free(E);
    free(w1row);
    return st;
}

/* ---------------------------------------------------------------------------
 * Verification (one sequence). P fp32 [B+1, V] target logits (row i scores the
 * token at block position i; row B is the bonus position), ell fp32 [B, V]
 * draft logits, tokens [B]. Output accept_len in 0..B and out_tokens [B+1]
 * (accepted drafts, then the correction or bonus token, then -1).
 *
 * Greedy: g_i = argmax P_i; a = number of leading positions with g_i == t_i;
 * emit t_1..t_a and g_{a+1}.
 *
 * Probabilistic (explicit uniforms so tests can enumerate them):
 *   accept t_i iff U_i * Eq_t * Sp < 2^32 * Ep_t * Sq  (exact 128-bit compare),
 *   i.e. U_i / 2^32 < p_i(t_i) / q_i(t_i);
 *   on the first reject draw from r_v = max(0, Ep_v * Sq - Eq_v * Sp) with Wres_i;
 *   if all are accepted draw the bonus from p_{B+1} with Wbonus.
 * With draft_greedy set, q_i is one-hot on t_i (Eq = [v == t_i], Sq = 1).
 * ------------------------------------------------------------------------- */
int oracle_verify_greedy(const float *P, const int32_t *tokens, int B, int V,
                         int32_t *accept_len, int32_t *out_tokens)
{
    int a = 0;
    int32_t g = 0;
    int st;
    for (int i = 0; i <= B; ++i) out_tokens[i] = -1;
    for (a = 0; a < B; ++a) {
        if (tokens[a] < 0 || tokens[a] >= V) return ERR_OOB;
        st = oracle_argmax(P + (size_t)a * V, V, &g);
        if (st) return st;
        if (g != tokens[a]) break;
        out_tokens[a] = tokens[a];
    }
    if (a == B) {
        st = oracle_argmax(P + (size_t)B * V, V, &g);
        if (st) return st;
    }
    out_tokens[a] = g;
    *accept_len = a;
    return OK;
}

int oracle_verify_prob_core(const float *P, const float *ell, const int32_t *tokens, int B, int V,
                            int draft_greedy, float T, float top_p,
                            const uint32_t *U, const uint32_t *Wres, uint32_t Wbonus,
                            int32_t *accept_len, int32_t *out_tokens)
{
    uint64_t *Ep = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)V);
    uint64_t *Eq = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)V);
    if (!Ep || !Eq) { free(Ep); free(Eq); return ERR_ALLOC; }
    int st = OK;
    for (int i = 0; i <= B; ++i) out_tokens[i] = -1;
    int i = 0;
    for (; i < B; ++i) {
        int32_t t = tokens[i];
        if (t < 0 || t >= V) { st = ERR_OOB; goto done; }
        oracle_nucleus_t np, nq;
        st = oracle_row_weights(P + (size_t)i * V, V, T, Ep);
        if (st) goto done;
        st = oracle_nucleus(Ep, V, top_p, &np);
        if (st) goto done;
        uint64_t Sq;
        if (draft_greedy) {
            for (int v = 0; v < V; ++v) Eq[v] = (v == t);
            Sq = 1;
            nq.kstar = 0;
        } else {
            st = oracle_row_weights(ell + (size_t)i * V, V, T, Eq);
            if (st) goto done;
            st = oracle_nucleus(Eq, V, top_p, &nq);
            if (st) goto done;
            Sq = nq.Sn;
        }
        uint64_t Sp = np.Sn;
        uint64_t ep = in_nucleus(Ep, t, np.kstar);
        uint64_t eq = draft_greedy ? 1 : in_nucleus(Eq, t, nq.kstar);
        u128 lhs = (u128)U[i] * (u128)eq * (u128)Sp;
        u128 rhs = ((u128)ep << 32) * (u128)Sq;
        if (lhs < rhs) {
            out_tokens[i] = t;
            continue;
        }
        /* first reject: residual max(0, p - q) scaled by Sp * Sq */
        u128 R = 0;
        for (int v = 0; v < V; ++v) {
            u128 a = (u128)in_nucleus(Ep, v, np.kstar) * Sq;
            u128 b = (u128)(draft_greedy ? (uint64_t)(v == t) : in_nucleus(Eq, v, nq.kstar)) * Sp;
            if (a > b) R += a - b;
        }
        u128 target = (R * (u128)(Wres[i] & 0xFFFFFFu)) >> 24;
        u128 cum = 0;
        int32_t pick = -1;
        for (int v = 0; v < V; ++v) {
            u128 a = (u128)in_nucleus(Ep, v, np.kstar) * Sq;
            u128 b = (u128)(draft_greedy ? (uint64_t)(v == t) : in_nucleus(Eq, v, nq.kstar)) * Sp;
            if (a > b) cum += a - b;
            if (cum > target) { pick = v; break; }
        }
        out_tokens[i] = pick;
        *accept_len = i;
        goto done;
    }
    {
        int32_t bonus;
        st = draw_from_logits(P + (size_t)B * V, V, T, top_p, Wbonus, Ep, &bonus);
        if (st) goto done;
        out_tokens[B] = bonus;
        *accept_len = B;
    }
done:
    free(Ep);
    free(Eq);
    return st;
}

int oracle_verify_prob(const float *P, const float *ell, const int32_t *tokens, int B, int V,
                       int draft_greedy, float T, float top_p, uint64_t seed, uint32_t seq,
                       uint32_t step, int32_t *accept_len, int32_t *out_tokens)
{
    uint32_t U[64], Wres[64];
    if (B > 64) return ERR_OOB;
    for (int i = 0; i < B; ++i) {
        U[i] = oracle_uniform_u32(seed, seq, step, (uint32_t)i, 2u);
        Wres[i] = oracle_uniform_u32(seed, seq, step, (uint32_t)i, 3u) >> 8;
    }
    uint32_t Wb = oracle_uniform_u32(seed, seq, step, (uint32_t)B, 4u) >> 8;
    return oracle_verify_prob_core(P, ell, tokens, B, V, draft_greedy, T, top_p, U, Wres, Wb,
                                   accept_len, out_tokens);
}

/* ---------------------------------------------------------------------------
 * Block verification ("Kimi-K3-DSpark-NVFP4", Quick Start / Sampling options:
 * rejection_sample_method "block" verifies the drafted block as a unit; the
 * method of Sun, Mendlovic, Leviathan, Aharoni, Beirami, Ro, Suresh, "Block
 * Verification Accelerates Speculative Decoding", 2024). With p(.) the target
 * rows and q(.) the draft rows of the sampling spec, X_1..X_B the drafted tokens:
 *   pi_0 = 1, pi_i = min(pi_{i-1} p_{i-1}(X_i) / q_{i-1}(X_i), 1)
 *   S_i  = sum_x max(pi_i p_i(x) - q_i(x), 0)                (i < B)
 *   h_i  = S_i / (S_i + 1 - pi_i) (i < B),  h_B = pi_B
 *   eta_i ~ Bernoulli(h_i) independently, tau = max {i : eta_i = 1} (0 if none)
 *   emit X_1..X_tau, then a token from max(pi_tau p_tau - q_tau, 0) (tau < B)
 *   or from p_B (tau = B).
 * Numerics (the paper gives none): p_i(x) and q_i(x) are the spec's exact
 * rationals E / S rounded once to double; every mass term is formed in double
 * (multiply, then subtract, no contraction), truncated to a multiple of 2^-80
 * and summed exactly in 128 bits, so the sums do not depend on the order of
 * summation. eta_i = (U_i < h_i * 2^32) with the 32-bit uniform U_i (purpose
 * 2, position i-1); the final token is drawn like the spec's other draws with
 * the 24-bit uniform of purpose 3 at position tau (the bonus: purpose 4).
 * ------------------------------------------------------------------------- */
static u128 fx80(double x)
{
    if (!(x > 0.0)) return 0;
    uint64_t b;
    memcpy(&b, &x, 8);
    const int e = (int)((b >> 52) & 0x7FF);
    if (e == 0) return 0; /* below 2^-1022 */
    const uint64_t m = (b & ((1ull << 52) - 1)) | (1ull << 52);
    const int sh = e - 995; /* x * 2^80 = m * 2^(e - 1075 + 80) */
    if (sh >= 0) return (u128)m << sh;
    if (sh <= -53) return 0;
    return (u128)(m >> (-sh));
}

/* The value of a 2^-80 fixed-point sum as a double: its top 53 bits, exactly. */
static double fx80_to_double(u128 s)
{
    if (s == 0) return 0.0;
    const uint64_t hi = (uint64_t)(s >> 64), lo = (uint64_t)s;
    const int n = hi ? 128 - __builtin_clzll(hi) : 64 - __builtin_clzll(lo);
    if (n <= 53) return ldexp((double)lo, -80);
    return ldexp((double)(uint64_t)(s >> (n - 53)), n - 53 - 80);
}

typedef struct {
    int B, V, dg;
    uint64_t *Ep, *Eq;   /* rows 0..B of p, 0..B-1 of q: in-nucleus weights (0 outside) */
    uint64_t Sp[65], Sq[65];
    const int32_t *tokens;
} brows_t;

static double bp(const brows_t *r, int i, int v) { return (double)r->Ep[(size_t)i * r->V + v] / (double)r->Sp[i]; }
static double bq(const brows_t *r, int i, int v)
{
    if (r->dg) return v == r->tokens[i] ? 1.0 : 0.0;
    return (double)r->Eq[(size_t)i * r->V + v] / (double)r->Sq[i];
}
static u128 bmass_term(const brows_t *r, int i, double pi, int v)
{
    double d = pi * bp(r, i, v);
    d = d - bq(r, i, v);
    return fx80(d);
}
static u128 bmass(const brows_t *r, int i, double pi)
{
    u128 s = 0;
    for (int v = 0; v < r->V; ++v) s += bmass_term(r, i, pi, v);
    return s;
}

static int brows_load(brows_t *r, const float *P, const float *ell, const int32_t *tokens, int B, int V, int dg,
                      float T, float top_p)
{
    r->B = B;
    r->V = V;
    r->dg = dg;
    r->tokens = tokens;
    r->Ep = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(B + 1) * V);
    r->Eq = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(B > 0 ? B : 1) * V);
    if (!r->Ep || !r->Eq) return ERR_ALLOC;
    for (int i = 0; i < B; ++i)
        if (tokens[i] < 0 || tokens[i] >= V) return ERR_OOB;
    for (int i = 0; i <= B; ++i) {
        uint64_t *E = r->Ep + (size_t)i * V;
        oracle_nucleus_t nu;
        int st = oracle_row_weights(P + (size_t)i * V, V, T, E);
        if (!st) st = oracle_nucleus(E, V, top_p, &nu);
        if (st) return st;
        for (int v = 0; v < V; ++v) E[v] = in_nucleus(E, v, nu.kstar);
        r->Sp[i] = nu.Sn;
    }
    for (int i = 0; i < B && !dg; ++i) {
        uint64_t *E = r->Eq + (size_t)i * V;
        oracle_nucleus_t nu;
        int st = oracle_row_weights(ell + (size_t)i * V, V, T, E);
        if (!st) st = oracle_nucleus(E, V, top_p, &nu);
        if (st) return st;
        for (int v = 0; v < V; ++v) E[v] = in_nucleus(E, v, nu.kstar);
        r->Sq[i] = nu.Sn;
    }
    return OK;
}

static void brows_free(brows_t *r)
{
    free(r->Ep);
    free(r->Eq);
}

/* pi_0..pi_B and h_1..h_B (h[0] = 0) of one sequence. */
static void bstats(const brows_t *r, double *pi, double *h)
{
    const int B = r->B;
    pi[0] = 1.0;
    h[0] = 0.0;
    for (int i = 1; i <= B; ++i) {
        const int t = r->tokens[i - 1];
        const double a = bp(r, i - 1, t), c = bq(r, i - 1, t);
        if (c == 0.0) {
            pi[i] = (a > 0.0 && pi[i - 1] > 0.0) ? 1.0 : 0.0;
        } else {
            const double x = pi[i - 1] * (a / c);
            pi[i] = x < 1.0 ? x : 1.0;
        }
    }
    for (int i = 1; i < B; ++i) {
        const double S = fx80_to_double(bmass(r, i, pi[i]));
        const double den = S + (1.0 - pi[i]);
        h[i] = den > 0.0 ? S / den : 0.0;
    }
    if (B > 0) h[B] = pi[B];
}

int oracle_verify_block_stats(const float *P, const float *ell, const int32_t *tokens, int B, int V,
                              int draft_greedy, float T, float top_p, double *pi, double *h)
{
    if (B > 64) return ERR_OOB;
    brows_t r;
    int st = brows_load(&r, P, ell, tokens, B, V, draft_greedy, T, top_p);
    if (!st) bstats(&r, pi, h);
    brows_free(&r);
    return st;
}

/* Residual weights at position i for the given pi (2^-80 fixed point, as lo/hi words). */
int oracle_block_residual_weights(const float *P, const float *ell, const int32_t *tokens, int B, int V,
                                  int draft_greedy, float T, float top_p, int i, double pi, uint64_t *w)
{
    if (B > 64 || i < 0 || i >= B) return ERR_OOB;
    brows_t r;
    int st = brows_load(&r, P, ell, tokens, B, V, draft_greedy, T, top_p);
    if (!st)
        for (int v = 0; v < V; ++v) {
            const u128 x = bmass_term(&r, i, pi, v);
            w[2 * v] = (uint64_t)x;
            w[2 * v + 1] = (uint64_t)(x >> 64);
        }
    brows_free(&r);
    return st;
}

int oracle_verify_block_core(const float *P, const float *ell, const int32_t *tokens, int B, int V,
                             int draft_greedy, float T, float top_p, const uint32_t *U, const uint32_t *Wres,
                             uint32_t Wbonus, int32_t *accept_len, int32_t *out_tokens)
{
    if (B > 64) return ERR_OOB;
    for (int i = 0; i <= B; ++i) out_tokens[i] = -1;
    brows_t r;
    int st = brows_load(&r, P, ell, tokens, B, V, draft_greedy, T, top_p);
    if (st) {
        brows_free(&r);
        return st;
    }
    double pi[65], h[65];
    bstats(&r, pi, h);
    int tau = 0;
    for (int i = 1; i <= B; ++i)
        if ((double)U[i - 1] < h[i] * 4294967296.0) tau = i;
    for (int i = 0; i < tau; ++i) out_tokens[i] = tokens[i];
    *accept_len = tau;
    if (tau == B) {
        int32_t bonus;
        st = draw_from_logits(P + (size_t)B * V, V, T, top_p, Wbonus, r.Ep, &bonus);
        if (!st) out_tokens[B] = bonus;
    } else {
        const u128 R = bmass(&r, tau, pi[tau]);
        const uint32_t W = Wres[tau] & 0xFFFFFFu;
        if (R == 0) {
            /* no residual mass left at 2^-80 resolution: draw from the target row */
            int32_t pick;
            st = draw_from_logits(P + (size_t)tau * V, V, T, top_p, W, r.Ep, &pick);
            if (!st) out_tokens[tau] = pick;
        } else {
            const u128 target = (R * (u128)W) >> 24;
            u128 cum = 0;
            int32_t pick = -1;
            for (int v = 0; v < V; ++v) {
                cum += bmass_term(&r, tau, pi[tau], v);
                if (cum > target) {
                    pick = v;
                    break;
                }
            }
            out_tokens[tau] = pick;
        }
    }
    brows_free(&r);
    return st;
}

int oracle_verify_block(const float *P, const float *ell, const int32_t *tokens, int B, int V, int draft_greedy,
                        float T, float top_p, uint64_t seed, uint32_t seq, uint32_t step, int32_t *accept_len,
                        int32_t *out_tokens)
{
    uint32_t U[64], Wres[64];
    if (B > 64) return ERR_OOB;
    for (int i = 0; i < B; ++i) {
        U[i] = oracle_uniform_u32(seed, seq, step, (uint32_t)i, 2u);
        Wres[i] = oracle_uniform_u32(seed, seq, step, (uint32_t)i, 3u) >> 8;
    }
    uint32_t Wb = oracle_uniform_u32(seed, seq, step, (uint32_t)B, 4u) >> 8;
    return oracle_verify_block_core(P, ell, tokens, B, V, draft_greedy, T, top_p, U, Wres, Wb, accept_len,
                                    out_tokens);
}
