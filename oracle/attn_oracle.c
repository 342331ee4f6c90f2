/*
 * attn_oracle.c -- plain, slow CPU oracle for the attention core under
 * selective activation recomputation.  TEST INFRASTRUCTURE ONLY: the tests,
 * the smoke check and the bench's CPU-baseline leg may call it; the product
 * library never does, and this file shares no code, header or constant
 * generator with the CUDA path.
 *
 * What it computes, and where the pages define it:
 *   - "Reducing Activation Recomputation in Large Transformer Models"
 *     (dmarx anthology of the SOTA, LIT-736), Key takeaways, fourth bullet:
 *     the attention core is QK^T, softmax, softmax dropout and attention
 *     over V; selective recomputation keeps everything except that core's
 *     activations, which the backward pass recomputes.
 *   - "Recomputing Activations" (curionode, Parallelism Plate 2), Workshop:
 *     per-token activation bytes 34d + 5HT (nothing recomputed), 34d
 *     (selective) and 2d (full); "Memory for compute, selectively": the
 *     Llama 3 70B worked example.
 * The pages fix no precision, no mask generator and no scaling; the readings
 * taken here (fp64 everywhere, Philox-4x32-10 with 8-bit draws, natural-log
 * LSE, top-left causal alignment, GQA head h -> h / (h_q/h_kv)) are listed in
 * the project's design notes and in the public ABI header.
 *
 * Query and key counts: s queries and s_kv keys (s_kv = 0 means s).  The
 * core's definition -- scores of every query against every visible key,
 * softmax over the keys, dropout, weighted sum of the value rows -- does not
 * need the two counts to be equal, so with s_kv != s the same functions give
 * cross-attention.  Causal masking is top-left: query i sees keys
 * 0 .. min(i, s_kv - 1).
 *
 * Every function works in double precision.  Inputs arrive as doubles (the
 * caller widens bf16 exactly).  Work is split over rows or heads with OpenMP;
 * there is no blocking, fusion or reordering beyond that.
 *
 * Stored-output model (flag stored_o_bf16): the method keeps only the bf16
 * output O from the forward pass, so its backward must form the softmax row
 * statistic sum_j P_ij dP_ij as dO_i . O_i from that stored O.  With the flag
 * set the oracle does the same with its own O rounded to bf16; without it the
 * exact row sum is used.  The two differ by (D_exact - D_stored) P_ij in every
 * dS_ij, an error set by bf16 storage, not by the kernels.
 *
 * Parity status: every function here is pinned by a CPU test (known-answer
 * vectors for Philox, textbook attention for p = 0, finite differences for
 * the gradients, the worked example for the byte counts, and the exact
 * first-order relation between the stored-output model and the exact
 * backward).  No function is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t b, h_q, h_kv, s, d;
    int32_t causal;     /* 1: key j is visible to query i only if j <= i */
    float p_drop;       /* softmax-dropout probability, [0, 1) */
    float scale;        /* score scale; <= 0 means 1/sqrt(d) in fp32 */
    uint64_t seed;      /* Philox key */
    uint64_t offset;    /* Philox stream offset, < 2^32 */
    int32_t stored_o_bf16; /* backward row statistic from the bf16-stored output (see below) */
    int32_t s_kv;       /* keys (and value rows) per KV head; 0 means s */
} oracle_params;

/* ------------------------------------------------------------------------
 * Philox-4x32-10, from Salmon, Moraes, Dror and Shaw, "Parallel Random
 * Numbers: As Easy as 1, 2, 3" (SC'11), section 3.2: each round multiplies
 * the even counter words by two fixed 32-bit constants, splits every product
 * into high and low halves, and XORs the high halves with the odd words and
 * the round key; the two key words are bumped by the Weyl constants (golden
 * ratio and sqrt(3)-1, scaled to 32 bits) between rounds.
 * ---------------------------------------------------------------------- */
#define PHILOX_MUL_A 0xD2511F53u
#define PHILOX_MUL_B 0xCD9E8D57u
#define PHILOX_WEYL_A 0x9E3779B9u
#define PHILOX_WEYL_B 0xBB67AE85u

void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t x0 = ctr_in[0], x1 = ctr_in[1], x2 = ctr_in[2], x3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t prod_a = (uint64_t)PHILOX_MUL_A * (uint64_t)x0;
        uint64_t prod_b = (uint64_t)PHILOX_MUL_B * (uint64_t)x2;
        uint32_t hi_a = (uint32_t)(prod_a >> 32), lo_a = (uint32_t)prod_a;
        uint32_t hi_b = (uint32_t)(prod_b >> 32), lo_b = (uint32_t)prod_b;
        uint32_t y0 = hi_b ^ x1 ^ k0;
        uint32_t y1 = lo_b;
        uint32_t y2 = hi_a ^ x3 ^ k1;
        uint32_t y3 = lo_a;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += PHILOX_WEYL_A;
        k1 += PHILOX_WEYL_B;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* Drop threshold on an 8-bit draw: round(p * 256), at most 255 (some draw
 * always survives).  An element is dropped iff its draw is below the
 * threshold, so the effective rate is threshold / 256. */
uint32_t oracle_drop_threshold(float p_drop)
{
    if (!(p_drop > 0.0f)) return 0u;
    long long t = llround((double)p_drop * 256.0);
    if (t > 255) t = 255;
    if (t < 0) t = 0;
    return (uint32_t)t;
}

/* The same on a 16-bit draw, round(p * 65536) and at most 65535: the
 * reading of the dropout + residual add + layer norm block's mask. */
uint32_t oracle_drop_threshold16(float p_drop)
{
    if (!(p_drop > 0.0f)) return 0u;
    long long t = llround((double)p_drop * 65536.0);
    if (t > 65535) t = 65535;
    if (t < 0) t = 0;
    return (uint32_t)t;
}

/* The 8-bit draw for element (query i, key j) of flattened query head bh:
 * counter (j / 16, i, bh, offset), key (seed low word, seed high word); the
 * sixteen draws of one call cover keys 16*(j/16) .. 16*(j/16)+15, key j
 * taking byte (j mod 4) (byte 0 = bits 0..7) of output word (j mod 16) / 4. */
uint32_t oracle_draw8(const oracle_params* p, int64_t bh, int64_t i, int64_t j)
{
    uint32_t ctr[4] = {(uint32_t)(j / 16), (uint32_t)i, (uint32_t)bh, (uint32_t)p->offset};
    uint32_t key[2] = {(uint32_t)(p->seed & 0xffffffffu), (uint32_t)(p->seed >> 32)};
    uint32_t w[4];
    oracle_philox4x32_10(ctr, key, w);
    int e = (int)(j % 16);
    return (w[e / 4] >> (8 * (e % 4))) & 0xffu;
}

/* 1 if element (i, j) of head bh survives softmax dropout, 0 if dropped. */
int oracle_keep(const oracle_params* p, int64_t bh, int64_t i, int64_t j)
{
    uint32_t thr = oracle_drop_threshold(p->p_drop);
    if (thr == 0) return 1;
    return oracle_draw8(p, bh, i, j) >= thr ? 1 : 0;
}

/* Z_ij = keep_ij / (1 - p_eff), p_eff = threshold / 256. */
static double keep_scale(const oracle_params* p)
{
    double p_eff = (double)oracle_drop_threshold(p->p_drop) / 256.0;
    return 1.0 / (1.0 - p_eff);
}

double oracle_resolved_scale(const oracle_params* p)
{
    if (p->scale > 0.0f) return (double)p->scale;
    float sc = 1.0f / sqrtf((float)p->d);
    return (double)sc;
}

/* Keys per KV head. */
static int64_t n_keys(const oracle_params* p)
{
    return p->s_kv > 0 ? (int64_t)p->s_kv : (int64_t)p->s;
}

/* Number of keys query i may attend to (keys 0 .. visible_keys - 1). */
static int64_t visible_keys(const oracle_params* p, int64_t i)
{
    const int64_t sk = n_keys(p);
    if (!p->causal) return sk;
    return i + 1 < sk ? i + 1 : sk;
}

/* KV head used by flattened query head bh. */
static int64_t kv_head_of(const oracle_params* p, int64_t bh)
{
    int64_t bi = bh / p->h_q, hq = bh % p->h_q;
    int64_t group = p->h_q / p->h_kv;
    return bi * p->h_kv + hq / group;
}

/* Round to the nearest bf16 value, ties to even (via fp32, which is exact for
 * every bf16 value; the double-to-float step rounds to nearest). */
static double round_bf16(double x)
{
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u) return (double)f;   /* inf / nan */
    u = (u + 0x7fffu + ((u >> 16) & 1u)) & 0xffff0000u;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* One query row of the core: scores S_ij = scale * q_i . k_j for visible j
 * (masked keys are -inf and are simply not formed: exp(-inf) = 0 exactly),
 * the softmax P_ij = exp(S_ij - m_i) / l_i, the dropout factors Z_ij, and
 * LSE_i = m_i + ln l_i.  S, P, Z have room for s_kv entries; entries past the
 * visible keys are set to -inf, 0 and 0. */
static void core_row(const oracle_params* p, const double* q, const double* k,
                     int64_t bh, int64_t i, double* S, double* P, double* Z, double* lse)
{
    const int64_t s = p->s, d = p->d, sk = n_keys(p);
    const double scale = oracle_resolved_scale(p);
    const double zs = keep_scale(p);
    const double* qi = q + (bh * s + i) * d;
    const double* kh = k + kv_head_of(p, bh) * sk * d;
    const int64_t nk = visible_keys(p, i);
    double m = -INFINITY;
    for (int64_t j = 0; j < sk; ++j) {
        if (j < nk) {
            double acc = 0.0;
            for (int64_t c = 0; c < d; ++c) acc += qi[c] * kh[j * d + c];
            S[j] = scale * acc;
            if (S[j] > m) m = S[j];
        } else {
            S[j] = -INFINITY;
        }
    }
    double l = 0.0;
    for (int64_t j = 0; j < nk; ++j) l += exp(S[j] - m);
    for (int64_t j = 0; j < sk; ++j) {
        if (j < nk) {
            P[j] = exp(S[j] - m) / l;
            Z[j] = oracle_keep(p, bh, i, j) ? zs : 0.0;
        } else {
            P[j] = 0.0;
            Z[j] = 0.0;
        }
    }
    if (lse) *lse = m + log(l);
}

/* Forward for a list of (flattened query head, row) pairs:
 * O_i = sum_j P_ij Z_ij v_j and LSE_i.  o has n*d entries, lse n. */
void oracle_fwd_rows(const oracle_params* p, const double* q, const double* k, const double* v,
                     int64_t n, const int64_t* bh_list, const int64_t* row_list,
                     double* o, double* lse)
{
    const int64_t d = p->d, sk = n_keys(p);
#pragma omp parallel
    {
        double* S = (double*)malloc(sizeof(double) * sk);
        double* P = (double*)malloc(sizeof(double) * sk);
        double* Z = (double*)malloc(sizeof(double) * sk);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n; ++r) {
            int64_t bh = bh_list[r], i = row_list[r];
            core_row(p, q, k, bh, i, S, P, Z, &lse[r]);
            const double* vh = v + kv_head_of(p, bh) * sk * d;
            double* oi = o + r * d;
            for (int64_t c = 0; c < d; ++c) oi[c] = 0.0;
            for (int64_t j = 0; j < sk; ++j) {
                double w = P[j] * Z[j];
                if (w == 0.0) continue;
                for (int64_t c = 0; c < d; ++c) oi[c] += w * vh[j * d + c];
            }
        }
        free(S); free(P); free(Z);
    }
}

/* Full forward: O [b, h_q, s, d], LSE [b, h_q, s]. */
void oracle_fwd(const oracle_params* p, const double* q, const double* k, const double* v,
                double* o, double* lse)
{
    const int64_t rows = (int64_t)p->b * p->h_q * p->s;
    int64_t* bh = (int64_t*)malloc(sizeof(int64_t) * rows);
    int64_t* ri = (int64_t*)malloc(sizeof(int64_t) * rows);
    for (int64_t r = 0; r < rows; ++r) { bh[r] = r / p->s; ri[r] = r % p->s; }
    oracle_fwd_rows(p, q, k, v, rows, bh, ri, o, lse);
    free(bh); free(ri);
}

/* Dense matrices of one query head (for self-tests): S, P and the 0/1 keep
 * mask M, each s*s_kv, row-major (query, key). */
void oracle_head_matrices(const oracle_params* p, const double* q, const double* k, int64_t bh,
                          double* S, double* P, uint8_t* M)
{
    const int64_t s = p->s, sk = n_keys(p);
    double* Z = (double*)malloc(sizeof(double) * sk);
    for (int64_t i = 0; i < s; ++i) {
        core_row(p, q, k, bh, i, S + i * sk, P + i * sk, Z, NULL);
        for (int64_t j = 0; j < sk; ++j)
            M[i * sk + j] = (uint8_t)((j < visible_keys(p, i)) ? oracle_keep(p, bh, i, j) : 0);
    }
    free(Z);
}

/* Keep mask of one query head for rows [i0, i1), all s_kv keys, row-major;
 * keys a causal mask hides are reported as 0. */
void oracle_mask_rows(const oracle_params* p, int64_t bh, int64_t i0, int64_t i1, uint8_t* M)
{
    const int64_t sk = n_keys(p);
#pragma omp parallel for schedule(static)
    for (int64_t i = i0; i < i1; ++i)
        for (int64_t j = 0; j < sk; ++j)
            M[(i - i0) * sk + j] = (uint8_t)((j < visible_keys(p, i)) ? oracle_keep(p, bh, i, j) : 0);
}

/* Backward quantities of one query row, given the upstream gradient dO:
 *   dPd_ij = dO_i . v_j        (gradient w.r.t. the dropped-out probabilities)
 *   dP_ij  = dPd_ij * Z_ij     (through the dropout)
 *   dS_ij  = P_ij (dP_ij - sum_k P_ik dP_ik)   (through the softmax)
 * dS has room for s_kv entries (zero past the visible keys). */
static void core_row_grad(const oracle_params* p, const double* v, const double* dout,
                          int64_t bh, int64_t i, const double* P, const double* Z, double* dS,
                          double* rowdot_out)
{
    const int64_t s = p->s, d = p->d, sk = n_keys(p);
    const double* vh = v + kv_head_of(p, bh) * sk * d;
    const double* gi = dout + (bh * s + i) * d;
    const int64_t nk = visible_keys(p, i);
    double rowdot = 0.0;
    for (int64_t j = 0; j < sk; ++j) {
        if (j < nk) {
            double acc = 0.0;
            for (int64_t c = 0; c < d; ++c) acc += gi[c] * vh[j * d + c];
            dS[j] = acc * Z[j];            /* dP_ij */
            rowdot += P[j] * dS[j];
        } else {
            dS[j] = 0.0;
        }
    }
    if (p->stored_o_bf16) {
        /* The method keeps only its output O (bf16) from the forward pass and
         * takes the row statistic from it: sum_j P_ij dP_ij = dO_i . O_i, with
         * O_i here the oracle's own output row rounded to bf16. */
        rowdot = 0.0;
        for (int64_t c = 0; c < d; ++c) {
            double oc = 0.0;
            for (int64_t j = 0; j < nk; ++j) oc += P[j] * Z[j] * vh[j * d + c];
            rowdot += gi[c] * round_bf16(oc);
        }
    }
    for (int64_t j = 0; j < nk; ++j) dS[j] = P[j] * (dS[j] - rowdot);
    if (rowdot_out) *rowdot_out = rowdot;
}

/* dQ for a list of (flattened query head, row) pairs:
 * dQ_i = scale * sum_j dS_ij k_j.  dq has n*d entries. */
void oracle_dq_rows(const oracle_params* p, const double* q, const double* k, const double* v,
                    const double* dout, int64_t n, const int64_t* bh_list, const int64_t* row_list,
                    double* dq)
{
    const int64_t d = p->d, sk = n_keys(p);
    const double scale = oracle_resolved_scale(p);
#pragma omp parallel
    {
        double* S = (double*)malloc(sizeof(double) * sk);
        double* P = (double*)malloc(sizeof(double) * sk);
        double* Z = (double*)malloc(sizeof(double) * sk);
        double* dS = (double*)malloc(sizeof(double) * sk);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n; ++r) {
            int64_t bh = bh_list[r], i = row_list[r];
            core_row(p, q, k, bh, i, S, P, Z, NULL);
            core_row_grad(p, v, dout, bh, i, P, Z, dS, NULL);
            const double* kh = k + kv_head_of(p, bh) * sk * d;
            double* gq = dq + r * d;
            for (int64_t c = 0; c < d; ++c) gq[c] = 0.0;
            for (int64_t j = 0; j < sk; ++j) {
                if (dS[j] == 0.0) continue;
                for (int64_t c = 0; c < d; ++c) gq[c] += dS[j] * kh[j * d + c];
            }
            for (int64_t c = 0; c < d; ++c) gq[c] *= scale;
        }
        free(S); free(P); free(Z); free(dS);
    }
}

/* dK and dV for a list of (flattened KV head, key row) pairs:
 *   dV_j = sum over the query heads of the group, sum_i P_ij Z_ij dO_i
 *   dK_j = scale * sum over the group, sum_i dS_ij q_i
 * with P_ij = exp(S_ij - LSE_i) and dS_ij = P_ij (dP_ij - r_i), where the
 * per-row LSE_i and r_i = sum_k P_ik dP_ik come from a first pass over the
 * query rows that can see the requested keys (all rows if not causal). */
void oracle_dkdv_rows(const oracle_params* p, const double* q, const double* k, const double* v,
                      const double* dout, int64_t n, const int64_t* bkv_list, const int64_t* row_list,
                      double* dk, double* dv)
{
    const int64_t s = p->s, d = p->d, sk = n_keys(p);
    const int64_t group = p->h_q / p->h_kv;
    const int64_t nbh = (int64_t)p->b * p->h_q;
    const double scale = oracle_resolved_scale(p);
    const double zs = keep_scale(p);

    /* first query row needed per query head */
    int64_t* first = (int64_t*)malloc(sizeof(int64_t) * nbh);
    for (int64_t bh = 0; bh < nbh; ++bh) first[bh] = s;
    for (int64_t r = 0; r < n; ++r) {
        int64_t bkv = bkv_list[r], j = row_list[r];
        int64_t bi = bkv / p->h_kv, hk = bkv % p->h_kv;
        for (int64_t g = 0; g < group; ++g) {
            int64_t bh = bi * p->h_q + hk * group + g;
            int64_t lo = p->causal ? j : 0;
            if (lo < first[bh]) first[bh] = lo;
        }
    }
    int64_t ntask = 0;
    for (int64_t bh = 0; bh < nbh; ++bh) ntask += s - first[bh];
    int64_t* task_bh = (int64_t*)malloc(sizeof(int64_t) * (ntask + 1));
    int64_t* task_i = (int64_t*)malloc(sizeof(int64_t) * (ntask + 1));
    ntask = 0;
    for (int64_t bh = 0; bh < nbh; ++bh)
        for (int64_t i = first[bh]; i < s; ++i) { task_bh[ntask] = bh; task_i[ntask] = i; ++ntask; }

    double* lse_all = (double*)malloc(sizeof(double) * nbh * s);
    double* rdot_all = (double*)malloc(sizeof(double) * nbh * s);
#pragma omp parallel
    {
        double* S = (double*)malloc(sizeof(double) * sk);
        double* P = (double*)malloc(sizeof(double) * sk);
        double* Z = (double*)malloc(sizeof(double) * sk);
        double* dS = (double*)malloc(sizeof(double) * sk);
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < ntask; ++t) {
            int64_t bh = task_bh[t], i = task_i[t];
            core_row(p, q, k, bh, i, S, P, Z, &lse_all[bh * s + i]);
            core_row_grad(p, v, dout, bh, i, P, Z, dS, &rdot_all[bh * s + i]);
        }
        free(S); free(P); free(Z); free(dS);
    }

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n; ++r) {
        int64_t bkv = bkv_list[r], j = row_list[r];
        int64_t bi = bkv / p->h_kv, hk = bkv % p->h_kv;
        const double* kj = k + (bkv * sk + j) * d;
        const double* vj = v + (bkv * sk + j) * d;
        double* gk = dk + r * d;
        double* gv = dv + r * d;
        for (int64_t c = 0; c < d; ++c) { gk[c] = 0.0; gv[c] = 0.0; }
        for (int64_t g = 0; g < group; ++g) {
            int64_t bh = bi * p->h_q + hk * group + g;
            for (int64_t i = 0; i < s; ++i) {
                if (j >= visible_keys(p, i)) continue;
                const double* qi = q + (bh * s + i) * d;
                const double* gi = dout + (bh * s + i) * d;
                double sc = 0.0, dpd = 0.0;
                for (int64_t c = 0; c < d; ++c) { sc += qi[c] * kj[c]; dpd += gi[c] * vj[c]; }
                double Pij = exp(scale * sc - lse_all[bh * s + i]);
                double Zij = oracle_keep(p, bh, i, j) ? zs : 0.0;
                double dSij = Pij * (dpd * Zij - rdot_all[bh * s + i]);
                for (int64_t c = 0; c < d; ++c) {
                    gv[c] += Pij * Zij * gi[c];
                    gk[c] += dSij * qi[c];
                }
            }
        }
        for (int64_t c = 0; c < d; ++c) gk[c] *= scale;
    }
    free(first); free(task_bh); free(task_i); free(lse_all); free(rdot_all);
}

/* Full backward: dQ [b, h_q, s, d], dK and dV [b, h_kv, s_kv, d].  One KV
 * head per task: every query row of its group is formed once and its dS row
 * is scattered into dK and dV. */
void oracle_bwd(const oracle_params* p, const double* q, const double* k, const double* v,
                const double* dout, double* dq, double* dk, double* dv)
{
    const int64_t s = p->s, d = p->d, sk = n_keys(p);
    const int64_t group = p->h_q / p->h_kv;
    const int64_t n_kv = (int64_t)p->b * p->h_kv;
    const double scale = oracle_resolved_scale(p);
#pragma omp parallel
    {
        double* S = (double*)malloc(sizeof(double) * sk);
        double* P = (double*)malloc(sizeof(double) * sk);
        double* Z = (double*)malloc(sizeof(double) * sk);
        double* dS = (double*)malloc(sizeof(double) * sk);
#pragma omp for schedule(dynamic, 1)
        for (int64_t bkv = 0; bkv < n_kv; ++bkv) {
            int64_t bi = bkv / p->h_kv, hk = bkv % p->h_kv;
            const double* kh = k + bkv * sk * d;
            double* gkh = dk + bkv * sk * d;
            double* gvh = dv + bkv * sk * d;
            memset(gkh, 0, sizeof(double) * sk * d);
            memset(gvh, 0, sizeof(double) * sk * d);
            for (int64_t g = 0; g < group; ++g) {
                int64_t bh = bi * p->h_q + hk * group + g;
                for (int64_t i = 0; i < s; ++i) {
                    core_row(p, q, k, bh, i, S, P, Z, NULL);
                    core_row_grad(p, v, dout, bh, i, P, Z, dS, NULL);
                    const double* qi = q + (bh * s + i) * d;
                    const double* gi = dout + (bh * s + i) * d;
                    double* gq = dq + (bh * s + i) * d;
                    for (int64_t c = 0; c < d; ++c) gq[c] = 0.0;
                    for (int64_t j = 0; j < visible_keys(p, i); ++j) {
                        double w = P[j] * Z[j];
                        for (int64_t c = 0; c < d; ++c) {
                            gq[c] += dS[j] * kh[j * d + c];
                            gkh[j * d + c] += scale * dS[j] * qi[c];
                            gvh[j * d + c] += w * gi[c];
                        }
                    }
                    for (int64_t c = 0; c < d; ++c) gq[c] *= scale;
                }
            }
        }
        free(S); free(P); free(Z); free(dS);
    }
}

/* ------------------------------------------------------------------------
 * Activation bytes (integer, exact).  "Recomputing Activations", Workshop:
 * per token per layer 34d + 5HT bytes with nothing recomputed, 34d with the
 * attention scores recomputed, 2d with only the layer input kept; here d is
 * the local hidden size h = a * d_head (one rank's shard), H the local head
 * count a and T the sequence length s, so a layer of s*b tokens holds
 * sbh(34 + 5as/h) bytes -- the form the anthology page's takeaways quote.
 * The layer terms describe a self-attention layer of s tokens; the core terms
 * count the actual tensors, with s_kv keys: 5 a s s_kv b score bytes avoided
 * and bf16 Q, O (s rows) and K, V (s_kv rows) kept.
 * ---------------------------------------------------------------------- */
typedef struct {
    int64_t layer_none;           /* 34 s b h + 5 a s^2 b */
    int64_t layer_selective;      /* 34 s b h */
    int64_t layer_full;           /* 2 s b h */
    int64_t core_scores_avoided;  /* 5 a s s_kv b */
    int64_t core_kept;            /* bf16 Q, K, V and O actually kept */
    int64_t core_recompute_state; /* fp32 LSE per query row + seed + offset */
} oracle_bytes;

void oracle_stored_bytes(const oracle_params* p, oracle_bytes* out)
{
    const int64_t s = p->s, sk = n_keys(p), b = p->b, a = p->h_q, akv = p->h_kv, dh = p->d;
    const int64_t h = a * dh;
    out->layer_selective = 34 * s * b * h;
    out->layer_none = out->layer_selective + 5 * a * s * s * b;
    out->layer_full = 2 * s * b * h;
    out->core_scores_avoided = 5 * a * s * sk * b;
    out->core_kept = 2 * dh * b * (2 * a * s + 2 * akv * sk);
    out->core_recompute_state = 4 * b * a * s + 16;
}
