/*
 * dropout_add_ln_oracle.c -- plain, slow CPU oracle for the dropout,
 * residual add and layer norm that sit on either side of the attention core.
 * TEST INFRASTRUCTURE ONLY (see attn_oracle.c): only the tests, the smoke
 * check and the bench's CPU-baseline leg call it; the product library shares
 * no code with it.
 *
 * Where the pages define it: "Reducing Activation Recomputation in Large
 * Transformer Models" (dmarx anthology, LIT-736), Key takeaways, first and
 * second bullets: the layer norms and the dropouts after the attention block
 * and the MLP are the part of a layer that tensor parallelism leaves
 * replicated (the 10sbh term), and they act on every sequence position
 * independently, which is why sequence parallelism can split them by rows.
 * The pages give no formula for the block; the reading taken is the standard
 * residual sub-layer boundary of a transformer layer:
 *     z = residual + dropout(x)                     (stored: next residual)
 *     y = gamma * (z - mean(z)) / sqrt(var(z) + eps) + beta   (next input)
 * per row (token) over the hidden dimension H, var the biased (1/H) variance.
 * Dropout uses Philox-4x32-10 with 16-bit draws (eight per call; the
 * attention core reads 8-bit ones), drop iff draw < round(p * 65536), kept
 * values scaled by 1 / (1 - p_eff), with counter (col / 8, row, 0xFFFFFFFF,
 * offset): word 2 is a value no attention head index takes.
 *
 * The backward takes dy (gradient of y) and, optionally, dz_next (the
 * gradient reaching z through the residual path) and returns
 *     dz = rstd * (g - mean(g) - xhat * mean(g * xhat)) + dz_next,
 *          g = dy * gamma, xhat = (z - mean) * rstd,
 *     d_residual = dz,  dx = dz * Z  (Z = keep / (1 - p_eff)),
 *     dgamma = sum over rows of dy * xhat,  dbeta = sum over rows of dy.
 * Everything is fp64; z is not rounded (the GPU stores it in bf16, an error
 * at bf16 resolution that the parity tolerance covers).
 *
 * Parity status: pinned by CPU tests against torch's fp64 layer_norm and its
 * autograd (p = 0, and p > 0 with this oracle's own mask), central finite
 * differences, a second statement of the mask mapping, and row invariants.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Philox-4x32-10 and the drop threshold, from attn_oracle.c (same library). */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]);
uint32_t oracle_drop_threshold16(float p_drop);

typedef struct {
    int32_t n_rows, hidden;
    float p_drop;
    float eps;
    uint64_t seed, offset;
} oracle_dal_params;

/* 1 if element (row, col) of x survives the dropout, 0 if dropped. */
int oracle_dal_keep(const oracle_dal_params* p, int64_t row, int64_t col)
{
    const uint32_t thr = oracle_drop_threshold16(p->p_drop);
    if (thr == 0) return 1;
    uint32_t ctr[4] = {(uint32_t)(col / 8), (uint32_t)row, 0xFFFFFFFFu, (uint32_t)p->offset};
    uint32_t key[2] = {(uint32_t)(p->seed & 0xffffffffu), (uint32_t)(p->seed >> 32)};
    uint32_t w[4];
    oracle_philox4x32_10(ctr, key, w);
    const int e = (int)(col % 8);
    const uint32_t draw = (e % 2 == 0) ? (w[e / 2] & 0xffffu) : (w[e / 2] >> 16);
    return draw >= thr ? 1 : 0;
}

static double dal_keep_scale(const oracle_dal_params* p)
{
    return 1.0 / (1.0 - (double)oracle_drop_threshold16(p->p_drop) / 65536.0);
}

/* z of one row, then its mean and 1/sqrt(var + eps). */
static void dal_row(const oracle_dal_params* p, const double* x, const double* r, int64_t row, double* z,
                    double* mean, double* rstd)
{
    const int64_t H = p->hidden;
    const double zs = dal_keep_scale(p);
    double m = 0.0;
    for (int64_t c = 0; c < H; ++c) {
        const double zc = r[row * H + c] + (oracle_dal_keep(p, row, c) ? zs * x[row * H + c] : 0.0);
        z[c] = zc;
        m += zc;
    }
    m /= (double)H;
    double v = 0.0;
    for (int64_t c = 0; c < H; ++c) v += (z[c] - m) * (z[c] - m);
    v /= (double)H;
    *mean = m;
    *rstd = 1.0 / sqrt(v + (double)p->eps);
}

/* Forward: z, y [n_rows, hidden]; mean, rstd [n_rows]. */
void oracle_dal_fwd(const oracle_dal_params* p, const double* x, const double* r, const double* gamma,
                    const double* beta, double* z, double* y, double* mean, double* rstd)
{
    const int64_t H = p->hidden;
#pragma omp parallel for schedule(static)
    for (int64_t row = 0; row < p->n_rows; ++row) {
        double* zr = z + row * H;
        dal_row(p, x, r, row, zr, &mean[row], &rstd[row]);
        for (int64_t c = 0; c < H; ++c) y[row * H + c] = gamma[c] * (zr[c] - mean[row]) * rstd[row] + beta[c];
    }
}

/* Backward: dx, dres [n_rows, hidden]; dgamma, dbeta [hidden].  dz_next may
 * be NULL (no gradient through the residual path). */
void oracle_dal_bwd(const oracle_dal_params* p, const double* x, const double* r, const double* gamma,
                    const double* dy, const double* dz_next, double* dx, double* dres, double* dgamma,
                    double* dbeta)
{
    const int64_t H = p->hidden, N = p->n_rows;
    const double zs = dal_keep_scale(p);
    double* xhat_all = (double*)malloc(sizeof(double) * N * H);
#pragma omp parallel
    {
        double* z = (double*)malloc(sizeof(double) * H);
        double* g = (double*)malloc(sizeof(double) * H);
#pragma omp for schedule(static)
        for (int64_t row = 0; row < N; ++row) {
            double mean, rstd;
            dal_row(p, x, r, row, z, &mean, &rstd);
            double* xh = xhat_all + row * H;
            double mg = 0.0, mgx = 0.0;
            for (int64_t c = 0; c < H; ++c) {
                xh[c] = (z[c] - mean) * rstd;
                g[c] = dy[row * H + c] * gamma[c];
                mg += g[c];
                mgx += g[c] * xh[c];
            }
            mg /= (double)H;
            mgx /= (double)H;
            for (int64_t c = 0; c < H; ++c) {
                double dz = rstd * (g[c] - mg - xh[c] * mgx);
                if (dz_next) dz += dz_next[row * H + c];
                dres[row * H + c] = dz;
                dx[row * H + c] = oracle_dal_keep(p, row, c) ? dz * zs : 0.0;
            }
        }
        free(z);
        free(g);
    }
    /* column sums over the rows, in row order */
    for (int64_t c = 0; c < H; ++c) {
        double sg = 0.0, sb = 0.0;
        for (int64_t row = 0; row < N; ++row) {
            sg += dy[row * H + c] * xhat_all[row * H + c];
            sb += dy[row * H + c];
        }
        dgamma[c] = sg;
        dbeta[c] = sb;
    }
    free(xhat_all);
}
