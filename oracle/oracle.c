/*
 * oracle.c -- plain, slow, double-precision CPU oracle for the Qwen3-style
 * RMSNorm forward and backward, its fused residual-add variant and (through
 * the same definition) its split-row forward.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load this library. The CUDA library shares no
 * code, header, helper, table or constant with it, and neither side includes
 * or calls the other.
 *
 * Sources, cited below by tag:
 *   [P1] "训推加速 Qwen3 实战：从“调包”到手写 Triton Kernel（含 backward）"
 *        (iqiancheng.github.io, posts/triton-kernel-fusion-practice)
 *   [P2] the article on hand-writing 21 Triton kernels for decoding a 0.8B
 *        Qwen model on one consumer GPU (trdm.cn, news/483216; the extracted
 *        page carries no title)
 *
 * Every function writes its definition out with plain loops in double
 * precision: no blocking, no fusion, no reordering beyond what the definition
 * states, so that it can be checked against the pages by eye. Inputs are read
 * in their stored format (fp32, bf16 or fp16 bit patterns, or fp64) and
 * decoded here,
 * exactly, to double. Results stay in double and are never rounded, except the
 * residual sum h, which the method stores in the input dtype.
 *
 * Parity status: every function below is pinned by the CPU tests (closed
 * forms, invariants, central finite differences, a library rounding routine);
 * none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F64 2
#define ORACLE_F16 3

/* ---------------------------------------------------------------- formats */

/* bfloat16 is the upper 16 bits of an IEEE binary32; widening is exact. */
double oracle_bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round a double to the nearest bfloat16, ties to even, in one step (no
 * intermediate rounding to binary32, which could round twice).
 * bfloat16 keeps 8 significant bits, normal exponents -126..127, subnormals
 * down to 2^-133.
 */
uint16_t oracle_bf16_from_double(double v)
{
    if (isnan(v))
        return (uint16_t)(signbit(v) ? 0xFFC0u : 0x7FC0u);
    if (v == 0.0)
        return (uint16_t)(signbit(v) ? 0x8000u : 0x0000u);
    int e;
    (void)frexp(v, &e);            /* |v| in [2^(e-1), 2^e) */
    int q = e - 8;                 /* spacing of 8-bit significands there */
    if (q < -133)
        q = -133;                  /* subnormal spacing */
    double scaled = ldexp(v, -q);  /* exact: a power-of-two scaling */
    double n = nearbyint(scaled);  /* default mode: nearest, ties to even */
    double r = ldexp(n, q);
    const double bf16_max = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
    if (fabs(r) > bf16_max)
        return (uint16_t)(v < 0 ? 0xFF80u : 0x7F80u);
    float f = (float)r;            /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* IEEE binary16: sign, 5-bit exponent with bias 15, 10 stored fraction
 * bits; exponent 0 holds subnormals (fraction * 2^-24), 31 infinities and
 * NaNs. Widening to double is exact. */
double oracle_f16_to_double(uint16_t bits)
{
    const int sign = bits >> 15;
    const int exp = (bits >> 10) & 0x1F;
    const int frac = bits & 0x3FF;
    double v;
    if (exp == 0)
        v = ldexp((double)frac, -24);
    else if (exp == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), exp - 25);
    return sign ? -v : v;
}

/*
 * Round a double to the nearest binary16, ties to even, in one step: 11
 * significant bits for normal numbers (exponents -14..15), spacing 2^-24 for
 * subnormals, infinity beyond the largest finite value 65504 (the tie at
 * 65520 goes to infinity, whose significand is even).
 */
uint16_t oracle_f16_from_double(double v)
{
    if (isnan(v))
        return (uint16_t)(signbit(v) ? 0xFE00u : 0x7E00u);
    const uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    int e;
    (void)frexp(a, &e);            /* a in [2^(e-1), 2^e) */
    int q = e - 11;                /* spacing of 11-bit significands there */
    if (q < -24)
        q = -24;                   /* subnormal spacing */
    double r = ldexp(nearbyint(ldexp(a, -q)), q);
    if (r > 65504.0)
        return (uint16_t)(sign | 0x7C00u);
    /* encode the representable r */
    if (r < ldexp(1.0, -14))
        return (uint16_t)(sign | (uint16_t)ldexp(r, 24));          /* subnormal */
    int re;
    double m = frexp(r, &re);      /* r = m 2^re, m in [0.5, 1) */
    int exp = re - 1 + 15;
    int frac = (int)ldexp(m, 11) - 1024;
    return (uint16_t)(sign | (exp << 10) | frac);
}

static double dec(const void *p, int dtype, int64_t i)
{
    switch (dtype) {
    case ORACLE_F32:
        return (double)((const float *)p)[i];
    case ORACLE_BF16:
        return oracle_bf16_to_double(((const uint16_t *)p)[i]);
    case ORACLE_F16:
        return oracle_f16_to_double(((const uint16_t *)p)[i]);
    default:
        return ((const double *)p)[i];
    }
}

/* Store v in the given format, rounding to nearest-even; returns the stored
 * value read back as a double. */
static double store_rounded(void *p, int dtype, int64_t i, double v)
{
    switch (dtype) {
    case ORACLE_F32: {
        float f = (float)v; /* C conversion in the default rounding mode */
        ((float *)p)[i] = f;
        return (double)f;
    }
    case ORACLE_BF16: {
        uint16_t b = oracle_bf16_from_double(v);
        ((uint16_t *)p)[i] = b;
        return oracle_bf16_to_double(b);
    }
    case ORACLE_F16: {
        uint16_t b = oracle_f16_from_double(v);
        ((uint16_t *)p)[i] = b;
        return oracle_f16_to_double(b);
    }
    default:
        ((double *)p)[i] = v;
        return v;
    }
}

/* ---------------------------------------------------------------- forward */

/*
 * [P1 §4.1]: per row i of x (M rows of H features) and a per-feature weight w,
 *   r_i   = 1 / sqrt( (1/H) * sum_j x_ij^2 + eps )
 *   y_ij  = w_j * x_ij * r_i
 * [P1 §4.2] divides the sum of squares by the true feature count H and adds
 * eps inside the square root. [P2 §3.2] computes the same sum of squares in
 * pieces and merges them; the merged value is this same sum, so the split-row
 * forward has this definition too.
 * y (M*H) and rstd (M) are outputs; either may be NULL.
 */
void oracle_rmsnorm_fwd(int64_t M, int64_t H, const void *x, const void *w,
                        int dtype, double eps, double *y, double *rstd)
{
    for (int64_t i = 0; i < M; ++i) {
        double ss = 0.0;
        for (int64_t j = 0; j < H; ++j) {
            double xv = dec(x, dtype, i * H + j);
            ss += xv * xv;
        }
        double ms = ss / (double)H;
        double r = 1.0 / sqrt(ms + eps);
        if (rstd)
            rstd[i] = r;
        if (y)
            for (int64_t j = 0; j < H; ++j)
                y[i * H + j] = dec(w, dtype, j) * dec(x, dtype, i * H + j) * r;
    }
}

/* --------------------------------------------------------------- backward */

/*
 * [P1 §5.3]: with wdy_j = w_j * dy_j and c = (1/H) * sum_j wdy_j * x_j,
 *   dx_ij = r_i * ( w_j * dy_ij - x_ij * r_i^2 * c_i )
 *   dw_j  = sum_i dy_ij * x_ij * r_i          (a sum over all rows)
 * with r_i recomputed from x as in the forward ([P1 §5.4] recomputes it).
 *
 * Optional error-scale outputs (sums of absolute values of the terms that
 * make up each result; used by the tests' tolerances):
 *   tdx_ij = |r_i w_j dy_ij| + |x_ij| r_i^3 (1/H) sum_k |w_k dy_ik x_ik|
 *   tdw_j  = sum_i |dy_ij x_ij r_i|
 * dx, dw, tdx, tdw may each be NULL. dw and tdw have H entries and are
 * overwritten (not accumulated into).
 */
void oracle_rmsnorm_bwd(int64_t M, int64_t H, const void *dy, const void *x,
                        const void *w, int dtype, double eps, double *dx,
                        double *dw, double *tdx, double *tdw)
{
    if (dw)
        for (int64_t j = 0; j < H; ++j)
            dw[j] = 0.0;
    if (tdw)
        for (int64_t j = 0; j < H; ++j)
            tdw[j] = 0.0;
    for (int64_t i = 0; i < M; ++i) {
        double ss = 0.0;
        for (int64_t j = 0; j < H; ++j) {
            double xv = dec(x, dtype, i * H + j);
            ss += xv * xv;
        }
        double r = 1.0 / sqrt(ss / (double)H + eps);

        double csum = 0.0, cabs = 0.0;
        for (int64_t j = 0; j < H; ++j) {
            double wdy = dec(w, dtype, j) * dec(dy, dtype, i * H + j);
            double xv = dec(x, dtype, i * H + j);
            csum += wdy * xv;
            cabs += fabs(wdy * xv);
        }
        double c = csum / (double)H;

        for (int64_t j = 0; j < H; ++j) {
            double xv = dec(x, dtype, i * H + j);
            double dyv = dec(dy, dtype, i * H + j);
            double wdy = dec(w, dtype, j) * dyv;
            if (dx)
                dx[i * H + j] = r * (wdy - xv * r * r * c);
            if (tdx)
                tdx[i * H + j] =
                    fabs(r * wdy) + fabs(xv) * r * r * r * (cabs / (double)H);
            if (dw)
                dw[j] += dyv * xv * r;
            if (tdw)
                tdw[j] += fabs(dyv * xv * r);
        }
    }
}

/* -------------------------------------------------------- residual variant */

/*
 * Residual add fused with the norm ([P1 §1] names "residual + next RMSNorm"
 * as the cross-block fusion a compiler misses; [P2 §2.1] lists residual_add
 * followed by rms_norm and plans their fused kernel):
 *   h_ij = round_to_dtype(x_ij + r_ij)       written out (the new residual)
 *   y, rstd = the forward above applied to the stored h
 * The sum of two bf16 (or two fp32) values is formed in double and rounded
 * once to the stored format. h has the input dtype; y and rstd are doubles.
 */
void oracle_residual_fwd(int64_t M, int64_t H, const void *x, const void *res,
                         const void *w, int dtype, double eps, void *h,
                         double *y, double *rstd)
{
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < H; ++j) {
            double s = dec(x, dtype, i * H + j) + dec(res, dtype, i * H + j);
            (void)store_rounded(h, dtype, i * H + j, s);
        }
    oracle_rmsnorm_fwd(M, H, h, w, dtype, eps, y, rstd);
}

/*
 * Backward of the residual variant. h = x + r feeds the norm and also flows
 * on as the residual stream, whose gradient dh_out arrives from the next
 * block (NULL means zero). Since dh/dx = dh/dr = identity, the gradient of
 * both x and r is
 *   dx_ij = (backward of the norm at h)_ij + dh_out_ij
 * and dw is the norm's dw at h ([P1 §5.3] applied to h).
 */
void oracle_residual_bwd(int64_t M, int64_t H, const void *dy,
                         const void *dh_out, const void *h, const void *w,
                         int dtype, double eps, double *dx, double *dw,
                         double *tdx, double *tdw)
{
    oracle_rmsnorm_bwd(M, H, dy, h, w, dtype, eps, dx, dw, tdx, tdw);
    if (dh_out)
        for (int64_t i = 0; i < M; ++i)
            for (int64_t j = 0; j < H; ++j) {
                double g = dec(dh_out, dtype, i * H + j);
                if (dx)
                    dx[i * H + j] += g;
                if (tdx)
                    tdx[i * H + j] += fabs(g);
            }
}

/* ---------------------------------------------------- double backward */

/*
 * Second derivatives ([P1 §5.6] lists double backward as what an autograd
 * wrapper must either implement or refuse). The backward of [P1 §5.3] maps
 * (dy, x, w) to dx and dw; given incoming gradients gx [M,H] on dx and gw [H]
 * on dw (either may be NULL: zero), this returns the gradients of
 *   L2 = sum_ij gx_ij dx_ij + sum_j gw_j dw_j
 * with respect to dy, x and w. Per row, with r = 1/sqrt(mean(x^2) + eps)
 * (a function of x), c = (1/H) sum_k w_k dy_k x_k and the row sums
 *   A = sum_k gx_k w_k dy_k,  B = sum_k gx_k x_k,  D = sum_k gw_k dy_k x_k,
 * differentiating dx_k = r w_k dy_k - r^3 c x_k and dw_k = sum dy_k x_k r
 * term by term (dr/dx_k = -r^3 x_k / H, dc/dx_k = w_k dy_k / H,
 * dc/ddy_k = w_k x_k / H, dc/dw_k = dy_k x_k / H) gives
 *   ddy_k = r w_k gx_k - (r^3 B / H) w_k x_k + r gw_k x_k
 *   dx2_k = (r^3 / H)(3 r^2 c B - A - D) x_k - (r^3 B / H) w_k dy_k
 *           - r^3 c gx_k + r gw_k dy_k
 *   dw2_k = sum over rows of  r gx_k dy_k - (r^3 B / H) dy_k x_k
 * Inputs dy, x, w, gx in the stored format; gw in double. Outputs in double;
 * t_* (each may be NULL) are the error scales, the sums of the absolute
 * values of the terms.
 */
void oracle_rmsnorm_bwd_bwd(int64_t M, int64_t H, const void *dy, const void *x,
                            const void *w, const void *gx, const double *gw,
                            int dtype, double eps, double *ddy, double *dx2,
                            double *dw2, double *t_ddy, double *t_dx2,
                            double *t_dw2)
{
    for (int64_t j = 0; j < H; ++j) {
        dw2[j] = 0.0;
        if (t_dw2)
            t_dw2[j] = 0.0;
    }
    for (int64_t i = 0; i < M; ++i) {
        double ss = 0.0, cs = 0.0, A = 0.0, B = 0.0, D = 0.0;
        double cabs = 0.0, Aabs = 0.0, Babs = 0.0, Dabs = 0.0;
        for (int64_t k = 0; k < H; ++k) {
            double xv = dec(x, dtype, i * H + k);
            double dyv = dec(dy, dtype, i * H + k);
            double wv = dec(w, dtype, k);
            double g = gx ? dec(gx, dtype, i * H + k) : 0.0;
            double gwv = gw ? gw[k] : 0.0;
            ss += xv * xv;
            cs += wv * dyv * xv;
            A += g * wv * dyv;
            B += g * xv;
            D += gwv * dyv * xv;
            cabs += fabs(wv * dyv * xv);
            Aabs += fabs(g * wv * dyv);
            Babs += fabs(g * xv);
            Dabs += fabs(gwv * dyv * xv);
        }
        double mean_sq = ss / (double)H;
        double r = 1.0 / sqrt(mean_sq + eps);
        double c = cs / (double)H;
        double r3 = r * r * r;
        for (int64_t k = 0; k < H; ++k) {
            double xv = dec(x, dtype, i * H + k);
            double dyv = dec(dy, dtype, i * H + k);
            double wv = dec(w, dtype, k);
            double g = gx ? dec(gx, dtype, i * H + k) : 0.0;
            double gwv = gw ? gw[k] : 0.0;
            double t1 = r * wv * g, t2 = (r3 * B / (double)H) * wv * xv, t3 = r * gwv * xv;
            ddy[i * H + k] = t1 - t2 + t3;
            double u1 = (r3 / (double)H) * (3.0 * r * r * c * B - A - D) * xv;
            double u2 = (r3 * B / (double)H) * wv * dyv;
            double u3 = r3 * c * g;
            double u4 = r * gwv * dyv;
            dx2[i * H + k] = u1 - u2 - u3 + u4;
            double v1 = r * g * dyv, v2 = (r3 * B / (double)H) * dyv * xv;
            dw2[k] += v1 - v2;
            if (t_ddy)
                t_ddy[i * H + k] = fabs(t1) + (r3 * Babs / (double)H) * fabs(wv * xv) + fabs(t3);
            if (t_dx2)
                t_dx2[i * H + k] =
                    (r3 / (double)H) * (3.0 * r * r * (cabs / (double)H) * Babs + Aabs + Dabs) *
                        fabs(xv) +
                    (r3 * Babs / (double)H) * fabs(wv * dyv) + r3 * (cabs / (double)H) * fabs(g) +
                    fabs(u4);
            if (t_dw2)
                t_dw2[k] += fabs(v1) + (r3 * Babs / (double)H) * fabs(dyv * xv);
        }
    }
}

/* ------------------------------------------------ norm, then projection */

/* v rounded to the given storage format (nearest, ties to even). */
static double round_to(int dtype, double v)
{
    switch (dtype) {
    case ORACLE_F32:
        return (double)(float)v;
    case ORACLE_BF16:
        return oracle_bf16_to_double(oracle_bf16_from_double(v));
    case ORACLE_F16:
        return oracle_f16_to_double(oracle_f16_from_double(v));
    default:
        return v;
    }
}

/*
 * The decode chain of [P2]: the norm (optionally after the residual add)
 * feeds the projection GEMVs -- q/k/v_proj, gate/up_proj ([P2 §2.1] ops
 * 3-5, 10-13; §3.1: a [1, 896] hidden state against the [1024, 896] q_proj
 * weight) -- and [P2 §6] names fusing these steps as the next optimisation.
 * The fused result is defined as the chain's: the norm's output y is stored
 * in the dtype (the separate rms_norm kernel writes it, the GEMV reads it
 * back), then, for a row-major weight A of N rows of H (a linear layer's
 * weight),
 *   out_in = sum_k y_ik A_nk          in double, unrounded.
 * res and h: the residual variant (both NULL for the plain norm), h as in
 * oracle_residual_fwd. y_store (may be NULL) receives the stored y; rstd
 * (may be NULL) as for the forward; tout (may be NULL) receives the error
 * scale sum_k |y_ik A_nk|. Returns 0, or -1 if scratch memory is short.
 */
int oracle_rmsnorm_gemv(int64_t M, int64_t H, int64_t N, const void *x,
                        const void *res, const void *w, const void *A,
                        int dtype, double eps, void *h, void *y_store,
                        double *out, double *rstd, double *tout)
{
    double *y = (double *)malloc((size_t)(M * H > 0 ? M * H : 1) * sizeof(double));
    if (!y)
        return -1;
    if (res)
        oracle_residual_fwd(M, H, x, res, w, dtype, eps, h, y, rstd);
    else
        oracle_rmsnorm_fwd(M, H, x, w, dtype, eps, y, rstd);
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < H; ++j) {
            y[i * H + j] = round_to(dtype, y[i * H + j]);
            if (y_store)
                (void)store_rounded(y_store, dtype, i * H + j, y[i * H + j]);
        }
    for (int64_t i = 0; i < M; ++i)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < H; ++k) {
                double term = y[i * H + k] * dec(A, dtype, n * H + k);
                acc += term;
                mag += fabs(term);
            }
            out[i * N + n] = acc;
            if (tout)
                tout[i * N + n] = mag;
        }
    free(y);
    return 0;
}
