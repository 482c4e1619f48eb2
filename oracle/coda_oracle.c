/*
 * CPU oracle for the CODA GEMM-epilogue block -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, unfused, fp64.  Nothing here is blocked, fused or reordered:
 * every routine is the textbook definition of one step of a pre-norm LLaMA
 * block as the CODA write-ups describe it, so a reader can check it by eye.
 * It shares no code, header or constant with the CUDA library and must only
 * be called from the tests, the package smoke check and the benchmark's CPU
 * baseline leg and reference arm.
 *
 * Sources (the CODA news write-ups, three translations of one article):
 *   - "CODA: the treasure hidden in the epilogue": the GEMM -> residual add ->
 *     RMSNorm -> GEMM pattern; RMSNorm's per-row scale r commutes with the
 *     next matmul; SwiGLU, RoPE and cross-entropy admit the same treatment.
 *   - "lazy tax of large-model training": the block's memory-bound operators
 *     (RMSNorm, SwiGLU, residual add) and the move to FP8 operands.
 *
 * Storage: row-major; weights in the mathematical orientation W [K x N]
 * so that a product reads Y = X . W exactly as the pages write it.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Thread count of the OpenMP loops below (n > 0 sets it; n <= 0 leaves it);
 * returns the count in effect.  For timing the oracle on one core: the
 * arithmetic and its order within each output element do not depend on it. */
int coda_oracle_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* C = R + A . W   (R may be NULL, meaning zero).
 * A [M x K], W [K x N], R and C [M x N].  i-k-j loops, fp64 accumulate.
 * With R this is the first GEMM of the block and its residual add ("the
 * treasure hidden in the epilogue"); with R == NULL it is a plain matmul. */
void coda_oracle_gemm(const double *A, const double *W, const double *R, double *C,
                      int64_t M, int64_t N, int64_t K)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        double *c = C + i * N;
        for (int64_t j = 0; j < N; ++j)
            c[j] = R ? R[i * N + j] : 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = A[i * K + k];
            const double *w = W + k * N;
            for (int64_t j = 0; j < N; ++j)
                c[j] += a * w[j];
        }
    }
}

/* RMSNorm (LLaMA form): ms_i = (1/N) sum_j h_ij^2 ; rstd_i = 1/sqrt(ms_i + eps);
 * y_ij = h_ij * rstd_i * gamma_j.  Y may be NULL when only rstd is wanted. */
void coda_oracle_rmsnorm(const double *H, const double *gamma, double eps,
                         int64_t M, int64_t N, double *Y, double *rstd)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        const double *h = H + i * N;
        double ss = 0.0;
        for (int64_t j = 0; j < N; ++j)
            ss += h[j] * h[j];
        const double r = 1.0 / sqrt(ss / (double)N + eps);
        rstd[i] = r;
        if (Y)
            for (int64_t j = 0; j < N; ++j)
                Y[i * N + j] = h[j] * r * gamma[j];
    }
}

/* silu(x) = x * sigmoid(x) = x / (1 + exp(-x)). */
double coda_oracle_silu(double x)
{
    return x / (1.0 + exp(-x));
}

/* SwiGLU gating of two already-computed projections: act = silu(G) * U. */
void coda_oracle_silu_mul(const double *G, const double *U, int64_t n, double *act)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        act[i] = coda_oracle_silu(G[i]) * U[i];
}

/* ---- OCP FP8 E4M3 ("fn": no infinities) -------------------------------
 * 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits.
 * Normal: (-1)^s * 2^(e-7) * (1 + m/8), e in 1..15, except e=15,m=7 = NaN.
 * Subnormal (e=0): (-1)^s * 2^-6 * (m/8).   Largest finite: 448. */
double coda_oracle_e4m3_decode(uint8_t code)
{
    const int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round to nearest, ties to even, saturating to +-448 ("satfinite"). */
uint8_t coda_oracle_e4m3_encode(double x)
{
    if (isnan(x))
        return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0)
        return sign | 0x7E;                 /* e=15, m=6: 448 */
    if (a < ldexp(1.0, -6)) {
        /* subnormal grid: multiples of 2^-9; q == 8 lands on 2^-6 (e=1,m=0) */
        const double q = nearbyint(a / ldexp(1.0, -9));
        return sign | (uint8_t)q;
    }
    int e2;
    (void)frexp(a, &e2);                    /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;                         /* a in [2^e, 2^(e+1)) */
    double q = nearbyint(a / ldexp(1.0, e - 3));  /* in [8, 16] */
    if (q >= 16.0) {
        q = 8.0;
        e += 1;
    }
    if (e + 7 > 15 || (e + 7 == 15 && q - 8.0 > 6.0))
        return sign | 0x7E;
    return sign | (uint8_t)(((e + 7) << 3) | (int)(q - 8.0));
}

/* Round to the nearest bfloat16 value, ties to even: 1 sign bit, 8 exponent
 * bits (the fp32 range), 8 significant bits.  A value a in [2^(e-1), 2^e)
 * lies on the grid k * 2^(e-8), k in [128, 256); below 2^-126 the grid is the
 * subnormal one, multiples of 2^-133.  Magnitudes past the largest finite
 * value, 255 * 2^120, round to infinity.  Zeros, infinities and NaNs pass. */
double coda_oracle_round_bf16(double x)
{
    if (x == 0.0 || !isfinite(x))
        return x;
    int e;
    (void)frexp(x, &e);                     /* |x| = f * 2^e, f in [0.5, 1) */
    int ulp_e = e - 8;
    if (ulp_e < -133)
        ulp_e = -133;
    const double y = ldexp(nearbyint(ldexp(x, -ulp_e)), ulp_e);  /* both scalings exact */
    if (fabs(y) > ldexp(255.0, 120))
        return copysign(INFINITY, x);
    return y;
}

void coda_oracle_round_bf16_array(const double *x, int64_t n, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = coda_oracle_round_bf16(x[i]);
}

/* max_i |x_i| */
double coda_oracle_amax(const double *x, int64_t n)
{
    double m = 0.0;
    for (int64_t i = 0; i < n; ++i)
        if (fabs(x[i]) > m)
            m = fabs(x[i]);
    return m;
}

/* Per-tensor FP8 quantise-dequantise: s = amax / 448 ; q_i = E4M3(x_i / s) ;
 * out_i = decode(q_i) * s.  Returns s (1 when the tensor is all zero). */
double coda_oracle_e4m3_fake_quant(const double *x, int64_t n, double *out)
{
    const double amax = coda_oracle_amax(x, n);
    const double s = amax > 0.0 ? amax / 448.0 : 1.0;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = coda_oracle_e4m3_decode(coda_oracle_e4m3_encode(x[i] / s)) * s;
    return s;
}

/* Rotary position embedding, the RoFormer definition with interleaved pairs
 * (the CODA write-up names RoPE among the operations that move into a GEMM
 * epilogue).  For row i at position pos[i], each head of `head_dim` columns
 * among the first `rot_cols` columns, and pair j < head_dim/2:
 *   phi = pos[i] * base^(-2j/head_dim)
 *   (z_2j, z_2j+1) -> (z_2j cos(phi) - z_2j+1 sin(phi), z_2j sin(phi) + z_2j+1 cos(phi))
 * Columns from rot_cols on (V in a fused QKV output) are left unchanged.
 * In place on Z [M x N]. */
void coda_oracle_rope(double *Z, int64_t M, int64_t N, int64_t rot_cols, int64_t head_dim,
                      const int64_t *pos, double base)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        double *z = Z + i * N;
        for (int64_t c = 0; c + 1 < rot_cols; c += 2) {
            const int64_t j = (c % head_dim) / 2;
            const double phi = (double)pos[i] * pow(base, -2.0 * (double)j / (double)head_dim);
            const double a = z[c], b = z[c + 1];
            z[c] = a * cos(phi) - b * sin(phi);
            z[c + 1] = a * sin(phi) + b * cos(phi);
        }
    }
}

/* Backward of RMSNorm (LLaMA form y = h r gamma, r = 1/sqrt(mean h^2 + eps))
 * for one upstream gradient dY [M x N]:
 *   dH_ij    = r_i gamma_j dY_ij - h_ij r_i^3 / N * sum_k gamma_k dY_ik h_ik
 *   dgamma_j = sum_i dY_ij h_ij r_i
 * (differentiating y_ij = h_ij r_i gamma_j with d r_i / d h_ik = -r_i^3 h_ik / N).
 * dgamma is written, not accumulated. */
void coda_oracle_rmsnorm_backward(const double *H, const double *gamma, double eps, const double *dY,
                                  int64_t M, int64_t N, double *dH, double *dgamma)
{
    for (int64_t j = 0; j < N; ++j)
        dgamma[j] = 0.0;
    for (int64_t i = 0; i < M; ++i) {
        const double *h = H + i * N, *dy = dY + i * N;
        double ss = 0.0, dot = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            ss += h[j] * h[j];
            dot += gamma[j] * dy[j] * h[j];
        }
        const double r = 1.0 / sqrt(ss / (double)N + eps);
        for (int64_t j = 0; j < N; ++j) {
            dH[i * N + j] = r * gamma[j] * dy[j] - h[j] * r * r * r / (double)N * dot;
            dgamma[j] += dy[j] * h[j] * r;
        }
    }
}

/* Backward of SwiGLU gating act = silu(G) * U, silu(x) = x sigmoid(x):
 *   dG = dAct * U * silu'(G),  silu'(x) = sigmoid(x) (1 + x (1 - sigmoid(x)))
 *   dU = dAct * silu(G) */
void coda_oracle_silu_mul_backward(const double *G, const double *U, const double *dAct, int64_t n,
                                   double *dG, double *dU)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        const double s = 1.0 / (1.0 + exp(-G[i]));
        dG[i] = dAct[i] * U[i] * s * (1.0 + G[i] * (1.0 - s));
        dU[i] = dAct[i] * G[i] * s;
    }
}
