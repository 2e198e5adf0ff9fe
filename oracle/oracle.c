/*
 * CPU oracle for the dense bf16 GEMM with a fused epilogue.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline / reference leg may load this library.  It
 * shares no code, header, table or helper with the CUDA path.
 *
 * What it computes.  The pages this library follows ("Automate performant
 * Hopper matmul", NVIDIA/Fuser issue #3819, sections "Persistent matmul" and
 * "Epilogue"; "Implement persistent matmul scheduling", NVIDIA/Fuser PR #3812,
 * description; "Translate MmaOp patterns properly on Hopper", NVIDIA/Fuser
 * PR #4072, review thread on the EPILOGUE_INPUT role and the commit "Fix llama
 * ffn horizontal fusion on Ampere") name the operations -- a matmul of two
 * bf16 operands, a linear layer with bias, an epilogue input added after the
 * product, and the Llama-FFN horizontal fusion -- without printing formulas.
 * This file writes out their plain definitions:
 *
 *   acc[m][n] = sum_{k=0}^{K-1} f32(A[m][k]) * f32(B[n][k])
 *               accumulated in fp32, in ascending k, one multiply and one add
 *               per term (the file is built with -ffp-contract=off, so no FMA);
 *               the product of two bf16 values is exact in fp32.
 *   linear :   v = acc;  v += f32(bias[n]) if bias;  v = act(v);
 *              v += f32(R[m][n]) if R;  D[m][n] = bf16_rne(v)
 *              optional second output (pre-activation): Z[m][n] = bf16_rne(acc + bias)
 *   ffn    :   a1 = acc(X, W1);  a3 = acc(X, W3);
 *              D[m][n] = bf16_rne( silu(a1) * a3 )
 *   dact   :   the activation-gradient product of a linear layer's backward pass
 *              (the consumer of the stored pre-activation Z):
 *              g[m][k] = sum_{n=0}^{N-1} f32(dY[m][n]) * f32(W[n][k])   (fp32, ascending n)
 *              D[m][k] = bf16_rne( g[m][k] * act'(f32(Z[m][k])) )
 *              with W the layer's [N,K] weight as the forward pass uses it.
 *
 *   act: 0 none, 1 GELU (tanh form, Hendrycks & Gimpel 2016:
 *        0.5 x (1 + tanh( sqrt(2/pi) (x + 0.044715 x^3) ))),
 *        2 SiLU (x / (1 + e^-x)), 3 ReLU (max(x, 0)).
 *   act' (derivatives, by the chain rule on the forms above):
 *        none 1;  ReLU 1 if x > 0 else 0;
 *        SiLU s (1 + x (1 - s)) with s = 1 / (1 + e^-x);
 *        GELU 0.5 (1 + t) + 0.5 x (1 - t^2) sqrt(2/pi) (1 + 3 * 0.044715 x^2)
 *             with t = tanh( sqrt(2/pi) (x + 0.044715 x^3) ).
 *
 * The *_entries functions evaluate the same definitions at a list of single
 * output entries, given each entry's operand rows gathered by the caller (row i
 * of A with row j of B; for dact row m of dY with column k of W): the checks of
 * outputs too large for the full oracle sample independent (i, j) pairs.
 *
 * Readings where the pages are silent: the activation is applied before the
 * epilogue input is added (act(acc + bias) + R); every epilogue step is fp32
 * with one rounding to bf16 at the end; bf16 rounding is round-to-nearest,
 * ties-to-even.
 *
 * The *_f64 twins evaluate the same expressions in float64 (products and sums
 * in double, epilogue in double) and return the unrounded value; they serve the
 * bf16-ULP diagnostic against the fp64 result and the error-bound pins.
 *
 * All indices are int64_t.  Rows are parallelised with OpenMP; each output
 * element is one independent sequential sum, so the thread count does not
 * change any result.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_ACT_NONE = 0, ORACLE_ACT_GELU_TANH = 1, ORACLE_ACT_SILU = 2, ORACLE_ACT_RELU = 3 };

/* ---- bf16 <-> binary32 / binary64 conversions -------------------------------- */

/* A bf16 value is the upper 16 bits of an IEEE binary32 value. */
static inline float bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

float oracle_bf16_to_f32(uint16_t h) { return bf16_to_f32(h); }

/* Round a binary32 value to bf16, nearest with ties to even. */
static inline uint16_t f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u); /* NaN stays NaN */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

uint16_t oracle_f32_to_bf16(float f) { return f32_to_bf16(f); }

/* Round a binary64 value straight to bf16 (nearest, ties to even), with no
 * intermediate rounding to binary32.  bf16 keeps 8 significant bits; below the
 * smallest normal (2^-126) the spacing is fixed at 2^-133. */
uint16_t oracle_f64_to_bf16(double x) {
    if (isnan(x)) return 0x7fc0u;
    if (x == 0.0) return signbit(x) ? 0x8000u : 0x0000u;
    if (isinf(x)) return signbit(x) ? 0xff80u : 0x7f80u;
    int e;
    (void)frexp(x, &e);               /* x = f * 2^e, 0.5 <= |f| < 1 */
    int qexp = e - 8;                  /* spacing of 8-bit significands at this binade */
    if (qexp < -133) qexp = -133;
    double r = nearbyint(ldexp(x, -qexp)); /* default rounding mode: ties to even */
    r = ldexp(r, qexp);
    if (fabs(r) >= ldexp(1.0, 128)) return signbit(x) ? 0xff80u : 0x7f80u;
    float f = (float)r;                /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* ---- activations ------------------------------------------------------------- */

static inline float act_f32(int act, float x) {
    switch (act) {
    case ORACLE_ACT_NONE: return x;
    case ORACLE_ACT_GELU_TANH: {
        const float c = 0.7978845608028654f; /* sqrt(2/pi) */
        const float a = 0.044715f;
        float inner = c * (x + a * x * x * x);
        return 0.5f * x * (1.0f + tanhf(inner));
    }
    case ORACLE_ACT_SILU: return x / (1.0f + expf(-x));
    case ORACLE_ACT_RELU: return x > 0.0f ? x : 0.0f;
    default: return NAN;
    }
}

static inline double act_f64(int act, double x) {
    switch (act) {
    case ORACLE_ACT_NONE: return x;
    case ORACLE_ACT_GELU_TANH: {
        const double c = 0.79788456080286535588; /* sqrt(2/pi) */
        const double a = 0.044715;
        return 0.5 * x * (1.0 + tanh(c * (x + a * x * x * x)));
    }
    case ORACLE_ACT_SILU: return x / (1.0 + exp(-x));
    case ORACLE_ACT_RELU: return x > 0.0 ? x : 0.0;
    default: return NAN;
    }
}

static inline float dact_f32(int act, float x) {
    switch (act) {
    case ORACLE_ACT_NONE: return 1.0f;
    case ORACLE_ACT_GELU_TANH: {
        const float c = 0.7978845608028654f; /* sqrt(2/pi) */
        const float a = 0.044715f;
        float t = tanhf(c * (x + a * x * x * x));
        return 0.5f * (1.0f + t) + 0.5f * x * (1.0f - t * t) * c * (1.0f + 3.0f * a * x * x);
    }
    case ORACLE_ACT_SILU: {
        float sg = 1.0f / (1.0f + expf(-x));
        return sg * (1.0f + x * (1.0f - sg));
    }
    case ORACLE_ACT_RELU: return x > 0.0f ? 1.0f : 0.0f;
    default: return NAN;
    }
}

static inline double dact_f64(int act, double x) {
    switch (act) {
    case ORACLE_ACT_NONE: return 1.0;
    case ORACLE_ACT_GELU_TANH: {
        const double c = 0.79788456080286535588; /* sqrt(2/pi) */
        const double a = 0.044715;
        double t = tanh(c * (x + a * x * x * x));
        return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * c * (1.0 + 3.0 * a * x * x);
    }
    case ORACLE_ACT_SILU: {
        double sg = 1.0 / (1.0 + exp(-x));
        return sg * (1.0 + x * (1.0 - sg));
    }
    case ORACLE_ACT_RELU: return x > 0.0 ? 1.0 : 0.0;
    default: return NAN;
    }
}

float oracle_act_f32(int act, float x) { return act_f32(act, x); }
double oracle_act_f64(int act, double x) { return act_f64(act, x); }

void oracle_act_f32_array(int act, const float* x, float* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = act_f32(act, x[i]);
}

void oracle_act_f64_array(int act, const double* x, double* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = act_f64(act, x[i]);
}

void oracle_dact_f32_array(int act, const float* x, float* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = dact_f32(act, x[i]);
}

void oracle_dact_f64_array(int act, const double* x, double* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = dact_f64(act, x[i]);
}

void oracle_f32_to_bf16_array(const float* x, uint16_t* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = f32_to_bf16(x[i]);
}

void oracle_f64_to_bf16_array(const double* x, uint16_t* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_f64_to_bf16(x[i]);
}

/* ---- the dot product ---------------------------------------------------------- */

static float dot_f32(const uint16_t* a, const uint16_t* b, int64_t K) {
    float acc = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
        float p = bf16_to_f32(a[k]) * bf16_to_f32(b[k]);
        acc = acc + p;
    }
    return acc;
}

/* The same sum with the second operand read at a stride (a column of a row-major matrix). */
static float dot_f32_strided(const uint16_t* a, const uint16_t* b, int64_t stride, int64_t K) {
    float acc = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
        float p = bf16_to_f32(a[k]) * bf16_to_f32(b[k * stride]);
        acc = acc + p;
    }
    return acc;
}

static double dot_f64_strided(const uint16_t* a, const uint16_t* b, int64_t stride, int64_t K) {
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double p = (double)bf16_to_f32(a[k]) * (double)bf16_to_f32(b[k * stride]);
        acc = acc + p;
    }
    return acc;
}

static double dot_f64(const uint16_t* a, const uint16_t* b, int64_t K) {
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double p = (double)bf16_to_f32(a[k]) * (double)bf16_to_f32(b[k]);
        acc = acc + p;
    }
    return acc;
}

/* Raw fp32 accumulator C[m][n] = acc[m][n] (no epilogue, no rounding to bf16). */
void oracle_acc_f32(const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                    float* C, int64_t ldc, int64_t M, int64_t N, int64_t K) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            C[m * ldc + n] = dot_f32(A + m * lda, B + n * ldb, K);
}

/* ---- linear: D = bf16( act(A.B^T + bias) + R ) -------------------------------- */

void oracle_linear_f32(const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                       const uint16_t* bias, const uint16_t* R, int64_t ldr, int act,
                       uint16_t* D, int64_t ldd, int64_t M, int64_t N, int64_t K) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            float v = dot_f32(A + m * lda, B + n * ldb, K);
            if (bias) v = v + bf16_to_f32(bias[n]);
            v = act_f32(act, v);
            if (R) v = v + bf16_to_f32(R[m * ldr + n]);
            D[m * ldd + n] = f32_to_bf16(v);
        }
    }
}

/* The same, also writing the pre-activation Z[m][n] = bf16_rne(acc + bias) (the
 * value a backward pass of the activation needs), before act and R. */
void oracle_linear_preact_f32(const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                              const uint16_t* bias, const uint16_t* R, int64_t ldr, int act,
                              uint16_t* D, int64_t ldd, uint16_t* Z, int64_t ldz,
                              int64_t M, int64_t N, int64_t K) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            float v = dot_f32(A + m * lda, B + n * ldb, K);
            if (bias) v = v + bf16_to_f32(bias[n]);
            Z[m * ldz + n] = f32_to_bf16(v);
            v = act_f32(act, v);
            if (R) v = v + bf16_to_f32(R[m * ldr + n]);
            D[m * ldd + n] = f32_to_bf16(v);
        }
    }
}

void oracle_linear_f64(const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                       const uint16_t* bias, const uint16_t* R, int64_t ldr, int act,
                       double* Y, int64_t ldy, int64_t M, int64_t N, int64_t K) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double v = dot_f64(A + m * lda, B + n * ldb, K);
            if (bias) v = v + (double)bf16_to_f32(bias[n]);
            v = act_f64(act, v);
            if (R) v = v + (double)bf16_to_f32(R[m * ldr + n]);
            Y[m * ldy + n] = v;
        }
    }
}

/* ---- Llama-FFN horizontal fusion: D = bf16( silu(X.W1^T) * (X.W3^T) ) ---------- */

void oracle_ffn_f32(const uint16_t* X, int64_t ldx, const uint16_t* W1, int64_t ldw1,
                    const uint16_t* W3, int64_t ldw3, uint16_t* D, int64_t ldd,
                    int64_t M, int64_t N, int64_t K) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            float a1 = dot_f32(X + m * ldx, W1 + n * ldw1, K);
            float a3 = dot_f32(X + m * ldx, W3 + n * ldw3, K);
            float v = act_f32(ORACLE_ACT_SILU, a1) * a3;
            D[m * ldd + n] = f32_to_bf16(v);
        }
    }
}

void oracle_ffn_f64(const uint16_t* X, int64_t ldx, const uint16_t* W1, int64_t ldw1,
                    const uint16_t* W3, int64_t ldw3, double* Y, int64_t ldy,
                    int64_t M, int64_t N, int64_t K) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double a1 = dot_f64(X + m * ldx, W1 + n * ldw1, K);
            double a3 = dot_f64(X + m * ldx, W3 + n * ldw3, K);
            Y[m * ldy + n] = act_f64(ORACLE_ACT_SILU, a1) * a3;
        }
    }
}

/* ---- activation gradient: D = bf16( (dY.W) * act'(Z) ) ---------------------------- */

/* dY [M,N], W [N,K] (the forward weight), Z [M,K]: the contraction runs over n. */
void oracle_dact_f32(const uint16_t* dY, int64_t lddy, const uint16_t* W, int64_t ldw,
                     const uint16_t* Z, int64_t ldz, int act,
                     uint16_t* D, int64_t ldd, int64_t M, int64_t N, int64_t K) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t k = 0; k < K; ++k) {
            float g = dot_f32_strided(dY + m * lddy, W + k, ldw, N);
            float v = g * dact_f32(act, bf16_to_f32(Z[m * ldz + k]));
            D[m * ldd + k] = f32_to_bf16(v);
        }
    }
}

void oracle_dact_f64(const uint16_t* dY, int64_t lddy, const uint16_t* W, int64_t ldw,
                     const uint16_t* Z, int64_t ldz, int act,
                     double* Y, int64_t ldy, int64_t M, int64_t N, int64_t K) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t k = 0; k < K; ++k) {
            double g = dot_f64_strided(dY + m * lddy, W + k, ldw, N);
            Y[m * ldy + k] = g * dact_f64(act, (double)bf16_to_f32(Z[m * ldz + k]));
        }
    }
}

/* ---- single entries: the definitions above at P listed output entries ----------------- */

/* Entry p of linear: row p of A (length K) with row p of B; bias and R are the
 * entry's own values (NULL: none).  out[p] = bf16(act(dot + bias[p]) + R[p]). */
void oracle_linear_entries_f32(const uint16_t* A, const uint16_t* B, int64_t K,
                               const uint16_t* bias, const uint16_t* R, int act,
                               uint16_t* out, int64_t P) {
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < P; ++p) {
        float v = dot_f32(A + p * K, B + p * K, K);
        if (bias) v = v + bf16_to_f32(bias[p]);
        v = act_f32(act, v);
        if (R) v = v + bf16_to_f32(R[p]);
        out[p] = f32_to_bf16(v);
    }
}

void oracle_linear_entries_f64(const uint16_t* A, const uint16_t* B, int64_t K,
                               const uint16_t* bias, const uint16_t* R, int act,
                               double* out, int64_t P) {
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < P; ++p) {
        double v = dot_f64(A + p * K, B + p * K, K);
        if (bias) v = v + (double)bf16_to_f32(bias[p]);
        v = act_f64(act, v);
        if (R) v = v + (double)bf16_to_f32(R[p]);
        out[p] = v;
    }
}

/* Entry p of the FFN fusion: row p of X with row p of W1 and row p of W3. */
void oracle_ffn_entries_f32(const uint16_t* X, const uint16_t* W1, const uint16_t* W3, int64_t K,
                            uint16_t* out, int64_t P) {
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < P; ++p) {
        float a1 = dot_f32(X + p * K, W1 + p * K, K);
        float a3 = dot_f32(X + p * K, W3 + p * K, K);
        out[p] = f32_to_bf16(act_f32(ORACLE_ACT_SILU, a1) * a3);
    }
}

void oracle_ffn_entries_f64(const uint16_t* X, const uint16_t* W1, const uint16_t* W3, int64_t K,
                            double* out, int64_t P) {
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < P; ++p) {
        double a1 = dot_f64(X + p * K, W1 + p * K, K);
        double a3 = dot_f64(X + p * K, W3 + p * K, K);
        out[p] = act_f64(ORACLE_ACT_SILU, a1) * a3;
    }
}

/* Entry p of dact: row p of dY (length N) with column p of W gathered as a row
 * (length N), and the entry's Z value. */
void oracle_dact_entries_f32(const uint16_t* dY, const uint16_t* Wcol, int64_t N,
                             const uint16_t* Z, int act, uint16_t* out, int64_t P) {
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < P; ++p) {
        float g = dot_f32(dY + p * N, Wcol + p * N, N);
        out[p] = f32_to_bf16(g * dact_f32(act, bf16_to_f32(Z[p])));
    }
}

void oracle_dact_entries_f64(const uint16_t* dY, const uint16_t* Wcol, int64_t N,
                             const uint16_t* Z, int act, double* out, int64_t P) {
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < P; ++p) {
        double g = dot_f64(dY + p * N, Wcol + p * N, N);
        out[p] = g * dact_f64(act, (double)bf16_to_f32(Z[p]));
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
