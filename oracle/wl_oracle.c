/*
 * wl_oracle.c -- plain fp64 CPU oracle for the weightless linear projection.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this file's library.  It shares no code,
 * header, table or helper with the CUDA library; the only thing both sides
 * consume is the seeded input generator (wl_synth), which holds none of the
 * method's arithmetic.
 *
 * What it computes (sources: the documentation pages of the "weightless"
 * framework):
 *   - "In-kernel reconstruction", formula section: the per-element expansion
 *       y[t,o] = s[o] * sum_i W0[o,i] x[t,i] + sum_k U[o,k] sum_i V[i,k] x[t,i]
 *   - "Serve and generate with weightless", "Set the fast path on NVIDIA":
 *       the effective weight W_eff = s * W0 + U V^T.
 *   - "What weightless inference costs", "Reconstruction fidelity":
 *       relative_frobenius_error = ||W - (diag(s) W0 + U V^T)||_F / ||W||_F.
 *   - "In-kernel reconstruction", "The GEMM path": the same output written as
 *       s[None,:] * (x @ W0.T) + (x @ V) @ U.T.
 *
 * Every floating-point quantity is converted exactly to double and the whole
 * computation runs in double with no intermediate rounding.  The result of the
 * method is, up to rounding, the plain linear map x -> x W_eff^T; the oracle
 * writes that definition out: it forms a row of W_eff, then multiplies.
 *
 * The one place that is NOT fp64 is orc_materialize_f32/_bf16: a bit-exact
 * fp32 reference with one fixed summation order (k ascending, fused
 * multiply-add, then one rounded product s*W0 and one rounded add).  The pages
 * give no order for the load-time materialisation; this file fixes it and the
 * CUDA materialize kernel must reproduce it bit for bit.  Build with
 * -ffp-contract=off so the compiler cannot fuse the product and the add.
 *
 * Layouts (row-major, PyTorch Linear convention, element names as on the
 * "In-kernel reconstruction" page):
 *   x  [T, in]   bf16 bits      W0 [out, in] bf16 bits     s [out] fp32
 *   U  [out, r]  bf16 bits      V  [in, r]   bf16 bits
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 -> double, exact: a bf16 value is the top 16 bits of an fp32. */
static double bf(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* fp32 -> bf16 bits, round to nearest, ties to even (NaN kept quiet). */
static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) /* NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

static float bf_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

void orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* W_eff[o, :] = s[o] * W0[o, :] + sum_k U[o,k] V[:, k]   (fp64, one row)     */
/* "Set the fast path on NVIDIA": W_eff = s*W0 + U V^T.                      */
/* ------------------------------------------------------------------------ */
static void weff_row(const uint16_t *W0, const float *s, const uint16_t *U,
                     const uint16_t *V, int64_t in, int64_t r, int64_t o,
                     double *row)
{
    for (int64_t i = 0; i < in; ++i) {
        double w = (double)s[o] * bf(W0[o * in + i]);
        for (int64_t k = 0; k < r; ++k)
            w += bf(U[o * r + k]) * bf(V[i * r + k]);
        row[i] = w;
    }
}

/* Full W_eff [out, in] in fp64. */
void orc_weff(const uint16_t *W0, const float *s, const uint16_t *U,
              const uint16_t *V, int64_t out, int64_t in, int64_t r,
              double *Weff)
{
#pragma omp parallel for schedule(static)
    for (int64_t o = 0; o < out; ++o)
        weff_row(W0, s, U, V, in, r, o, Weff + o * in);
}

/*
 * y = x W_eff^T in fp64, for a chosen set of tokens and outputs.
 *   tok[nt]  token indices (NULL: all T tokens, nt ignored)
 *   col[no]  output indices (NULL: all out outputs, no ignored)
 *   y        [nt, no] row-major
 * Explicit-W_eff form: for each output o build W_eff[o,:], then dot it with
 * each selected token row ("In-kernel reconstruction", formula section).
 */
void orc_linear_sel(const uint16_t *x, const uint16_t *W0, const float *s,
                    const uint16_t *U, const uint16_t *V, int64_t T,
                    int64_t in, int64_t out, int64_t r, const int64_t *tok,
                    int64_t nt, const int64_t *col, int64_t no, double *y)
{
    if (!tok) nt = T;
    if (!col) no = out;
#pragma omp parallel
    {
        double *row = (double *)malloc((size_t)(in > 0 ? in : 1) * sizeof(double));
#pragma omp for schedule(dynamic, 4)
        for (int64_t j = 0; j < no; ++j) {
            int64_t o = col ? col[j] : j;
            weff_row(W0, s, U, V, in, r, o, row);
            for (int64_t a = 0; a < nt; ++a) {
                int64_t t = tok ? tok[a] : a;
                double acc = 0.0;
                for (int64_t i = 0; i < in; ++i)
                    acc += bf(x[t * in + i]) * row[i];
                y[a * no + j] = acc;
            }
        }
        free(row);
    }
}

/* All tokens, all outputs: y [T, out]. */
void orc_linear(const uint16_t *x, const uint16_t *W0, const float *s,
                const uint16_t *U, const uint16_t *V, int64_t T, int64_t in,
                int64_t out, int64_t r, double *y)
{
    orc_linear_sel(x, W0, s, U, V, T, in, out, r, NULL, 0, NULL, 0, y);
}

/*
 * Same map, fp64 input x (used for the MLP's down projection, whose input h
 * is never rounded in the oracle).  x64 [T, in].
 */
void orc_linear_f64in(const double *x64, const uint16_t *W0, const float *s,
                      const uint16_t *U, const uint16_t *V, int64_t T,
                      int64_t in, int64_t out, int64_t r, const int64_t *col,
                      int64_t no, double *y)
{
    if (!col) no = out;
#pragma omp parallel
    {
        double *row = (double *)malloc((size_t)(in > 0 ? in : 1) * sizeof(double));
#pragma omp for schedule(dynamic, 4)
        for (int64_t j = 0; j < no; ++j) {
            int64_t o = col ? col[j] : j;
            weff_row(W0, s, U, V, in, r, o, row);
            for (int64_t t = 0; t < T; ++t) {
                double acc = 0.0;
                for (int64_t i = 0; i < in; ++i)
                    acc += x64[t * in + i] * row[i];
                y[t * no + j] = acc;
            }
        }
        free(row);
    }
}

/*
 * fp32-encoded bundles ("Serve and generate with weightless", "Supported
 * encodings and devices": the architectures also support float32): x, W0, U,
 * V and s as fp32, each converted to fp64 exactly; then the same
 * explicit-W_eff form in fp64:
 *   W_eff[o,i] = s[o] W0[o,i] + sum_k U[o,k] V[i,k],  y[t,o] = sum_i x[t,i] W_eff[o,i].
 */
void orc_linear_f32w(const float *x, const float *W0, const float *s, const float *U,
                     const float *V, int64_t T, int64_t in, int64_t out, int64_t r,
                     double *y)
{
#pragma omp parallel
    {
        double *row = (double *)malloc((size_t)(in > 0 ? in : 1) * sizeof(double));
#pragma omp for schedule(dynamic, 4)
        for (int64_t o = 0; o < out; ++o) {
            for (int64_t i = 0; i < in; ++i) {
                double w = (double)s[o] * (double)W0[o * in + i];
                for (int64_t k = 0; k < r; ++k)
                    w += (double)U[o * r + k] * (double)V[i * r + k];
                row[i] = w;
            }
            for (int64_t t = 0; t < T; ++t) {
                double acc = 0.0;
                for (int64_t i = 0; i < in; ++i)
                    acc += (double)x[t * in + i] * row[i];
                y[t * out + o] = acc;
            }
        }
        free(row);
    }
}

/*
 * Factored form, used only to pin the explicit form against a second,
 * independent evaluation ("In-kernel reconstruction", "The GEMM path"):
 *   y = s[None,:] * (x @ W0.T) + (x @ V) @ U.T
 * Computed as written: P = x W0^T, z = x V, then the combine.
 */
void orc_linear_factored(const uint16_t *x, const uint16_t *W0, const float *s,
                         const uint16_t *U, const uint16_t *V, int64_t T,
                         int64_t in, int64_t out, int64_t r, double *y)
{
    double *z = (double *)calloc((size_t)(T * r > 0 ? T * r : 1), sizeof(double));
    for (int64_t t = 0; t < T; ++t)
        for (int64_t k = 0; k < r; ++k) {
            double a = 0.0;
            for (int64_t i = 0; i < in; ++i)
                a += bf(x[t * in + i]) * bf(V[i * r + k]);
            z[t * r + k] = a;
        }
#pragma omp parallel for schedule(static)
    for (int64_t o = 0; o < out; ++o)
        for (int64_t t = 0; t < T; ++t) {
            double p = 0.0;
            for (int64_t i = 0; i < in; ++i)
                p += bf(x[t * in + i]) * bf(W0[o * in + i]);
            double d = 0.0;
            for (int64_t k = 0; k < r; ++k)
                d += z[t * r + k] * bf(U[o * r + k]);
            y[t * out + o] = (double)s[o] * p + d;
        }
    free(z);
}

/*
 * tanh-form GELU in fp64:
 *   gelu(v) = 0.5 v (1 + tanh( sqrt(2/pi) (v + 0.044715 v^3) ))
 * The fused MLP ("In-kernel reconstruction", custom-op path: gate, up,
 * activation, down in one dispatch) applies it to the gate projection.
 */
double orc_gelu_tanh(double v)
{
    const double c = sqrt(2.0 / 3.14159265358979323846);
    return 0.5 * v * (1.0 + tanh(c * (v + 0.044715 * v * v * v)));
}

/*
 * GeGLU MLP of the weightless layer, fp64 throughout:
 *   g = x W_eff_gate^T,  u = x W_eff_up^T   [T, inter]
 *   h = gelu_tanh(g) * u                    [T, inter]  (never rounded)
 *   y = h W_eff_down^T                      [T, hidden]
 * tok[nt] selects tokens (NULL: all), col[no] selects outputs of y (NULL: all).
 * h_out (optional, [nt, inter]) receives h.
 */
void orc_mlp_geglu(const uint16_t *x,
                   const uint16_t *Wg, const float *sg, const uint16_t *Ug, const uint16_t *Vg,
                   const uint16_t *Wu, const float *su, const uint16_t *Uu, const uint16_t *Vu,
                   const uint16_t *Wd, const float *sd, const uint16_t *Ud, const uint16_t *Vd,
                   int64_t T, int64_t hidden, int64_t inter, int64_t r,
                   const int64_t *tok, int64_t nt, const int64_t *col, int64_t no,
                   double *y, double *h_out)
{
    if (!tok) nt = T;
    size_t nh = (size_t)(nt * inter > 0 ? nt * inter : 1);
    double *g = (double *)malloc(nh * sizeof(double));
    double *u = (double *)malloc(nh * sizeof(double));
    double *h = (double *)malloc(nh * sizeof(double));
    orc_linear_sel(x, Wg, sg, Ug, Vg, T, hidden, inter, r, tok, nt, NULL, 0, g);
    orc_linear_sel(x, Wu, su, Uu, Vu, T, hidden, inter, r, tok, nt, NULL, 0, u);
    for (int64_t a = 0; a < nt * inter; ++a)
        h[a] = orc_gelu_tanh(g[a]) * u[a];
    if (h_out) memcpy(h_out, h, (size_t)(nt * inter) * sizeof(double));
    orc_linear_f64in(h, Wd, sd, Ud, Vd, nt, inter, hidden, r, col, no, y);
    free(g);
    free(u);
    free(h);
}

/*
 * Bit-exact fp32 materialisation with one fixed order (the pages leave the
 * order open; this is the one the library commits to):
 *   d = +0.0f; for k = 0 .. r-1: d = fmaf(U[o,k], V[i,k], d)
 *   w = s[o] * W0[o,i]               (one fp32 multiply, round to nearest)
 *   if r > 0: w = w + d              (one fp32 add, round to nearest)
 * W_eff [out, in] fp32.
 */
void orc_materialize_f32(const uint16_t *W0, const float *s, const uint16_t *U,
                         const uint16_t *V, int64_t out, int64_t in, int64_t r,
                         float *Weff)
{
#pragma omp parallel for schedule(static)
    for (int64_t o = 0; o < out; ++o)
        for (int64_t i = 0; i < in; ++i) {
            float d = 0.0f;
            for (int64_t k = 0; k < r; ++k)
                d = fmaf(bf_f32(U[o * r + k]), bf_f32(V[i * r + k]), d);
            float w = s[o] * bf_f32(W0[o * in + i]);
            if (r > 0) w = w + d;
            Weff[o * in + i] = w;
        }
}

/* Same value, then rounded to bf16 (nearest, ties to even). */
void orc_materialize_bf16(const uint16_t *W0, const float *s, const uint16_t *U,
                          const uint16_t *V, int64_t out, int64_t in, int64_t r,
                          uint16_t *Weff)
{
#pragma omp parallel for schedule(static)
    for (int64_t o = 0; o < out; ++o)
        for (int64_t i = 0; i < in; ++i) {
            float d = 0.0f;
            for (int64_t k = 0; k < r; ++k)
                d = fmaf(bf_f32(U[o * r + k]), bf_f32(V[i * r + k]), d);
            float w = s[o] * bf_f32(W0[o * in + i]);
            if (r > 0) w = w + d;
            Weff[o * in + i] = f32_to_bf16_rne(w);
        }
}

/* Plain fp32 -> bf16 rounding, exposed so tests can pin it on its own. */
void orc_f32_to_bf16(const float *a, int64_t n, uint16_t *b)
{
    for (int64_t j = 0; j < n; ++j) b[j] = f32_to_bf16_rne(a[j]);
}

/*
 * fp64 -> bf16 bits, one correct rounding (nearest, ties to even).  The
 * method ends with a cast of the fp32 combine to the output dtype
 * ("In-kernel reconstruction", custom-op path and "The GEMM path"); for a
 * bf16 output the reference value is the exact result after that cast.
 * Rounds the 53-bit significand to 8 bits on the bit pattern; the kept value
 * is then exact in fp32.  Normal range only (tiny values below 2^-126 are
 * outside what this library produces); zero and sign are kept.
 */
void orc_f64_to_bf16(const double *a, int64_t n, uint16_t *b)
{
    for (int64_t j = 0; j < n; ++j) {
        uint64_t u;
        memcpy(&u, &a[j], sizeof u);
        if ((u & 0x7fffffffffffffffull) > 0x7ff0000000000000ull) { /* NaN */
            b[j] = 0x7fc0u;
            continue;
        }
        const uint64_t lsb = (u >> 45) & 1ull;
        u += (1ull << 44) - 1ull + lsb;
        u &= ~((1ull << 45) - 1ull);
        double d;
        memcpy(&d, &u, sizeof d);
        float f = (float)d; /* exact: at most 8 significant bits */
        uint32_t fb;
        memcpy(&fb, &f, sizeof fb);
        b[j] = (uint16_t)(fb >> 16);
    }
}

/*
 * relative_frobenius_error ("What weightless inference costs",
 * "Reconstruction fidelity"):
 *   ||W - (diag(s) W0 + U V^T)||_F / ||W||_F,  W [out, in] given in fp64.
 */
double orc_rel_frobenius(const double *W, const uint16_t *W0, const float *s,
                         const uint16_t *U, const uint16_t *V, int64_t out,
                         int64_t in, int64_t r)
{
    double num = 0.0, den = 0.0;
    double *row = (double *)malloc((size_t)(in > 0 ? in : 1) * sizeof(double));
    for (int64_t o = 0; o < out; ++o) {
        weff_row(W0, s, U, V, in, r, o, row);
        for (int64_t i = 0; i < in; ++i) {
            double e = W[o * in + i] - row[i];
            num += e * e;
            den += W[o * in + i] * W[o * in + i];
        }
    }
    free(row);
    return sqrt(num) / sqrt(den);
}

/*
 * Band selection: G shared W0 blocks per projection family over L layers,
 * contiguous bands, layer l uses block floor(l * G / L).  G = L gives one W0
 * per layer (passthrough, "Set the fast path on NVIDIA"); G = 1 shares one
 * block across the stack ("What weightless inference costs", Compression).
 * Returns -1 for arguments outside 0 <= l < L, 1 <= G <= L.
 */
int64_t orc_band_of_layer(int64_t l, int64_t L, int64_t G)
{
    if (L < 1 || G < 1 || G > L || l < 0 || l >= L) return -1;
    return (l * G) / L;
}
