// decompose.cu -- dense projection weights -> theta bundles, one band of
// layers of one projection family per call.
//
// The pages give the decomposition by its results: the weight adapter
// auto-decomposes a checkpoint into the bundle ("Serve and generate with
// weightless", "How the custom architecture loads"); the bundle is a W0 per
// band, a per-row scale s and a rank-r delta U V^T (overview); at the
// passthrough point G = num_layers the reconstruction equals the original
// ("Set the fast path on NVIDIA").  The steps computed here:
//   1. W0 = mean of the band's weights (fp32 sum in layer order), stored bf16;
//   2. per layer, s[o] = <W[o], W0[o]> / <W0[o], W0[o]> against the stored
//      W0 (1 where the W0 row is zero), fp32;
//   3. per layer, U and V from the rank-r truncated SVD of the residual
//      R = W - diag(s) W0, split evenly (U = U_r S^1/2, V = V_r S^1/2), bf16.
// Step 3 is randomized subspace iteration (Halko, Martinsson and Tropp,
// "Finding structure with randomness", 2011): Y = R Omega for a caller-drawn
// Gaussian Omega with k = r + p columns, q rounds of Y <- R (R^T Y) with
// re-orthonormalisation (shifted CholeskyQR2), then Rayleigh-Ritz: B = Q^T R,
// the eigenpairs of B B^T (parallel cyclic Jacobi in one CTA), U = Q E_r
// L^1/4, V = B^T E_r L^-1/4.  R is never stored: every pass over it re-forms
// it from W, W0 and s.  At G = L: W0 = W, s = 1, R = 0 and U = V = 0.
#include <algorithm>
#include <cmath>

#include "wl_internal.cuh"

namespace wl {

struct DcLayers {
    const bf16 *W[kDecompMaxLayers];
};

// ---- 1. band mean -------------------------------------------------------
__global__ void dc_mean_kernel(const __grid_constant__ DcLayers L, int n, int64_t total8, bf16 *W0)
{
    const float inv = 1.0f / (float)n;
    for (int64_t c = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; c < total8; c += (int64_t)gridDim.x * blockDim.x) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int l = 0; l < n; ++l) {
            const uint4 v = reinterpret_cast<const uint4 *>(L.W[l])[c];
            acc[0] += bf_lo(v.x); acc[1] += bf_hi(v.x); acc[2] += bf_lo(v.y); acc[3] += bf_hi(v.y);
            acc[4] += bf_lo(v.z); acc[5] += bf_hi(v.z); acc[6] += bf_lo(v.w); acc[7] += bf_hi(v.w);
        }
        uint32_t p[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[2 * b] * inv, acc[2 * b + 1] * inv);
            p[b] = *reinterpret_cast<const uint32_t *>(&h2);
        }
        reinterpret_cast<uint4 *>(W0)[c] = make_uint4(p[0], p[1], p[2], p[3]);
    }
}

// ---- 2. least-squares row scale (one warp per row) ----------------------
__global__ void dc_scale_kernel(const bf16 *__restrict__ W, const bf16 *__restrict__ W0, int out, int in, float *s)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= out) return;
    const uint4 *w = reinterpret_cast<const uint4 *>(W + (int64_t)warp * in);
    const uint4 *w0 = reinterpret_cast<const uint4 *>(W0 + (int64_t)warp * in);
    float num = 0.f, den = 0.f;
    for (int c = lane; c < in / 8; c += 32) {
        const uint4 a = w[c], b = w0[c];
        const float av[8] = {bf_lo(a.x), bf_hi(a.x), bf_lo(a.y), bf_hi(a.y), bf_lo(a.z), bf_hi(a.z), bf_lo(a.w), bf_hi(a.w)};
        const float bv[8] = {bf_lo(b.x), bf_hi(b.x), bf_lo(b.y), bf_hi(b.y), bf_lo(b.z), bf_hi(b.z), bf_lo(b.w), bf_hi(b.w)};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            num = fmaf(av[e], bv[e], num);
            den = fmaf(bv[e], bv[e], den);
        }
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        num += __shfl_xor_sync(0xffffffffu, num, m);
        den += __shfl_xor_sync(0xffffffffu, den, m);
    }
    if (lane == 0) s[warp] = den > 0.f ? num / den : 1.0f;
}

// ---- products with the implicit residual --------------------------------
// TR = 0:  C[m, j] = sum_t R[m, t] B[t, j]   (Y = R X;   m < out, t < in)
// TR = 1:  C[m, j] = sum_t R[t, m] B[t, j]   (Z = R^T Y; m < in,  t < out)
// with R[o, i] = W[o, i] - s[o] W0[o, i].  B [nt, k] and C [nm, k] fp32
// row-major.  CTA: 32 values of m x all k columns, 16 x 16 threads (2 m x
// KT columns each), the contraction in chunks of 32.  The contraction is
// split over blockIdx.y (tsplit rows of t each): split q writes its partial
// sums to C + q nm k, summed afterwards in split order (dc_sum_splits), so
// that the result does not depend on timing.
template <int TR, int KT>
__global__ void __launch_bounds__(256) dc_rmul_kernel(const bf16 *__restrict__ W, const bf16 *__restrict__ W0,
                                                      const float *__restrict__ s, const float *__restrict__ B,
                                                      float *__restrict__ C, int out, int in, int k, int tsplit)
{
    constexpr int BM = 32, BK = 32, KP = 16 * KT;
    __shared__ __align__(16) float As[BK][BM + 1];
    __shared__ __align__(16) float Bs[BK][KP + 4];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int nm = TR ? in : out;
    const int m0 = blockIdx.x * BM;
    const int tb = blockIdx.y * tsplit;
    const int nt = min(TR ? out : in, tb + tsplit);
    C += (size_t)blockIdx.y * nm * k;
    float acc[2][KT];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < KT; ++b) acc[a][b] = 0.f;
    for (int t0 = tb; t0 < nt; t0 += BK) {
        for (int e = tid; e < BM * BK; e += 256) {
            int m, t;
            if (TR) {  // rows o = t of R, consecutive threads along i = m
                t = e / BM;
                m = e - t * BM;
            } else {  // rows o = m of R, consecutive threads along i = t
                m = e / BK;
                t = e - m * BK;
            }
            const int gm = m0 + m, gt = t0 + t;
            float v = 0.f;
            if (gm < nm && gt < nt) {
                const int o = TR ? gt : gm, i = TR ? gm : gt;
                const int64_t idx = (int64_t)o * in + i;
                v = bf2f(W[idx]) - s[o] * bf2f(W0[idx]);
            }
            As[t][m] = v;
        }
        for (int e = tid; e < BK * KP; e += 256) {
            const int t = e / KP, j = e - t * KP;
            Bs[t][j] = (t0 + t < nt && j < k) ? B[(int64_t)(t0 + t) * k + j] : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int t = 0; t < BK; ++t) {
            const float a0 = As[t][ty * 2], a1 = As[t][ty * 2 + 1];
#pragma unroll
            for (int b = 0; b < KT; ++b) {
                const float bv = Bs[t][tx + 16 * b];
                acc[0][b] = fmaf(a0, bv, acc[0][b]);
                acc[1][b] = fmaf(a1, bv, acc[1][b]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < 2; ++a) {
        const int m = m0 + ty * 2 + a;
        if (m >= nm) continue;
#pragma unroll
        for (int b = 0; b < KT; ++b) {
            const int j = tx + 16 * b;
            if (j < k) C[(int64_t)m * k + j] = acc[a][b];
        }
    }
}

// C[e] = sum over q < nsplit of P[q n + e], in q order
__global__ void dc_sum_splits_kernel(const float *__restrict__ P, int nsplit, int64_t n, float *__restrict__ C)
{
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
        float v = 0.f;
        for (int q = 0; q < nsplit; ++q) v += P[(size_t)q * n + e];
        C[e] = v;
    }
}

// ---- Gram matrices Y^T Y (k x k) of a tall Y [n, k] -----------------------
// partial Gram of rows [blockIdx.x * rows, ...) per CTA, then a fixed-order sum
// (rows staged through shared memory 32 at a time, read coalesced; a
// thread's entries summed over the rows in order)
constexpr int kGramChunk = 32;
constexpr int kGramRows = 64;  // rows of Y per CTA (partial Gram matrices: n / 64 of them)
template <int EPT>  // entries per thread: k * k <= 256 * EPT
__global__ void __launch_bounds__(256) dc_gram_partial_kernel(const float *__restrict__ Y, int n, int k, int rows,
                                                              float *__restrict__ part)
{
    extern __shared__ float ys[];  // [kGramChunk][k]
    const int r0 = blockIdx.x * rows, r1 = min(n, r0 + rows);
    float *P = part + (size_t)blockIdx.x * k * k;
    float v[EPT];
    const int ne = k * k;
#pragma unroll
    for (int j = 0; j < EPT; ++j) v[j] = 0.f;
    for (int c0 = r0; c0 < r1; c0 += kGramChunk) {
        const int nr = min(kGramChunk, r1 - c0);
        __syncthreads();
        for (int e = threadIdx.x; e < nr * k; e += blockDim.x) ys[e] = Y[(int64_t)c0 * k + e];
        __syncthreads();
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
            const int e = threadIdx.x + j * 256;
            if (e < ne) {
                const int a = e / k, b = e - a * k;
                if (b >= a) {
                    float acc = v[j];
                    for (int i = 0; i < nr; ++i) acc = fmaf(ys[i * k + a], ys[i * k + b], acc);
                    v[j] = acc;
                }
            }
        }
    }
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
        const int e = threadIdx.x + j * 256;
        if (e < ne) P[e] = v[j];
    }
}

__global__ void dc_gram_reduce_kernel(const float *__restrict__ part, int nparts, int k, float *__restrict__ Gm)
{
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < k * k; e += gridDim.x * blockDim.x) {
        const int a = e / k, b = e - a * k;
        const int src = b >= a ? e : b * k + a;  // upper triangle mirrored
        float v = 0.f;
        for (int p = 0; p < nparts; ++p) v += part[(size_t)p * k * k + src];
        Gm[e] = v;
    }
}

// ---- small dense problems in one CTA ------------------------------------
// mode 0 (orthonormalisation): M = L^-T for G + shift I = L L^T (shifted
// Cholesky; the shift keeps it positive definite when Y is rank-deficient);
// M = 0 when G = 0 (Y = 0).
// mode 1 (Rayleigh-Ritz): eigenpairs of G = B B^T by parallel cyclic Jacobi;
// MU = E_r diag(l^1/4), MV = E_r diag(l^-1/4) for the r largest eigenvalues
// (a column is zero where l is not above a relative floor).
__global__ void __launch_bounds__(1024) dc_small_kernel(const float *__restrict__ Gin, int k, int r, int mode,
                                                        float *__restrict__ M, float *__restrict__ MU,
                                                        float *__restrict__ MV, unsigned *status)
{
    extern __shared__ float sm[];
    const int kk = (k + 1) & ~1;  // even size for the Jacobi pairing (padding row/column of zeros)
    float *A = sm;                // [kk][kk]
    float *E = A + kk * kk;       // [kk][kk] eigenvectors (columns) / L^-1
    float *aux = E + kk * kk;     // [kk * 4]
    const int tid = threadIdx.x, nth = blockDim.x;
    for (int e = tid; e < kk * kk; e += nth) {
        const int a = e / kk, b = e - a * kk;
        A[e] = (a < k && b < k) ? Gin[a * k + b] : 0.f;
        E[e] = a == b ? 1.f : 0.f;
    }
    __syncthreads();
    if (mode == 0) {
        // shifted Cholesky, column by column (rows below the pivot in parallel)
        __shared__ float tr;
        if (tid == 0) {
            float t = 0.f;
            for (int a = 0; a < k; ++a) t += A[a * kk + a];
            tr = t;
        }
        __syncthreads();
        const float shift = 1e-6f * tr / (float)k;
        if (tr <= 0.f) {
            for (int e = tid; e < k * k; e += nth) M[e] = 0.f;
            return;
        }
        for (int a = tid; a < k; a += nth) A[a * kk + a] += shift;
        __syncthreads();
        for (int c = 0; c < k; ++c) {
            if (tid == 0) A[c * kk + c] = sqrtf(fmaxf(A[c * kk + c], 1e-30f));
            __syncthreads();
            const float d = A[c * kk + c];
            for (int a = c + 1 + tid; a < k; a += nth) A[a * kk + c] /= d;
            __syncthreads();
            // trailing update A[a][b] -= L[a][c] L[b][c] for c < b <= a
            for (int e = tid; e < (k - c - 1) * (k - c - 1); e += nth) {
                const int a = c + 1 + e / (k - c - 1), b = c + 1 + e % (k - c - 1);
                if (b <= a) A[a * kk + b] -= A[a * kk + c] * A[b * kk + c];
            }
            __syncthreads();
        }
        // L^-1 by forward substitution, one column of the inverse per thread
        for (int j = tid; j < k; j += nth) {
            for (int a = 0; a < k; ++a) {
                float v = a == j ? 1.f : 0.f;
                for (int b = j; b < a; ++b) v -= A[a * kk + b] * E[b * kk + j];
                E[a * kk + j] = a >= j ? v / A[a * kk + a] : 0.f;
            }
        }
        __syncthreads();
        // M = (L^-1)^T
        for (int e = tid; e < k * k; e += nth) {
            const int a = e / k, b = e - a * k;
            M[e] = E[b * kk + a];
        }
        return;
    }
    // parallel cyclic Jacobi: kk/2 disjoint pairs per step (round-robin), kk-1 steps per sweep
    float *cs = aux;                 // [kk/2] cos
    float *sn = aux + kk / 2;        // [kk/2] sin
    int *pp = reinterpret_cast<int *>(aux + kk);          // [kk/2]
    int *qq = reinterpret_cast<int *>(aux + kk + kk / 2);  // [kk/2]
    __shared__ float off, diag;
    const int npair = kk / 2;
    for (int sweep = 0; sweep < 30; ++sweep) {
        if (tid == 0) {
            float o = 0.f, d = 0.f;
            for (int a = 0; a < kk; ++a)
                for (int b = 0; b < kk; ++b) {
                    const float v = A[a * kk + b] * A[a * kk + b];
                    if (a == b) d += v;
                    else o += v;
                }
            off = o;
            diag = d;
        }
        __syncthreads();
        if (off <= 1e-14f * diag || diag == 0.f) break;
        for (int step = 0; step < kk - 1; ++step) {
            // pairing: position 0 fixed, the others rotate
            for (int i = tid; i < npair; i += nth) {
                auto at = [&](int pos) { return pos == 0 ? 0 : 1 + (pos - 1 + step) % (kk - 1); };
                int p = at(i), q = at(kk - 1 - i);
                if (p > q) { const int t = p; p = q; q = t; }
                pp[i] = p;
                qq[i] = q;
                const float app = A[p * kk + p], aqq = A[q * kk + q], apq = A[p * kk + q];
                float c = 1.f, sv = 0.f;
                if (fabsf(apq) > 1e-30f) {
                    const float th = (aqq - app) / (2.f * apq);
                    const float t = (th >= 0.f ? 1.f : -1.f) / (fabsf(th) + sqrtf(1.f + th * th));
                    c = rsqrtf(1.f + t * t);
                    sv = t * c;
                }
                cs[i] = c;
                sn[i] = sv;
            }
            __syncthreads();
            // rows p, q of A
            for (int e = tid; e < npair * kk; e += nth) {
                const int i = e / kk, b = e - i * kk;
                const int p = pp[i], q = qq[i];
                const float c = cs[i], sv = sn[i];
                const float x = A[p * kk + b], y = A[q * kk + b];
                A[p * kk + b] = c * x - sv * y;
                A[q * kk + b] = sv * x + c * y;
            }
            __syncthreads();
            // columns p, q of A and of E
            for (int e = tid; e < npair * kk; e += nth) {
                const int i = e / kk, a = e - i * kk;
                const int p = pp[i], q = qq[i];
                const float c = cs[i], sv = sn[i];
                float x = A[a * kk + p], y = A[a * kk + q];
                A[a * kk + p] = c * x - sv * y;
                A[a * kk + q] = sv * x + c * y;
                x = E[a * kk + p];
                y = E[a * kk + q];
                E[a * kk + p] = c * x - sv * y;
                E[a * kk + q] = sv * x + c * y;
            }
            __syncthreads();
        }
    }
    // the r largest eigenvalues (selection by rank: ties broken by index)
    float *lam = aux;  // reuse [kk]
    int *order = reinterpret_cast<int *>(aux + kk);
    for (int a = tid; a < kk; a += nth) lam[a] = a < k ? fmaxf(A[a * kk + a], 0.f) : -1.f;
    __syncthreads();
    for (int a = tid; a < kk; a += nth) {
        int rank = 0;
        for (int b = 0; b < kk; ++b)
            if (lam[b] > lam[a] || (lam[b] == lam[a] && b < a)) ++rank;
        order[rank] = a;
    }
    __syncthreads();
    const float lmax = lam[order[0]];
    for (int e = tid; e < k * r; e += nth) {
        const int a = e / r, j = e - a * r;  // row a of E, output column j
        const int col = order[j];
        const float l = lam[col];
        const bool keep = l > 1e-10f * lmax && l > 0.f;
        const float q4 = keep ? sqrtf(sqrtf(l)) : 0.f;
        MU[e] = keep ? E[a * kk + col] * q4 : 0.f;
        MV[e] = keep ? E[a * kk + col] / q4 : 0.f;
    }
    (void)status;
}

// ---- C [n, kc] = A [n, k] M [k, kc]; fp32 out (ob == 0) or bf16 out ------
__global__ void __launch_bounds__(256) dc_apply_kernel(const float *__restrict__ A, int n, int k,
                                                       const float *__restrict__ M, int kc, void *out, int ob)
{
    extern __shared__ float Ms[];  // [k][kc]
    for (int e = threadIdx.x; e < k * kc; e += blockDim.x) Ms[e] = M[e];
    __syncthreads();
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < (int64_t)n * kc;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = e / kc;
        const int j = (int)(e - row * kc);
        float v = 0.f;
        for (int t = 0; t < k; ++t) v = fmaf(A[row * k + t], Ms[t * kc + j], v);
        if (ob) static_cast<bf16 *>(out)[e] = __float2bfloat16_rn(v);
        else static_cast<float *>(out)[e] = v;
    }
}

// ------------------------------------------------------------------ host
struct DcWs {
    float *Y, *Y2, *Z, *Z2, *part, *G, *M, *MU, *MV, *split;
    int nparts;
    int64_t split_floats;
};

// Partial sums of the split contraction: up to 16 splits, at most 8 Mi floats.
static int64_t dc_split_floats(int64_t out, int64_t in, int64_t k)
{
    return std::min<int64_t>(16 * std::max(out, in) * k, (int64_t)1 << 23);
}

static size_t dc_carve(int64_t out, int64_t in, int64_t k, int64_t r, char *base, DcWs *w)
{
    size_t off = 0;
    auto take = [&](size_t bytes) {
        off = (off + 255) / 256 * 256;
        const size_t o = off;
        off += bytes;
        return o;
    };
    const int nparts = (int)((std::max(out, in) + kGramRows - 1) / kGramRows);
    const size_t oY = take(4 * out * k), oY2 = take(4 * out * k), oZ = take(4 * in * k), oZ2 = take(4 * in * k);
    const size_t oP = take(4 * (size_t)nparts * k * k), oG = take(4 * k * k), oM = take(4 * k * k);
    const size_t oMU = take(4 * k * r), oMV = take(4 * k * r);
    const int64_t nsplit_f = dc_split_floats(out, in, k);
    const size_t oS = take(4 * (size_t)nsplit_f);
    if (base) {
        w->split = reinterpret_cast<float *>(base + oS);
        w->split_floats = nsplit_f;
        w->Y = reinterpret_cast<float *>(base + oY);
        w->Y2 = reinterpret_cast<float *>(base + oY2);
        w->Z = reinterpret_cast<float *>(base + oZ);
        w->Z2 = reinterpret_cast<float *>(base + oZ2);
        w->part = reinterpret_cast<float *>(base + oP);
        w->G = reinterpret_cast<float *>(base + oG);
        w->M = reinterpret_cast<float *>(base + oM);
        w->MU = reinterpret_cast<float *>(base + oMU);
        w->MV = reinterpret_cast<float *>(base + oMV);
        w->nparts = nparts;
    }
    return take(0);
}

size_t decompose_workspace_bytes(int64_t out, int64_t in, int64_t r, int64_t p)
{
    return dc_carve(out, in, r + p, r, nullptr, nullptr);
}

static int kt_of(int k) { return k <= 16 ? 1 : k <= 32 ? 2 : k <= 64 ? 4 : k <= 96 ? 6 : k <= 128 ? 8 : 10; }

// The contraction is split so that the grid holds about four CTAs per SM
// (the m strips alone are too few where m runs over the shorter side), each
// split a multiple of 32 rows of t, within the workspace's partial buffer.
template <int TR>
static void rmul(const bf16 *W, const bf16 *W0, const float *s, const float *B, float *C, int out, int in, int k,
                 const DcWs &w, const DeviceInfo *di, cudaStream_t st)
{
    const int nm = TR ? in : out, nt = TR ? out : in;
    const int mt = (nm + 31) / 32;
    int nsplit = std::max(1, (4 * di->sm_count + mt - 1) / mt);
    nsplit = std::min(nsplit, (nt + 31) / 32);
    nsplit = (int)std::min<int64_t>(nsplit, std::max<int64_t>(1, w.split_floats / ((int64_t)nm * k)));
    int tsplit = (nt + nsplit - 1) / nsplit;
    tsplit = (tsplit + 31) / 32 * 32;
    nsplit = (nt + tsplit - 1) / tsplit;
    float *dst = nsplit > 1 ? w.split : C;
    const dim3 grid((unsigned)mt, (unsigned)nsplit);
    switch (kt_of(k)) {
    case 1: dc_rmul_kernel<TR, 1><<<grid, 256, 0, st>>>(W, W0, s, B, dst, out, in, k, tsplit); break;
    case 2: dc_rmul_kernel<TR, 2><<<grid, 256, 0, st>>>(W, W0, s, B, dst, out, in, k, tsplit); break;
    case 4: dc_rmul_kernel<TR, 4><<<grid, 256, 0, st>>>(W, W0, s, B, dst, out, in, k, tsplit); break;
    case 6: dc_rmul_kernel<TR, 6><<<grid, 256, 0, st>>>(W, W0, s, B, dst, out, in, k, tsplit); break;
    case 8: dc_rmul_kernel<TR, 8><<<grid, 256, 0, st>>>(W, W0, s, B, dst, out, in, k, tsplit); break;
    default: dc_rmul_kernel<TR, 10><<<grid, 256, 0, st>>>(W, W0, s, B, dst, out, in, k, tsplit); break;
    }
    if (nsplit > 1) {
        const int64_t n = (int64_t)nm * k;
        dc_sum_splits_kernel<<<(unsigned)std::min<int64_t>((n + 255) / 256, 4 * di->sm_count), 256, 0, st>>>(
            w.split, nsplit, n, C);
    }
}

static void gram(const float *Y, int n, int k, const DcWs &w, cudaStream_t st)
{
    const int rows = kGramRows;
    const int parts = (n + rows - 1) / rows;
    const size_t sm = (size_t)kGramChunk * k * 4;
    if (k * k <= 256 * 4)
        dc_gram_partial_kernel<4><<<parts, 256, sm, st>>>(Y, n, k, rows, w.part);
    else if (k * k <= 256 * 16)
        dc_gram_partial_kernel<16><<<parts, 256, sm, st>>>(Y, n, k, rows, w.part);
    else
        dc_gram_partial_kernel<100><<<parts, 256, sm, st>>>(Y, n, k, rows, w.part);
    dc_gram_reduce_kernel<<<(k * k + 255) / 256, 256, 0, st>>>(w.part, parts, k, w.G);
}

static int small_smem(int k) { const int kk = (k + 1) & ~1; return (2 * kk * kk + 4 * kk) * 4; }

// Y [n, k] -> an orthonormal basis of its columns (shifted CholeskyQR, twice),
// result in *Y (tmp: a buffer of the same size)
static void orth(float **Y, float **tmp, int n, int k, const DcWs &w, const DeviceInfo *di, cudaStream_t st)
{
    for (int pass = 0; pass < 2; ++pass) {
        gram(*Y, n, k, w, st);
        dc_small_kernel<<<1, 1024, small_smem(k), st>>>(w.G, k, 0, 0, w.M, w.MU, w.MV, di->status);
        const int64_t tot = (int64_t)n * k;
        dc_apply_kernel<<<(unsigned)std::min<int64_t>((tot + 255) / 256, 4096), 256, k * k * 4, st>>>(*Y, n, k, w.M, k,
                                                                                                    *tmp, 0);
        float *t = *Y;
        *Y = *tmp;
        *tmp = t;
    }
}

wl_status launch_decompose(const bf16 *const *Wl, int n, int out, int in, int r, int p, int iters, const float *omega,
                           bf16 *W0, float *s, bf16 *U, bf16 *V, void *ws, size_t ws_bytes, cudaStream_t st)
{
    wl_status stt = WL_OK;
    const DeviceInfo *di = device_info(&stt);
    if (!di) return stt;
    const int k = r + p;
    DcWs w;
    if (decompose_workspace_bytes(out, in, r, p) > ws_bytes)
        return fail(WL_ERR_WORKSPACE, "wl_decompose_band: workspace too small");
    dc_carve(out, in, k, r, static_cast<char *>(ws), &w);
    // dynamic shared memory of the largest sizes (k = kDecompMaxK)
    cudaError_t ea = cudaFuncSetAttribute(dc_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          small_smem(kDecompMaxK));
    if (ea == cudaSuccess)
        ea = cudaFuncSetAttribute(dc_apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kDecompMaxK * kDecompMaxK * 4);
    if (ea != cudaSuccess) return cuda_fail(ea, "wl_decompose_band: cudaFuncSetAttribute");
    DcLayers L = {};
    for (int l = 0; l < n; ++l) L.W[l] = Wl[l];
    const int64_t total8 = (int64_t)out * in / 8;
    dc_mean_kernel<<<(unsigned)std::min<int64_t>((total8 + 255) / 256, 8 * di->sm_count), 256, 0, st>>>(L, n, total8, W0);
    for (int l = 0; l < n; ++l) {
        float *sl = s + (int64_t)l * out;
        dc_scale_kernel<<<(out + 7) / 8, 256, 0, st>>>(Wl[l], W0, out, in, sl);
        if (r == 0) continue;
        float *Y = w.Y, *Y2 = w.Y2, *Z = w.Z, *Z2 = w.Z2;
        rmul<0>(Wl[l], W0, sl, omega, Y, out, in, k, w, di, st);  // Y = R Omega
        orth(&Y, &Y2, out, k, w, di, st);
        for (int it = 0; it < iters; ++it) {
            rmul<1>(Wl[l], W0, sl, Y, Z, out, in, k, w, di, st);  // Z = R^T Q
            orth(&Z, &Z2, in, k, w, di, st);
            rmul<0>(Wl[l], W0, sl, Z, Y, out, in, k, w, di, st);  // Y = R Z
            orth(&Y, &Y2, out, k, w, di, st);
        }
        rmul<1>(Wl[l], W0, sl, Y, Z, out, in, k, w, di, st);  // B^T = R^T Q
        gram(Z, in, k, w, st);                          // B B^T
        dc_small_kernel<<<1, 1024, small_smem(k), st>>>(w.G, k, r, 1, w.M, w.MU, w.MV, di->status);
        const int64_t nu = (int64_t)out * r, nv = (int64_t)in * r;
        dc_apply_kernel<<<(unsigned)std::min<int64_t>((nu + 255) / 256, 4096), 256, k * r * 4, st>>>(
            Y, out, k, w.MU, r, U + (int64_t)l * out * r, 1);
        dc_apply_kernel<<<(unsigned)std::min<int64_t>((nv + 255) / 256, 4096), 256, k * r * 4, st>>>(
            Z, in, k, w.MV, r, V + (int64_t)l * in * r, 1);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "wl_decompose_band launch");
    return WL_OK;
}

}  // namespace wl
