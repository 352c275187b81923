// f32_linear.cu -- weightless projections with fp32-encoded bundles and
// inputs ("Serve and generate with weightless", "Supported encodings and
// devices": the architectures default to bfloat16 and also support float32).
//
//     y[t,o] = s[o] * sum_i W0[o,i] x[t,i] + sum_k U[o,k] z[t,k],
//     z[t,k] = sum_i x[t,i] V[i,k]
//
// fp32 inputs keep fp32 arithmetic: the bf16 tensor-core forms would round
// every operand to 8 significant bits, far outside the fp32 output tolerance,
// and the fp32 tensor-core form (tf32) keeps only 11.  So this is a tiled
// CUDA-core GEMM with fp32 FMAs: a CTA computes a BM-token x BN-row tile of y
// over the whole K, staging x, W0 and the matching V rows through shared
// memory BK columns at a time; z of the CTA's tokens is accumulated in the
// same K loop (the x tile is already staged), and the epilogue applies the
// scale and U z.  One launch per call; Q/K/V are segments of one grid, so x
// is read once per token tile.
#include "wl_internal.cuh"

namespace wl {

struct F32Seg {
    const float *W0, *s, *U, *V;
    void *y;
    int out;
    int nt0;  // first N tile of this segment
};

struct F32Args {
    F32Seg seg[3];
    int nseg;
    const float *x;
    int T, in, r, ydt;
};

// BM tokens x BN rows per CTA, BK columns per step, TM x TN outputs per
// thread (16 x 16 threads), z as (BM/16) tokens x ZTN ranks per thread
// (ranks up to 16 * ZTN).
template <int BM, int BN, int BK, int TM, int TN, int ZTN>
__global__ void __launch_bounds__(256) f32_linear_kernel(const __grid_constant__ F32Args a)
{
    constexpr int RP = 16 * ZTN;  // padded ranks
    constexpr int ZTM = BM / 16;
    // K-loop tiles (k-major), then z of the tile's tokens in the same memory
    constexpr int XS = BM + 4, WS = BN + 4, VS = RP + 4, ZS = RP + 1;
    constexpr int LOOP_F = BK * (XS + WS + VS), Z_F = BM * ZS;
    __shared__ __align__(16) float smf[LOOP_F > Z_F ? LOOP_F : Z_F];
    float(*xs)[XS] = reinterpret_cast<float(*)[XS]>(smf);
    float(*ws)[WS] = reinterpret_cast<float(*)[WS]>(smf + BK * XS);
    float(*vs)[VS] = reinterpret_cast<float(*)[VS]>(smf + BK * (XS + WS));
    float(*zs)[ZS] = reinterpret_cast<float(*)[ZS]>(smf);

    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int nt = blockIdx.x;
    const int si = (a.nseg > 2 && nt >= a.seg[2].nt0) ? 2 : (a.nseg > 1 && nt >= a.seg[1].nt0) ? 1 : 0;
    const F32Seg &sg = a.seg[si];
    const float *__restrict__ W0 = sg.W0;
    const float *__restrict__ V = sg.V;
    const float *__restrict__ x = a.x;
    const int out = sg.out, in = a.in, T = a.T, r = a.r;
    const int o0 = (nt - sg.nt0) * BN;
    const int t0 = blockIdx.y * BM;

    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
    float zacc[ZTM][ZTN > 0 ? ZTN : 1];
#pragma unroll
    for (int i = 0; i < ZTM; ++i)
#pragma unroll
        for (int j = 0; j < (ZTN > 0 ? ZTN : 1); ++j) zacc[i][j] = 0.f;

    for (int k0 = 0; k0 < in; k0 += BK) {
        // x tile [BM tokens][BK] and W0 tile [BN rows][BK], stored k-major;
        // consecutive threads read consecutive columns of a row
        for (int e = tid; e < BM * BK; e += 256) {
            const int t = e / BK, k = e - t * BK;
            xs[k][t] = (t0 + t < T && k0 + k < in) ? x[(int64_t)(t0 + t) * in + k0 + k] : 0.f;
        }
        for (int e = tid; e < BN * BK; e += 256) {
            const int o = e / BK, k = e - o * BK;
            ws[k][o] = (o0 + o < out && k0 + k < in) ? W0[(int64_t)(o0 + o) * in + k0 + k] : 0.f;
        }
        if (ZTN > 0) {
            for (int e = tid; e < BK * RP; e += 256) {
                const int k = e / RP, j = e - k * RP;
                vs[k][j] = (j < r && k0 + k < in) ? V[(int64_t)(k0 + k) * r + j] : 0.f;
            }
        }
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < BK; ++kk) {
            float av[TM], bv[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) av[i] = xs[kk][ty * TM + i];
#pragma unroll
            for (int j = 0; j < TN; ++j) bv[j] = ws[kk][tx * TN + j];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
            if (ZTN > 0) {
                float zx[ZTM], zv[ZTN > 0 ? ZTN : 1];
#pragma unroll
                for (int i = 0; i < ZTM; ++i) zx[i] = xs[kk][ty * ZTM + i];
#pragma unroll
                for (int j = 0; j < ZTN; ++j) zv[j] = vs[kk][tx * ZTN + j];
#pragma unroll
                for (int i = 0; i < ZTM; ++i)
#pragma unroll
                    for (int j = 0; j < ZTN; ++j) zacc[i][j] = fmaf(zx[i], zv[j], zacc[i][j]);
            }
        }
        __syncthreads();
    }

    // z of the tile's tokens (over the K-loop tiles: the loop ended with a
    // barrier), then y = s * acc + U z
    if (ZTN > 0) {
#pragma unroll
        for (int i = 0; i < ZTM; ++i)
#pragma unroll
            for (int j = 0; j < ZTN; ++j) zs[ty * ZTM + i][tx * ZTN + j] = zacc[i][j];
        __syncthreads();
    }
#pragma unroll
    for (int j = 0; j < TN; ++j) {
        const int o = o0 + tx * TN + j;
        if (o >= out) continue;
        const float sv = sg.s[o];
        const float *Ur = sg.U + (int64_t)o * r;
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int tl = ty * TM + i, t = t0 + tl;
            if (t >= T) continue;
            float v = sv * acc[i][j];
            if (ZTN > 0)
                for (int k = 0; k < r; ++k) v = fmaf(Ur[k], zs[tl][k], v);
            store_out(sg.y, a.ydt, (int64_t)t * out + o, v);
        }
    }
}

typedef void (*f32_fn)(F32Args);

template <int BM, int BN, int BK, int TM, int TN>
static f32_fn pick_rank(int r)
{
    if (r == 0) return f32_linear_kernel<BM, BN, BK, TM, TN, 0>;
    if (r <= 16) return f32_linear_kernel<BM, BN, BK, TM, TN, 1>;
    if (r <= 32) return f32_linear_kernel<BM, BN, BK, TM, TN, 2>;
    if (r <= 64) return f32_linear_kernel<BM, BN, BK, TM, TN, 4>;
    return f32_linear_kernel<BM, BN, BK, TM, TN, 8>;
}

// Few tokens: 16 x 32 tiles (enough CTAs to keep HBM busy on W0); many
// tokens: 64 x 128 tiles (32 outputs per thread).
wl_status launch_f32_linear(const float *x, const wl_proj_f32 *proj, int nproj, void *const *y, int64_t T,
                            int64_t in, int64_t r, int ydt, cudaStream_t st)
{
    const bool small = T <= 16;
    const int BM = small ? 16 : 64, BN = small ? 32 : 128;
    F32Args a = {};
    a.x = x;
    a.T = (int)T;
    a.in = (int)in;
    a.r = (int)r;
    a.ydt = ydt;
    a.nseg = nproj;
    int ntiles = 0;
    for (int j = 0; j < nproj; ++j) {
        F32Seg &sg = a.seg[j];
        sg.W0 = proj[j].W0;
        sg.s = proj[j].s;
        sg.U = proj[j].U;
        sg.V = proj[j].V;
        sg.y = y[j];
        sg.out = (int)proj[j].out;
        sg.nt0 = ntiles;
        ntiles += (int)((proj[j].out + BN - 1) / BN);
    }
    const int64_t mt = (T + BM - 1) / BM;
    if (mt > 65535) return fail(WL_ERR_UNSUPPORTED, "fp32 linear: T too large (%lld)", (long long)T);
    const dim3 grid((unsigned)ntiles, (unsigned)mt);
    const f32_fn fn = small ? pick_rank<16, 32, 32, 1, 2>((int)r) : pick_rank<64, 128, 16, 4, 8>((int)r);
    fn<<<grid, 256, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "fp32 linear launch");
    return WL_OK;
}

}  // namespace wl
