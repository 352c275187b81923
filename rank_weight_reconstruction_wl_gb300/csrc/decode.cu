// decode.cu -- decode-size (small T) weightless projections on CUDA cores.
//
// Computes, for each output row o of a projection ("In-kernel
// reconstruction", formula section):
//     y[t,o] = s[o] * sum_i W0[o,i] x[t,i] + sum_k U[o,k] z[t,k],
//     z[t,k] = sum_i V[i,k] x[t,i]
// in ONE launch per call: W0 is streamed from HBM exactly once with 16-byte
// loads, z is formed in the same launch, and the scale and the rank-r delta
// are applied in the epilogue.  At decode sizes the work is bound by the
// HBM stream of W0 (one multiply-add per two bytes at T = 1), so these
// kernels use CUDA cores, not the tensor cores.
//
// Work split.  A launch covers a set of projections ("segments": one for
// wl_linear, three for Q/K/V fusion).  Output rows are cut into row blocks;
// each row block is handled by a thread-block cluster of KS CTAs that split
// the input dimension K.  Every CTA computes, over its own K range,
//     p[t,o] = s[o] * sum_{i in range} W0[o,i] x[t,i] + sum_k U[o,k] z_range[t,k]
// (both terms are linear in the K split, so the ranges add up to y), then the
// cluster adds the KS partials through distributed shared memory in a fixed
// rank order (deterministic, no global atomics, no scratch memory).
//
// The fused GeGLU MLP ("In-kernel reconstruction", custom-op path: gate, up,
// activation and down in one dispatch) runs as one persistent launch in two
// phases separated by a bounded grid barrier: phase 1 produces h = gelu(g)*u
// and the down projection's low-rank partials z_down = h V_down, phase 2
// streams W_down.
#include <cooperative_groups.h>
#include <stdio.h>

#include <mutex>
#include <unordered_map>

#include "wl_internal.cuh"

namespace cg = cooperative_groups;

namespace wl {

// ------------------------------------------------------------------------
// Shared device pieces
// ------------------------------------------------------------------------

// Stage x[t, k0:k0+klen) (bf16, row stride `ld`) into xs[t*Kc + j] as fp32;
// rows t >= T are zero.  klen % 8 == 0.
template <int TT>
__device__ __forceinline__ void stage_x_bf16(const bf16 *__restrict__ x, int64_t ld, int T,
                                             int k0, int klen, int Kc, float *xs)
{
    const int nck = klen >> 3;
    for (int idx = threadIdx.x; idx < TT * nck; idx += kThreads) {
        const int t = idx / nck, c = idx - t * nck;
        float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
        if (t < T) {
            const uint4 v = *reinterpret_cast<const uint4 *>(x + t * ld + k0 + 8 * c);
            lo = make_float4(bf_lo(v.x), bf_hi(v.x), bf_lo(v.y), bf_hi(v.y));
            hi = make_float4(bf_lo(v.z), bf_hi(v.z), bf_lo(v.w), bf_hi(v.w));
        }
        *reinterpret_cast<float4 *>(xs + t * Kc + 8 * c) = lo;
        *reinterpret_cast<float4 *>(xs + t * Kc + 8 * c + 4) = hi;
    }
}

// Same from an fp32 source written earlier in this launch (L2-coherent loads).
template <int TT>
__device__ __forceinline__ void stage_x_f32(const float *x, int64_t ld, int T, int k0, int klen,
                                            int Kc, float *xs)
{
    const int nq = klen >> 2;
    for (int idx = threadIdx.x; idx < TT * nq; idx += kThreads) {
        const int t = idx / nq, c = idx - t * nq;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < T) v = __ldcg(reinterpret_cast<const float4 *>(x + t * ld + k0 + 4 * c));
        *reinterpret_cast<float4 *>(xs + t * Kc + 4 * c) = v;
    }
}

// Raw dot products acc[v*TT + t] = sum_{c < nck} W0row(v)[8c..8c+7] . xs[t][8c..]
// for the virtual rows v in [0, nv).  row_ptr(v) returns the address of the
// K-range start of virtual row v.  LPR lanes share one row; a warp works on
// (32/LPR)*RPI rows at a time.
template <int TT, int LPR, typename RowPtr>
__device__ __forceinline__ void stream_rows(RowPtr row_ptr, int nv, int nck, const float *xs,
                                            int Kc, float *acc)
{
    constexpr int G = 32 / LPR;
    constexpr int RPI = (TT <= 2) ? 4 : 2;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int gi = lane / LPR, sl = lane % LPR;
    for (int rb = warp * G * RPI; rb < nv; rb += kWarps * G * RPI) {
        float a[RPI][TT];
        const bf16 *wp[RPI];
        bool ok[RPI];
#pragma unroll
        for (int j = 0; j < RPI; ++j) {
            const int v = rb + gi * RPI + j;
            ok[j] = v < nv;
            wp[j] = row_ptr(ok[j] ? v : 0);
#pragma unroll
            for (int t = 0; t < TT; ++t) a[j][t] = 0.f;
        }
#pragma unroll 2
        for (int c = sl; c < nck; c += LPR) {
            uint4 w[RPI];
#pragma unroll
            for (int j = 0; j < RPI; ++j)
                w[j] = ok[j] ? ld_stream16(wp[j] + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int t = 0; t < TT; ++t) {
                const float4 xa = *reinterpret_cast<const float4 *>(xs + t * Kc + 8 * c);
                const float4 xb = *reinterpret_cast<const float4 *>(xs + t * Kc + 8 * c + 4);
#pragma unroll
                for (int j = 0; j < RPI; ++j) {
                    float s = a[j][t];
                    s = fmaf(bf_lo(w[j].x), xa.x, s);
                    s = fmaf(bf_hi(w[j].x), xa.y, s);
                    s = fmaf(bf_lo(w[j].y), xa.z, s);
                    s = fmaf(bf_hi(w[j].y), xa.w, s);
                    s = fmaf(bf_lo(w[j].z), xb.x, s);
                    s = fmaf(bf_hi(w[j].z), xb.y, s);
                    s = fmaf(bf_lo(w[j].w), xb.z, s);
                    s = fmaf(bf_hi(w[j].w), xb.w, s);
                    a[j][t] = s;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < RPI; ++j)
#pragma unroll
            for (int t = 0; t < TT; ++t) {
                float s = a[j][t];
#pragma unroll
                for (int off = LPR / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
                a[j][t] = s;
            }
        if (sl == 0) {
#pragma unroll
            for (int j = 0; j < RPI; ++j)
                if (ok[j]) {
                    const int v = rb + gi * RPI + j;
#pragma unroll
                    for (int t = 0; t < TT; ++t) acc[v * TT + t] = a[j][t];
                }
        }
    }
}

// out[t*ostride + k] = sum_{i < n} src[t*sstride + i] * V[i*r + k], k < r.
// All threads of the CTA take part (contains __syncthreads).  zred holds
// kWarps*TT*32 floats.
template <int TT>
__device__ __forceinline__ void block_xV(const float *src, int sstride, int n,
                                         const bf16 *__restrict__ V, int r, float *out,
                                         int ostride, float *zred)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int kb = 0; kb < r; kb += 32) {
        const int k = kb + lane;
        float part[TT];
#pragma unroll
        for (int t = 0; t < TT; ++t) part[t] = 0.f;
        if (k < r) {
            for (int i = warp; i < n; i += kWarps) {
                const float v = bf2f(V[(int64_t)i * r + k]);
#pragma unroll
                for (int t = 0; t < TT; ++t) part[t] = fmaf(src[t * sstride + i], v, part[t]);
            }
        }
#pragma unroll
        for (int t = 0; t < TT; ++t) zred[(warp * TT + t) * 32 + lane] = part[t];
        __syncthreads();
        for (int idx = threadIdx.x; idx < TT * 32; idx += kThreads) {
            const int t = idx >> 5, l = idx & 31;
            if (kb + l < r) {
                float s = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) s += zred[(w * TT + t) * 32 + l];
                out[t * ostride + kb + l] = s;
            }
        }
        __syncthreads();
    }
}

__device__ __forceinline__ float gelu_tanh_f32(float v)
{
    const float c = 0.7978845608028654f;  // sqrt(2/pi)
    return 0.5f * v * (1.0f + tanhf(c * (v + 0.044715f * v * v * v)));
}

// ------------------------------------------------------------------------
// wl_linear / wl_qkv_fused decode kernel
// ------------------------------------------------------------------------
struct DecSeg {
    const bf16 *W0;
    const float *s;
    const bf16 *U;
    const bf16 *V;
    void *y;
    int out;
    int blk0;  // first row block of this segment
    int nblk;  // row blocks of this segment
};

struct DecArgs {
    const bf16 *x;
    int T, in, r, ydt;
    int KS, Kc;  // K splits (= cluster size) and K elements per split
    int rmax;    // largest row block
    int nseg;
    DecSeg seg[3];
};

template <int TT>
__host__ __device__ constexpr int dec_zred_floats() { return kWarps * TT * 32; }

template <int TT, int LPR>
__global__ void __launch_bounds__(kThreads, 2) dec_linear_kernel(const __grid_constant__ DecArgs a)
{
    extern __shared__ __align__(16) float smem[];
    const int KS = a.KS;
    const int q = (int)(blockIdx.x % (unsigned)KS);  // rank in the cluster
    const int b = (int)(blockIdx.x / (unsigned)KS);  // row block
    const int si = (a.nseg > 2 && b >= a.seg[2].blk0) ? 2 : (a.nseg > 1 && b >= a.seg[1].blk0) ? 1 : 0;
    const DecSeg sg = si == 0 ? a.seg[0] : (si == 1 ? a.seg[1] : a.seg[2]);
    const int lb = b - sg.blk0;
    const int r0 = (int)((int64_t)lb * sg.out / sg.nblk);
    const int nrows = (int)((int64_t)(lb + 1) * sg.out / sg.nblk) - r0;
    const int k0 = q * a.Kc;
    const int klen = max(0, min(a.in, k0 + a.Kc) - k0);
    const int rp = a.r > 0 ? a.r : 1;

    float *xs = smem;
    float *acc = xs + TT * a.Kc;
    float *zp = acc + a.rmax * TT;
    float *zred = zp + TT * rp;

    stage_x_bf16<TT>(a.x, a.in, a.T, k0, klen, a.Kc, xs);
    __syncthreads();

    const bf16 *W0 = sg.W0 + (int64_t)r0 * a.in + k0;
    const int64_t ld = a.in;
    stream_rows<TT, LPR>([&](int v) { return W0 + v * ld; }, nrows, klen >> 3, xs, a.Kc, acc);

    if (a.r > 0) block_xV<TT>(xs, a.Kc, klen, sg.V + (int64_t)k0 * a.r, a.r, zp, rp, zred);
    __syncthreads();

    // epilogue: p = s*acc + U z_range
    for (int row = threadIdx.x; row < nrows; row += kThreads) {
        const int o = r0 + row;
        const float sv = sg.s[o];
        float yv[TT];
#pragma unroll
        for (int t = 0; t < TT; ++t) yv[t] = sv * acc[row * TT + t];
        const bf16 *Ur = sg.U + (int64_t)o * a.r;
        for (int k = 0; k < a.r; ++k) {
            const float u = bf2f(Ur[k]);
#pragma unroll
            for (int t = 0; t < TT; ++t) yv[t] = fmaf(u, zp[t * rp + k], yv[t]);
        }
        if (KS == 1) {
#pragma unroll
            for (int t = 0; t < TT; ++t)
                if (t < a.T) store_out(sg.y, a.ydt, (int64_t)t * sg.out + o, yv[t]);
        } else {
#pragma unroll
            for (int t = 0; t < TT; ++t) acc[row * TT + t] = yv[t];
        }
    }
    if (KS > 1) {
        cg::cluster_group cl = cg::this_cluster();
        cl.sync();
        const int lo = (int)((int64_t)q * nrows / KS);
        const int n = (int)((int64_t)(q + 1) * nrows / KS) - lo;
        for (int idx = threadIdx.x; idx < n * a.T; idx += kThreads) {
            const int t = idx / n, row = lo + (idx - t * n);
            float v = 0.f;
            for (int p = 0; p < KS; ++p) v += cl.map_shared_rank(acc, p)[row * TT + t];
            store_out(sg.y, a.ydt, (int64_t)t * sg.out + r0 + row, v);
        }
        cl.sync();
    }
}

// ------------------------------------------------------------------------
// fused GeGLU MLP decode kernel (persistent, two phases)
// ------------------------------------------------------------------------
struct MlpArgs {
    const bf16 *x;
    int T, hidden, inter, r, ydt;
    const bf16 *Wg, *Wu, *Wd;
    const float *sg, *su, *sd;
    const bf16 *Ug, *Uu, *Ud, *Vg, *Vu, *Vd;
    void *y;
    float *h;          // workspace [kDecodeTT][inter] fp32
    float *zd;         // workspace [NB1][kDecodeTT][rp] fp32
    unsigned *bar;     // workspace [2]: arrival count, generation
    unsigned *status;  // library status word
    int KS, Kc1, Kc2, NB1, NB2, rmax1, rmax2, hmax, nclus;
    int xs_f, acc_f;   // smem region sizes (floats)
};

// Grid-wide barrier over all CTAs of the launch (all co-resident).  Bounded:
// after kWaitLimitNs it records kStatusTimeout and returns false.
__device__ bool grid_barrier(unsigned *bar, unsigned nblocks, unsigned *status)
{
    __shared__ int ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        volatile unsigned *vgen = bar + 1;
        const unsigned gen = *vgen;
        __threadfence();
        const unsigned prev = atomicAdd(bar, 1u);
        ok = 1;
        if (prev == nblocks - 1) {
            atomicExch(bar, 0u);
            __threadfence();
            atomicAdd(bar + 1, 1u);
        } else {
            const uint64_t t0 = globaltimer_ns();
            while (*vgen == gen) {
                __nanosleep(100);
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    atomicOr(status, kStatusTimeout);
                    ok = 0;
                    break;
                }
            }
        }
        __threadfence();
    }
    __syncthreads();
    return ok != 0;
}

template <int TT, int LPR1, int LPR2>
__global__ void __launch_bounds__(kThreads, 2) dec_mlp_kernel(const __grid_constant__ MlpArgs a)
{
    extern __shared__ __align__(16) float smem[];
    cg::cluster_group cl = cg::this_cluster();
    const int KS = a.KS;
    const int q = (int)(blockIdx.x % (unsigned)KS);
    const int cid = (int)(blockIdx.x / (unsigned)KS);
    const int rp = a.r > 0 ? a.r : 1;

    float *xs = smem;
    float *acc = xs + a.xs_f;
    float *zp = acc + a.acc_f;       // [2][TT][rp]
    float *zred = zp + 2 * TT * rp;  // [kWarps*TT*32]
    float *zdl = zred + dec_zred_floats<TT>();  // [TT][rp]
    float *hl = zdl + TT * rp;       // [TT][hmax]

    // ---- phase 1: g, u -> h, and z_down partials -----------------------
    for (int b = cid; b < a.NB1; b += a.nclus) {
        const int j0 = (int)((int64_t)b * a.inter / a.NB1);
        const int nr = (int)((int64_t)(b + 1) * a.inter / a.NB1) - j0;
        const int k0 = q * a.Kc1;
        const int klen = max(0, min(a.hidden, k0 + a.Kc1) - k0);

        stage_x_bf16<TT>(a.x, a.hidden, a.T, k0, klen, a.Kc1, xs);
        __syncthreads();
        const bf16 *Wg = a.Wg + (int64_t)j0 * a.hidden + k0;
        const bf16 *Wu = a.Wu + (int64_t)j0 * a.hidden + k0;
        const int64_t ld = a.hidden;
        stream_rows<TT, LPR1>(
            [&](int v) { return v < nr ? Wg + v * ld : Wu + (v - nr) * ld; }, 2 * nr,
            klen >> 3, xs, a.Kc1, acc);
        if (a.r > 0) {
            block_xV<TT>(xs, a.Kc1, klen, a.Vg + (int64_t)k0 * a.r, a.r, zp, rp, zred);
            block_xV<TT>(xs, a.Kc1, klen, a.Vu + (int64_t)k0 * a.r, a.r, zp + TT * rp, rp, zred);
        }
        __syncthreads();
        for (int v = threadIdx.x; v < 2 * nr; v += kThreads) {
            const bool up = v >= nr;
            const int j = j0 + (up ? v - nr : v);
            const float sv = up ? a.su[j] : a.sg[j];
            const bf16 *Ur = (up ? a.Uu : a.Ug) + (int64_t)j * a.r;
            const float *z = zp + (up ? TT * rp : 0);
            float yv[TT];
#pragma unroll
            for (int t = 0; t < TT; ++t) yv[t] = sv * acc[v * TT + t];
            for (int k = 0; k < a.r; ++k) {
                const float u = bf2f(Ur[k]);
#pragma unroll
                for (int t = 0; t < TT; ++t) yv[t] = fmaf(u, z[t * rp + k], yv[t]);
            }
#pragma unroll
            for (int t = 0; t < TT; ++t) acc[v * TT + t] = yv[t];
        }
        cl.sync();
        // my share of the rows: complete g, u -> h
        const int lo = (int)((int64_t)q * nr / KS);
        const int n = (int)((int64_t)(q + 1) * nr / KS) - lo;
        for (int idx = threadIdx.x; idx < n * TT; idx += kThreads) {
            const int t = idx / n, v = lo + (idx - t * n);
            float g = 0.f, u = 0.f;
            for (int p = 0; p < KS; ++p) {
                const float *pa = cl.map_shared_rank(acc, p);
                g += pa[v * TT + t];
                u += pa[(nr + v) * TT + t];
            }
            const float hv = t < a.T ? gelu_tanh_f32(g) * u : 0.f;
            hl[t * a.hmax + (v - lo)] = hv;
            if (t < a.T) a.h[(int64_t)t * a.inter + j0 + v] = hv;
        }
        __syncthreads();
        if (a.r > 0) block_xV<TT>(hl, a.hmax, n, a.Vd + (int64_t)(j0 + lo) * a.r, a.r, zdl, rp, zred);
        cl.sync();
        if (q == 0 && a.r > 0) {
            float *dst = a.zd + (int64_t)b * kDecodeTT * rp;
            for (int idx = threadIdx.x; idx < TT * a.r; idx += kThreads) {
                const int t = idx / a.r, k = idx - t * a.r;
                float s = 0.f;
                for (int p = 0; p < KS; ++p) s += cl.map_shared_rank(zdl, p)[t * rp + k];
                dst[t * rp + k] = s;
            }
        }
        cl.sync();
    }

    // On a timeout the status word is set and the CTA carries on (its output
    // is then meaningless): returning early could strand cluster peers at a
    // cluster barrier, while carrying on keeps every wait bounded.
    grid_barrier(a.bar, gridDim.x, a.status);

    // ---- phase 2: y = wl(h; down) ---------------------------------------
    for (int b = cid; b < a.NB2; b += a.nclus) {
        const int o0 = (int)((int64_t)b * a.hidden / a.NB2);
        const int nr = (int)((int64_t)(b + 1) * a.hidden / a.NB2) - o0;
        const int k0 = q * a.Kc2;
        const int klen = max(0, min(a.inter, k0 + a.Kc2) - k0);

        stage_x_f32<TT>(a.h, a.inter, a.T, k0, klen, a.Kc2, xs);
        if (q == 0 && a.r > 0) {
            for (int idx = threadIdx.x; idx < TT * a.r; idx += kThreads) {
                const int t = idx / a.r, k = idx - t * a.r;
                float s = 0.f;
                for (int p = 0; p < a.NB1; ++p) s += __ldcg(a.zd + ((int64_t)p * kDecodeTT + t) * rp + k);
                zp[t * rp + k] = s;
            }
        }
        __syncthreads();
        const bf16 *Wd = a.Wd + (int64_t)o0 * a.inter + k0;
        const int64_t ld = a.inter;
        stream_rows<TT, LPR2>([&](int v) { return Wd + v * ld; }, nr, klen >> 3, xs, a.Kc2, acc);
        __syncthreads();
        const int rr = (q == 0) ? a.r : 0;  // the low-rank term is added once
        for (int row = threadIdx.x; row < nr; row += kThreads) {
            const int o = o0 + row;
            const float sv = a.sd[o];
            float yv[TT];
#pragma unroll
            for (int t = 0; t < TT; ++t) yv[t] = sv * acc[row * TT + t];
            const bf16 *Ur = a.Ud + (int64_t)o * a.r;
            for (int k = 0; k < rr; ++k) {
                const float u = bf2f(Ur[k]);
#pragma unroll
                for (int t = 0; t < TT; ++t) yv[t] = fmaf(u, zp[t * rp + k], yv[t]);
            }
#pragma unroll
            for (int t = 0; t < TT; ++t) acc[row * TT + t] = yv[t];
        }
        cl.sync();
        const int lo = (int)((int64_t)q * nr / KS);
        const int n = (int)((int64_t)(q + 1) * nr / KS) - lo;
        for (int idx = threadIdx.x; idx < n * a.T; idx += kThreads) {
            const int t = idx / n, row = lo + (idx - t * n);
            float v = 0.f;
            for (int p = 0; p < KS; ++p) v += cl.map_shared_rank(acc, p)[row * TT + t];
            store_out(a.y, a.ydt, (int64_t)t * a.hidden + o0 + row, v);
        }
        cl.sync();
    }
}

// ------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------
static inline int round_up(int v, int m) { return (v + m - 1) / m * m; }
static inline int lpr_for(int nck) { return nck >= 64 ? 32 : (nck >= 32 ? 16 : 8); }
static inline int lpr_index(int lpr) { return lpr == 32 ? 2 : (lpr == 16 ? 1 : 0); }
static inline int tt_for(int64_t T) { return T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8; }
static inline int tt_index(int tt) { return tt == 1 ? 0 : tt == 2 ? 1 : tt == 4 ? 2 : 3; }

typedef void (*dec_fn)(DecArgs);
typedef void (*mlp_fn)(MlpArgs);

template <int TT>
static void fill_dec(dec_fn *row)
{
    row[0] = dec_linear_kernel<TT, 8>;
    row[1] = dec_linear_kernel<TT, 16>;
    row[2] = dec_linear_kernel<TT, 32>;
}
static dec_fn g_dec[4][3];

template <int TT, int L1>
static void fill_mlp2(mlp_fn *row)
{
    row[0] = dec_mlp_kernel<TT, L1, 8>;
    row[1] = dec_mlp_kernel<TT, L1, 16>;
    row[2] = dec_mlp_kernel<TT, L1, 32>;
}
template <int TT>
static void fill_mlp(mlp_fn (*tab)[3])
{
    fill_mlp2<TT, 8>(tab[0]);
    fill_mlp2<TT, 16>(tab[1]);
    fill_mlp2<TT, 32>(tab[2]);
}
static mlp_fn g_mlp[4][3][3];

static std::mutex g_mu;
static std::unordered_map<uint64_t, int> g_smem_set;  // (device, fn) -> bytes set

static wl_status ensure_smem(const void *fn, int bytes, const DeviceInfo *di)
{
    if (bytes > di->max_smem_optin)
        return fail(WL_ERR_UNSUPPORTED, "decode kernel needs %d bytes of shared memory, device allows %d",
                    bytes, di->max_smem_optin);
    std::lock_guard<std::mutex> lk(g_mu);
    const uint64_t key = ((uint64_t)di->device << 56) ^ (uint64_t)(uintptr_t)fn;
    auto it = g_smem_set.find(key);
    if (it != g_smem_set.end() && it->second >= bytes) return WL_OK;
    const int want = di->max_smem_optin;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic smem)");
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(non-portable cluster)");
    g_smem_set[key] = want;
    return WL_OK;
}

static void init_tables()
{
    static std::once_flag once;
    std::call_once(once, [] {
        fill_dec<1>(g_dec[0]);
        fill_dec<2>(g_dec[1]);
        fill_dec<4>(g_dec[2]);
        fill_dec<8>(g_dec[3]);
        fill_mlp<1>(g_mlp[0]);
        fill_mlp<2>(g_mlp[1]);
        fill_mlp<4>(g_mlp[2]);
        fill_mlp<8>(g_mlp[3]);
    });
}

static wl_status launch_with_cluster(const void *fn, int grid, int KS, int smem, cudaStream_t st,
                                     void **args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)KS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
    return WL_OK;
}

// One launch over up to kDecodeTT tokens.
static wl_status dec_linear_once(const bf16 *x, const wl_proj *proj, int nproj, void *const *y,
                                 int T, int in, int r, int ydt, cudaStream_t st,
                                 const DeviceInfo *di)
{
    const int TT = tt_for(T);
    int64_t rows = 0;
    for (int j = 0; j < nproj; ++j) rows += proj[j].out;
    const int target = 2 * di->sm_count;

    // K split (cluster size): enough row work per CTA, x slice small enough
    // for shared memory, and few enough row blocks that the rank-r operand V
    // (re-read by every row block) stays small next to W0.
    int KS = 1;
    auto kc_of = [&](int ks) { return round_up((in + ks - 1) / ks, 8); };
    while (KS < 8 && TT * kc_of(KS) * 4 > 96 * 1024) KS *= 2;
    while (KS < 8) {
        const int64_t nb = target / KS;
        const bool few_rows = rows / nb < 16;
        const bool v_heavy = r > 0 && nb * 4 * (int64_t)r > rows;
        if ((few_rows || v_heavy) && kc_of(2 * KS) >= 64) KS *= 2;
        else break;
    }
    const int Kc = kc_of(KS);
    int64_t nb_total = target / KS;
    if (nb_total < nproj) nb_total = nproj;

    DecArgs a = {};
    a.x = x;
    a.T = T;
    a.in = in;
    a.r = r;
    a.ydt = ydt;
    a.KS = KS;
    a.Kc = Kc;
    a.nseg = nproj;
    int blk = 0, rmax = 1;
    for (int j = 0; j < nproj; ++j) {
        int nblk = (int)((nb_total * proj[j].out + rows - 1) / rows);
        if (nblk < 1) nblk = 1;
        if (nblk > proj[j].out) nblk = (int)proj[j].out;
        DecSeg &sg = a.seg[j];
        sg.W0 = static_cast<const bf16 *>(proj[j].W0);
        sg.s = proj[j].s;
        sg.U = static_cast<const bf16 *>(proj[j].U);
        sg.V = static_cast<const bf16 *>(proj[j].V);
        sg.y = y[j];
        sg.out = (int)proj[j].out;
        sg.blk0 = blk;
        sg.nblk = nblk;
        blk += nblk;
        const int rm = (int)((proj[j].out + nblk - 1) / nblk);
        if (rm > rmax) rmax = rm;
    }
    a.rmax = rmax;
    const int rp = r > 0 ? r : 1;
    const int smem = 4 * (TT * Kc + rmax * TT + TT * rp + kWarps * TT * 32);
    const dec_fn fn = g_dec[tt_index(TT)][lpr_index(lpr_for(Kc / 8))];
    wl_status s = ensure_smem((const void *)fn, smem, di);
    if (s != WL_OK) return s;
    void *args[] = {&a};
    return launch_with_cluster((const void *)fn, blk * KS, KS, smem, st, args);
}

wl_status launch_decode_linear(const bf16 *x, const wl_proj *proj, int nproj, void *const *y,
                               int64_t T, int64_t in, int64_t r, int ydt, cudaStream_t st)
{
    init_tables();
    wl_status s = WL_OK;
    const DeviceInfo *di = device_info(&s);
    if (!di) return s;
    const int es = ydt == WL_OUT_F32 ? 4 : 2;
    for (int64_t t0 = 0; t0 < T; t0 += kDecodeTT) {
        const int Tc = (int)((T - t0) < kDecodeTT ? (T - t0) : kDecodeTT);
        void *yc[3];
        for (int j = 0; j < nproj; ++j)
            yc[j] = static_cast<char *>(y[j]) + (size_t)t0 * (size_t)proj[j].out * es;
        s = dec_linear_once(x + t0 * in, proj, nproj, yc, Tc, (int)in, (int)r, ydt, st, di);
        if (s != WL_OK) return s;
    }
    return WL_OK;
}

// ---- MLP ---------------------------------------------------------------
static constexpr int kMlpKS = 8;
static constexpr int kMaxNB1 = 512;

size_t decode_mlp_workspace_bytes(int64_t hidden, int64_t inter, int64_t r)
{
    (void)hidden;
    const int64_t rp = r > 0 ? r : 1;
    auto al = [](int64_t v) { return (v + 255) / 256 * 256; };
    return (size_t)(256 + al(kDecodeTT * inter * 4) + al((int64_t)kMaxNB1 * kDecodeTT * rp * 4));
}

static std::unordered_map<uint64_t, int> g_max_clusters;

static wl_status max_active_clusters(const void *fn, int smem, const DeviceInfo *di, int *out)
{
    const uint64_t key = ((uint64_t)di->device << 56) ^ ((uint64_t)(uintptr_t)fn << 8) ^ (uint64_t)smem;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_max_clusters.find(key);
        if (it != g_max_clusters.end()) {
            *out = it->second;
            return WL_OK;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kMlpKS * 64);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kMlpKS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveClusters");
    if (n < 1) return fail(WL_ERR_UNSUPPORTED, "MLP kernel cannot place a cluster of %d CTAs", kMlpKS);
    std::lock_guard<std::mutex> lk(g_mu);
    g_max_clusters[key] = n;
    *out = n;
    return WL_OK;
}

static wl_status dec_mlp_once(const bf16 *x, const wl_proj &gate, const wl_proj &up,
                              const wl_proj &down, void *y, int T, int hidden, int inter, int r,
                              char *ws, int ydt, cudaStream_t st, const DeviceInfo *di)
{
    const int TT = tt_for(T);
    const int KS = kMlpKS;
    const int Kc1 = round_up((hidden + KS - 1) / KS, 8);
    const int Kc2 = round_up((inter + KS - 1) / KS, 8);
    const int rp = r > 0 ? r : 1;

    int nclus = (2 * di->sm_count) / KS;
    int NB1 = nclus < kMaxNB1 ? nclus : kMaxNB1;
    if (NB1 > inter) NB1 = inter;
    int NB2 = nclus < hidden ? nclus : hidden;
    const int rmax1 = (inter + NB1 - 1) / NB1;
    const int rmax2 = (hidden + NB2 - 1) / NB2;
    const int hmax = (rmax1 + KS - 1) / KS + 1;
    MlpArgs a = {};
    a.x = x;
    a.T = T;
    a.hidden = hidden;
    a.inter = inter;
    a.r = r;
    a.ydt = ydt;
    a.Wg = static_cast<const bf16 *>(gate.W0);
    a.Wu = static_cast<const bf16 *>(up.W0);
    a.Wd = static_cast<const bf16 *>(down.W0);
    a.sg = gate.s;
    a.su = up.s;
    a.sd = down.s;
    a.Ug = static_cast<const bf16 *>(gate.U);
    a.Uu = static_cast<const bf16 *>(up.U);
    a.Ud = static_cast<const bf16 *>(down.U);
    a.Vg = static_cast<const bf16 *>(gate.V);
    a.Vu = static_cast<const bf16 *>(up.V);
    a.Vd = static_cast<const bf16 *>(down.V);
    a.y = y;
    a.bar = reinterpret_cast<unsigned *>(ws);
    a.h = reinterpret_cast<float *>(ws + 256);
    a.zd = reinterpret_cast<float *>(ws + 256 + ((int64_t)kDecodeTT * inter * 4 + 255) / 256 * 256);
    a.status = di->status;
    a.KS = KS;
    a.Kc1 = Kc1;
    a.Kc2 = Kc2;
    a.NB1 = NB1;
    a.NB2 = NB2;
    a.rmax1 = rmax1;
    a.rmax2 = rmax2;
    a.hmax = hmax;
    a.xs_f = TT * (Kc1 > Kc2 ? Kc1 : Kc2);
    a.acc_f = TT * (2 * rmax1 > rmax2 ? 2 * rmax1 : rmax2);
    const int smem = 4 * (a.xs_f + a.acc_f + 2 * TT * rp + kWarps * TT * 32 + TT * rp + TT * hmax);
    const mlp_fn fn = g_mlp[tt_index(TT)][lpr_index(lpr_for(Kc1 / 8))][lpr_index(lpr_for(Kc2 / 8))];
    wl_status s = ensure_smem((const void *)fn, smem, di);
    if (s != WL_OK) return s;
    int maxc = 0;
    s = max_active_clusters((const void *)fn, smem, di, &maxc);
    if (s != WL_OK) return s;
    // every CTA of the launch must be resident at once (grid barrier)
    if (nclus > maxc) nclus = maxc;
    a.nclus = nclus;
    void *args[] = {&a};
    return launch_with_cluster((const void *)fn, nclus * KS, KS, smem, st, args);
}

wl_status launch_decode_mlp(const bf16 *x, const wl_proj &gate, const wl_proj &up,
                            const wl_proj &down, void *y, int64_t T, int64_t hidden,
                            int64_t inter, int64_t r, void *ws, size_t ws_bytes, int ydt,
                            cudaStream_t st)
{
    init_tables();
    wl_status s = WL_OK;
    const DeviceInfo *di = device_info(&s);
    if (!di) return s;
    if (ws_bytes < decode_mlp_workspace_bytes(hidden, inter, r))
        return fail(WL_ERR_WORKSPACE, "MLP workspace too small");
    const int es = ydt == WL_OUT_F32 ? 4 : 2;
    for (int64_t t0 = 0; t0 < T; t0 += kDecodeTT) {
        const int Tc = (int)((T - t0) < kDecodeTT ? (T - t0) : kDecodeTT);
        s = dec_mlp_once(x + t0 * hidden, gate, up, down,
                         static_cast<char *>(y) + (size_t)t0 * (size_t)hidden * es, Tc,
                         (int)hidden, (int)inter, (int)r, static_cast<char *>(ws), ydt, st, di);
        if (s != WL_OK) return s;
    }
    return WL_OK;
}

}  // namespace wl
