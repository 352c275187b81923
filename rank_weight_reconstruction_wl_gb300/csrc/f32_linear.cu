// f32_linear.cu -- weightless projections with fp32-encoded bundles and
// inputs ("Serve and generate with weightless", "Supported encodings and
// devices": the architectures default to bfloat16 and also support float32).
//
//     y[t,o] = s[o] * sum_i W0[o,i] x[t,i] + sum_k U[o,k] z[t,k],
//     z[t,k] = sum_i x[t,i] V[i,k]
//
// fp32 inputs keep fp32 arithmetic: the bf16 tensor-core forms would round
// every operand to 8 significant bits, far outside the fp32 output tolerance,
// and the fp32 tensor-core form (tf32) keeps only 11.  So these are CUDA-core
// kernels with fp32 FMAs, one launch per call, Q/K/V as segments of one grid:
//   T <= 8 (T r <= 64): f32_decode_kernel, shaped by the weight stream (a
//     warp per output row, z split over a cluster of 8 CTAs);
//   more tokens, r <= 64: f32_gemm_kernel, a double-buffered 128-token x
//     64-row tile;
//   otherwise f32_linear_kernel: a CTA computes a BM-token x BN-row tile of y
//     over the whole K, staging x, W0 and the matching V rows through shared
//     memory BK columns at a time.
// In the tiled forms z of the CTA's tokens is accumulated in the same K loop
// (the x tile is already staged), and the epilogue applies the scale and U z.
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

// ---------------------------------------------------------------- decode --
// Few tokens (T <= 8): the call streams W0 once and the work per weight is
// T multiply-adds, so the layout follows the weight stream instead of a GEMM
// tile: one warp per output row reads the row with 16-byte loads (all of a
// lane's loads in flight before the sums), x comes from L1.  z = x V is split
// over a cluster of 8 CTAs by K (each CTA sums 1/8 of the rows of V), and every
// CTA adds the 8 partial z in rank order from distributed shared memory, so all
// rows of a projection see the same z.  A projection's CTAs are padded to a
// multiple of 8 so that a cluster never spans two projections.
constexpr int kF32DecRows = 8;   // output rows per CTA: one per warp
constexpr int kF32DecCl = 8;     // CTAs per cluster
constexpr int kF32DecZ = 64;     // T * r limit (z sums held per thread)

__device__ __forceinline__ float ld_peer_f32(const float *p, uint32_t rank)
{
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
    return v;
}

__device__ __forceinline__ void f32_cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int TT, int RR>
__global__ void __cluster_dims__(kF32DecCl, 1, 1) __launch_bounds__(256)
    f32_decode_kernel(const __grid_constant__ F32Args a)
{
    __shared__ float zred[8][kF32DecZ];  // per-warp partial z, then the CTA's partial (row 0)
    __shared__ float zs[kF32DecZ];       // z of the projection: [t][k]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cl = blockIdx.x / kF32DecCl;
    const uint32_t crank = (uint32_t)(blockIdx.x % kF32DecCl);
    // segment: seg.nt0 counts clusters
    const int si = (a.nseg > 2 && cl >= a.seg[2].nt0) ? 2 : (a.nseg > 1 && cl >= a.seg[1].nt0) ? 1 : 0;
    const F32Seg &sg = a.seg[si];
    const int in = a.in, r = a.r;
    const int o = ((cl - sg.nt0) * kF32DecCl + (int)crank) * kF32DecRows + warp;
    const bool row_ok = o < sg.out;
    const float *__restrict__ x = a.x;

    // this warp's row: the first loads in flight before z
    const float4 *wrow = reinterpret_cast<const float4 *>(sg.W0 + (int64_t)(row_ok ? o : 0) * in);
    const int nq = in >> 2;  // float4 per row
    float dot[TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) dot[t] = 0.f;
    constexpr int PF = 8;
    float4 wq[PF];
#pragma unroll
    for (int u = 0; u < PF; ++u) wq[u] = (row_ok && lane + 32 * u < nq) ? __ldg(wrow + lane + 32 * u) : make_float4(0.f, 0.f, 0.f, 0.f);

    if (RR > 0) {
        // z partial over this CTA's eighth of K: thread rows i = k0 + tid, + 256, ...
        const int k0 = (int)(((int64_t)in * crank) / kF32DecCl), k1 = (int)(((int64_t)in * (crank + 1)) / kF32DecCl);
        constexpr int RA = RR > 0 ? RR : 1;
        float zp[TT][RA];
#pragma unroll
        for (int t = 0; t < TT; ++t)
#pragma unroll
            for (int k = 0; k < RR; ++k) zp[t][k] = 0.f;
        for (int i = k0 + tid; i < k1; i += 256) {
            const float *vr = sg.V + (int64_t)i * r;
            float vv[RA];
#pragma unroll
            for (int k = 0; k < RR; ++k) vv[k] = k < r ? __ldg(vr + k) : 0.f;
#pragma unroll
            for (int t = 0; t < TT; ++t) {
                const float xv = t < a.T ? __ldg(x + (int64_t)t * in + i) : 0.f;
#pragma unroll
                for (int k = 0; k < RR; ++k) zp[t][k] = fmaf(xv, vv[k], zp[t][k]);
            }
        }
#pragma unroll
        for (int t = 0; t < TT; ++t)
#pragma unroll
            for (int k = 0; k < RR; ++k) {
                float v = zp[t][k];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                if (lane == 0) zred[warp][t * RR + k] = v;
            }
        __syncthreads();
        if (tid < TT * RR) {
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) v += zred[w][tid];
            zred[0][tid] = v;  // this CTA's partial (row 0 is read by the cluster)
        }
        f32_cluster_sync();
        if (tid < TT * RR) {
            float v = 0.f;
            for (uint32_t c = 0; c < (uint32_t)kF32DecCl; ++c) v += ld_peer_f32(&zred[0][tid], c);
            zs[tid] = v;
        }
        // no CTA leaves (or rewrites zred) before every CTA has read it
        f32_cluster_sync();
    }

    // the row's dot products with x
    for (int q0 = 0; q0 < nq; q0 += 32 * PF) {
#pragma unroll
        for (int u = 0; u < PF; ++u) {
            const int q = q0 + lane + 32 * u;
            if (q < nq) {
                const float4 w = wq[u];
#pragma unroll
                for (int t = 0; t < TT; ++t) {
                    if (t < a.T) {
                        const float4 xv = __ldg(reinterpret_cast<const float4 *>(x + (int64_t)t * in) + q);
                        dot[t] = fmaf(w.x, xv.x, dot[t]);
                        dot[t] = fmaf(w.y, xv.y, dot[t]);
                        dot[t] = fmaf(w.z, xv.z, dot[t]);
                        dot[t] = fmaf(w.w, xv.w, dot[t]);
                    }
                }
            }
            const int qn = q + 32 * PF;
            wq[u] = (row_ok && qn < nq) ? __ldg(wrow + qn) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
#pragma unroll
    for (int t = 0; t < TT; ++t)
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot[t] += __shfl_xor_sync(0xffffffffu, dot[t], off);
    if (!row_ok) return;
    // lane t writes token t
#pragma unroll
    for (int t = 0; t < TT; ++t) {
        if (lane == t && t < a.T) {
            float v = sg.s[o] * dot[t];
            if (RR > 0)
                for (int k = 0; k < r; ++k) v = fmaf(sg.U[(int64_t)o * r + k], zs[t * RR + k], v);
            store_out(sg.y, a.ydt, (int64_t)t * sg.out + o, v);
        }
    }
}

typedef void (*f32_dec_fn)(F32Args);

template <int TT>
static f32_dec_fn pick_dec_rank(int r)
{
    if (r == 0) return f32_decode_kernel<TT, 0>;
    if (r <= 4) return f32_decode_kernel<TT, 4>;
    if (r <= 8 && TT * 8 <= kF32DecZ) return f32_decode_kernel<TT, (TT * 8 <= kF32DecZ ? 8 : 4)>;
    if (r <= 16 && TT * 16 <= kF32DecZ) return f32_decode_kernel<TT, (TT * 16 <= kF32DecZ ? 16 : 4)>;
    if (r <= 32 && TT * 32 <= kF32DecZ) return f32_decode_kernel<TT, (TT * 32 <= kF32DecZ ? 32 : 4)>;
    if (r <= 64 && TT * 64 <= kF32DecZ) return f32_decode_kernel<TT, (TT * 64 <= kF32DecZ ? 64 : 4)>;
    return nullptr;
}

static f32_dec_fn pick_dec(int64_t T, int64_t r)
{
    switch (T) {
    case 1: return pick_dec_rank<1>((int)r);
    case 2: return pick_dec_rank<2>((int)r);
    case 3:
    case 4: return pick_dec_rank<4>((int)r);
    case 5:
    case 6:
    case 7:
    case 8: return pick_dec_rank<8>((int)r);
    default: return nullptr;
    }
}

// ------------------------------------------------------------ many tokens --
// 128 tokens x 64 rows per CTA, 8 x 4 outputs per thread (16 x 16 threads),
// K in steps of 16 through two shared-memory buffers: the next step's x (two
// 16-byte loads per thread), W0 (one) and V rows are fetched into registers
// while the current step is multiplied, then stored to the other buffer, one
// barrier per step.  x and W0 tiles are stored k-major (transposed), so a
// thread reads its 8 tokens as two 16-byte words, its 4 rows as one.  z of
// the tile's tokens (8 tokens x ZTN ranks per thread) comes from the same x
// words.  The sums over k run in order, as in the form above.
constexpr int kGBM = 128, kGBN = 64, kGBK = 16;

template <int ZTN>
__global__ void __launch_bounds__(256, ZTN >= 4 ? 1 : 2) f32_gemm_kernel(const __grid_constant__ F32Args a)
{
    constexpr int RP = 16 * ZTN;  // padded ranks
    constexpr int AS = kGBM + 4, BS = kGBN + 4, VSS = RP + 4, ZS = RP + 1;
    constexpr int STAGE_F = kGBK * (AS + BS + VSS);
    constexpr int Z_F = kGBM * ZS;
    __shared__ __align__(16) float smf[2 * STAGE_F > Z_F ? 2 * STAGE_F : Z_F];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int nt = blockIdx.x;
    const int si = (a.nseg > 2 && nt >= a.seg[2].nt0) ? 2 : (a.nseg > 1 && nt >= a.seg[1].nt0) ? 1 : 0;
    const F32Seg &sg = a.seg[si];
    const float *__restrict__ W0 = sg.W0;
    const float *__restrict__ V = sg.V;
    const float *__restrict__ x = a.x;
    const int out = sg.out, in = a.in, T = a.T, r = a.r;
    const int o0 = (nt - sg.nt0) * kGBN;
    const int t0 = blockIdx.y * kGBM;

    // this thread's loads of a step: x row lr (tokens), k words kq..kq+3 and
    // kq+8..kq+11; W0 row wr, k words wq..wq+3
    const int lr = tid >> 1, kq = (tid & 1) * 4;
    const int wr = tid >> 2, wq = (tid & 3) * 4;
    const bool xok = t0 + lr < T, wok = o0 + wr < out;
    const float *xp = x + (int64_t)(xok ? t0 + lr : 0) * in + kq;
    const float *wp = W0 + (int64_t)(wok ? o0 + wr : 0) * in + wq;
    // V rows of a step: RP ranks x 16 k, (16 * RP) / 256 values per thread
    constexpr int VPT = (kGBK * RP + 255) / 256;

    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    float zacc[8][ZTN > 0 ? ZTN : 1];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < (ZTN > 0 ? ZTN : 1); ++j) zacc[i][j] = 0.f;

    auto load = [&](int k0, float4 (&xa)[2], float4 &wa, float (&vr)[VPT > 0 ? VPT : 1]) {
        // in % 8 == 0: a word of 4 is all in or all out
#pragma unroll
        for (int h = 0; h < 2; ++h)
            xa[h] = (xok && k0 + 8 * h + kq < in) ? __ldg(reinterpret_cast<const float4 *>(xp + k0 + 8 * h))
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        wa = (wok && k0 + wq < in) ? __ldg(reinterpret_cast<const float4 *>(wp + k0)) : make_float4(0.f, 0.f, 0.f, 0.f);
        if (ZTN > 0) {
#pragma unroll
            for (int u = 0; u < VPT; ++u) {
                const int e = tid + 256 * u, k = e / RP, j = e - k * RP;
                vr[u] = (e < kGBK * RP && j < r && k0 + k < in) ? __ldg(V + (int64_t)(k0 + k) * r + j) : 0.f;
            }
        }
    };
    auto store = [&](int b, const float4 (&xa)[2], const float4 &wa, const float (&vr)[VPT > 0 ? VPT : 1]) {
        float *As = smf + b * STAGE_F, *Bs = As + kGBK * AS, *Vs = Bs + kGBK * BS;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int kk = kq + 8 * h;
            As[(kk + 0) * AS + lr] = xa[h].x;
            As[(kk + 1) * AS + lr] = xa[h].y;
            As[(kk + 2) * AS + lr] = xa[h].z;
            As[(kk + 3) * AS + lr] = xa[h].w;
        }
        Bs[(wq + 0) * BS + wr] = wa.x;
        Bs[(wq + 1) * BS + wr] = wa.y;
        Bs[(wq + 2) * BS + wr] = wa.z;
        Bs[(wq + 3) * BS + wr] = wa.w;
        if (ZTN > 0) {
#pragma unroll
            for (int u = 0; u < VPT; ++u) {
                const int e = tid + 256 * u, k = e / RP, j = e - k * RP;
                if (e < kGBK * RP) Vs[k * VSS + j] = vr[u];
            }
        }
    };

    float4 xa[2], wa;
    float vr[VPT > 0 ? VPT : 1];
    load(0, xa, wa, vr);
    store(0, xa, wa, vr);
    __syncthreads();
    int b = 0;
    for (int k0 = 0; k0 < in; k0 += kGBK) {
        const bool more = k0 + kGBK < in;
        if (more) load(k0 + kGBK, xa, wa, vr);
        const float *As = smf + b * STAGE_F, *Bs = As + kGBK * AS, *Vs = Bs + kGBK * BS;
#pragma unroll
        for (int k = 0; k < kGBK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4 *>(As + k * AS + ty * 8);
            const float4 a1 = *reinterpret_cast<const float4 *>(As + k * AS + ty * 8 + 4);
            const float4 b0 = *reinterpret_cast<const float4 *>(Bs + k * BS + tx * 4);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[4] = {b0.x, b0.y, b0.z, b0.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
            if (ZTN > 0) {
#pragma unroll
                for (int j = 0; j < ZTN; ++j) {
                    const float zv = Vs[k * VSS + tx * ZTN + j];
#pragma unroll
                    for (int i = 0; i < 8; ++i) zacc[i][j] = fmaf(av[i], zv, zacc[i][j]);
                }
            }
        }
        if (more) store(b ^ 1, xa, wa, vr);
        __syncthreads();
        b ^= 1;
    }

    // z of the tile's tokens, then y = s * acc + U z
    float(*zs)[ZS] = reinterpret_cast<float(*)[ZS]>(smf);
    if (ZTN > 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < ZTN; ++j) zs[ty * 8 + i][tx * ZTN + j] = zacc[i][j];
        __syncthreads();
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int o = o0 + tx * 4 + j;
        if (o >= out) continue;
        const float sv = sg.s[o];
        const float *Ur = sg.U + (int64_t)o * r;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int tl = ty * 8 + i, t = t0 + tl;
            if (t >= T) continue;
            float v = sv * acc[i][j];
            if (ZTN > 0)
                for (int k = 0; k < r; ++k) v = fmaf(Ur[k], zs[tl][k], v);
            store_out(sg.y, a.ydt, (int64_t)t * out + o, v);
        }
    }
}

typedef void (*f32_fn)(F32Args);

// ranks up to 64 (above, the tiled form: the z stash of 128 tokens would
// not fit the static shared memory)
static f32_fn pick_gemm(int r)
{
    if (r == 0) return f32_gemm_kernel<0>;
    if (r <= 16) return f32_gemm_kernel<1>;
    if (r <= 32) return f32_gemm_kernel<2>;
    if (r <= 64) return f32_gemm_kernel<4>;
    return nullptr;
}

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
    // few tokens: the weight-streaming form (16-byte rows: in a multiple of 4)
    const f32_dec_fn dfn = (in % 4 == 0) ? pick_dec(T, r) : nullptr;
    if (dfn) {
        F32Args a = {};
        a.x = x;
        a.T = (int)T;
        a.in = (int)in;
        a.r = (int)r;
        a.ydt = ydt;
        a.nseg = nproj;
        int ncl = 0;
        for (int j = 0; j < nproj; ++j) {
            F32Seg &sg = a.seg[j];
            sg.W0 = proj[j].W0;
            sg.s = proj[j].s;
            sg.U = proj[j].U;
            sg.V = proj[j].V;
            sg.y = y[j];
            sg.out = (int)proj[j].out;
            sg.nt0 = ncl;
            ncl += (int)((proj[j].out + kF32DecRows * kF32DecCl - 1) / (kF32DecRows * kF32DecCl));
        }
        dfn<<<ncl * kF32DecCl, 256, 0, st>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "fp32 decode launch");
        return WL_OK;
    }
    const bool small = T <= 16;
    const bool gemm = !small && r <= 64;
    const int BM = small ? 16 : gemm ? kGBM : 64, BN = small ? 32 : gemm ? kGBN : 128;
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
    const f32_fn fn = small ? pick_rank<16, 32, 32, 1, 2>((int)r)
                            : gemm ? pick_gemm((int)r) : pick_rank<64, 128, 16, 4, 8>((int)r);
    fn<<<grid, 256, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "fp32 linear launch");
    return WL_OK;
}

}  // namespace wl
