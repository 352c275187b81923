// materialize.cu -- W_eff = s*W0 + U V^T, formed once ("Serve and generate
// with weightless", "Set the fast path on NVIDIA": the effective weight is
// materialised at load time and every projection becomes one dense matmul).
//
// Bit-exact contract, per element (the pages give no order; this one is the
// library's):
//     d = +0; for k = 0..r-1 ascending: d = fma(U[o,k], V[i,k], d)
//     w = fl(s[o] * W0[o,i]); if r > 0: w = fl(w + d)
// and, for a bf16 result, one round-to-nearest-even.  The tensor cores are
// not used: their accumulation order is not this one.
//
// Tiling: a CTA owns a 32 x 256 tile of W_eff (4 rows x 8 columns per
// thread, 80 registers, three CTAs per SM: with 64-row tiles and 127 registers
// only two fit, and an SM's HBM requests stall between one CTA's loads and the
// next's).  Each thread loads its W0 chunks before anything else, so that
// their HBM round trip overlaps the rank-r work.  U and V are staged through
// shared memory in chunks of 32 ranks (read row-major, coalesced; stored
// transposed, so each k step reads one float4 pair of V and of U), which keeps
// the rank-r operands out of HBM after their first read: V is re-read once
// per 32 output rows, U once per 256 input columns, both from L2.
#include "wl_internal.cuh"

namespace wl {

constexpr int kMatRowsPerThread = 4;
constexpr int kMatRows = 8 * kMatRowsPerThread;  // tile rows: 8 row groups of the thread's rows
constexpr int kMatCols = 256;
constexpr int kMatK = 32;
constexpr int kUStr = kMatRows + 4;  // padded row strides (floats), multiples of 4
constexpr int kVStr = kMatCols + 4;

template <int F32OUT>
__global__ void __launch_bounds__(kThreads, 3) materialize_kernel(
    const bf16 *__restrict__ W0, const float *__restrict__ s, const bf16 *__restrict__ U,
    const bf16 *__restrict__ V, void *__restrict__ Weff, int out, int in, int r)
{
    __shared__ __align__(16) float Us[kMatK * kUStr];
    __shared__ __align__(16) float Vs[kMatK * kVStr];
    const int o_base = blockIdx.y * kMatRows;
    const int i_base = blockIdx.x * kMatCols;
    const int tr = threadIdx.x >> 5;  // rows o_base + tr*RPT .. +RPT-1
    const int tc = threadIdx.x & 31;  // cols i_base + tc*8 .. +7
    const int i0 = i_base + tc * 8;
    const bool col_ok = i0 < in;      // in % 8 == 0: a chunk of 8 columns is all in or all out

    // the thread's W0 chunks and row scales first: their round trips overlap
    // the staging of U and V and the rank-r products (loaded later, inside the
    // row loop with its early exit, the scales would cost one round trip per row)
    constexpr int RPT = kMatRowsPerThread;
    uint4 wv[RPT];
    float sv[RPT];
#pragma unroll
    for (int a = 0; a < RPT; ++a) {
        const int o = o_base + tr * RPT + a;
        const bool ok = col_ok && o < out;
        wv[a] = ok ? *reinterpret_cast<const uint4 *>(W0 + (int64_t)o * in + i0) : make_uint4(0u, 0u, 0u, 0u);
        sv[a] = ok ? s[o] : 0.f;
    }

    float d[RPT][8];
#pragma unroll
    for (int a = 0; a < RPT; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) d[a][b] = 0.0f;

    for (int k0 = 0; k0 < r; k0 += kMatK) {
        const int kn = min(kMatK, r - k0);
        // U rows o_base.., ranks k0..k0+kn-1, and V rows i_base.., the same
        // ranks, walked in row-major order: consecutive threads read
        // consecutive ranks of a row, then the next row
        for (int e = threadIdx.x; e < kMatRows * kn; e += kThreads) {
            const int o = e / kn, k = e - o * kn;
            Us[k * kUStr + o] = o_base + o < out ? bf2f(U[(int64_t)(o_base + o) * r + k0 + k]) : 0.f;
        }
        for (int e = threadIdx.x; e < kMatCols * kn; e += kThreads) {
            const int i = e / kn, k = e - i * kn;
            Vs[k * kVStr + i] = i_base + i < in ? bf2f(V[(int64_t)(i_base + i) * r + k0 + k]) : 0.f;
        }
        __syncthreads();
        for (int k = 0; k < kn; ++k) {
            const float4 u0 = *reinterpret_cast<const float4 *>(Us + k * kUStr + tr * RPT);
            const float4 v0 = *reinterpret_cast<const float4 *>(Vs + k * kVStr + tc * 8);
            const float4 v1 = *reinterpret_cast<const float4 *>(Vs + k * kVStr + tc * 8 + 4);
            const float uu[4] = {u0.x, u0.y, u0.z, u0.w};
            const float vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int a = 0; a < RPT; ++a)
#pragma unroll
                for (int b = 0; b < 8; ++b) d[a][b] = __fmaf_rn(uu[a], vv[b], d[a][b]);
        }
        __syncthreads();
    }

    if (!col_ok) return;
#pragma unroll
    for (int a = 0; a < RPT; ++a) {
        const int o = o_base + tr * RPT + a;
        if (o >= out) break;
        const float w0[8] = {bf_lo(wv[a].x), bf_hi(wv[a].x), bf_lo(wv[a].y), bf_hi(wv[a].y),
                             bf_lo(wv[a].z), bf_hi(wv[a].z), bf_lo(wv[a].w), bf_hi(wv[a].w)};
        float w[8];
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            w[b] = __fmul_rn(sv[a], w0[b]);
            if (r > 0) w[b] = __fadd_rn(w[b], d[a][b]);
        }
        if (F32OUT) {
            float *dst = static_cast<float *>(Weff) + (int64_t)o * in + i0;
            reinterpret_cast<float4 *>(dst)[0] = make_float4(w[0], w[1], w[2], w[3]);
            reinterpret_cast<float4 *>(dst)[1] = make_float4(w[4], w[5], w[6], w[7]);
        } else {
            uint32_t p[4];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(w[2 * b], w[2 * b + 1]);
                p[b] = *reinterpret_cast<const uint32_t *>(&h2);
            }
            bf16 *dst = static_cast<bf16 *>(Weff) + (int64_t)o * in + i0;
            *reinterpret_cast<uint4 *>(dst) = make_uint4(p[0], p[1], p[2], p[3]);
        }
    }
}

wl_status launch_materialize(const bf16 *W0, const float *s, const bf16 *U, const bf16 *V,
                             void *W_eff, int64_t out, int64_t in, int64_t r, int dt,
                             cudaStream_t st)
{
    const dim3 grid((unsigned)((in + kMatCols - 1) / kMatCols),
                    (unsigned)((out + kMatRows - 1) / kMatRows));
    if (grid.y > 65535u) return fail(WL_ERR_UNSUPPORTED, "materialize: out too large (%lld)", (long long)out);
    if (dt == WL_OUT_F32)
        materialize_kernel<1><<<grid, kThreads, 0, st>>>(W0, s, U, V, W_eff, (int)out, (int)in, (int)r);
    else
        materialize_kernel<0><<<grid, kThreads, 0, st>>>(W0, s, U, V, W_eff, (int)out, (int)in, (int)r);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "materialize launch");
    return WL_OK;
}

}  // namespace wl
