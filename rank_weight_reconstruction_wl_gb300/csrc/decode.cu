// decode.cu -- decode-size (small T) weightless projections.
//
// Computes, for each output row o of a projection ("In-kernel
// reconstruction", formula section):
//     y[t,o] = s[o] * sum_i W0[o,i] x[t,i] + sum_k U[o,k] z[t,k],
//     z[t,k] = sum_i V[i,k] x[t,i]
// in ONE launch per call: W0 is streamed from HBM exactly once, z is formed in
// the same launch, and the scale and the rank-r delta are applied in the
// epilogue.  At decode sizes the cost is the HBM stream of W0.
//
// CTA organisation (288 threads):
//   warp 8      producer: one thread streams W0 as 64-row x 64-column tiles
//               (TMA 2D, 128-byte swizzle) into a ring of shared-memory stages
//               (two tiles = 16 KB per stage), each completed by an mbarrier
//               transaction count.  It waits only for a free stage, so HBM
//               stays busy through the consumers' synchronisation points.
//   warps 0..7  consumers: stage x, form z over their K range, then multiply
//               each stage on the tensor cores (mma.sync m16n8k16, bf16 in,
//               fp32 accumulate) with the W0 rows as the M side and the tokens
//               as the N side (8 columns per n-tile), and run the epilogue.
//               One tensor-core instruction covers 16 rows x 16 columns of W0,
//               which keeps the consumers well ahead of the HBM stream.
//
// Work split.  Output rows are cut into groups of 64-row tiles; a group is
// handled by a thread-block cluster of KS CTAs that split the input dimension
// K.  Every CTA computes over its K range
//     p[t,o] = s[o] * sum_{i in range} W0[o,i] x[t,i] + sum_k U[o,k] z_range[t,k]
// (both terms are linear in the split, so the ranges add up to y).  The KS
// partials are added through distributed shared memory in a fixed rank order
// (deterministic, no atomics, no scratch memory); readiness is signalled with
// remote mbarrier arrivals, so the producer warp never joins a cluster barrier.
//
// The fused GeGLU MLP ("In-kernel reconstruction", custom-op path: gate, up,
// activation and down in one dispatch) is one call made of two launches
// chained by programmatic dependent launch: the first forms h = gelu(g)*u and
// partial sums of z_down = h V_down; the second streams W_down from the moment
// its CTAs are resident and reads h once the first launch has finished.  (A
// single persistent launch would need every CTA resident at once for a grid
// barrier; with overlapping launches that is not guaranteed.)  The second
// launch takes h as a pair of bf16 columns per token (hi and lo parts), so its
// tensor-core product keeps fp32 accuracy.
//
// Launches use programmatic dependent launch: a kernel lets the next one on
// the stream start once all its CTAs run; the next kernel's producer streams
// weights at once, and its consumers wait (griddepcontrol.wait) for the
// previous kernel to finish before reading its input or writing any output.
#include <cooperative_groups.h>

#include <algorithm>
#include <mutex>
#include <unordered_map>

#include "dec_ptx.cuh"

namespace cg = cooperative_groups;

namespace wl {

constexpr int kDecThreads = kThreads + 32;  // 8 consumer warps + 1 producer warp
constexpr int kBR = 64;                     // W0 rows per tile
constexpr int kBK = 64;                     // W0 columns per TMA box (128 bytes)
constexpr int kBoxBytes = kBR * kBK * 2;    // 8 KB
constexpr int kStageBytes = 2 * kBoxBytes;  // two boxes (k-tiles) per ring stage
constexpr int kTokChunk = 8;                // tokens per pass of the rank-r helpers

// ------------------------------------------------------------------------
// Rank-r helpers (consumer threads 0..255)
// ------------------------------------------------------------------------

// How 8 consecutive rank values of a row can be loaded: 2 = one 16-byte
// load, 1 = two 8-byte loads, 0 = element by element.
__device__ __forceinline__ int vec_mode(const bf16 *p, int r)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    if (r % 8 == 0 && a % 16 == 0) return 2;
    if (r % 4 == 0 && a % 8 == 0) return 1;
    return 0;
}

// v[e] = M[i*r + kc + e] as fp32 for e < 8 (0 where kc + e >= r); M may be in
// global or shared memory.
__device__ __forceinline__ void load8(const bf16 *__restrict__ M, int64_t i, int r, int kc, int vm,
                                      float v[8])
{
    const bf16 *p = M + i * r + kc;
    if (vm == 2) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        v[0] = bf_lo(u.x); v[1] = bf_hi(u.x); v[2] = bf_lo(u.y); v[3] = bf_hi(u.y);
        v[4] = bf_lo(u.z); v[5] = bf_hi(u.z); v[6] = bf_lo(u.w); v[7] = bf_hi(u.w);
    } else if (vm == 1) {
        const uint2 a = *reinterpret_cast<const uint2 *>(p);
        const uint2 b = (kc + 4 < r) ? *reinterpret_cast<const uint2 *>(p + 4) : make_uint2(0u, 0u);
        v[0] = bf_lo(a.x); v[1] = bf_hi(a.x); v[2] = bf_lo(a.y); v[3] = bf_hi(a.y);
        v[4] = bf_lo(b.x); v[5] = bf_hi(b.x); v[6] = bf_lo(b.y); v[7] = bf_hi(b.y);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = (kc + e < r) ? bf2f(p[e]) : 0.f;
    }
}

// Warp reduce-scatter of 8 values: returns, in lane l, the sum over all 32
// lanes of value index l >> 2 (9 shuffles instead of 40).
__device__ __forceinline__ float warp_reduce8(const float v[8])
{
    const int lane = threadIdx.x & 31;
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float a[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float send = b4 ? v[j] : v[j + 4];
        const float keep = b4 ? v[j + 4] : v[j];
        a[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
    float c[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float send = b3 ? a[j] : a[j + 2];
        const float keep = b3 ? a[j + 2] : a[j];
        c[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    const float send = b2 ? c[0] : c[1];
    const float keep = b2 ? c[1] : c[0];
    float d = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    d += __shfl_xor_sync(0xffffffffu, d, 2);
    d += __shfl_xor_sync(0xffffffffu, d, 1);
    return d;
}

// Coalesced x V for r = 8*RG ranks, RG a power of two up to 16 (16-byte
// aligned V): a CTA's V slice [n][r] is one contiguous block, read as 16-byte
// chunks with thread tid on rank group g = tid % RG (8 ranks) of rows
// tid / RG, tid / RG + kThreads / RG, ...; a warp's loads then cover whole
// 128-byte lines.  Returns RG, or 0 where the layout does not allow it.
__device__ __forceinline__ int zlin_groups(const bf16 *V, int r)
{
    const int RG = r >> 3;
    const bool ok = r > 0 && (r & 7) == 0 && RG <= 16 && (RG & (RG - 1)) == 0 &&
                    (reinterpret_cast<uintptr_t>(V) & 15) == 0;
    return ok ? RG : 0;
}

__device__ __forceinline__ void unpack8(const uint4 u, float v[8])
{
    v[0] = bf_lo(u.x); v[1] = bf_hi(u.x); v[2] = bf_lo(u.y); v[3] = bf_hi(u.y);
    v[4] = bf_lo(u.z); v[5] = bf_hi(u.z); v[6] = bf_lo(u.w); v[7] = bf_hi(u.w);
}

// p[t][e] += src(t, i) * V[i*r + 8g + e] over this thread's rows i in
// [i0, i1) (lg = log2 RG); tid, nthr: this thread's index among the nthr
// threads that share the work.
template <int TT, int UR, typename Src>
__device__ __forceinline__ void zlin_rows(Src src, const uint4 *__restrict__ Vq, int RG, int lg, int i0, int i1,
                                          float p[TT][8], int tid, int nthr)
{
    const int g = tid & (RG - 1);
#pragma unroll UR
    for (int i = i0 + (tid >> lg); i < i1; i += nthr >> lg) {
        float v[8];
        unpack8(Vq[(int64_t)i * RG + g], v);
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            const float xv = src(t, i);
#pragma unroll
            for (int e = 0; e < 8; ++e) p[t][e] = fmaf(xv, v[e], p[t][e]);
        }
    }
}

// out[t*ostride + 8g + e] = the sum of p[t][e] over the threads of rank group
// g: a butterfly over the lanes of a group, then the warps' sums in a fixed
// order through zred (512 floats), 64 ranks at a time.  Contains consumer
// barriers.
template <int TT>
__device__ __forceinline__ void zlin_finish(float p[TT][8], int RG, int r, float *out, int ostride, float *zred)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int off = RG; off < 32; off <<= 1)
#pragma unroll
        for (int t = 0; t < TT; ++t)
#pragma unroll
            for (int e = 0; e < 8; ++e) p[t][e] += __shfl_xor_sync(0xffffffffu, p[t][e], off);
#pragma unroll
    for (int t = 0; t < TT; ++t)
        for (int kb = 0; kb < r; kb += 64) {
            if (lane < RG && 8 * lane >= kb && 8 * lane < kb + 64)
#pragma unroll
                for (int e = 0; e < 8; ++e) zred[warp * 64 + 8 * lane - kb + e] = p[t][e];
            consumer_sync();
            if (threadIdx.x < min(64, r - kb)) {
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) sum += zred[w * 64 + threadIdx.x];
                out[t * ostride + kb + threadIdx.x] = sum;
            }
            consumer_sync();
        }
}

// One token, r <= 64 (RG <= 8): the warp's sums of p over the lanes of each
// rank group, stored as part[8*g + e] (64 floats per warp).
__device__ __forceinline__ void zlin_warp_store(float p[1][8], int RG, float *part)
{
    const int lane = threadIdx.x & 31;
    for (int off = RG; off < 32; off <<= 1)
#pragma unroll
        for (int e = 0; e < 8; ++e) p[0][e] += __shfl_xor_sync(0xffffffffu, p[0][e], off);
    if (lane < RG)
#pragma unroll
        for (int e = 0; e < 8; ++e) part[8 * lane + e] = p[0][e];
}

// out[t*ostride + k] = sum_{i < n} src(t, i) * V[i*r + k] for t < TT,
// k < r (out may be shared or global memory).  The coalesced form above where
// the layout allows it; otherwise one thread per row i of V, eight ranks per
// load, partial sums reduced across the warp, then across warps in shared
// memory (zred: 512 floats).  Contains consumer barriers.
template <int TT, typename Src>
__device__ __forceinline__ void block_xV(Src src, int n, const bf16 *__restrict__ V, int r,
                                         float *out, int ostride, float *zred)
{
    constexpr int UR = TT == 1 ? 8 : TT <= 2 ? 4 : 1;  // rows in flight (registers)
    const int RG = zlin_groups(V, r);
    if (RG) {
        float p[TT][8];
#pragma unroll
        for (int t = 0; t < TT; ++t)
#pragma unroll
            for (int e = 0; e < 8; ++e) p[t][e] = 0.f;
        zlin_rows<TT, UR>(src, reinterpret_cast<const uint4 *>(V), RG, __ffs(RG) - 1, 0, n, p, threadIdx.x,
                          kThreads);
        zlin_finish<TT>(p, RG, r, out, ostride, zred);
        return;
    }
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int vm = vec_mode(V, r);
    for (int kc = 0; kc < r; kc += 8) {
        float p[TT][8];
#pragma unroll
        for (int t = 0; t < TT; ++t)
#pragma unroll
            for (int e = 0; e < 8; ++e) p[t][e] = 0.f;
#pragma unroll UR
        for (int i = tid; i < n; i += kThreads) {
            float v[8];
            load8(V, i, r, kc, vm, v);
#pragma unroll
            for (int t = 0; t < TT; ++t) {
                const float xv = src(t, i);
#pragma unroll
                for (int e = 0; e < 8; ++e) p[t][e] = fmaf(xv, v[e], p[t][e]);
            }
        }
#pragma unroll
        for (int t = 0; t < TT; ++t) {
            const float sum = warp_reduce8(p[t]);
            if ((lane & 3) == 0) zred[(warp * TT + t) * 8 + (lane >> 2)] = sum;
        }
        consumer_sync();
        for (int idx = tid; idx < TT * 8; idx += kThreads) {
            const int t = idx >> 3, j = idx & 7;
            if (kc + j < r) {
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) sum += zred[(w * TT + t) * 8 + j];
                out[t * ostride + kc + j] = sum;
            }
        }
        consumer_sync();
    }
}

// y[t] += sum_k U[o*r + k] * z[t*zs + k], t < TT (loads of eight ranks at a
// time, issued ahead of their use).
template <int TT>
__device__ __forceinline__ void add_delta(const bf16 *__restrict__ U, int64_t o, int r, int vm,
                                          const float *z, int zs, float yv[TT])
{
    // at few tokens every rank group's load is issued before the first
    // multiply (the loop is latency-bound: U is read once, cold)
    constexpr int UR = TT <= 2 ? 8 : 2;
#pragma unroll UR
    for (int kc = 0; kc < r; kc += 8) {
        float u[8];
        load8(U, o, r, kc, vm, u);
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (kc + e < r)
#pragma unroll
                for (int t = 0; t < TT; ++t) yv[t] = fmaf(u[e], z[t * zs + kc + e], yv[t]);
    }
}

// ------------------------------------------------------------------------
// Ring of 16 KB stages shared by the producer thread and the consumer warps
// ------------------------------------------------------------------------
struct Ring {
    char *base;       // nst stages of kStageBytes, 1024-byte aligned
    uint64_t *full;   // [nst]: producer -> consumers (transaction bytes)
    uint64_t *empty;  // [nst]: consumers -> producer (one arrival per consumer warp)
    int nst;
    int s;            // current stage
    unsigned ph;      // parity of the current pass over the ring
    __device__ __forceinline__ void advance()
    {
        if (++s == nst) {
            s = 0;
            ph ^= 1u;
        }
    }
};

// Producer (one thread): rows [row0, row0 + 64) x columns [k0, k0 + 64*ktiles)
// of `map`, two 64x64 boxes per stage.  Rows or columns past the matrix are
// filled with zeros by the TMA unit.  blk: `map` is the k-block view (K a
// multiple of 64), and one copy fills the stage: a TMA copy costs a fixed few
// hundred ns, so two 8 KB copies per stage would hold the stream to about 60 %
// of HBM.  An odd last tile then also loads the next 64 columns, which the
// consumers skip.
__device__ __forceinline__ bool produce_tile(Ring &rg, const CUtensorMap *map, int row0, int k0,
                                             int ktiles, unsigned *status, bool blk)
{
    for (int kt = 0; kt < ktiles; kt += 2) {
        if (!mbar_wait(&rg.empty[rg.s], rg.ph ^ 1u, status, kWaitRingEmpty)) return false;
        char *dst = rg.base + (size_t)rg.s * kStageBytes;
        if (blk) {
            mbar_expect_tx(&rg.full[rg.s], (unsigned)kStageBytes);
            tma_load_3d(dst, map, 0, row0, k0 / kBK + kt, &rg.full[rg.s]);
        } else {
            const int nb = min(2, ktiles - kt);
            mbar_expect_tx(&rg.full[rg.s], (unsigned)(nb * kBoxBytes));
            for (int b = 0; b < nb; ++b)
                tma_load_2d(dst + b * kBoxBytes, map, k0 + (kt + b) * kBK, row0, &rg.full[rg.s]);
        }
        rg.advance();
    }
    return true;
}

// Consumers: the tile's stages on the tensor cores.  KW = 2: warps 0-7, warp w
// owns rows 16*(w&3) .. +15 of the tile and the k-steps of parity (w>>2) of
// each stage; the two warps of a row group are added at the end (consumer
// barriers).  KW = 1: warps 0-3 only, warp w owns rows 16*w .. +15 and all
// eight k-steps of each stage (no barrier; the ring's empty barriers then
// count four arrivals).  xb: the tile's x as
// bf16 pairs, row n (token) at xb + n*xs32 (u32 units) for n < nx, column 0 =
// the CTA's k0, zero past its K range; the MMA columns n >= nx are zeros that
// are not stored (at one token x takes an eighth of the shared memory).
// acc[row*ald + n] receives the raw dot products of the 64 rows with the 8*NT
// columns.  red: 512*NT floats.
template <int NT, int KW = 2>
__device__ __forceinline__ bool consume_tile(Ring &rg, int ktiles, const uint32_t *xb, int xs32, int nx,
                                             float *red, float *acc, int ald, unsigned *status)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rw = warp & 3, kw = KW == 2 ? warp >> 2 : 0;
    const int g = lane >> 2, t4 = lane & 3;
    float c[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) c[nt][0] = c[nt][1] = c[nt][2] = c[nt][3] = 0.f;
    // ldmatrix row/chunk of this lane (swizzled 128-byte rows)
    const int lrow = rw * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int lchunk = lane >> 4;
    // B operands (token rows of x) by shared address
    const uint32_t xb_ln = smem_u32(xb) + (uint32_t)((g * xs32 + t4) * 4);
    bool ok = true;
    for (int kt = 0; kt < ktiles; kt += 2) {
        int w_ok = 1;
        if (lane == 0) w_ok = mbar_wait(&rg.full[rg.s], rg.ph, status, kWaitRingFull);
        w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
        if (!w_ok) {
            ok = false;
            break;
        }
        const uint32_t sb = smem_u32(rg.base + (size_t)rg.s * kStageBytes);
        // the stage's fragments first (A of four k steps of this warp, then
        // their B words), then the MMAs; KW = 1 takes two such passes
#pragma unroll
        for (int h = 0; h < 8 / KW; h += 4) {
        uint32_t a[4][4], bw[4][NT][2];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int step = KW == 2 ? kw + 2 * q : h + q;  // 0..7 within the stage
            const int box = step >> 2;      // which 64-column box
            const int kin = step & 3;       // 16-column step inside the box
            if (kt + box >= ktiles) continue;
            const int chunk = kin * 2 + lchunk;
            ldmatrix_x4(a[q], sb + box * kBoxBytes + lrow * 128 + ((chunk ^ (lrow & 7)) << 4));
            const int kk = (kt + box) * kBK + kin * 16;  // column relative to k0
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint32_t xa = xb_ln + (uint32_t)((nt * 8 * xs32 + (kk >> 1)) * 4);
                const bool v = nt * 8 + g < nx;
                bw[q][nt][0] = v ? lds_u32(xa) : 0u;
                bw[q][nt][1] = v ? lds_u32(xa + 16) : 0u;
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int box = (KW == 2 ? kw + 2 * q : h + q) >> 2;
            if (kt + box >= ktiles) continue;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_16816(c[nt], a[q], bw[q][nt][0], bw[q][nt][1]);
        }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&rg.empty[rg.s]);
        rg.advance();
    }
    if (KW == 1) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int row = rw * 16 + g, col = nt * 8 + 2 * t4;
            acc[row * ald + col] = c[nt][0];
            acc[row * ald + col + 1] = c[nt][1];
            acc[(row + 8) * ald + col] = c[nt][2];
            acc[(row + 8) * ald + col + 1] = c[nt][3];
        }
        return ok;
    }
    // add the two k-halves of every row group and store
    if (kw == 1) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) red[((rw * NT + nt) * 4 + e) * 32 + lane] = c[nt][e];
    }
    consumer_sync();
    if (kw == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) c[nt][e] += red[((rw * NT + nt) * 4 + e) * 32 + lane];
            const int row = rw * 16 + g, col = nt * 8 + 2 * t4;
            acc[row * ald + col] = c[nt][0];
            acc[row * ald + col + 1] = c[nt][1];
            acc[(row + 8) * ald + col] = c[nt][2];
            acc[(row + 8) * ald + col + 1] = c[nt][3];
        }
    }
    consumer_sync();
    return ok;
}

// Deterministic cluster reduction of per-CTA partials held in shared memory.
// publish: all CTAs signal every peer, then wait until every peer signalled.
// release: after reading the peers' partials, tell every peer.
// reclaim: before the CTA exits, wait until every peer has released it.
struct Exchange {
    uint64_t *ready;
    uint64_t *done;
};

__device__ __forceinline__ void exchange_publish(const Exchange &ex, int KS, unsigned *status)
{
    cluster_wait();  // every CTA of the cluster has initialised its barriers
    consumer_sync();
    if (threadIdx.x == 0)
        for (int p = 0; p < KS; ++p) mbar_arrive_remote(ex.ready, (unsigned)p);
    mbar_wait_cluster(ex.ready, 0, status);
}

__device__ __forceinline__ void exchange_release(const Exchange &ex, int KS)
{
    consumer_sync();
    if (threadIdx.x == 0)
        for (int p = 0; p < KS; ++p) mbar_arrive_remote(ex.done, (unsigned)p);
}

__device__ __forceinline__ void exchange_reclaim(const Exchange &ex, unsigned *status)
{
    mbar_wait_cluster(ex.done, 0, status);
}

// Shared memory: ring (1024-byte aligned) | barriers | floats.
struct Carve {
    Ring rg;
    Exchange ex;
    char *rest;  // 16-byte aligned, after the barriers
};

__host__ __device__ constexpr int carve_head_bytes(int nst) { return 1024 + nst * kStageBytes + (2 * nst + 2) * 8 + 16; }

__device__ __forceinline__ Carve carve(char *smem_raw, int nst)
{
    // 128-byte swizzled TMA tiles want 1024-byte aligned stages
    char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Carve c;
    c.rg.base = smem;
    c.rg.nst = nst;
    c.rg.s = 0;
    c.rg.ph = 0;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)nst * kStageBytes);
    c.rg.full = bars;
    c.rg.empty = bars + nst;
    c.ex.ready = bars + 2 * nst;
    c.ex.done = bars + 2 * nst + 1;
    c.rest = reinterpret_cast<char *>(bars + 2 * nst + 2);
    c.rest = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(c.rest) + 15) & ~uintptr_t(15));
    return c;
}

// cw: consumer warps that release each ring stage
__device__ __forceinline__ void init_barriers(Carve &c, int KS, int cw = kWarps)
{
    for (int i = 0; i < c.rg.nst; ++i) {
        mbar_init(&c.rg.full[i], 1);
        mbar_init(&c.rg.empty[i], cw);
    }
    mbar_init(c.ex.ready, KS);
    mbar_init(c.ex.done, KS);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// x[t, k0:k0+klen) (bf16, row stride ld) -> xb rows (bf16, xs32 u32 per row),
// width 64*ktiles (zero past klen); rows T <= t < nrow zero.
__device__ __forceinline__ void stage_x(const bf16 *__restrict__ x, int64_t ld, int T, int k0, int klen,
                                        int width, int nrow, uint32_t *xb, int xs32)
{
    const int nq = width >> 3;  // 16-byte chunks per row
    for (int idx = threadIdx.x; idx < nrow * nq; idx += kThreads) {
        const int t = idx / nq, c = idx - t * nq;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (t < T && 8 * c < klen) v = *reinterpret_cast<const uint4 *>(x + t * ld + k0 + 8 * c);
        *reinterpret_cast<uint4 *>(xb + t * xs32 + 4 * c) = v;
    }
}

// ------------------------------------------------------------------------
// wl_linear / wl_qkv_fused decode kernel
// ------------------------------------------------------------------------
struct DecSeg {
    CUtensorMap map;  // W0 [out, in], box 64 x 64
    const float *s;
    const bf16 *U;
    const bf16 *V;
    void *y;
    int out;
    int grp0;  // first row group of this segment
    int ngrp;  // row groups of this segment
};

struct DecArgs {
    DecSeg seg[3];
    const bf16 *x;
    int T, in, r, ydt;
    int KS, Kc;  // K splits (= cluster size), K elements per split (multiple of 64)
    int tpc;     // 64-row tiles per row group
    int nseg, nst, xs32;
    int vbuf, ubuf;  // shared-memory bytes for the prefetched V slice and U rows (0: read in place)
    int blk;  // 1: the W0 maps are k-block views (one 16 KB copy per ring stage)
    unsigned *status;
};

// ZW (one token, r = 8*RG <= 64, RG a power of two, V 16-byte aligned):
// warps 0-3 stream W0 while warps 4-7 form z = x V over the CTA's K range, so
// the rank-r reads overlap the W0 stream instead of following it.
template <int NT, int TC, bool ZW = false>
__global__ void __launch_bounds__(kDecThreads, 2) dec_linear_kernel(const __grid_constant__ DecArgs a)
{
    extern __shared__ __align__(1024) char smem_raw[];
    const int KS = a.KS;
    const int q = (int)(blockIdx.x % (unsigned)KS);
    const int gi = (int)(blockIdx.x / (unsigned)KS);
    const int si = (a.nseg > 2 && gi >= a.seg[2].grp0) ? 2 : (a.nseg > 1 && gi >= a.seg[1].grp0) ? 1 : 0;
    const DecSeg &sg = a.seg[si];
    const int r0 = (gi - sg.grp0) * a.tpc * kBR;
    const int nrows = min(sg.out - r0, a.tpc * kBR);
    const int ntl = (nrows + kBR - 1) / kBR;
    const int k0 = q * a.Kc;
    const int klen = max(0, min(a.in, k0 + a.Kc) - k0);
    const int ktiles = (klen + kBK - 1) / kBK;
    const int rp = a.r > 0 ? a.r : 1;
    constexpr int ald = 8 * NT;

    Carve c = carve(smem_raw, a.nst);
    uint32_t *xb = reinterpret_cast<uint32_t *>(c.rest);
    float *acc = reinterpret_cast<float *>(xb + a.T * a.xs32);  // x: T rows
    float *red = acc + a.tpc * kBR * ald;
    float *zp = red + 512 * NT;  // [ceil8(T)][rp]
    float *zred = zp + ((a.T + 7) / 8) * 8 * rp;
    char *sbuf = reinterpret_cast<char *>(zred + 512);
    char *vbuf = sbuf + a.tpc * kBR * 4 + 16;
    char *ubuf = vbuf + a.vbuf;

    if (threadIdx.x == 0) {
        init_barriers(c, KS, ZW ? 4 : kWarps);
        pdl_trigger();
    }
    __syncthreads();           // barriers initialised (this CTA)
    if (KS > 1) cluster_arrive();  // peers may arrive remotely once all have passed this

    if (threadIdx.x >= kThreads) {  // ---------------- producer thread
        if (threadIdx.x == kThreads && ktiles > 0)
            for (int tl = 0; tl < ntl; ++tl)
                if (!produce_tile(c.rg, &sg.map, r0 + tl * kBR, k0, ktiles, a.status, a.blk)) break;
        return;
    }

    // ------------------------------------------------ consumer warps
    // weight-side operands first (they do not depend on the previous kernel),
    // so their round trips overlap the x load and the W0 stream
    const float *sv_p = reinterpret_cast<const float *>(prefetch(sbuf, sg.s + r0, nrows * 4));
    const bf16 *Vp = sg.V + (int64_t)k0 * a.r;
    const bf16 *Up = sg.U + (int64_t)r0 * a.r;
    if (a.r > 0 && a.vbuf > 0) Vp = reinterpret_cast<const bf16 *>(prefetch(vbuf, Vp, klen * a.r * 2));
    if (a.r > 0 && a.ubuf > 0) Up = reinterpret_cast<const bf16 *>(prefetch(ubuf, Up, nrows * a.r * 2));
    pdl_wait();  // x comes from the previous kernel on the stream
    stage_x(a.x, a.in, a.T, k0, klen, ktiles * kBK, a.T, xb, a.xs32);
    consumer_sync();
    const bf16 *xbh = reinterpret_cast<const bf16 *>(xb);
    const int xsh = 2 * a.xs32;
    if constexpr (ZW) {
        const int warp = threadIdx.x >> 5;
        const int RG = a.r >> 3;
        if (warp < 4) {
            for (int tl = 0; tl < ntl && ktiles > 0; ++tl)
                consume_tile<NT, 1>(c.rg, ktiles, xb, a.xs32, a.T, red, acc + tl * kBR * ald, ald, a.status);
        } else {
            float p[1][8];
#pragma unroll
            for (int e = 0; e < 8; ++e) p[0][e] = 0.f;
            zlin_rows<1, 16>([&](int, int i) { return bf2f(xbh[i]); }, reinterpret_cast<const uint4 *>(Vp), RG,
                             __ffs(RG) - 1, 0, klen, p, threadIdx.x - 128, 128);
            zlin_warp_store(p, RG, zred + (warp - 4) * 64);
        }
        cp_async_wait_all();
        consumer_sync();
        for (int k = threadIdx.x; k < a.r; k += kThreads)
            zp[k] = (zred[k] + zred[64 + k]) + (zred[128 + k] + zred[192 + k]);
        consumer_sync();
    } else {
    // W0 first: the ring has been filling since the kernel started
    for (int tl = 0; tl < ntl && ktiles > 0; ++tl)
        consume_tile<NT>(c.rg, ktiles, xb, a.xs32, a.T, red, acc + tl * kBR * ald, ald, a.status);
    cp_async_wait_all();
    consumer_sync();
    if (a.r > 0)
        for (int t0 = 0; t0 < a.T; t0 += TC)
            block_xV<TC>([&](int t, int i) { return t0 + t < a.T ? bf2f(xbh[(t0 + t) * xsh + i]) : 0.f; },
                         klen, Vp, a.r, zp + t0 * rp, rp, zred);
    }

    // epilogue: p = s*acc + U z_range
    const int vmU = vec_mode(Up, a.r);
    for (int row = threadIdx.x; row < nrows; row += kThreads) {
        const int o = r0 + row;
        const float sv = sv_p[row];
        for (int t0 = 0; t0 < a.T; t0 += TC) {
            float yv[TC];
#pragma unroll
            for (int j = 0; j < TC; ++j) yv[j] = (ktiles > 0 && t0 + j < ald) ? sv * acc[row * ald + t0 + j] : 0.f;
            if (a.r > 0) add_delta<TC>(Up, row, a.r, vmU, zp + t0 * rp, rp, yv);
#pragma unroll
            for (int j = 0; j < TC; ++j) {
                if (t0 + j >= a.T) break;
                if (KS == 1)
                    store_out(sg.y, a.ydt, (int64_t)(t0 + j) * sg.out + o, yv[j]);
                else
                    acc[row * ald + t0 + j] = yv[j];
            }
        }
    }
    if (KS > 1) {
        cg::cluster_group cl = cg::this_cluster();
        exchange_publish(c.ex, KS, a.status);
        const int lo = (int)((int64_t)q * nrows / KS);
        const int n = (int)((int64_t)(q + 1) * nrows / KS) - lo;
        for (int idx = threadIdx.x; idx < n * a.T; idx += kThreads) {
            const int t = idx / n, row = lo + (idx - t * n);
            float v = 0.f;
            for (int p = 0; p < KS; ++p) v += cl.map_shared_rank(acc, p)[row * ald + t];
            store_out(sg.y, a.ydt, (int64_t)t * sg.out + r0 + row, v);
        }
        exchange_release(c.ex, KS);
        exchange_reclaim(c.ex, a.status);  // peers are done with this CTA's memory
    }
}

// ------------------------------------------------------------------------
// fused GeGLU MLP decode: launch 1 (gate, up -> h, partials of h V_down)
// ------------------------------------------------------------------------
struct GateUpArgs {
    CUtensorMap mapg, mapu;
    const bf16 *x;
    int T, hidden, inter, r;
    const float *sg, *su;
    const bf16 *Ug, *Uu, *Vg, *Vu, *Vd;
    float *h;   // workspace [kTokChunk][inter] fp32
    float *zd;  // workspace [ngrp*KS][kTokChunk][rp] fp32
    int KS, Kc, tpc, nst, xs32, hmax;
    int vbuf, ubuf, dbuf;  // shared-memory bytes per prefetched V slice / U block / V_down rows (0: in place)
    int blk;  // 1: the W0 maps are k-block views (one 16 KB copy per ring stage)
    unsigned *status;
};

// ZW: as for dec_linear_kernel (warps 4-7 form z_gate and z_up while warps
// 0-3 stream the gate and up tiles).
template <int TC, bool ZW = false>
__global__ void __launch_bounds__(kDecThreads, 2) dec_gateup_kernel(const __grid_constant__ GateUpArgs a)
{
    constexpr int NT = 1, ald = 8;
    extern __shared__ __align__(1024) char smem_raw[];
    const int KS = a.KS;
    const int q = (int)(blockIdx.x % (unsigned)KS);
    const int gi = (int)(blockIdx.x / (unsigned)KS);
    const int rp = a.r > 0 ? a.r : 1;
    const int j0 = gi * a.tpc * kBR;
    const int nr = min(a.inter - j0, a.tpc * kBR);
    const int ntl = (nr + kBR - 1) / kBR;
    const int k0 = q * a.Kc;
    const int klen = max(0, min(a.hidden, k0 + a.Kc) - k0);
    const int ktiles = (klen + kBK - 1) / kBK;

    Carve c = carve(smem_raw, a.nst);
    uint32_t *xb = reinterpret_cast<uint32_t *>(c.rest);
    float *accg = reinterpret_cast<float *>(xb + a.T * a.xs32);  // x: T rows
    float *accu = accg + a.tpc * kBR * ald;
    float *red = accu + a.tpc * kBR * ald;
    float *zg = red + 512 * NT;   // [8][rp]
    float *zu = zg + 8 * rp;      // [8][rp]
    float *zred = zu + 8 * rp;    // [512]
    float *hl = zred + 512;       // [8][hmax]
    char *sgb = reinterpret_cast<char *>(hl + 8 * a.hmax);
    char *sub = sgb + a.tpc * kBR * 4 + 16;
    char *vgb = sub + a.tpc * kBR * 4 + 16;
    char *vub = vgb + a.vbuf;
    char *ugb = vub + a.vbuf;
    char *uub = ugb + a.ubuf;
    char *vdb = uub + a.ubuf;

    if (threadIdx.x == 0) {
        init_barriers(c, KS, ZW ? 4 : kWarps);
        pdl_trigger();
    }
    __syncthreads();           // barriers initialised (this CTA)
    if (KS > 1) cluster_arrive();  // peers may arrive remotely once all have passed this

    if (threadIdx.x >= kThreads) {  // ---------------- producer thread
        if (threadIdx.x == kThreads && ktiles > 0)
            for (int tl = 0; tl < ntl; ++tl) {
                if (!produce_tile(c.rg, &a.mapg, j0 + tl * kBR, k0, ktiles, a.status, a.blk)) break;
                if (!produce_tile(c.rg, &a.mapu, j0 + tl * kBR, k0, ktiles, a.status, a.blk)) break;
            }
        return;
    }

    // ------------------------------------------------ consumer warps
    const int lo = (int)((int64_t)q * nr / KS);
    const int n = (int)((int64_t)(q + 1) * nr / KS) - lo;
    const float *sgp = reinterpret_cast<const float *>(prefetch(sgb, a.sg + j0, nr * 4));
    const float *sup = reinterpret_cast<const float *>(prefetch(sub, a.su + j0, nr * 4));
    const bf16 *Vgp = a.Vg + (int64_t)k0 * a.r, *Vup = a.Vu + (int64_t)k0 * a.r;
    const bf16 *Ugp = a.Ug + (int64_t)j0 * a.r, *Uup = a.Uu + (int64_t)j0 * a.r;
    const bf16 *Vdp = a.Vd + (int64_t)(j0 + lo) * a.r;
    if (a.r > 0 && a.vbuf > 0 && a.dbuf > 0) {
        if (!ZW) {
            Vgp = reinterpret_cast<const bf16 *>(prefetch(vgb, Vgp, klen * a.r * 2));
            Vup = reinterpret_cast<const bf16 *>(prefetch(vub, Vup, klen * a.r * 2));
        }
        Ugp = reinterpret_cast<const bf16 *>(prefetch(ugb, Ugp, nr * a.r * 2));
        Uup = reinterpret_cast<const bf16 *>(prefetch(uub, Uup, nr * a.r * 2));
        Vdp = reinterpret_cast<const bf16 *>(prefetch(vdb, Vdp, n * a.r * 2));
    }
    pdl_wait();
    stage_x(a.x, a.hidden, a.T, k0, klen, ktiles * kBK, a.T, xb, a.xs32);
    consumer_sync();
    const bf16 *xbh = reinterpret_cast<const bf16 *>(xb);
    const int xsh = 2 * a.xs32;
    auto xsrc = [&](int t, int i) { return t < a.T ? bf2f(xbh[t * xsh + i]) : 0.f; };
    if constexpr (ZW) {
        const int warp = threadIdx.x >> 5;
        const int RG = a.r >> 3;
        if (warp < 4) {
            for (int tl = 0; tl < ntl && ktiles > 0; ++tl) {
                consume_tile<NT, 1>(c.rg, ktiles, xb, a.xs32, a.T, red, accg + tl * kBR * ald, ald, a.status);
                consume_tile<NT, 1>(c.rg, ktiles, xb, a.xs32, a.T, red, accu + tl * kBR * ald, ald, a.status);
            }
        } else {
            auto x1 = [&](int, int i) { return bf2f(xbh[i]); };
            float p[1][8];
#pragma unroll
            for (int e = 0; e < 8; ++e) p[0][e] = 0.f;
            zlin_rows<1, 16>(x1, reinterpret_cast<const uint4 *>(Vgp), RG, __ffs(RG) - 1, 0, klen, p,
                             threadIdx.x - 128, 128);
            zlin_warp_store(p, RG, zred + (warp - 4) * 64);
#pragma unroll
            for (int e = 0; e < 8; ++e) p[0][e] = 0.f;
            zlin_rows<1, 16>(x1, reinterpret_cast<const uint4 *>(Vup), RG, __ffs(RG) - 1, 0, klen, p,
                             threadIdx.x - 128, 128);
            zlin_warp_store(p, RG, zred + 256 + (warp - 4) * 64);
        }
        cp_async_wait_all();
        consumer_sync();
        for (int k = threadIdx.x; k < a.r; k += kThreads) {
            zg[k] = (zred[k] + zred[64 + k]) + (zred[128 + k] + zred[192 + k]);
            zu[k] = (zred[256 + k] + zred[320 + k]) + (zred[384 + k] + zred[448 + k]);
        }
        consumer_sync();
    } else {
        for (int tl = 0; tl < ntl && ktiles > 0; ++tl) {
            consume_tile<NT>(c.rg, ktiles, xb, a.xs32, a.T, red, accg + tl * kBR * ald, ald, a.status);
            consume_tile<NT>(c.rg, ktiles, xb, a.xs32, a.T, red, accu + tl * kBR * ald, ald, a.status);
        }
        cp_async_wait_all();
        consumer_sync();
        if (a.r > 0) {
            block_xV<TC>(xsrc, klen, Vgp, a.r, zg, rp, zred);
            block_xV<TC>(xsrc, klen, Vup, a.r, zu, rp, zred);
        }
    }
    // partial g, u over this K range: s*acc + U z_range (in place)
    const int vmUg = vec_mode(Ugp, a.r), vmUu = vec_mode(Uup, a.r);
    for (int v = threadIdx.x; v < 2 * nr; v += kThreads) {
        const bool up = v >= nr;
        const int row = up ? v - nr : v;
        float *acc = up ? accu : accg;
        const float sv = up ? sup[row] : sgp[row];
        float yv[TC];
#pragma unroll
        for (int t = 0; t < TC; ++t) yv[t] = ktiles > 0 ? sv * acc[row * ald + t] : 0.f;
        if (a.r > 0) add_delta<TC>(up ? Uup : Ugp, row, a.r, up ? vmUu : vmUg, up ? zu : zg, rp, yv);
#pragma unroll
        for (int t = 0; t < TC; ++t) acc[row * ald + t] = yv[t];
    }
    // complete g, u for this CTA's share of the rows, then h = gelu(g) * u
    if (KS > 1) {
        cg::cluster_group cl = cg::this_cluster();
        exchange_publish(c.ex, KS, a.status);
        for (int idx = threadIdx.x; idx < n * TC; idx += kThreads) {
            const int t = idx / n, v = lo + (idx - t * n);
            float g = 0.f, u = 0.f;
            for (int p = 0; p < KS; ++p) {
                g += cl.map_shared_rank(accg, p)[v * ald + t];
                u += cl.map_shared_rank(accu, p)[v * ald + t];
            }
            const float hv = t < a.T ? gelu_tanh_f32(g) * u : 0.f;
            hl[t * a.hmax + (v - lo)] = hv;
            if (t < a.T) a.h[(int64_t)t * a.inter + j0 + v] = hv;
        }
        exchange_release(c.ex, KS);
    } else {
        consumer_sync();
        for (int idx = threadIdx.x; idx < n * TC; idx += kThreads) {
            const int t = idx / n, v = lo + (idx - t * n);
            const float hv = t < a.T ? gelu_tanh_f32(accg[v * ald + t]) * accu[v * ald + t] : 0.f;
            hl[t * a.hmax + (v - lo)] = hv;
            if (t < a.T) a.h[(int64_t)t * a.inter + j0 + v] = hv;
        }
        consumer_sync();
    }
    // partial z_down = sum over this CTA's rows of h V_down, to the workspace
    if (a.r > 0)
        block_xV<TC>([&](int t, int i) { return hl[t * a.hmax + i]; }, n, Vdp, a.r,
                     a.zd + ((int64_t)gi * KS + q) * kTokChunk * rp, rp, zred);
    if (KS > 1) exchange_reclaim(c.ex, a.status);
}

// ------------------------------------------------------------------------
// fused GeGLU MLP decode: launch 2 (y = wl(h; down))
// ------------------------------------------------------------------------
struct DownArgs {
    CUtensorMap mapd;
    const float *h;   // [kTokChunk][inter] fp32, written by launch 1
    const float *zd;  // [nzd][kTokChunk][rp] partials of h V_down
    int nzd;
    int T, inter, hidden, r, ydt;
    const float *sd;
    const bf16 *Ud;
    void *y;
    int KS, Kc, tpc, nst, xs32;
    int ubuf;  // shared-memory bytes for the prefetched U rows (0: read in place)
    int blk;  // 1: the W0 maps are k-block views (one 16 KB copy per ring stage)
    unsigned *status;
};

// x columns of the down product: token t's h as bf16 (column t) plus the
// rounding remainder h - bf16(h) as bf16 (column T + t); their sum carries h
// to about 16 bits, enough for fp32-output accuracy.
template <int NT, int TC>
__global__ void __launch_bounds__(kDecThreads, 2) dec_down_kernel(const __grid_constant__ DownArgs a)
{
    constexpr int ald = 8 * NT;
    extern __shared__ __align__(1024) char smem_raw[];
    const int KS = a.KS;
    const int q = (int)(blockIdx.x % (unsigned)KS);
    const int gi = (int)(blockIdx.x / (unsigned)KS);
    const int rp = a.r > 0 ? a.r : 1;
    const int o0 = gi * a.tpc * kBR;
    const int nr = min(a.hidden - o0, a.tpc * kBR);
    const int ntl = (nr + kBR - 1) / kBR;
    const int k0 = q * a.Kc;
    const int klen = max(0, min(a.inter, k0 + a.Kc) - k0);
    const int ktiles = (klen + kBK - 1) / kBK;

    Carve c = carve(smem_raw, a.nst);
    uint32_t *xb = reinterpret_cast<uint32_t *>(c.rest);
    float *acc = reinterpret_cast<float *>(xb + 2 * a.T * a.xs32);  // x: 2T rows (hi, lo)
    float *red = acc + a.tpc * kBR * ald;
    float *zp = red + 512 * NT;    // [8][rp]
    float *zred = zp + 8 * rp;     // [kThreads]
    char *sbuf = reinterpret_cast<char *>(zred + kThreads);
    char *ubuf = sbuf + a.tpc * kBR * 4 + 16;

    if (threadIdx.x == 0) {
        init_barriers(c, KS);
        pdl_trigger();
    }
    __syncthreads();           // barriers initialised (this CTA)
    if (KS > 1) cluster_arrive();  // peers may arrive remotely once all have passed this

    if (threadIdx.x >= kThreads) {  // ---------------- producer: W_down does not depend on h
        if (threadIdx.x == kThreads && ktiles > 0)
            for (int tl = 0; tl < ntl; ++tl)
                if (!produce_tile(c.rg, &a.mapd, o0 + tl * kBR, k0, ktiles, a.status, a.blk)) break;
        return;
    }

    // ------------------------------------------------ consumer warps
    // every CTA of a K split forms z_down; the low-rank term of a row is added
    // by the CTA that stores the row
    const int rr = a.r;
    const float *sdp = reinterpret_cast<const float *>(prefetch(sbuf, a.sd + o0, nr * 4));
    const bf16 *Udp = a.Ud + (int64_t)o0 * a.r;
    if (rr > 0 && a.ubuf > 0) Udp = reinterpret_cast<const bf16 *>(prefetch(ubuf, Udp, nr * a.r * 2));
    pdl_wait();  // h and the partials come from launch 1
    {
        const int width = ktiles * kBK;
        const int nq = width >> 2;  // 4-column groups
        bf16 *xbh = reinterpret_cast<bf16 *>(xb);
        const int xsh = 2 * a.xs32;
        for (int idx = threadIdx.x; idx < 2 * a.T * nq; idx += kThreads) {
            const int n = idx / nq, cq = idx - n * nq;
            const int t = n < a.T ? n : n - a.T;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (4 * cq < klen)
                v = __ldcg(reinterpret_cast<const float4 *>(a.h + (int64_t)t * a.inter + k0 + 4 * cq));
            const float e[4] = {v.x, v.y, v.z, v.w};
            for (int j = 0; j < 4; ++j) {
                const bf16 hi = __float2bfloat16_rn(e[j]);
                xbh[n * xsh + 4 * cq + j] = n < a.T ? hi : __float2bfloat16_rn(e[j] - __bfloat162float(hi));
            }
        }
    }
    const int vmU = vec_mode(Udp, a.r);
    // z_down[t][k] = sum over the nzd partials in a fixed order.  One token,
    // r = 4*RQ <= 64 (RQ a power of two): thread tid adds 16-byte chunk
    // tid % RQ of partials tid / RQ, tid / RQ + kThreads / RQ, ... (sixteen
    // loads in flight), then the lanes of a chunk and the warps are added in a
    // fixed order (red is free before the W0 stream).  Otherwise threads split
    // the partials into chunks of scalar loads, added in chunk order.
    const int nout = TC * rr;
    const int RQ = rr >> 2;
    if (TC == 1 && rr > 0 && (rr & 3) == 0 && rr <= 64 && (RQ & (RQ - 1)) == 0) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, lq = __ffs(RQ) - 1;
        const int g4 = threadIdx.x & (RQ - 1);
        float4 sm = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 16
        for (int p = threadIdx.x >> lq; p < a.nzd; p += kThreads >> lq) {
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.zd + (int64_t)p * kTokChunk * rp) + g4);
            sm.x += v.x;
            sm.y += v.y;
            sm.z += v.z;
            sm.w += v.w;
        }
        for (int off = RQ; off < 32; off <<= 1) {
            sm.x += __shfl_xor_sync(0xffffffffu, sm.x, off);
            sm.y += __shfl_xor_sync(0xffffffffu, sm.y, off);
            sm.z += __shfl_xor_sync(0xffffffffu, sm.z, off);
            sm.w += __shfl_xor_sync(0xffffffffu, sm.w, off);
        }
        if (lane < RQ) reinterpret_cast<float4 *>(red + warp * 64)[lane] = sm;
        consumer_sync();
        for (int k = threadIdx.x; k < rr; k += kThreads) {
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) v += red[w * 64 + k];
            zp[k] = v;
        }
    } else if (nout > 0 && nout <= kThreads) {
        const int nch = kThreads / nout;
        const int ch = threadIdx.x / nout, cc = threadIdx.x - ch * nout;
        if (ch < nch) {
            const int t = cc / rr, k = cc - t * rr;
            float s = 0.f;
#pragma unroll 16
            for (int p = ch; p < a.nzd; p += nch) s += __ldcg(a.zd + ((int64_t)p * kTokChunk + t) * rp + k);
            zred[ch * nout + cc] = s;
        }
        consumer_sync();
        for (int c2 = threadIdx.x; c2 < nout; c2 += kThreads) {
            float s = 0.f;
            for (int j = 0; j < nch; ++j) s += zred[j * nout + c2];
            zp[(c2 / rr) * rp + (c2 % rr)] = s;
        }
    } else if (nout > 0) {
        for (int c2 = threadIdx.x; c2 < nout; c2 += kThreads) {
            const int t = c2 / rr, k = c2 - t * rr;
            float s = 0.f;
#pragma unroll 4
            for (int p = 0; p < a.nzd; ++p) s += __ldcg(a.zd + ((int64_t)p * kTokChunk + t) * rp + k);
            zp[t * rp + k] = s;
        }
    }
    cp_async_wait_all();
    consumer_sync();
    for (int tl = 0; tl < ntl && ktiles > 0; ++tl)
        consume_tile<NT>(c.rg, ktiles, xb, a.xs32, 2 * a.T, red, acc + tl * kBR * ald, ald, a.status);
    for (int row = threadIdx.x; row < nr; row += kThreads) {
        const int o = o0 + row;
        const float sv = sdp[row];
        float yv[TC];
#pragma unroll
        for (int t = 0; t < TC; ++t)
            yv[t] = (ktiles > 0 && t < a.T) ? sv * (acc[row * ald + t] + acc[row * ald + a.T + t]) : 0.f;
        if (rr > 0 && KS == 1) add_delta<TC>(Udp, row, rr, vmU, zp, rp, yv);
#pragma unroll
        for (int t = 0; t < TC; ++t) {
            if (t >= a.T) break;
            if (KS == 1)
                store_out(a.y, a.ydt, (int64_t)t * a.hidden + o, yv[t]);
            else
                acc[row * ald + t] = yv[t];
        }
    }
    if (KS > 1) {
        cg::cluster_group cl = cg::this_cluster();
        exchange_publish(c.ex, KS, a.status);
        const int lo = (int)((int64_t)q * nr / KS);
        const int n = (int)((int64_t)(q + 1) * nr / KS) - lo;
        for (int idx = threadIdx.x; idx < n * a.T; idx += kThreads) {
            const int t = idx / n, row = lo + (idx - t * n);
            float v = 0.f;
            for (int p = 0; p < KS; ++p) v += cl.map_shared_rank(acc, p)[row * ald + t];
            if (rr > 0) add_delta<1>(Udp, row, rr, vmU, zp + t * rp, rp, &v);
            store_out(a.y, a.ydt, (int64_t)t * a.hidden + o0 + row, v);
        }
        exchange_release(c.ex, KS);
        exchange_reclaim(c.ex, a.status);
    }
}

// ------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------
static inline int round_up(int v, int m) { return (v + m - 1) / m * m; }
static inline int cdiv(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

constexpr int kSmemTarget = 112 * 1024;  // two CTAs (of successive kernels) share an SM
constexpr int kMaxPartials = 512;        // z_down partials (one per gate/up CTA)
constexpr int kPrefetchBudget = 24 * 1024;  // shared memory for prefetched rank-r operands

typedef void (*dec_fn)(DecArgs);
typedef void (*gu_fn)(GateUpArgs);
typedef void (*dn_fn)(DownArgs);
// [token chunk 1 or 8][n-tiles 1, 2, 4, 8]; one token uses the TC = 1 forms
static dec_fn g_dec[2][4] = {{dec_linear_kernel<1, 1>, nullptr, nullptr, nullptr},
                             {dec_linear_kernel<1, 8>, dec_linear_kernel<2, 8>, dec_linear_kernel<4, 8>,
                              dec_linear_kernel<8, 8>}};
static gu_fn g_gu[2] = {dec_gateup_kernel<1>, dec_gateup_kernel<8>};
// one token with separate x V warps
static dec_fn g_dec_zw = dec_linear_kernel<1, 1, true>;
static gu_fn g_gu_zw = dec_gateup_kernel<1, true>;

// The ZW forms apply: one token, r = 8*RG <= 64 with RG a power of two, every
// V 16-byte aligned.
static bool zw_ok(int64_t T, int64_t r, const void *const *V, int nv)
{
    if (T != 1 || r <= 0 || r > 64 || r % 8) return false;
    const int RG = (int)(r / 8);
    if (RG & (RG - 1)) return false;
    for (int j = 0; j < nv; ++j)
        if (reinterpret_cast<uintptr_t>(V[j]) % 16) return false;
    return true;
}
static dn_fn g_dn[2][2] = {{dec_down_kernel<1, 1>, nullptr}, {dec_down_kernel<1, 8>, dec_down_kernel<2, 8>}};

static inline int nt_index(int nt) { return nt <= 1 ? 0 : nt <= 2 ? 1 : nt <= 4 ? 2 : 3; }
static inline int nt_round(int nt) { return nt <= 1 ? 1 : nt <= 2 ? 2 : nt <= 4 ? 4 : 8; }

static std::mutex g_mu;
static std::unordered_map<uint64_t, int> g_attr_set;  // (device, fn) -> done

static wl_status ensure_attrs(const void *fn, int bytes, const DeviceInfo *di)
{
    if (bytes > di->max_smem_optin)
        return fail(WL_ERR_UNSUPPORTED, "decode kernel needs %d bytes of shared memory, device allows %d",
                    bytes, di->max_smem_optin);
    std::lock_guard<std::mutex> lk(g_mu);
    const uint64_t key = ((uint64_t)di->device << 56) ^ (uint64_t)(uintptr_t)fn;
    if (g_attr_set.count(key)) return WL_OK;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, di->max_smem_optin);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic smem)");
    g_attr_set[key] = 1;
    return WL_OK;
}

static wl_status launch(const void *fn, int grid, int KS, int smem, cudaStream_t st, void **args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)KS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
    return WL_OK;
}

// Work split of a launch's 64-row tiles with K = in (see plan_balanced):
//   tpc   tiles per row group: each group forms z = x V once, so more tiles
//         per group keep the rank-r operand's traffic small next to W0;
//   KS    K splits (cluster size);
//   Kc    K elements per split, a multiple of 64 (whole TMA boxes).
struct Split {
    int tpc, ngrp, KS, Kc;
};

// Plans are computed once per (launch kind, device, shape) and reused.
static std::mutex g_plan_mu;
static std::unordered_map<uint64_t, Split> g_plans;
static uint64_t plan_key(int kind, int dev, int64_t a, int64_t b, int64_t c, int64_t d)
{
    uint64_t h = (uint64_t)kind * 0x9E3779B97F4A7C15ull ^ (uint64_t)dev;
    for (int64_t v : {a, b, c, d}) h = (h ^ (uint64_t)v) * 0x100000001B3ull + (h >> 29);
    return h;
}

// Ring stages that fit next to `other` bytes of shared memory.
static int ring_stages(int other, const DeviceInfo *di)
{
    int n = (kSmemTarget - other - 1024) / kStageBytes;
    if (n > 6) n = 6;
    if (n < 3) {  // does not fit next to another CTA: use one SM's worth
        n = (di->max_smem_optin - other - 1024) / kStageBytes;
        if (n > 6) n = 6;
    }
    return n;
}

// x row stride in u32: 16-byte multiple, odd number of 16-byte units (keeps
// the tensor-core operand reads free of shared-memory bank conflicts).
static inline int x_stride32(int width)
{
    int u16 = width / 8;  // 16-byte units of bf16
    if ((u16 & 1) == 0) u16 += 1;
    return u16 * 4;
}

// CTAs of `fn` that can be resident at once in clusters of ks with `smem`
// bytes of shared memory each (cached per device, kernel, ks, smem).
static int cluster_capacity(const void *fn, int ks, int smem, const DeviceInfo *di)
{
    static std::mutex mu;
    static std::unordered_map<uint64_t, int> cache;
    const uint64_t key = ((uint64_t)di->device << 58) ^ ((uint64_t)(uintptr_t)fn << 8) ^ ((uint64_t)smem << 24) ^ (uint64_t)ks;
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(ks * di->sm_count));
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    int cap;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) == cudaSuccess && n > 0) {
        cap = n * ks;
    } else {
        cudaGetLastError();
        cap = (di->sm_count / ks) * ks * (smem <= kSmemTarget ? 2 : 1);
    }
    std::lock_guard<std::mutex> lk(mu);
    cache[key] = cap;
    return cap;
}

// Expected time of a launch plan, in microseconds, from a model calibrated on
// GB300 decode timings (T = 1, forced plans):
//   * a CTA keeps its ring's stages in flight, one round trip of a 16 KB stage
//     taking about kStageLatUs, so an SM streams at min(its share of HBM,
//     stages resident on it * 16 KB / kStageLatUs);
//   * CTAs beyond one per SM share that SM's stream; beyond what can be
//     resident at once (cluster placement included) they run as further
//     rounds;
//   * a K split costs a cluster exchange, about 0.7 us per split;
//   * x V that follows the stream reads the V slice at about 40 GB/s per CTA;
//     formed by four separate warps during the stream (zw) it runs at about
//     12 GB/s and costs only what the stream does not hide;
//   * clusters of 5, 7 or 8 CTAs place unevenly on the GPCs and measured far
//     slower than this predicts; they are used only where no other size fits.
constexpr double kHbmBytesPerUs = 6.8e6;
constexpr double kStageLatUs = 2.34;
constexpr double kZBytesPerUs = 4.0e4;    // x V after the stream, 8 warps
constexpr double kZwBytesPerUs = 1.2e4;   // x V by 4 warps during the stream

// The split of the segments' 64-row tiles (seg_tiles[0..nseg)) by `in` columns
// with the least expected time.  A row group of tpc tiles of one segment and a
// K split of Kc columns make one CTA, which streams pair*tpc tiles (gate and
// up: pair = 2) and reads nzv V slices of r ranks.  smem_of(tpc, Kc, &nst)
// gives the launch's shared memory and ring stages (< 0: does not fit).
template <class SmemOf>
static bool plan_balanced(const int *seg_tiles, int nseg, int in, int r, int pair, int nzv, bool zw, int max_kc,
                          int tpc_max, int max_ctas, const void *fn, SmemOf smem_of, const DeviceInfo *di,
                          Split *out)
{
    double best = 1e30;
    int best_ctas = 0;
    bool found = false;
    const int S = di->sm_count;
    // the preferred cluster sizes first; 5, 7 and 8 only where nothing else fits
    for (int pass = 0; pass < 2 && !found; ++pass)
    for (int tpc = 1; tpc <= tpc_max; ++tpc) {
        int ngrp = 0;
        for (int j = 0; j < nseg; ++j) ngrp += cdiv(seg_tiles[j], tpc);
        for (int ks = 1; ks <= 8; ++ks) {
            if ((ks == 5 || ks > 6) != (pass == 1)) continue;
            const int Kc = round_up(cdiv(in, ks), kBK);
            if (Kc > max_kc || cdiv(in, Kc) != ks) continue;
            const int ctas = ngrp * ks;
            if (ctas > max_ctas) continue;
            int nst = 0;
            const int smem = smem_of(tpc, Kc, &nst);
            if (smem < 0) continue;
            const int cap = cluster_capacity(fn, ks, smem, di);
            if (cap <= 0) continue;
            const int res = ctas < cap ? ctas : cap;
            const int rounds = cdiv(ctas, cap);
            const int k = cdiv(res, S);
            const int busy = res < S ? res : S;
            const double bw = (double)pair * tpc * kBR * Kc * 2;
            const double rate = std::min(kHbmBytesPerUs / busy, (double)k * nst * kStageBytes / kStageLatUs);
            const double t_stream = k * bw / rate;
            const double vb = (double)nzv * Kc * r * 2;
            const double t_z = r <= 0 ? 0.0 : zw ? std::max(0.0, vb / kZwBytesPerUs - t_stream) : vb / kZBytesPerUs;
            const double cost = rounds * (t_stream + t_z) + (ks > 1 ? 0.7 * ks : 0.0) + 1.0;
            if (cost < best * 0.999 || (cost < best * 1.001 && ctas < best_ctas)) {
                best = cost;
                best_ctas = ctas;
                *out = Split{tpc, ngrp, ks, Kc};
                found = true;
            }
        }
    }
    return found;
}

// The W0 map of a projection for the ring: the k-block view (one copy per
// 16 KB stage) when K is a multiple of 64, else 64 x 64 boxes (two copies).
static wl_status w0_map(const void *W0, int64_t K, int64_t out, CUtensorMap *m, int *blk)
{
    if (K % kBK == 0) {
        *blk = 1;
        return tmap_kblocks_bf16(W0, K, out, kBR, 2, m);
    }
    *blk = 0;
    return tmap_2d_bf16(W0, K, out, K, kBK, kBR, m);
}

// plan_only: find (and cache) the launch plan, launch nothing; WL_ERR_UNSUPPORTED
// when no plan fits shared memory.
static wl_status dec_linear_once(const bf16 *x, const wl_proj *proj, int nproj, void *const *y,
                                 int64_t T, int64_t in, int64_t r, int ydt, cudaStream_t st,
                                 const DeviceInfo *di, bool plan_only = false)
{
    wl_status s = WL_OK;
    const int NT = nt_round(cdiv(T, 8));
    // keep x (T rows of K columns) within about 48 KB; where the staged x
    // and the per-tile partial sums still leave no room for two ring stages
    // (many tokens, long K, large rank), take fewer tiles per row group and
    // narrower K splits
    int max_kc = (48 * 1024) / ((int)T * 2);
    max_kc = max_kc < kBK ? kBK : (max_kc / kBK) * kBK;
    const int rp0 = r > 0 ? (int)r : 1;
    const void *vs[3] = {};
    int seg_tiles[3] = {};
    for (int j = 0; j < nproj; ++j) {
        vs[j] = proj[j].V;
        seg_tiles[j] = cdiv(proj[j].out, kBR);
    }
    const bool zw = zw_ok(T, r, vs, nproj);
    const dec_fn fn = zw ? g_dec_zw : g_dec[T == 1 ? 0 : 1][nt_index(NT)];
    // shared memory of a (tpc, Kc) plan, as laid out below
    auto smem_of = [&](int tpc, int Kc, int *nst_out) {
        const int xs = x_stride32(Kc);
        int pre = 0;
        const int vb = round_up(Kc * (int)r * 2 + 16, 16), ub = round_up(tpc * kBR * (int)r * 2 + 16, 16);
        if (r > 0 && zw && ub <= kPrefetchBudget) pre = ub;  // the z warps read V in place
        else if (r > 0 && vb + ub <= kPrefetchBudget) pre = vb + ub;
        const int other = (int)T * xs * 4 + 4 * (tpc * kBR * 8 * NT + 512 * NT + cdiv(T, 8) * 8 * rp0 + 512) +
                          tpc * kBR * 4 + 16 + pre;
        const int nst = ring_stages(other, di);
        *nst_out = nst;
        return nst < 2 ? -1 : carve_head_bytes(nst) + other;
    };
    s = ensure_attrs((const void *)fn, 0, di);
    if (s != WL_OK) return s;
    Split sp;
    {
        std::lock_guard<std::mutex> lk(g_plan_mu);
        const uint64_t key = plan_key(1, di->device, ((int64_t)seg_tiles[0] << 40) ^ ((int64_t)seg_tiles[1] << 20) ^ seg_tiles[2],
                                      in, r, T * 2 + (zw ? 1 : 0));
        auto it = g_plans.find(key);
        if (it != g_plans.end()) {
            sp = it->second;
        } else {
            if (!plan_balanced(seg_tiles, nproj, (int)in, (int)r, 1, 1, zw, max_kc, 8, 1 << 20, (const void *)fn,
                               smem_of, di, &sp))
                return fail(WL_ERR_UNSUPPORTED, "decode: shapes too large for shared memory");
            g_plans[key] = sp;
        }
    }

    if (plan_only) return WL_OK;
    DecArgs a = {};
    a.x = x;
    a.T = (int)T;
    a.in = (int)in;
    a.r = (int)r;
    a.ydt = ydt;
    a.KS = sp.KS;
    a.Kc = sp.Kc;
    a.tpc = sp.tpc;
    a.nseg = nproj;
    a.status = di->status;
    a.xs32 = x_stride32(sp.Kc);
    int grp = 0;
    for (int j = 0; j < nproj; ++j) {
        DecSeg &sg = a.seg[j];
        s = w0_map(proj[j].W0, in, proj[j].out, &sg.map, &a.blk);
        if (s != WL_OK) return s;
        sg.s = proj[j].s;
        sg.U = static_cast<const bf16 *>(proj[j].U);
        sg.V = static_cast<const bf16 *>(proj[j].V);
        sg.y = y[j];
        sg.out = (int)proj[j].out;
        sg.grp0 = grp;
        sg.ngrp = cdiv(cdiv(proj[j].out, kBR), sp.tpc);
        grp += sg.ngrp;
    }
    const int rp = r > 0 ? (int)r : 1;
    // prefetch the V slice and U rows into shared memory when they are small
    const int vb = round_up(sp.Kc * (int)r * 2 + 16, 16), ub = round_up(sp.tpc * kBR * (int)r * 2 + 16, 16);
    if (r > 0 && zw && ub <= kPrefetchBudget) {
        a.ubuf = ub;
    } else if (r > 0 && vb + ub <= kPrefetchBudget) {
        a.vbuf = vb;
        a.ubuf = ub;
    }
    const int other = (int)T * a.xs32 * 4 + 4 * (sp.tpc * kBR * 8 * NT + 512 * NT + cdiv(T, 8) * 8 * rp + 512) +
                      sp.tpc * kBR * 4 + 16 + a.vbuf + a.ubuf;
    a.nst = ring_stages(other, di);
    const int smem = carve_head_bytes(a.nst) + other;
    if (a.nst < 2) return fail(WL_ERR_UNSUPPORTED, "decode: shapes too large for shared memory");
    s = ensure_attrs((const void *)fn, smem, di);
    if (s != WL_OK) return s;
    void *args[] = {&a};
    return launch((const void *)fn, grp * sp.KS, sp.KS, smem, st, args);
}

// Decode path for up to 64 tokens per launch (W0 streamed once per launch).
constexpr int64_t kDecodeMaxT = 64;

wl_status launch_decode_linear(const bf16 *x, const wl_proj *proj, int nproj, void *const *y,
                               int64_t T, int64_t in, int64_t r, int ydt, cudaStream_t st)
{
    wl_status s = WL_OK;
    const DeviceInfo *di = device_info(&s);
    if (!di) return s;
    const int es = ydt == WL_OUT_F32 ? 4 : 2;
    for (int64_t t0 = 0; t0 < T; t0 += kDecodeMaxT) {
        const int64_t Tc = (T - t0) < kDecodeMaxT ? (T - t0) : kDecodeMaxT;
        void *yc[3];
        for (int j = 0; j < nproj; ++j)
            yc[j] = static_cast<char *>(y[j]) + (size_t)t0 * (size_t)proj[j].out * es;
        s = dec_linear_once(x + t0 * in, proj, nproj, yc, Tc, in, r, ydt, st, di);
        if (s != WL_OK) return s;
    }
    return WL_OK;
}

bool decode_linear_fits(const wl_proj *proj, int nproj, int64_t T, int64_t in, int64_t r, int ydt)
{
    wl_status s = WL_OK;
    const DeviceInfo *di = device_info(&s);
    if (!di) return false;
    const int64_t Tc = T < kDecodeMaxT ? T : kDecodeMaxT;
    void *ys[3] = {};
    const bool ok = dec_linear_once(nullptr, proj, nproj, ys, Tc, in, r, ydt, nullptr, di, true) == WL_OK;
    clear_error();
    return ok;
}

// ---- MLP ---------------------------------------------------------------
size_t decode_mlp_workspace_bytes(int64_t hidden, int64_t inter, int64_t r)
{
    (void)hidden;
    const int64_t rp = r > 0 ? r : 1;
    auto al = [](int64_t v) { return (v + 255) / 256 * 256; };
    return (size_t)(256 + al(kTokChunk * inter * 4) + al((int64_t)kMaxPartials * kTokChunk * rp * 4));
}

// Both launches are planned before either is made; plan_only: find (and cache)
// the plans, launch nothing; WL_ERR_UNSUPPORTED when one does not fit.
static wl_status dec_mlp_once(const bf16 *x, const wl_proj &gate, const wl_proj &up,
                              const wl_proj &down, void *y, int T, int hidden, int inter, int r,
                              char *ws, int ydt, cudaStream_t st, const DeviceInfo *di,
                              bool plan_only = false)
{
    const int rp = r > 0 ? r : 1;

    // launch 1: gate and up tiles, h, partials of h V_down
    GateUpArgs g = {};
    const void *gv[2] = {gate.V, up.V};
    const bool gzw = zw_ok(T, r, gv, 2);
    const gu_fn gfn = gzw ? g_gu_zw : g_gu[T == 1 ? 0 : 1];
    wl_status s = ensure_attrs((const void *)gfn, 0, di);
    if (s != WL_OK) return s;
    // shared memory of a gate/up plan (tpc, Kc), as laid out below
    auto gsmem_of = [&](int tpc, int Kc, int *nst_out) {
        const int ks = cdiv(hidden, Kc);
        const int xs = x_stride32(Kc), hmax = cdiv(tpc * kBR, ks) + 1;
        const int vb = round_up(Kc * r * 2 + 16, 16), ub = round_up(tpc * kBR * r * 2 + 16, 16);
        const int db = round_up(hmax * r * 2 + 16, 16);
        const int pre = (r > 0 && 2 * vb + 2 * ub + db <= kPrefetchBudget) ? 2 * vb + 2 * ub + db : 0;
        const int other = T * xs * 4 + 4 * (2 * tpc * kBR * 8 + 512 + 16 * rp + 512 + 8 * hmax) +
                          2 * (tpc * kBR * 4 + 16) + pre;
        const int nst = ring_stages(other, di);
        *nst_out = nst;
        return nst < 2 ? -1 : carve_head_bytes(nst) + other;
    };
    Split sg;
    {
        std::lock_guard<std::mutex> lk(g_plan_mu);
        const uint64_t key = plan_key(2, di->device, inter, hidden, r, T * 2 + (gzw ? 1 : 0));
        auto it = g_plans.find(key);
        if (it != g_plans.end()) {
            sg = it->second;
        } else {
            // gate and up tiles are a pair per CTA: twice the W0 stream and rank work per tile
            const int gt = cdiv(inter, kBR);
            if (!plan_balanced(&gt, 1, hidden, r, 2, 2, gzw, 48 * 1024 / (2 * T) / kBK * kBK, 8, kMaxPartials,
                               (const void *)gfn,
                               gsmem_of, di, &sg))
                return fail(WL_ERR_UNSUPPORTED, "MLP decode: shapes too large for shared memory");
            g_plans[key] = sg;
        }
    }
    // launch 2: down tiles, input h as bf16 hi/lo columns
    DownArgs d = {};
    const int NT = nt_round(cdiv(2 * T, 8));
    const dn_fn dfn = g_dn[T == 1 ? 0 : 1][NT <= 1 ? 0 : 1];
    s = ensure_attrs((const void *)dfn, 0, di);
    if (s != WL_OK) return s;
    auto dsmem_of = [&](int tpc, int Kc, int *nst_out) {
        const int xs = x_stride32(Kc);
        const int ub = round_up(tpc * kBR * r * 2 + 16, 16);
        const int pre = (r > 0 && ub <= kPrefetchBudget) ? ub : 0;
        const int other = 2 * T * xs * 4 + 4 * (tpc * kBR * 8 * NT + 512 * NT + 8 * rp + kThreads) + tpc * kBR * 4 + 16 + pre;
        const int nst = ring_stages(other, di);
        *nst_out = nst;
        return nst < 2 ? -1 : carve_head_bytes(nst) + other;
    };
    Split sd;
    {
        std::lock_guard<std::mutex> lk(g_plan_mu);
        const uint64_t key = plan_key(3, di->device, hidden, inter, r, T);
        auto it = g_plans.find(key);
        if (it != g_plans.end()) {
            sd = it->second;
        } else {
            const int dt = cdiv(hidden, kBR);
            if (!plan_balanced(&dt, 1, inter, r, 1, 0, false, (48 * 1024) / (2 * T * 2) / kBK * kBK, 8, 1 << 20,
                               (const void *)dfn, dsmem_of, di, &sd))
                return fail(WL_ERR_UNSUPPORTED, "MLP decode: shapes too large for shared memory");
            g_plans[key] = sd;
        }
    }
    if (plan_only) return WL_OK;  // both launches have a plan
    float *h = reinterpret_cast<float *>(ws + 256);
    float *zd = reinterpret_cast<float *>(ws + 256 + ((int64_t)kTokChunk * inter * 4 + 255) / 256 * 256);
    s = w0_map(gate.W0, hidden, inter, &g.mapg, &g.blk);
    if (s != WL_OK) return s;
    s = w0_map(up.W0, hidden, inter, &g.mapu, &g.blk);
    if (s != WL_OK) return s;
    g.x = x;
    g.T = T;
    g.hidden = hidden;
    g.inter = inter;
    g.r = r;
    g.sg = gate.s;
    g.su = up.s;
    g.Ug = static_cast<const bf16 *>(gate.U);
    g.Uu = static_cast<const bf16 *>(up.U);
    g.Vg = static_cast<const bf16 *>(gate.V);
    g.Vu = static_cast<const bf16 *>(up.V);
    g.Vd = static_cast<const bf16 *>(down.V);
    g.h = h;
    g.zd = zd;
    g.KS = sg.KS;
    g.Kc = sg.Kc;
    g.tpc = sg.tpc;
    g.xs32 = x_stride32(sg.Kc);
    g.hmax = cdiv(sg.tpc * kBR, sg.KS) + 1;
    g.status = di->status;
    {
        const int vb = round_up(sg.Kc * r * 2 + 16, 16), ub = round_up(sg.tpc * kBR * r * 2 + 16, 16);
        const int db = round_up(g.hmax * r * 2 + 16, 16);
        if (r > 0 && 2 * vb + 2 * ub + db <= kPrefetchBudget) {
            g.vbuf = vb;
            g.ubuf = ub;
            g.dbuf = db;
        }
    }
    const int gother = T * g.xs32 * 4 + 4 * (2 * sg.tpc * kBR * 8 + 512 + 16 * rp + 512 + 8 * g.hmax) +
                       2 * (sg.tpc * kBR * 4 + 16) + 2 * g.vbuf + 2 * g.ubuf + g.dbuf;
    g.nst = ring_stages(gother, di);
    if (g.nst < 2) return fail(WL_ERR_UNSUPPORTED, "MLP decode: shapes too large for shared memory");
    const int gsmem = carve_head_bytes(g.nst) + gother;
    s = ensure_attrs((const void *)gfn, gsmem, di);
    if (s != WL_OK) return s;
    void *gargs[] = {&g};
    s = launch((const void *)gfn, sg.ngrp * sg.KS, sg.KS, gsmem, st, gargs);
    if (s != WL_OK) return s;

    s = w0_map(down.W0, inter, hidden, &d.mapd, &d.blk);
    if (s != WL_OK) return s;
    d.h = h;
    d.zd = zd;
    d.nzd = sg.ngrp * sg.KS;
    d.T = T;
    d.inter = inter;
    d.hidden = hidden;
    d.r = r;
    d.ydt = ydt;
    d.sd = down.s;
    d.Ud = static_cast<const bf16 *>(down.U);
    d.y = y;
    d.KS = sd.KS;
    d.Kc = sd.Kc;
    d.tpc = sd.tpc;
    d.xs32 = x_stride32(sd.Kc);
    d.status = di->status;
    {
        const int ub = round_up(sd.tpc * kBR * r * 2 + 16, 16);
        if (r > 0 && ub <= kPrefetchBudget) d.ubuf = ub;
    }
    const int dother = 2 * T * d.xs32 * 4 + 4 * (sd.tpc * kBR * 8 * NT + 512 * NT + 8 * rp + kThreads) +
                       sd.tpc * kBR * 4 + 16 + d.ubuf;
    d.nst = ring_stages(dother, di);
    if (d.nst < 2) return fail(WL_ERR_UNSUPPORTED, "MLP decode: shapes too large for shared memory");
    const int dsmem = carve_head_bytes(d.nst) + dother;
    s = ensure_attrs((const void *)dfn, dsmem, di);
    if (s != WL_OK) return s;
    void *dargs[] = {&d};
    return launch((const void *)dfn, sd.ngrp * sd.KS, sd.KS, dsmem, st, dargs);
}

bool decode_mlp_fits(const wl_proj &gate, const wl_proj &up, const wl_proj &down, int64_t T, int64_t hidden,
                     int64_t inter, int64_t r, int ydt)
{
    wl_status s = WL_OK;
    const DeviceInfo *di = device_info(&s);
    if (!di) return false;
    const int Tc = (int)(T < kTokChunk ? T : kTokChunk);
    const bool ok = dec_mlp_once(nullptr, gate, up, down, nullptr, Tc, (int)hidden, (int)inter, (int)r, nullptr,
                                 ydt, nullptr, di, true) == WL_OK;
    clear_error();
    return ok;
}

wl_status launch_decode_mlp(const bf16 *x, const wl_proj &gate, const wl_proj &up,
                            const wl_proj &down, void *y, int64_t T, int64_t hidden,
                            int64_t inter, int64_t r, void *ws, size_t ws_bytes, int ydt,
                            cudaStream_t st)
{
    wl_status s = WL_OK;
    const DeviceInfo *di = device_info(&s);
    if (!di) return s;
    if (ws_bytes < decode_mlp_workspace_bytes(hidden, inter, r))
        return fail(WL_ERR_WORKSPACE, "MLP workspace too small");
    const int es = ydt == WL_OUT_F32 ? 4 : 2;
    for (int64_t t0 = 0; t0 < T; t0 += kTokChunk) {
        const int Tc = (int)((T - t0) < kTokChunk ? (T - t0) : kTokChunk);
        s = dec_mlp_once(x + t0 * hidden, gate, up, down,
                         static_cast<char *>(y) + (size_t)t0 * (size_t)hidden * es, Tc,
                         (int)hidden, (int)inter, (int)r, static_cast<char *>(ws), ydt, st, di);
        if (s != WL_OK) return s;
    }
    return WL_OK;
}

}  // namespace wl
