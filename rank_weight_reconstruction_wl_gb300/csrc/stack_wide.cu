// stack_wide.cu -- a whole stack of weightless decoder layers for 5..32
// tokens (batched decode) in ONE persistent launch per up to 24 layers.
//
// The phases of a layer are those of the one-to-four-token stack kernel
// ("In-kernel reconstruction", formula section, per projection):
//     QKV  x_l -> q, k, v     O  q -> o     GU  o -> g, u; h = gelu_tanh(g) u
//     D    h -> x_{l+1}
// and the weight stream is the same: the producer warp walks every phase's
// 64 x 64 W0 boxes (with the matching V^T rows) through a ring of
// shared-memory stages, waiting only for free stages.  What changes with the
// token count is what a box costs and how outputs travel between phases:
//
//   * All eight consumer warps work on every box: warp w multiplies the
//     box's rows 16 (w % 4) .. +16 with token group w / 4 (mma.sync
//     m16n8k16, W0 rows as M, tokens as N), and keeps its sums in registers
//     for the whole piece (the CTA's boxes of one row tile).  z = x V of the
//     piece's k range is formed the same way from the V^T rows of each stage.
//     No warp ever holds another warp's rows, so no cross-warp reduction is
//     needed.
//   * At the end of a piece, p = s * acc + U z_range (both terms linear in the
//     K split) is stored as an fp32 partial of the row tile.  The last CTA to
//     contribute to a row tile (an atomic count of contributions) sums the
//     partials in slot order, rounds to bf16 and writes the row tile's output
//     (for GU: h = gelu(g) u as a bf16 pair hi + lo, so that h keeps fp32
//     accuracy), then raises the row tile's flag.
//   * A phase starts by polling the flags of the input blocks its boxes need,
//     then copies those bf16 blocks into shared memory (cp.async).  D stages
//     h as two rows per token (hi, lo): an MMA lane then holds both columns of
//     a token, and their sum is the product with h.
//
// At 32 tokens every CTA needs about 80 KB of its phase input; reading it as
// bf16 outputs, summed once per row tile, costs a fraction of what summing
// the split-K partials in every reader would.
//
// Every wait is bounded (status word + the CTA winds down).  Flags and
// counts are cleared by the small kernel that also writes V^T before every
// step, so a step that gave up leaves nothing behind for the next one.
// Co-residency of all CTAs (needed for waits on other CTAs) is guaranteed by a
// cooperative launch of one CTA per SM.
#include <algorithm>
#include <cstring>
#include <vector>

#include "dec_ptx.cuh"

namespace wl {

constexpr int kWdThreads = kThreads + 32;  // 8 consumer warps + 1 producer warp
constexpr int kWdBox = 64;
constexpr int kWdBoxBytes = kWdBox * kWdBox * 2;
constexpr int kWdMaxPh = 96;    // phases per launch (24 layers)
constexpr int kWdRecHead = 8;   // record header ints
constexpr int kWdPiece = 12;    // ints per piece record

enum WdKind { kWdQKV = 0, kWdO = 1, kWdGU = 2, kWdD = 3 };

struct WdSeg {
    const CUtensorMap *map;    // W0 [out, K], box 64 x 64
    const CUtensorMap *vtmap;  // V^T [rpad, K], box 64 x rpad
    const float *s;
    const bf16 *U;
    bf16 *y;  // output [T, out] (GU: unused)
    int out, rt0, nrt;
};

struct WdPhase {
    WdSeg seg[3];
    int nseg, kind, K, KB, nrt, bpr, nbox, ncta, nsub;
    const bf16 *xin;          // input [T, K] (null: the launch's x)
    const unsigned *in_flag;  // flags of the producing phase (block kb = its row tile kb); null: no wait
    unsigned *flag;           // [nrt] 1 once the row tile's output is written
    unsigned *cnt;            // [nrt] partials stored so far
    float *part;              // [slot][nsub][T][64]
    bf16 *h;                  // GU: h [2][T, nrt * 64] (hi, then the rounding remainder lo)
    const bf16 *xin_lo;       // D: the lo part of h [T, K]
};

struct WdArgs {
    WdPhase ph[kWdMaxPh];
    int nph;
    const bf16 *x;  // [T, hidden]: input of the chunk's first layer
    int T, r, rpad;
    int nst, stage_bytes;
    int maxp, us_bytes, us_soff;
    int off_us, off_xs, off_z, off_rec, off_flags;  // shared-memory carve (bytes from the ring's base)
    int zstride;    // floats per z row (rpad + 1)
    const int *rec;  // per (phase, CTA) records, rec_ints each
    int rec_ints;
    unsigned *status;
};
static_assert(sizeof(WdArgs) <= 31 * 1024, "kernel parameter space");

// CTA c < n of a phase takes boxes [nbox*c/n, nbox*(c+1)/n).
__device__ __forceinline__ int wd_lo(int nbox, int c, int n) { return (int)((int64_t)nbox * (c < n ? c : n) / n); }

// Poll a row tile's flag (bounded); on success the flag's writes are visible
// to this thread (fence after the observation).
__device__ __forceinline__ bool wd_poll_flag(const unsigned *f, unsigned *status)
{
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    if (v == 0) {
        const long long t0 = wait_clock();
        for (;;) {
            asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
            if (v != 0) break;
            if (wait_clock() - t0 > kWaitLimitCycles) {
                atomicOr(status, kStatusTimeout | kWaitExchange);
                return false;
            }
        }
    }
    __threadfence();
    return true;
}

__device__ __forceinline__ float4 ld_cg4(const float *p) { return __ldcg(reinterpret_cast<const float4 *>(p)); }

// The last contributor of row tile rt: sum its np partials (slots slot0..)
// in slot order and write the row tile's bf16 output (GU: h).  All consumer
// threads.
__device__ __noinline__ void wd_finish(const WdPhase &P, int rt, int np, int slot0, int T)
{
    const size_t sstride = (size_t)P.nsub * T * kWdBox;
    const float *base = P.part + (size_t)slot0 * sstride;
    if (P.kind == kWdGU) {
        const int inter = P.nrt * kWdBox;
        bf16 *const h = P.h;
        for (int i = threadIdx.x; i < T * 16; i += kThreads) {
            const int t = i >> 4, r4 = (i & 15) * 4;
            float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
            for (int j = 0; j < np; ++j) {
                const float *p = base + j * sstride + t * kWdBox + r4;
                const float4 a = ld_cg4(p), b = ld_cg4(p + (size_t)T * kWdBox);
                g.x += a.x; g.y += a.y; g.z += a.z; g.w += a.w;
                u.x += b.x; u.y += b.y; u.z += b.z; u.w += b.w;
            }
            const float hf[4] = {gelu_tanh_f32(g.x) * u.x, gelu_tanh_f32(g.y) * u.y, gelu_tanh_f32(g.z) * u.z,
                                 gelu_tanh_f32(g.w) * u.w};
            __align__(8) bf16 hi[4];
            __align__(8) bf16 lo[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                hi[q] = __float2bfloat16_rn(hf[q]);
                lo[q] = __float2bfloat16_rn(hf[q] - __bfloat162float(hi[q]));
            }
            bf16 *hp = h + (size_t)t * inter + rt * kWdBox + r4;
            *reinterpret_cast<uint2 *>(hp) = *reinterpret_cast<uint2 *>(hi);
            *reinterpret_cast<uint2 *>(hp + (size_t)T * inter) = *reinterpret_cast<uint2 *>(lo);
        }
    } else {
        int si = 0;
        while (si + 1 < P.nseg && rt >= P.seg[si + 1].rt0) ++si;
        const WdSeg &sg = P.seg[si];
        const int row0 = (rt - sg.rt0) * kWdBox;
        const int out = sg.out;
        bf16 *const yb = sg.y;
        for (int i = threadIdx.x; i < T * 16; i += kThreads) {
            const int t = i >> 4, r4 = (i & 15) * 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j = 0; j < np; ++j) {
                const float4 a = ld_cg4(base + j * sstride + t * kWdBox + r4);
                v.x += a.x; v.y += a.y; v.z += a.z; v.w += a.w;
            }
            const float e[4] = {v.x, v.y, v.z, v.w};
            bf16 *y = yb + (size_t)t * out + row0 + r4;
            if (row0 + r4 + 4 <= out && ((out & 3) == 0)) {
                __align__(8) bf16 hv[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) hv[q] = __float2bfloat16_rn(e[q]);
                *reinterpret_cast<uint2 *>(y) = *reinterpret_cast<uint2 *>(hv);
            } else {
                for (int q = 0; q < 4; ++q)
                    if (row0 + r4 + q < out) y[q] = __float2bfloat16_rn(e[q]);
            }
        }
    }
}

// The boxes, partials and finishing of one phase (consumer threads).  NTW:
// n-tiles of 8 staged rows per warp; DL: the D phase, whose staged rows are
// (hi, lo) pairs per token.  false: a wait gave up (all consumer threads
// return false together).
template <int NTW, bool DL>
__device__ __forceinline__ bool wd_phase(const WdArgs &a, const WdPhase &P, const int *rec, int qbase, char *ring,
                                         uint64_t *full, uint64_t *empty, const char *aux_us, const uint32_t *xst,
                                         int xs32, float *zbuf, volatile int *flags)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8, lchunk = lane >> 4;
    const int mt = warp & 3, tg = warp >> 2;
    // Launch fields in registers: read through the parameter's address they
    // are generic loads, which the memory clobbers of the barrier operations
    // would otherwise force to repeat for every box.
    const int T = a.T, r = a.r, zs = a.zstride, nst = a.nst, sbytes = a.stage_bytes, KB = P.KB;
    const int us_bytes = a.us_bytes, us_soff = a.us_soff, nsub = P.nsub, kind = P.kind;
    unsigned *const status = a.status;
    float *const part = P.part;
    const int Tp = DL ? 2 * T : T;  // staged rows
    const int NT = (Tp + 7) >> 3;
    constexpr int ZPW = DL ? 2 : 1;      // z tiles per warp
    const int nzp = (a.rpad >> 4) * NT;  // z tiles (16 ranks x 8 rows): at most 8 (D: 16)
    const int npc = rec[2], kbs = rec[3];
    const int *pcs = rec + kWdRecHead;
    // B operands (staged rows = tokens, k contiguous) by ldmatrix: lane l
    // addresses row l % 8 of matrix l / 8; matrices alternate the k halves
    // (b0, b1) of consecutive n-tiles.  Rows past the staged ones hold stale
    // values that only reach output columns the epilogue ignores.
    const uint32_t xs_lane = smem_u32(xst) + (uint32_t)(((lane & 7) * xs32 + ((lane >> 3) & 1) * 4) * 4);
    const uint32_t xs_row8 = (uint32_t)(8 * xs32 * 4);  // bytes per n-tile of rows
    const int bnt = tg * NTW + (lane >> 4);             // n-tile of this lane's x4 address
    int zm[ZPW], zn[ZPW];
#pragma unroll
    for (int z = 0; z < ZPW; ++z) {
        zm[z] = (warp + 8 * z) / NT;
        zn[z] = warp + 8 * z - zm[z] * NT;
    }
    // ring position of the phase's first box (boxes are consumed in order)
    int s = qbase % nst;
    unsigned ph = (unsigned)((qbase / nst) & 1);
    const uint32_t ring0 = smem_u32(ring);

    for (int p = 0; p < npc; ++p) {
        const int *pc = pcs + p * kWdPiece;
        const int rt = pc[0], sub = pc[1], si = pc[2], row0 = pc[3], nb = pc[5], kb0 = pc[6];
        const int slot = pc[7], np = pc[8], slot0 = pc[9];
        float acc[NTW][4];
        float zacc[ZPW][4];
#pragma unroll
        for (int n = 0; n < NTW; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
        for (int z = 0; z < ZPW; ++z) zacc[z][0] = zacc[z][1] = zacc[z][2] = zacc[z][3] = 0.f;
        // staged position of the box's input block: (kb - kbs) mod KB
        int pos = kb0 - kbs;
        if (pos < 0) pos += KB;
        for (int j = 0; j < nb; ++j, pos = (pos + 1 == KB) ? 0 : pos + 1) {
            int w_ok = 1;
            if (lane == 0) w_ok = !flags[0] && ring_wait(&full[s], ph, status);
            w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
            if (!w_ok) {
                if (lane == 0) flags[0] = 1;
                break;
            }
            const uint32_t sb = ring0 + (uint32_t)(s * sbytes);
            const uint32_t xb = xs_lane + (uint32_t)(pos * 128);
            // KS k steps at a time: every fragment load of the group is issued
            // before its MMAs, so the loads' latency is paid once per group
            // (two steps where the fragments fit the register budget)
            constexpr int KS = (NTW >= 4) ? 1 : 2;
#pragma unroll
            for (int k2 = 0; k2 < 4; k2 += KS) {
                uint32_t af[KS][4], bf[KS][NTW < 2 ? 2 : NTW][2], av[KS][ZPW][4], bz[KS][ZPW][2];
#pragma unroll
                for (int h = 0; h < KS; ++h) {
                    const int kin = k2 + h;
                    const int chunk = kin * 2 + lchunk;
                    const int arow = mt * 16 + lrow;
                    ldmatrix_x4(af[h], sb + arow * 128 + ((chunk ^ (arow & 7)) << 4));
#pragma unroll
                    for (int n = 0; n < NTW; n += 2) {
                        if (tg * NTW + n < NT) {
                            if (NTW >= 2) {
                                uint32_t q4[4];
                                ldmatrix_x4(q4, xb + (uint32_t)(bnt + n) * xs_row8 + kin * 32);
                                bf[h][n][0] = q4[0];
                                bf[h][n][1] = q4[1];
                                bf[h][n + 1 < NTW ? n + 1 : n][0] = q4[2];
                                bf[h][n + 1 < NTW ? n + 1 : n][1] = q4[3];
                            } else {
                                ldmatrix_x2(bf[h][n], xb + (uint32_t)(tg * NTW) * xs_row8 + kin * 32);
                            }
                        }
                    }
#pragma unroll
                    for (int z = 0; z < ZPW; ++z) {
                        if (warp + 8 * z < nzp) {
                            const int zrow = zm[z] * 16 + lrow;
                            ldmatrix_x4(av[h][z], sb + kWdBoxBytes + zrow * 128 + ((chunk ^ (zrow & 7)) << 4));
                            ldmatrix_x2(bz[h][z], xb + (uint32_t)zn[z] * xs_row8 + kin * 32);
                        }
                    }
                }
#pragma unroll
                for (int h = 0; h < KS; ++h) {
#pragma unroll
                    for (int n = 0; n < NTW; ++n)
                        if (tg * NTW + n < NT) mma_16816(acc[n], af[h], bf[h][n][0], bf[h][n][1]);
#pragma unroll
                    for (int z = 0; z < ZPW; ++z)
                        if (warp + 8 * z < nzp) mma_16816(zacc[z], av[h][z], bz[h][z][0], bz[h][z][1]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            if (++s == nst) {
                s = 0;
                ph ^= 1u;
            }
        }
        // z tiles -> zbuf [staged row][rank]
#pragma unroll
        for (int z = 0; z < ZPW; ++z) {
            if (warp + 8 * z < nzp) {
                const int col = zn[z] * 8 + 2 * t4, rank = zm[z] * 16 + g;
                if (col < Tp) {
                    zbuf[col * zs + rank] = zacc[z][0];
                    zbuf[col * zs + rank + 8] = zacc[z][2];
                }
                if (col + 1 < Tp) {
                    zbuf[(col + 1) * zs + rank] = zacc[z][1];
                    zbuf[(col + 1) * zs + rank + 8] = zacc[z][3];
                }
            }
        }
        consumer_sync();
        if (flags[0]) return false;

        // p = s * acc + U z for this warp's rows and tokens
        const WdSeg &sg = P.seg[si];
        const char *us = aux_us + (size_t)p * us_bytes;
        const bf16 *Ur = reinterpret_cast<const bf16 *>(us + (reinterpret_cast<uintptr_t>(sg.U + (size_t)row0 * r) & 15));
        const float *sr = reinterpret_cast<const float *>(us + us_soff + (reinterpret_cast<uintptr_t>(sg.s + row0) & 15));
        const int sout = sg.out;
        float *dst = part + ((size_t)slot * nsub + sub) * T * kWdBox;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int row = mt * 16 + g + 8 * hh;
            const bool rv = row0 + row < sout;
            const float sv = rv ? sr[row] : 0.f;
#pragma unroll
            for (int n = 0; n < NTW; ++n) {
                const int nt = tg * NTW + n;
                if (nt >= NT) continue;
                if (DL) {
                    // columns 2 t4 (hi) and 2 t4 + 1 (lo) are the two parts of token nt * 4 + t4
                    const int t = nt * 4 + t4;
                    if (t >= T) continue;
                    float v = 0.f;
                    if (rv) {
                        v = sv * (acc[n][2 * hh] + acc[n][2 * hh + 1]);
                        const float *zh = zbuf + (2 * t) * zs, *zl = zh + zs;
                        for (int k = 0; k < r; ++k) v = fmaf(__bfloat162float(Ur[row * r + k]), zh[k] + zl[k], v);
                    }
                    dst[t * kWdBox + row] = v;
                } else {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int t = nt * 8 + 2 * t4 + e;
                        if (t >= T) continue;
                        float v = 0.f;
                        if (rv) {
                            v = sv * acc[n][2 * hh + e];
                            const float *zt = zbuf + t * zs;
                            for (int k = 0; k < r; ++k) v = fmaf(__bfloat162float(Ur[row * r + k]), zt[k], v);
                        }
                        dst[t * kWdBox + row] = v;
                    }
                }
            }
        }
        // GU: a CTA holding one part of a pair stores zeros for the other
        const bool next_same = p + 1 < npc && pcs[(p + 1) * kWdPiece] == rt;
        if (kind == kWdGU) {
            const bool has_other = sub == 0 ? next_same : (p > 0 && pcs[(p - 1) * kWdPiece] == rt);
            if (!has_other) {
                float *o = part + ((size_t)slot * nsub + (1 - sub)) * T * kWdBox;
                for (int i = tid; i < T * kWdBox; i += kThreads) o[i] = 0.f;
            }
        }
        consumer_sync();  // partials stored; zbuf free for the next piece
        if (!next_same) {
            // count this CTA's contribution; the last contributor finishes the row tile
            if (tid == 0) {
                __threadfence();
                const unsigned old = atomicAdd(P.cnt + rt, 1u);
                const int fin = old == (unsigned)(np - 1);
                if (fin) __threadfence();
                flags[1] = fin;
            }
            consumer_sync();
            if (flags[1]) {
                wd_finish(P, rt, np, slot0, T);
                consumer_sync();
                if (tid == 0) {
                    __threadfence();
                    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(P.flag + rt), "r"(1u) : "memory");
                }
            }
        }
    }
    return true;
}

__device__ __forceinline__ void wd_fetch_rec(int *recbuf, const int *rec, int rec_ints, int ph_i, int G, int c)
{
    const int *src = rec + ((size_t)ph_i * G + c) * rec_ints;
    int *dst = recbuf + (ph_i & 1) * rec_ints;
    for (int i = threadIdx.x; i < rec_ints / 4; i += kThreads) cp_async16(dst + 4 * i, src + 4 * i);
}

// NTW / NTWD: n-tiles per warp in the phases other than D / in D (twice the
// staged rows).  Nine warps put three on one SM sub-partition, whose 16K
// registers then allow at most 168 per thread.
template <int NTW, int NTWD>
__global__ void __launch_bounds__(kWdThreads, 1) stack_wide_kernel(const __grid_constant__ WdArgs a)
{
    extern __shared__ __align__(1024) char smem_raw[];
    char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, G = gridDim.x;
    const int T = a.T;

    char *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + (size_t)a.nst * a.stage_bytes);
    uint64_t *empty = full + a.nst;
    char *aux_us = smem + a.off_us;
    uint32_t *xst = reinterpret_cast<uint32_t *>(smem + a.off_xs);
    float *zbuf = reinterpret_cast<float *>(smem + a.off_z);
    int *recbuf = reinterpret_cast<int *>(smem + a.off_rec);
    // [0] consumers gave up, [1] finisher decision, [2] producer gave up
    volatile int *flags = reinterpret_cast<volatile int *>(smem + a.off_flags);

    if (tid == 0) {
        for (int i = 0; i < a.nst; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        flags[0] = flags[1] = flags[2] = 0;
    }
    __syncthreads();

    if (warp == kWarps) {
        // ------------------------------------------------------- producer
        if (lane != 0) return;
        const uint32_t w_base = smem_u32(ring);
        const int nst = a.nst, nph = a.nph, rpad = a.rpad;
        const unsigned sbytes = (unsigned)a.stage_bytes;
        unsigned *const status = a.status;
        int s = 0;
        unsigned ph = 0;
        int issued = 0;
        bool ok = true;
        for (int phi = 0; phi < nph && ok; ++phi) {
            const WdPhase &P = a.ph[phi];
            const int nbox = P.nbox, ncta = P.ncta;
            const int b0 = wd_lo(nbox, c, ncta), b1 = wd_lo(nbox, c + 1, ncta);
            if (b0 >= b1) continue;
            const bool gu = P.kind == kWdGU;
            const int KB = P.KB, bpr = P.bpr, nseg = P.nseg;
            const CUtensorMap *map[3], *vtm[3];
            int rt0[3];
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                map[j] = P.seg[j].map;
                vtm[j] = P.seg[j].vtmap;
                rt0[j] = j < nseg ? P.seg[j].rt0 : 0x7fffffff;
            }
            int rt = b0 / bpr, w = b0 - rt * bpr;
            for (int b = b0; b < b1; ++b) {
                int si, kb, row0;
                if (gu) {
                    si = w >= KB ? 1 : 0;
                    kb = w - si * KB;
                    row0 = rt * kWdBox;
                } else {
                    si = rt >= rt0[2] ? 2 : (rt >= rt0[1] ? 1 : 0);
                    kb = w;
                    row0 = (rt - (si == 2 ? rt0[2] : si == 1 ? rt0[1] : 0)) * kWdBox;
                }
                const CUtensorMap *m = si == 2 ? map[2] : si == 1 ? map[1] : map[0];
                const CUtensorMap *vm = si == 2 ? vtm[2] : si == 1 ? vtm[1] : vtm[0];
                if (flags[0] || !ring_wait_empty(&empty[s], ph ^ 1u, status)) {
                    ok = false;
                    break;
                }
                uint64_t *fb = &full[s];
                mbar_expect_tx(fb, sbytes);
                const uint32_t sdst = w_base + (uint32_t)s * sbytes;
                tma_load_2d_u32(sdst, m, kb * kWdBox, row0, fb);
                if (rpad) tma_load_2d_u32(sdst + kWdBoxBytes, vm, kb * kWdBox, 0, fb);
                ++issued;
                if (++s == nst) {
                    s = 0;
                    ph ^= 1u;
                }
                if (++w == bpr) {
                    w = 0;
                    ++rt;
                }
            }
        }
        if (!ok) {
            // let the copies in flight land before the CTA exits; a drain wait
            // that gives up is recorded with its own bit
            flags[2] = 1;
            const int n = issued < nst ? issued : nst;
            for (int i = 0; i < n; ++i) {
                s = (s == 0 ? nst : s) - 1;
                if (s == nst - 1) ph ^= 1u;
                if (!mbar_wait(&full[s], ph, status, kWaitRingFull)) atomicOr(status, kWaitDrain);
            }
        }
        return;
    }

    // ----------------------------------------------------------- consumers
    int qbase = 0;
    wd_fetch_rec(recbuf, a.rec, a.rec_ints, 0, G, c);
    cp_async_wait_all();
    consumer_sync();

    for (int phi = 0; phi < a.nph && !flags[0]; ++phi) {
        const WdPhase &P = a.ph[phi];
        const int *rec = recbuf + (phi & 1) * a.rec_ints;
        const int nbx = rec[1];
        if (phi + 1 < a.nph) wd_fetch_rec(recbuf, a.rec, a.rec_ints, phi + 1, G, c);  // lands by the phase's end
        if (nbx > 0) {
            const int npc = rec[2], kbs = rec[3], nk = rec[4];
            const int *pcs = rec + kWdRecHead;
            // U rows and s of every piece (independent of the input)
            for (int i = 0; i < npc; ++i) {
                const int *pc = pcs + i * kWdPiece;
                const WdSeg &sg = P.seg[pc[2]];
                const int row0 = pc[3];
                const int rows = min(kWdBox, sg.out - row0);
                char *dst = aux_us + (size_t)i * a.us_bytes;
                if (a.r > 0) prefetch(dst, sg.U + (size_t)row0 * a.r, rows * a.r * 2);
                prefetch(dst + a.us_soff, sg.s + row0, rows * 4);
            }
            // wait until the producing phase has written the input blocks
            if (P.in_flag) {
                const unsigned *const in_flag = P.in_flag;
                const int KB = P.KB;
                for (int i = tid; i < nk; i += kThreads) {
                    int kb = kbs + i;
                    if (kb >= KB) kb -= KB;
                    if (!wd_poll_flag(in_flag + kb, a.status)) {
                        flags[0] = 1;
                        break;
                    }
                }
                consumer_sync();
                if (flags[0]) break;
            }
            // stage input blocks kbs .. kbs + nk - 1 (mod KB) at positions 0 .. nk - 1;
            // D: row 2t holds h_hi of token t, row 2t + 1 its h_lo
            const bool dl = P.kind == kWdD;
            const int rows = dl ? 2 * T : T;
            const int xs32 = 32 * nk + 36;  // 4 mod 32: conflict-free B-operand reads
            const bf16 *const src = P.xin ? P.xin : a.x;
            const bf16 *const src_lo = P.xin_lo;
            const int K = P.K, KB = P.KB;
            const int nch = rows * nk * 8;
            for (int i = tid; i < nch; i += kThreads) {
                const int row = i / (nk * 8);
                const int rem = i - row * nk * 8;
                const int pos = rem >> 3, cc = rem & 7;
                int kb = kbs + pos;
                if (kb >= KB) kb -= KB;
                const int t = dl ? row >> 1 : row;
                const bf16 *sp = (dl && (row & 1)) ? src_lo : src;
                cp_async16(xst + row * xs32 + pos * 32 + cc * 4, sp + (size_t)t * K + kb * kWdBox + cc * 8);
            }
            cp_async_wait_all();
            consumer_sync();
            const bool ok = dl ? wd_phase<NTWD, true>(a, P, rec, qbase, ring, full, empty, aux_us, xst, xs32, zbuf, flags)
                               : wd_phase<NTW, false>(a, P, rec, qbase, ring, full, empty, aux_us, xst, xs32, zbuf, flags);
            qbase += nbx;
            if (!ok) break;
        }
        cp_async_wait_all();  // the next phase's record
        consumer_sync();
    }
    cp_async_wait_all();
}

// Before every step: V^T of every projection (padded with zero rows to rpad)
// and the flags and counts of the step cleared.
struct WdVtJob {
    const bf16 *V;  // [K, r]
    bf16 *VT;       // [rpad, K]
    int K;
};

__global__ void wd_prep_kernel(const WdVtJob *__restrict__ jobs, int njobs, int r, int rpad, unsigned *zero, int nzero)
{
    if ((int)blockIdx.y < njobs) {
        const WdVtJob jb = jobs[blockIdx.y];
        const int i = blockIdx.x * blockDim.x + threadIdx.x;
        if (i >= jb.K) return;
        for (int j = 0; j < rpad; ++j)
            jb.VT[(size_t)j * jb.K + i] = j < r ? jb.V[(size_t)i * r + j] : __float2bfloat16_rn(0.f);
    } else {
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nzero; i += gridDim.x * blockDim.x) zero[i] = 0u;
    }
}

// ------------------------------------------------------------------- host
struct WidePlan {
    int device = -1;
    int L = 0, T = 0, r = 0, rpad = 0, G = 0, smem = 0;
    std::vector<WdArgs> chunks;
    std::vector<const bf16 *> chunk_x;  // input of each chunk (null: the caller's x)
    const WdVtJob *jobs = nullptr;
    int njobs = 0, vt_maxk = 0;
    unsigned *zero = nullptr;
    int nzero = 0;
    void *dmem = nullptr;
};

static int wd_cdiv(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// n-tiles of 8 staged rows per warp (two token groups of four warps) for T
// tokens; D stages twice the rows.
static int wide_ntw(int T, bool d)
{
    if (d) return T <= 8 ? 1 : (T <= 16 ? 2 : 4);
    return T <= 16 ? 1 : 2;
}

// The instantiation for T tokens (template arguments as wide_ntw).
static const void *wide_kernel(int T)
{
    if (T <= 8) return (const void *)stack_wide_kernel<1, 1>;
    if (T <= 16) return (const void *)stack_wide_kernel<1, 2>;
    return (const void *)stack_wide_kernel<2, 4>;
}

wl_status wide_stack_create(WidePlan **out, const wl_layer *layers, const wl_layer_out *outs, int64_t L, int64_t T,
                            int64_t hidden, int64_t r, const DeviceInfo *di)
{
    *out = nullptr;
    const int64_t qd = layers[0].q.out, inter = layers[0].gate.out;
    const int G = di->sm_count;
    const int rpad = r == 0 ? 0 : (r <= 16 ? 16 : 32);

    // ---- phases: geometry, partial slots per row tile
    struct HP {
        WdPhase P;
        const wl_proj *proj[3];
        std::vector<int> np, slot0;
        int nslots;
    };
    std::vector<HP> hp(4 * L);
    for (int64_t l = 0; l < L; ++l) {
        const wl_layer &ly = layers[l];
        const wl_layer_out &o = outs[l];
        for (int k = 0; k < 4; ++k) {
            HP &h = hp[4 * l + k];
            WdPhase &P = h.P;
            memset(&P, 0, sizeof(P));
            P.kind = k;
            int64_t K = 0;
            if (k == kWdQKV) {
                K = hidden;
                P.nseg = 3;
                h.proj[0] = &ly.q;
                h.proj[1] = &ly.k;
                h.proj[2] = &ly.v;
                P.seg[0].y = static_cast<bf16 *>(o.yq);
                P.seg[1].y = static_cast<bf16 *>(o.yk);
                P.seg[2].y = static_cast<bf16 *>(o.yv);
            } else if (k == kWdO) {
                K = qd;
                P.nseg = 1;
                h.proj[0] = &ly.o;
                P.seg[0].y = static_cast<bf16 *>(o.yo);
            } else if (k == kWdGU) {
                K = hidden;
                P.nseg = 2;
                h.proj[0] = &ly.gate;
                h.proj[1] = &ly.up;
            } else {
                K = inter;
                P.nseg = 1;
                h.proj[0] = &ly.down;
                P.seg[0].y = static_cast<bf16 *>(o.ym);
            }
            P.K = (int)K;
            P.KB = (int)(K / kWdBox);
            int rt = 0;
            for (int j = 0; j < P.nseg; ++j) {
                P.seg[j].out = (int)h.proj[j]->out;
                P.seg[j].s = h.proj[j]->s;
                P.seg[j].U = static_cast<const bf16 *>(h.proj[j]->U);
                P.seg[j].nrt = wd_cdiv(h.proj[j]->out, kWdBox);
                P.seg[j].rt0 = (k == kWdGU) ? 0 : rt;
                if (k != kWdGU) rt += P.seg[j].nrt;
            }
            if (k == kWdGU) {
                P.nrt = P.seg[0].nrt;
                P.bpr = 2 * P.KB;
                P.nsub = 2;
            } else {
                P.nrt = rt;
                P.bpr = P.KB;
                P.nsub = 1;
            }
            P.nbox = P.nrt * P.bpr;
            const int want = (k == kWdO) ? (G + 1) / 2 : G;  // O is small: half the CTAs
            P.ncta = P.nbox < want ? P.nbox : want;
            h.np.resize(P.nrt);
            h.slot0.resize(P.nrt);
            int ns = 0;
            for (int t = 0; t < P.nrt; ++t) {
                const int bfirst = t * P.bpr, blast = bfirst + P.bpr - 1;
                const int c0 = (int)((((int64_t)bfirst + 1) * P.ncta - 1) / P.nbox);
                const int c1 = (int)((((int64_t)blast + 1) * P.ncta - 1) / P.nbox);
                h.np[t] = c1 - c0 + 1;
                h.slot0[t] = ns;
                ns += h.np[t];
            }
            h.nslots = ns;
        }
    }

    // ---- per (phase, CTA) work: pieces and staged input blocks
    auto owner = [](int b, int nbox, int n) { return (int)((((int64_t)b + 1) * n - 1) / nbox); };
    int maxp = 1, xs_max = 16;
    for (auto &h : hp) {
        const WdPhase &P = h.P;
        for (int cc = 0; cc < P.ncta; ++cc) {
            const int b0 = (int)((int64_t)P.nbox * cc / P.ncta), b1 = (int)((int64_t)P.nbox * (cc + 1) / P.ncta);
            if (b0 >= b1) continue;
            int n = 0;
            for (int b = b0; b < b1;) {
                const int rt = b / P.bpr, w = b - rt * P.bpr;
                int end = (rt + 1) * P.bpr;
                if (P.kind == kWdGU && w < P.KB) end = rt * P.bpr + P.KB;
                b = std::min(end, b1);
                ++n;
            }
            maxp = std::max(maxp, n);
            const int nk = std::min(b1 - b0, P.KB);
            // every row the B-operand loads can address: two token groups of NTW n-tiles
            const int rows = 16 * wide_ntw((int)T, P.kind == kWdD);
            xs_max = std::max(xs_max, rows * (32 * nk + 36) * 4);
        }
    }
    const int rec_ints = (kWdRecHead + kWdPiece * maxp + 3) / 4 * 4;
    auto make_rec = [&](int gi, int cc, int *rec) {
        const WdPhase &P = hp[gi].P;
        const int b0 = (int)((int64_t)P.nbox * std::min(cc, P.ncta) / P.ncta);
        const int b1 = (int)((int64_t)P.nbox * std::min(cc + 1, P.ncta) / P.ncta);
        memset(rec, 0, sizeof(int) * rec_ints);
        rec[0] = b0;
        rec[1] = b1 - b0;
        if (b1 <= b0) return;
        int n = 0;
        for (int b = b0; b < b1;) {
            const int rt = b / P.bpr, w = b - rt * P.bpr;
            const int sub = P.kind == kWdGU ? w / P.KB : 0;
            int end = (rt + 1) * P.bpr;
            if (P.kind == kWdGU && sub == 0) end = rt * P.bpr + P.KB;
            if (end > b1) end = b1;
            int si = sub;
            if (P.kind != kWdGU)
                while (si + 1 < P.nseg && rt >= P.seg[si + 1].rt0) ++si;
            int *pc = rec + kWdRecHead + kWdPiece * n;
            pc[0] = rt;
            pc[1] = sub;
            pc[2] = si;
            pc[3] = P.kind == kWdGU ? rt * kWdBox : (rt - P.seg[si].rt0) * kWdBox;
            pc[4] = b - b0;
            pc[5] = end - b;
            pc[6] = w - sub * P.KB;
            pc[7] = hp[gi].slot0[rt] + (cc - owner(rt * P.bpr, P.nbox, P.ncta));
            pc[8] = hp[gi].np[rt];
            pc[9] = hp[gi].slot0[rt];
            ++n;
            b = end;
        }
        rec[2] = n;
        rec[3] = (b0 % P.bpr) % P.KB;  // kbs
        rec[4] = std::min(b1 - b0, P.KB);  // nk
    };

    // ---- shared memory carve
    auto r16 = [](int v) { return (v + 15) / 16 * 16; };
    const int us_soff = r16((int)(kWdBox * r * 2) + 16);
    const int us_bytes = us_soff + r16(kWdBox * 4 + 16);
    const int zstride = rpad + 1;
    const int stage_bytes = kWdBoxBytes + rpad * 128;  // a 1024-byte multiple
    const int zbytes = r16(2 * (int)T * zstride * 4);
    const int fixed_tail = maxp * us_bytes + xs_max + zbytes + 2 * rec_ints * 4 + 16;
    int nst = (di->max_smem_optin - 1024 - fixed_tail) / (stage_bytes + 16);
    if (nst > 32) nst = 32;
    if (nst < 4)
        return fail(WL_ERR_UNSUPPORTED, "wl_stack_create: these shapes leave room for %d ring stages at T = %lld", nst,
                    (long long)T);
    int off = nst * stage_bytes + 16 * nst;
    const int off_us = off;
    off += maxp * us_bytes;
    const int off_xs = off;
    off += xs_max;
    const int off_z = off;
    off += zbytes;
    const int off_rec = off;
    off += 2 * rec_ints * 4;
    const int off_flags = off;
    off += 16;
    const int smem = 1024 + off;

    // ---- device memory
    size_t doff = 0;
    auto take = [&](size_t bytes, size_t align) {
        doff = (doff + align - 1) / align * align;
        const size_t o = doff;
        doff += bytes;
        return o;
    };
    const size_t o_maps = take(sizeof(CUtensorMap) * 7 * L, 128);
    const size_t o_vtmaps = take(sizeof(CUtensorMap) * 7 * L, 128);
    const size_t o_jobs = take(sizeof(WdVtJob) * 7 * L, 16);
    const size_t o_rec = take(sizeof(int) * (size_t)rec_ints * 4 * L * G, 256);
    const size_t o_tables_end = take(0, 256);
    std::vector<size_t> o_flag(4 * L), o_cnt(4 * L);
    for (size_t i = 0; i < hp.size(); ++i) {
        o_flag[i] = take(sizeof(unsigned) * hp[i].P.nrt, 4);
        o_cnt[i] = take(sizeof(unsigned) * hp[i].P.nrt, 4);
    }
    const size_t o_zero_end = take(0, 256);
    const int64_t kin[7] = {hidden, hidden, hidden, qd, hidden, hidden, inter};
    std::vector<size_t> o_vt(7 * L), o_part(4 * L), o_h(L);
    for (int64_t l = 0; l < L; ++l)
        for (int j = 0; j < 7; ++j) o_vt[7 * l + j] = take((size_t)rpad * kin[j] * 2, 256);
    for (size_t i = 0; i < hp.size(); ++i)
        o_part[i] = take(sizeof(float) * (size_t)hp[i].nslots * hp[i].P.nsub * T * kWdBox, 256);
    for (int64_t l = 0; l < L; ++l) o_h[l] = take((size_t)2 * T * inter * 2, 256);
    const size_t total = doff;

    void *dmem = nullptr;
    cudaError_t e = cudaMalloc(&dmem, total);
    if (e != cudaSuccess) return cuda_fail(e, "wl_stack_create: cudaMalloc of the stack's tables and scratch");
    char *base = static_cast<char *>(dmem);
    std::vector<char> host(o_tables_end, 0);
    for (int gi = 0; gi < 4 * L; ++gi)
        for (int cc = 0; cc < G; ++cc)
            make_rec(gi, cc, reinterpret_cast<int *>(host.data() + o_rec) + ((size_t)gi * G + cc) * rec_ints);
    CUtensorMap *hmaps = reinterpret_cast<CUtensorMap *>(host.data() + o_maps);
    CUtensorMap *hvt = reinterpret_cast<CUtensorMap *>(host.data() + o_vtmaps);
    WdVtJob *hjobs = reinterpret_cast<WdVtJob *>(host.data() + o_jobs);
    wl_status st = WL_OK;
    for (int64_t l = 0; l < L && st == WL_OK; ++l) {
        const wl_proj *pj[7] = {&layers[l].q, &layers[l].k, &layers[l].v, &layers[l].o,
                                &layers[l].gate, &layers[l].up, &layers[l].down};
        for (int j = 0; j < 7 && st == WL_OK; ++j) {
            st = tmap_2d_bf16(pj[j]->W0, kin[j], pj[j]->out, kin[j], kWdBox, kWdBox, &hmaps[7 * l + j]);
            if (st == WL_OK && rpad > 0) {
                bf16 *vt = reinterpret_cast<bf16 *>(base + o_vt[7 * l + j]);
                st = tmap_2d_bf16(vt, kin[j], rpad, kin[j], kWdBox, rpad, &hvt[7 * l + j]);
                hjobs[7 * l + j] = WdVtJob{static_cast<const bf16 *>(pj[j]->V), vt, (int)kin[j]};
            }
        }
    }
    if (st != WL_OK) {
        cudaFree(dmem);
        return st;
    }
    const int mj[4][3] = {{0, 1, 2}, {3, -1, -1}, {4, 5, -1}, {6, -1, -1}};
    for (size_t i = 0; i < hp.size(); ++i) {
        WdPhase &P = hp[i].P;
        const int64_t l = (int64_t)i / 4;
        const int k = (int)(i % 4);
        for (int j = 0; j < P.nseg; ++j) {
            P.seg[j].map = reinterpret_cast<const CUtensorMap *>(base + o_maps) + 7 * l + mj[k][j];
            P.seg[j].vtmap = rpad ? reinterpret_cast<const CUtensorMap *>(base + o_vtmaps) + 7 * l + mj[k][j] : nullptr;
        }
        P.flag = reinterpret_cast<unsigned *>(base + o_flag[i]);
        P.cnt = reinterpret_cast<unsigned *>(base + o_cnt[i]);
        P.part = reinterpret_cast<float *>(base + o_part[i]);
        if (k == kWdGU) P.h = reinterpret_cast<bf16 *>(base + o_h[l]);
        // the input: the previous phase's output (layer 0's QKV: the launch's x)
        if (k == kWdQKV) {
            P.xin = l > 0 ? static_cast<const bf16 *>(outs[l - 1].ym) : nullptr;
        } else if (k == kWdO) {
            P.xin = static_cast<const bf16 *>(outs[l].yq);  // q is QKV's first segment: block kb = row tile kb
        } else if (k == kWdGU) {
            P.xin = static_cast<const bf16 *>(outs[l].yo);
        } else {
            P.xin = reinterpret_cast<const bf16 *>(base + o_h[l]);
            P.xin_lo = P.xin + (size_t)T * inter;
        }
        P.in_flag = i > 0 ? reinterpret_cast<const unsigned *>(base + o_flag[i - 1]) : nullptr;
    }
    e = cudaMemcpy(dmem, host.data(), o_tables_end, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(base + o_tables_end, 0, total - o_tables_end);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaFree(dmem);
        return cuda_fail(e, "wl_stack_create: table upload");
    }
    const void *kern = wide_kernel((int)T);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, di->max_smem_optin);
    if (e != cudaSuccess) {
        cudaFree(dmem);
        return cuda_fail(e, "cudaFuncSetAttribute(stack_wide_kernel)");
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWdThreads, (size_t)smem);
    if (e != cudaSuccess || per_sm < 1) {
        cudaFree(dmem);
        return fail(WL_ERR_UNSUPPORTED, "wl_stack_create: the stack kernel does not fit on an SM (%d bytes)", smem);
    }

    WidePlan *pl = new (std::nothrow) WidePlan;
    if (!pl) {
        cudaFree(dmem);
        return fail(WL_ERR_INVALID_ARG, "wl_stack_create: out of host memory");
    }
    pl->device = di->device;
    pl->L = (int)L;
    pl->T = (int)T;
    pl->r = (int)r;
    pl->rpad = rpad;
    pl->G = G;
    pl->smem = smem;
    pl->dmem = dmem;
    pl->jobs = reinterpret_cast<const WdVtJob *>(base + o_jobs);
    pl->njobs = rpad ? (int)(7 * L) : 0;
    pl->vt_maxk = (int)std::max(hidden, std::max(qd, inter));
    pl->zero = reinterpret_cast<unsigned *>(base + o_flag[0]);
    pl->nzero = (int)((o_zero_end - o_flag[0]) / sizeof(unsigned));

    // launches: chunks of at most kWdMaxPh / 4 layers, of about equal size
    const int lmax = kWdMaxPh / 4;
    const int nchunk = wd_cdiv(L, lmax);
    WdArgs a;
    memset(&a, 0, sizeof(a));
    a.T = (int)T;
    a.r = (int)r;
    a.rpad = rpad;
    a.nst = nst;
    a.stage_bytes = stage_bytes;
    a.maxp = maxp;
    a.us_bytes = us_bytes;
    a.us_soff = us_soff;
    a.off_us = off_us;
    a.off_xs = off_xs;
    a.off_z = off_z;
    a.off_rec = off_rec;
    a.off_flags = off_flags;
    a.zstride = zstride;
    a.rec_ints = rec_ints;
    a.status = di->status;
    for (int ch = 0; ch < nchunk; ++ch) {
        const int l0 = (int)(L * ch / nchunk), l1 = (int)(L * (ch + 1) / nchunk);
        const int base_ph = 4 * l0;
        a.nph = 4 * (l1 - l0);
        a.rec = reinterpret_cast<const int *>(base + o_rec) + (size_t)base_ph * G * rec_ints;
        for (int i = 0; i < a.nph; ++i) {
            WdPhase P = hp[base_ph + i].P;
            if (i == 0) {
                // the chunk's input: x, or the previous chunk's output (complete:
                // that launch has finished)
                P.xin = nullptr;
                P.in_flag = nullptr;
            }
            a.ph[i] = P;
        }
        pl->chunks.push_back(a);
        pl->chunk_x.push_back(l0 == 0 ? nullptr : static_cast<const bf16 *>(outs[l0 - 1].ym));
    }
    *out = pl;
    return WL_OK;
}

wl_status wide_stack_decode(WidePlan *pl, const void *x, cudaStream_t stream)
{
    {
        // V^T of this step's V, flags and counts cleared
        const int gx = std::max(1, (pl->vt_maxk + 255) / 256);
        dim3 grid((unsigned)gx, (unsigned)(pl->njobs + 1));
        wd_prep_kernel<<<grid, 256, 0, stream>>>(pl->jobs, pl->njobs, pl->r, pl->rpad, pl->zero, pl->nzero);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "wl_stack_decode: prep launch");
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl->G);
    cfg.blockDim = dim3(kWdThreads);
    cfg.dynamicSmemBytes = (size_t)pl->smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const void *kern = wide_kernel(pl->T);
    for (size_t ch = 0; ch < pl->chunks.size(); ++ch) {
        WdArgs a = pl->chunks[ch];
        a.x = pl->chunk_x[ch] ? pl->chunk_x[ch] : static_cast<const bf16 *>(x);
        void *args[] = {&a};
        cudaError_t e = cudaLaunchKernelExC(&cfg, kern, args);
        if (e != cudaSuccess) return cuda_fail(e, "wl_stack_decode: launch");
    }
    return WL_OK;
}

void wide_stack_destroy(WidePlan *pl)
{
    if (!pl) return;
    if (pl->dmem) cudaFree(pl->dmem);
    delete pl;
}

int wide_stack_device(const WidePlan *pl) { return pl->device; }

}  // namespace wl
