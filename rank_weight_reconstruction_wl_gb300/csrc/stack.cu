// stack.cu -- a whole stack of weightless decoder layers at decode size
// (T <= 4 tokens) in ONE persistent launch.
//
// Each layer runs four projection phases ("In-kernel reconstruction", formula
// section, per projection):
//     QKV  x_l  -> q, k, v          (three bundles sharing x_l)
//     O    q    -> o                (q stands in for the attention output)
//     GU   o    -> g, u;  h = gelu_tanh(g) * u
//     D    h    -> x_{l+1}
// At decode size the cost is streaming every W0 from HBM once; with one
// launch per projection the fixed cost of each launch (start-up, the wait
// for x behind the weight stream, the epilogue) dominates ("What weightless
// inference costs": extra dispatches, not arithmetic, dominate at batch 1).
// Here the weights of all layers form one stream that never waits for the
// data dependencies between projections:
//
//   producer warp   walks the CTA's share of every phase in order and loads
//                   each 64x64 W0 box with the matching 64 columns of V^T
//                   (both TMA, 128-byte swizzle) into a ring of shared-memory
//                   stages, waiting only for free stages;
//   8 consumer warps  per phase: gather the phase input; then each warp takes
//                   whole boxes (box j of the phase goes to warp j % 8) and
//                   multiplies them on the tensor cores (mma.sync m16n8k16,
//                   W0 rows, and the rank rows of V^T for z = x V, as M;
//                   tokens as N); at the end of the phase the warps' sums are added
//                   in warp order and p = s * acc + U z_range goes to a
//                   global partial slot per (row tile, CTA).
//
// Work split.  A phase's boxes are numbered row tile by row tile (for GU a
// row tile is a pair: the gate tile's boxes, then the up tile's) and the
// phase's n CTAs take equal contiguous ranges: every CTA streams about the
// same number of bytes.  A row tile is shared by the few CTAs whose ranges
// touch it; each adds one partial (both terms of the projection are linear
// in the K split).
//
// Publication without fences.  Every partial value is stored as one 64-bit
// word holding the value and the launch's epoch.  A consumer polls the words
// it needs until all carry the current epoch, then sums them in slot order
// (every CTA sums in the same order, so all agree bit for bit) and rounds to
// bf16 as the projection output is defined.  The CTA that owns box kb of the
// phase's first row tile also stores input block kb to the previous phase's
// output buffer, so every output element is written exactly once; k, v and
// the last layer's output, which no phase reads, are stored by CTAs assigned
// to them after their own work.  Slots and outputs are distinct per layer
// and phase, so no write can overtake a read of an earlier layer, and the
// epoch makes values left by an earlier launch invisible.
//
// The down projection takes h as two bf16 columns per token (h = hi + lo), so
// its tensor-core product keeps fp32 accuracy (for z as well).
//
// V^T: each launch is preceded by a small kernel that writes V^T of every
// projection, padded to 16 or 32 rank rows, into the stack's scratch, so that
// V is read when the step runs and its 64-column blocks are TMA tiles.
//
// Every wait (ring stages, partial words) is bounded; a wait that gives up
// sets the status word and the CTA winds down after its copies in flight
// land.  Co-residency of all CTAs (needed for the waits on other CTAs'
// partials) is guaranteed by a cooperative launch of one CTA per SM.
#include <cstring>
#include <mutex>
#include <vector>

#include "dec_ptx.cuh"

namespace wl {

// Ring stages for `warps` consumer warps that take boxes round-robin: a
// multiple of the warp count.  Box j of a phase goes to warp j % warps and to
// stage (phase start + j) % nst, so every use of a stage within a phase falls
// to one warp, in order.  Otherwise a warp could wait for a stage's next use
// before the previous one (another warp's box) has landed, and a parity wait
// cannot tell that phase from the one two uses back: it would return at once,
// read the stage early and release it out of turn.  wl_stack_decode checks
// the rule again before every launch.
static inline int round_ring_to_warps(int nst, int warps) { return nst / warps * warps; }

constexpr int kStThreads = kThreads + 32;  // 8 consumer warps + 1 producer warp
constexpr int kStMaxT = 4;                 // tokens per launch
constexpr int kStMaxR = 32;                // rank
constexpr int kStBox = 64;                 // rows and columns of a W0 box
constexpr int kStBoxBytes = kStBox * kStBox * 2;

enum StKind { kQKV = 0, kO = 1, kGU = 2, kD = 3 };

struct StSeg {
    const CUtensorMap *map;    // W0 [out, K], box 64 x 64 (device memory)
    const CUtensorMap *vtmap;  // V^T [rpad, K] (padded with zero rows), box 64 x rpad
    const float *s;
    const bf16 *U;
    bf16 *y;   // output [T, out] (bf16)
    int out;
    int rt0;   // first row tile of this segment within the phase
    int nrt;   // row tiles
};

struct StPhase {
    StSeg seg[3];
    int nseg, kind;
    int K, KB;     // input length and 64-wide k blocks
    int nrt;       // row tiles (GU: gate/up pairs)
    int bpr;       // boxes per row tile (GU: 2 * KB)
    int nbox;      // nrt * bpr
    int ncta;      // CTAs sharing the phase (<= grid, <= nbox: none has an empty range)
    int nsub;      // parts per slot (GU: 2, gate and up)
    int prev;      // phase producing the input, -1: the launch's x
    bf16 *wy;      // the input vector's buffer (owner of box kb stores block kb), or null
    int xw_ph, xw_rt0, xw_n;  // after its work, CTA c stores row tiles xw_rt0 + c (+ grid...) of phase xw_ph
    const int *np;     // [nrt] partials per row tile
    const int *slot0;  // [nrt] first slot of the row tile
    unsigned long long *part;  // [slot][nsub][T][64] words: epoch << 32 | fp32 bits
};

// Phases per launch: the descriptors travel as a kernel parameter (read
// through the constant cache; shared memory leaves little L1 for tables in
// global memory), and the parameter space holds 24 layers.
constexpr int kStMaxPh = 96;

struct StArgs {
    StPhase ph[kStMaxPh];
    int nph;
    const bf16 *x;  // [T, hidden] input of layer 0
    int T, r;
    unsigned epoch;
    int nst;        // ring stages
    int maxp;       // most pieces of one CTA in one phase
    int xs32;       // x stage row stride (u32)
    int us_bytes;   // bytes per piece in the U/s area
    int wb_floats;  // floats per (piece, warp) partial block: [2T][64] sums, then [2T][rpad] z
    int wb_zoff;    // offset of the z part (2T * 64)
    int rpad;       // V^T rows per box (0, 16 or 32)
    int stage_bytes;  // W0 box + V^T box
    int maxnk;      // most input blocks one CTA stages in one phase
    const int *rec; // per (phase, CTA) work records, rec_ints each (see Piece)
    int rec_ints;
    unsigned *status;
};
static_assert(sizeof(StPhase) <= 256, "phase descriptor grew");
static_assert(sizeof(StArgs) <= 31 * 1024, "kernel parameter space");

// ----------------------------------------------------------- small helpers
// A phase's nbox boxes are shared by its first n CTAs: CTA c < n takes
// [nbox*c/n, nbox*(c+1)/n) (at least one box, as n <= nbox); the others none.
// The CTA holding box b is ((b + 1) * n - 1) / nbox.
__device__ __forceinline__ int st_lo(int nbox, int c, int n)
{
    return (int)((int64_t)nbox * (c < n ? c : n) / n);
}

// Partial words: one 64-bit store carries the value and the epoch together.
__device__ __forceinline__ void st_word(unsigned long long *p, float v, unsigned epoch)
{
    const unsigned long long w = ((unsigned long long)epoch << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ ulonglong2 ld_words2(const unsigned long long *p)
{
    ulonglong2 v;
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_word(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ float word_val(unsigned long long w) { return __uint_as_float((unsigned)w); }
__device__ __forceinline__ bool word_ok(unsigned long long w, unsigned epoch) { return (unsigned)(w >> 32) == epoch; }

// One element (part 0) of a row tile of phase Q (n partials from slot0),
// polled until it carries the epoch (bounded).
__device__ __forceinline__ float sum1(const StPhase &Q, int n, int slot0, int t, int i, int T, unsigned epoch,
                                      bool *ok_out, unsigned *status)
{
    const size_t stride = (size_t)Q.nsub * T * kStBox;
    const unsigned long long *p = Q.part + (size_t)slot0 * Q.nsub * T * kStBox + t * kStBox + i;
    long long t0 = -1;
    for (;;) {
        float s = 0.f;
        bool ok = true;
#pragma unroll 4
        for (int j = 0; j < n; ++j) {
            const unsigned long long w = ld_word(p + j * stride);
            ok = ok && word_ok(w, epoch);
            s += word_val(w);
        }
        if (ok) return s;
        if (t0 < 0) t0 = wait_clock();
        else if (wait_clock() - t0 > kWaitLimitCycles) {
            atomicOr(status, kStatusTimeout | kWaitExchange);
            *ok_out = false;
            return 0.f;
        }
    }
}

// This warp's sums for one piece into its partial block (zeros: the warp had
// no box of the piece).  Column c of the MMA result is token c (D: c >= T are
// the lo columns); rows of zc are ranks.
__device__ __forceinline__ void flush_piece(float *wb, int zoff, const float (&cacc)[4][4], const float (&zc)[2][4],
                                            bool zeros, int Tp, int rpad, int lane)
{
    const int g = lane >> 2, t4 = lane & 3;
    const int col = 2 * t4;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const int row = m * 16 + g;
        if (col < Tp) {
            wb[col * kStBox + row] = zeros ? 0.f : cacc[m][0];
            wb[col * kStBox + row + 8] = zeros ? 0.f : cacc[m][2];
        }
        if (col + 1 < Tp) {
            wb[(col + 1) * kStBox + row] = zeros ? 0.f : cacc[m][1];
            wb[(col + 1) * kStBox + row + 8] = zeros ? 0.f : cacc[m][3];
        }
    }
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        if (m * 16 < rpad) {
            float *wz = wb + zoff;  // [2T][rpad]
            const int j = m * 16 + g;
            if (col < Tp) {
                wz[col * rpad + j] = zeros ? 0.f : zc[m][0];
                wz[col * rpad + j + 8] = zeros ? 0.f : zc[m][2];
            }
            if (col + 1 < Tp) {
                wz[(col + 1) * rpad + j] = zeros ? 0.f : zc[m][1];
                wz[(col + 1) * rpad + j + 8] = zeros ? 0.f : zc[m][3];
            }
        }
    }
}

// Sums of partial words for NQ groups of 4 rows (i0 ..) of token t and NS
// parts of a row tile of phase Q (n partials from slot0).  The loads of up to
// CH slots are issued before any of them is used, and the epochs are checked
// without branching, so a ready input costs one L2 round trip per CH slots
// rather than one per slot pair (the poll sits on the path between phases).
// Sums run in slot order.  false: gave up (status set).
template <int NQ, int NS>
__device__ __forceinline__ bool sumq(const StPhase &Q, int n, int slot0, int t, int i0, int T, unsigned epoch,
                                     float (&out)[NS][NQ * 4], unsigned *status)
{
    constexpr int CH = 4 / (NQ * NS) > 0 ? 4 / (NQ * NS) : 1;  // slots in flight: 8 loads of 16 bytes
    const size_t stride = (size_t)Q.nsub * T * kStBox;
    const unsigned long long *base = Q.part + (size_t)slot0 * Q.nsub * T * kStBox + t * kStBox + i0;
    long long t0 = -1;
    for (;;) {
        float acc[NS][NQ * 4];
#pragma unroll
        for (int ps = 0; ps < NS; ++ps)
#pragma unroll
            for (int e = 0; e < NQ * 4; ++e) acc[ps][e] = 0.f;
        unsigned bad = 0;
        for (int j0 = 0; j0 < n; j0 += CH) {
            ulonglong2 w[CH][NS][NQ][2];
#pragma unroll
            for (int jj = 0; jj < CH; ++jj)
#pragma unroll
                for (int ps = 0; ps < NS; ++ps)
#pragma unroll
                    for (int q = 0; q < NQ; ++q) {
                        if (j0 + jj < n) {
                            const unsigned long long *pp = base + (j0 + jj) * stride + (size_t)ps * T * kStBox + 4 * q;
                            w[jj][ps][q][0] = ld_words2(pp);
                            w[jj][ps][q][1] = ld_words2(pp + 2);
                        }
                    }
#pragma unroll
            for (int jj = 0; jj < CH; ++jj) {
                if (j0 + jj < n)
#pragma unroll
                for (int ps = 0; ps < NS; ++ps)
#pragma unroll
                    for (int q = 0; q < NQ; ++q) {
                        const ulonglong2 u = w[jj][ps][q][0], v = w[jj][ps][q][1];
                        bad |= ((unsigned)(u.x >> 32) ^ epoch) | ((unsigned)(u.y >> 32) ^ epoch) |
                               ((unsigned)(v.x >> 32) ^ epoch) | ((unsigned)(v.y >> 32) ^ epoch);
                        acc[ps][4 * q] += word_val(u.x);
                        acc[ps][4 * q + 1] += word_val(u.y);
                        acc[ps][4 * q + 2] += word_val(v.x);
                        acc[ps][4 * q + 3] += word_val(v.y);
                    }
            }
        }
        if (!bad) {
#pragma unroll
            for (int ps = 0; ps < NS; ++ps)
#pragma unroll
                for (int e = 0; e < NQ * 4; ++e) out[ps][e] = acc[ps][e];
            return true;
        }
        if (t0 < 0) t0 = wait_clock();
        else if (wait_clock() - t0 > kWaitLimitCycles) {
            atomicOr(status, kStatusTimeout | kWaitExchange);
            return false;
        }
    }
}

// The phase input from the previous phase's partials: items of NQ groups of 4
// elements of one token of one staged block (consumer threads).  D forms
// h = gelu(g) u from the gate and up parts and stages it as bf16 hi + lo;
// the others round to bf16, and the owner of box kb of the first row tile
// stores block kb to the previous phase's output.  false: a wait gave up.
template <int NQ>
__device__ __forceinline__ bool gather_items(const StPhase &P, const StPhase &Q, const int *gnp, const int *gs0,
                                             int kbs, int nk, int T, int b0, int b1, bf16 *xs, int xsb,
                                             unsigned epoch, unsigned *status)
{
    constexpr int per_tok = 16 / NQ;  // items per token and block
    const int KB = P.KB;
    for (int it = threadIdx.x; it < nk * T * per_tok; it += kThreads) {
        const int pos = it / (T * per_tok);
        const int rem = it - pos * T * per_tok;
        const int t = rem / per_tok, i0 = (rem % per_tok) * 4 * NQ;
        int kb = kbs + pos;
        if (kb >= KB) kb -= KB;
        const int col = pos * kStBox + i0;
        const int qn = gnp[pos], qs = gs0[pos];
        if (P.kind == kD) {
            float gu[2][NQ * 4];
            if (!sumq<NQ, 2>(Q, qn, qs, t, i0, T, epoch, gu, status)) return false;
#pragma unroll
            for (int e = 0; e < NQ * 4; ++e) {
                const float hv = gelu_tanh_f32(gu[0][e]) * gu[1][e];
                const bf16 hi = __float2bfloat16_rn(hv);
                xs[t * xsb + col + e] = hi;
                xs[(T + t) * xsb + col + e] = __float2bfloat16_rn(hv - __bfloat162float(hi));
            }
        } else {
            float v[1][NQ * 4];
            if (!sumq<NQ, 1>(Q, qn, qs, t, i0, T, epoch, v, status)) return false;
            const bool wr = P.wy && kb >= b0 && kb < b1;
#pragma unroll
            for (int e = 0; e < NQ * 4; ++e) {
                const bf16 b = __float2bfloat16_rn(v[0][e]);
                xs[t * xsb + col + e] = b;
                if (wr) P.wy[(size_t)t * P.K + (size_t)kb * kStBox + i0 + e] = b;
            }
        }
    }
    return true;
}

// ------------------------------------------------------------------ kernel
// Start copying the record of phase ph_i of CTA c into its buffer (consumer
// threads; completes with cp_async_wait_all).
__device__ __forceinline__ void fetch_rec(int *recbuf, const int *rec, int rec_ints, int ph_i, int G, int c)
{
    const int *src = rec + ((size_t)ph_i * G + c) * rec_ints;
    int *dst = recbuf + (ph_i & 1) * rec_ints;
    for (int i = threadIdx.x; i < rec_ints / 4; i += kThreads) cp_async16(dst + 4 * i, src + 4 * i);
}

struct Piece {
    int rt, sub, si, row0, j0, nb, kb0;  // boxes j0 .. j0+nb-1 of the CTA's phase range, k blocks kb0..
    int slot;                            // this CTA's partial slot of the row tile
};

// A CTA's work in one phase, worked out on the host (int32 words):
//   [0] b0  [1] boxes  [2] pieces  [3] kbs  [4] nk  [5..7] unused
//   [8 ..]            maxp Pieces (8 words each)
//   then              maxnk partial counts of the staged input blocks
//   then              maxnk first slots of the staged input blocks
// Records are fetched one phase ahead into shared memory (cp.async), so no
// table lookup in global memory sits on the path between two phases.
constexpr int kRecHead = 8;

__global__ void __launch_bounds__(kStThreads, 1) stack_kernel(const __grid_constant__ StArgs a)
{
    extern __shared__ __align__(1024) char smem_raw[];
    char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, G = gridDim.x;
    const int T = a.T, r = a.r;
    const int sbytes_stage = a.stage_bytes;

    // shared memory carve
    char *ring_w = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(ring_w + (size_t)a.nst * sbytes_stage);
    uint64_t *empty = full + a.nst;
    char *aux_us = reinterpret_cast<char *>(empty + a.nst);
    uint32_t *xst = reinterpret_cast<uint32_t *>(aux_us + (size_t)a.maxp * a.us_bytes);
    float *wbuf = reinterpret_cast<float *>(xst + (size_t)(2 * T) * a.xs32);  // [maxp][8][wb_floats]
    float *zsum = wbuf + (size_t)a.maxp * kWarps * a.wb_floats;                     // [maxp][T][r] (r > 8)
    int *recbuf = reinterpret_cast<int *>(zsum + a.maxp * kStMaxT * kStMaxR);  // 2 x rec_ints
    // [0] consumers gave up (written only by consumers; read for control
    // right after a consumer barrier), [2] producer gave up
    volatile int *flags = reinterpret_cast<volatile int *>(recbuf + 2 * a.rec_ints);

    if (tid == 0) {
        for (int i = 0; i < a.nst; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        flags[0] = flags[1] = flags[2] = 0;
    }
    __syncthreads();

    if (warp == kWarps) {
        // ------------------------------------------------------- producer
        // Per box only register arithmetic and the copies: the phase's fields
        // are read once per phase, box coordinates advance incrementally.
        if (lane != 0) return;
        const unsigned sbytes = (unsigned)sbytes_stage;
        const uint32_t w_base = smem_u32(ring_w);
        int s = 0;
        unsigned ph = 0;
        int issued = 0;
        bool ok = true;
        for (int phi = 0; phi < a.nph && ok; ++phi) {
            const int nbox = a.ph[phi].nbox, ncta = a.ph[phi].ncta;
            const int b0 = st_lo(nbox, c, ncta), b1 = st_lo(nbox, c + 1, ncta);
            if (b0 >= b1) continue;
            const bool gu = a.ph[phi].kind == kGU;
            const int KB = a.ph[phi].KB, bpr = a.ph[phi].bpr, nseg = a.ph[phi].nseg;
            const CUtensorMap *map[3], *vtm[3];
            int rt0[3];
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                map[j] = a.ph[phi].seg[j].map;
                vtm[j] = a.ph[phi].seg[j].vtmap;
                rt0[j] = j < nseg ? a.ph[phi].seg[j].rt0 : 0x7fffffff;
            }
            // Every box of the phase beyond one ring's worth, into L2 now: the
            // producer reaches a phase while the consumers are still on the
            // previous one or waiting for its partial sums, when HBM has little
            // else to do; the ring's refill for those boxes then comes from L2.
            // Only W0, and only with a ring of 16 stages or more: with a short
            // ring (large ranks) the extra copies cost more than they save.
            if (a.nst >= 16 && b1 - b0 > a.nst) {
                int rtq = (b0 + a.nst) / bpr, wq = (b0 + a.nst) - rtq * bpr;
                for (int bq = b0 + a.nst; bq < b1; ++bq) {
                    int sq, kq, rq;
                    if (gu) {
                        sq = wq >= KB ? 1 : 0;
                        kq = wq - sq * KB;
                        rq = rtq * kStBox;
                    } else {
                        sq = rtq >= rt0[2] ? 2 : (rtq >= rt0[1] ? 1 : 0);
                        kq = wq;
                        rq = (rtq - (sq == 2 ? rt0[2] : sq == 1 ? rt0[1] : 0)) * kStBox;
                    }
                    tma_prefetch_2d(sq == 2 ? map[2] : sq == 1 ? map[1] : map[0], kq * kStBox, rq);
                    if (++wq == bpr) {
                        wq = 0;
                        ++rtq;
                    }
                }
            }
            int rt = b0 / bpr, w = b0 - rt * bpr;
            for (int b = b0; b < b1; ++b) {
                // segment, row offset and k block of box (rt, w)
                int si, kb, row0;
                if (gu) {
                    si = w >= KB ? 1 : 0;
                    kb = w - si * KB;
                    row0 = rt * kStBox;
                } else {
                    si = rt >= rt0[2] ? 2 : (rt >= rt0[1] ? 1 : 0);
                    kb = w;
                    row0 = (rt - (si == 2 ? rt0[2] : si == 1 ? rt0[1] : 0)) * kStBox;
                }
                const CUtensorMap *m = si == 2 ? map[2] : si == 1 ? map[1] : map[0];
                const CUtensorMap *vm = si == 2 ? vtm[2] : si == 1 ? vtm[1] : vtm[0];
                if (flags[0] || !ring_wait_empty(&empty[s], ph ^ 1u, a.status)) {
                    ok = false;
                    break;
                }
                uint64_t *fb = &full[s];
                mbar_expect_tx(fb, sbytes);
                const uint32_t sdst = w_base + (uint32_t)s * (uint32_t)sbytes_stage;
                tma_load_2d_u32(sdst, m, kb * kStBox, row0, fb);
                if (a.rpad) tma_load_2d_u32(sdst + kStBoxBytes, vm, kb * kStBox, 0, fb);
                ++issued;
                if (++s == a.nst) {
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
            // let the copies in flight land before the CTA exits
            flags[2] = 1;
            const int n = issued < a.nst ? issued : a.nst;
            for (int i = 0; i < n; ++i) {
                s = (s == 0 ? a.nst : s) - 1;
                if (s == a.nst - 1) ph ^= 1u;
                if (!mbar_wait(&full[s], ph, a.status, kWaitRingFull)) atomicOr(a.status, kWaitDrain);
            }
        }
        return;
    }

    // ----------------------------------------------------------- consumers
    const int g = lane >> 2, t4 = lane & 3;
    const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8;  // ldmatrix row within a 16-row group
    const int lchunk = lane >> 4;
    int qbase = 0;  // CTA-local sequence number of the phase's first box
    fetch_rec(recbuf, a.rec, a.rec_ints, 0, G, c);
    cp_async_wait_all();
    consumer_sync();

    for (int phi = 0; phi < a.nph && !flags[0]; ++phi) {
        const StPhase &P = a.ph[phi];
        const int *rec = recbuf + (phi & 1) * a.rec_ints;
        const int b0 = rec[0], nbx = rec[1];
        const int b1 = b0 + nbx;
        const int kind = P.kind, KB = P.KB, Tp = kind == kD ? 2 * T : T;
        if (phi + 1 < a.nph) fetch_rec(recbuf, a.rec, a.rec_ints, phi + 1, G, c);  // lands by the phase's end
        if (nbx > 0) {
            // input blocks kbs .. kbs + nk - 1 (mod KB), staged at positions 0..nk-1
            const int npc = rec[2], kbs = rec[3], nk = rec[4];
            const Piece *pcs = reinterpret_cast<const Piece *>(rec + kRecHead);
            const int *gnp = rec + kRecHead + 8 * a.maxp;  // partials of each staged input block
            const int *gs0 = gnp + a.maxnk;                 // their first slot

            // prefetch U rows and s of every piece (independent of the input)
            for (int i = 0; i < npc; ++i) {
                const Piece pc = pcs[i];
                const StSeg &sg = P.seg[pc.si];
                const int rows = min(kStBox, sg.out - pc.row0);
                char *dst = aux_us + (size_t)i * a.us_bytes;
                if (r > 0) prefetch(dst, sg.U + (size_t)pc.row0 * r, rows * r * 2);
                prefetch(dst + ((kStBox * r * 2 + 16 + 15) & ~15), sg.s + pc.row0, rows * 4);
            }

            bf16 *xs = reinterpret_cast<bf16 *>(xst);
            const int xsb = 2 * a.xs32;  // x stage row stride (bf16)
            if (P.prev >= 0) {
                const StPhase &Q = a.ph[P.prev];
                // one item per thread where possible (a ready input then costs
                // one round trip): 8 elements per item when 4 would not fit
                const bool ok = (nk * T * 16 > kThreads)
                                    ? gather_items<2>(P, Q, gnp, gs0, kbs, nk, T, b0, b1, xs, xsb, a.epoch, a.status)
                                    : gather_items<1>(P, Q, gnp, gs0, kbs, nk, T, b0, b1, xs, xsb, a.epoch, a.status);
                if (!ok) flags[0] = 1;
            } else {
                for (int it = tid; it < nk * T * kStBox; it += kThreads) {
                    const int pos = it / (T * kStBox);
                    const int rem = it - pos * T * kStBox;
                    const int t = rem / kStBox, i = rem - t * kStBox;
                    int kb = kbs + pos;
                    if (kb >= KB) kb -= KB;
                    xs[t * xsb + pos * kStBox + i] = a.x[(size_t)t * P.K + (size_t)kb * kStBox + i];
                }
            }
            cp_async_wait_all();
            consumer_sync();
            if (flags[0]) break;  // every thread has passed its input waits

            // ---- boxes: box j of the range goes to warp j % 8
            float cacc[4][4];
            float zc[2][4];
#pragma unroll
            for (int m = 0; m < 4; ++m) cacc[m][0] = cacc[m][1] = cacc[m][2] = cacc[m][3] = 0.f;
#pragma unroll
            for (int m = 0; m < 2; ++m) zc[m][0] = zc[m][1] = zc[m][2] = zc[m][3] = 0.f;
            const int rpad = a.rpad, nst = a.nst;
            int cur = -1;  // piece of the accumulators
            int pi = 0;
            float *wbw = wbuf + (size_t)warp * a.wb_floats;
            const size_t wbp = (size_t)kWarps * a.wb_floats;  // stride between pieces
            // the current piece's first box and k block, and where the next piece starts
            int pj0 = pcs[0].j0, pkb0 = pcs[0].kb0, nj0 = npc > 1 ? pcs[1].j0 : 0x7fffffff;
            // ring position of this warp's first box: boxes j = warp, warp + 8, ... and
            // a ring of a multiple of 8 stages
            int s = (qbase + warp) % nst;
            unsigned ph = (unsigned)(((qbase + warp) / nst) & 1);
            // B operand (token row g of the staged input): by shared address
            const uint32_t xs_ln = smem_u32(xst) + (uint32_t)((g * a.xs32 + t4) * 4);
            for (int j = warp; j < nbx; j += kWarps) {
                while (j >= nj0) {
                    ++pi;
                    pj0 = nj0;
                    pkb0 = pcs[pi].kb0;
                    nj0 = pi + 1 < npc ? pcs[pi + 1].j0 : 0x7fffffff;
                }
                if (pi != cur) {
                    if (cur >= 0) flush_piece(wbw + cur * wbp, a.wb_zoff, cacc, zc, false, Tp, rpad, lane);
                    for (int p = cur + 1; p < pi; ++p)
                        flush_piece(wbw + p * wbp, a.wb_zoff, cacc, zc, true, Tp, rpad, lane);
#pragma unroll
                    for (int m = 0; m < 4; ++m) cacc[m][0] = cacc[m][1] = cacc[m][2] = cacc[m][3] = 0.f;
#pragma unroll
                    for (int m = 0; m < 2; ++m) zc[m][0] = zc[m][1] = zc[m][2] = zc[m][3] = 0.f;
                    cur = pi;
                }
                int w_ok = 1;
                if (lane == 0) w_ok = !flags[0] && ring_wait(&full[s], ph, a.status);
                w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
                if (!w_ok) {
                    if (lane == 0) flags[0] = 1;
                    break;
                }
                int pos = pkb0 + (j - pj0) - kbs;
                if (pos < 0) pos += KB;
                const uint32_t sb = smem_u32(ring_w) + (uint32_t)(s * sbytes_stage);
                // the box's B fragments (8 words) first, then per k step the A
                // fragments of the four row groups and the V^T rows, then the MMAs
                uint32_t bfr[4][2];
#pragma unroll
                for (int kin = 0; kin < 4; ++kin) {
                    bfr[kin][0] = bfr[kin][1] = 0u;
                    if (g < Tp) {
                        const uint32_t xa = xs_ln + (uint32_t)((pos * (kStBox / 2) + kin * 8) * 4);
                        bfr[kin][0] = lds_u32(xa);
                        bfr[kin][1] = lds_u32(xa + 16);
                    }
                }
#pragma unroll
                for (int kin = 0; kin < 4; ++kin) {
                    const int chunk = kin * 2 + lchunk;
                    uint32_t af[4][4], zf[2][4];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const int row = m * 16 + lrow;
                        ldmatrix_x4(af[m], sb + row * 128 + ((chunk ^ (row & 7)) << 4));
                    }
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        if (m * 16 < rpad) {
                            const int row = m * 16 + lrow;
                            ldmatrix_x4(zf[m], sb + kStBoxBytes + row * 128 + ((chunk ^ (row & 7)) << 4));
                        }
                    }
#pragma unroll
                    for (int m = 0; m < 4; ++m) mma_16816(cacc[m], af[m], bfr[kin][0], bfr[kin][1]);
                    // z = x V: the V^T rows (ranks) as M, the same token columns
#pragma unroll
                    for (int m = 0; m < 2; ++m)
                        if (m * 16 < rpad) mma_16816(zc[m], zf[m], bfr[kin][0], bfr[kin][1]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                s += kWarps;
                if (s >= nst) {
                    s -= nst;
                    ph ^= 1u;
                }
            }
            qbase += nbx;
            if (cur >= 0) flush_piece(wbw + cur * wbp, a.wb_zoff, cacc, zc, false, Tp, rpad, lane);
            for (int p = cur + 1; p < npc; ++p)
                flush_piece(wbw + p * wbp, a.wb_zoff, cacc, zc, true, Tp, rpad, lane);
            consumer_sync();
            if (flags[0]) break;  // every box loop has ended: all threads agree

            // ---- phase end: p = s * acc + U z per row, the warps' sums added in
            // warp order.  Small r: z over the warps inside the rank loop; larger
            // r: z summed once per (piece, token, rank) first.
            // the warps' z sums, once per (piece, token, rank); then each row's
            // acc, its scale and U z.  All reads by shared address.
            const int wbf = a.wb_floats, wzo = a.wb_zoff;
            const uint32_t wb_s = smem_u32(wbuf), zs_s = smem_u32(zsum);
            if (r > 0) {
                for (int it = tid; it < npc * T * r; it += kThreads) {
                    const int p = it / (T * r), rem = it - p * T * r;
                    const int t = rem / r, j = rem - t * r;
                    const uint32_t za = wb_s + (uint32_t)(((p * kWarps) * wbf + wzo + t * rpad + j) * 4);
                    float zw[kWarps], zl[kWarps];
#pragma unroll
                    for (int w = 0; w < kWarps; ++w) {
                        zw[w] = lds_f32(za + (uint32_t)(w * wbf * 4));
                        zl[w] = kind == kD ? lds_f32(za + (uint32_t)((w * wbf + T * rpad) * 4)) : 0.f;
                    }
                    float sum = 0.f;
#pragma unroll
                    for (int w = 0; w < kWarps; ++w) {
                        sum += zw[w];
                        if (kind == kD) sum += zl[w];
                    }
                    zsum[p * kStMaxT * kStMaxR + rem] = sum;
                }
                consumer_sync();
            }
            const int us_soff = (kStBox * r * 2 + 16 + 15) & ~15;
            for (int it = tid; it < npc * T * kStBox; it += kThreads) {
                const int p = it / (T * kStBox), rem = it - p * T * kStBox;
                const int t = rem >> 6, row = rem & 63;
                const Piece pc = pcs[p];
                const StSeg &sg = P.seg[pc.si];
                const uint32_t wa = wb_s + (uint32_t)(((p * kWarps) * wbf + t * kStBox + row) * 4);
                float aw[kWarps], al[kWarps];
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    aw[w] = lds_f32(wa + (uint32_t)(w * wbf * 4));
                    al[w] = kind == kD ? lds_f32(wa + (uint32_t)((w * wbf + T * kStBox) * 4)) : 0.f;
                }
                float acc = 0.f, acc_lo = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    acc += aw[w];
                    if (kind == kD) acc_lo += al[w];
                }
                acc += acc_lo;
                float v = 0.f;
                if (pc.row0 + row < sg.out) {
                    const uint32_t us = smem_u32(aux_us) + (uint32_t)(p * a.us_bytes);
                    const uint32_t Ur = us + (uint32_t)(reinterpret_cast<uintptr_t>(sg.U + (size_t)pc.row0 * r) & 15) +
                                        (uint32_t)(row * r * 2);
                    const uint32_t sr = us + (uint32_t)us_soff + (uint32_t)(reinterpret_cast<uintptr_t>(sg.s + pc.row0) & 15);
                    v = lds_f32(sr + (uint32_t)(row * 4)) * acc;
                    const uint32_t zp = zs_s + (uint32_t)((p * kStMaxT * kStMaxR + t * r) * 4);
                    for (int k = 0; k < r; ++k) v = fmaf(lds_bf16(Ur + (uint32_t)(k * 2)), lds_f32(zp + (uint32_t)(k * 4)), v);
                }
                unsigned long long *sp = P.part + (size_t)pc.slot * P.nsub * T * kStBox;
                st_word(sp + ((size_t)pc.sub * T + t) * kStBox + row, v, a.epoch);
                // GU: a CTA holding one part of a pair adds zeros for the other
                if (kind == kGU) {
                    const bool has_other = pc.sub == 0 ? (p + 1 < npc && pcs[p + 1].rt == pc.rt)
                                                       : (p > 0 && pcs[p - 1].rt == pc.rt);
                    if (!has_other) st_word(sp + ((size_t)(1 - pc.sub) * T + t) * kStBox + row, 0.f, a.epoch);
                }
            }
        }

        // ---- outputs no phase reads (k, v; the last layer's): assigned row
        // tiles, counted from the last CTA (O leaves the upper half idle)
        if (P.xw_n > 0) {
            const StPhase &X = a.ph[P.xw_ph];
            for (int w = G - 1 - c; w < P.xw_n; w += G) {
                const int rt = P.xw_rt0 + w;
                int si = 0;
                while (si + 1 < X.nseg && rt >= X.seg[si + 1].rt0) ++si;
                const StSeg &sg = X.seg[si];
                const int row0 = (rt - sg.rt0) * kStBox;
                if (tid < T * kStBox) {
                    const int t = tid >> 6, row = tid & 63;
                    bool ok = true;
                    const float v = sum1(X, X.np[rt], X.slot0[rt], t, row, T, a.epoch, &ok, a.status);
                    if (!ok) flags[0] = 1;
                    else if (row0 + row < sg.out)
                        sg.y[(size_t)t * sg.out + row0 + row] = __float2bfloat16_rn(v);
                }
            }
        }
        cp_async_wait_all();  // the next phase's record
        consumer_sync();
    }
    cp_async_wait_all();
}

// V^T of every projection, padded with zero rows to rpad: VT[j][i] = V[i][j]
// (j < r), 0 (r <= j < rpad).  One block row per projection, 256 columns i per
// block; the writes of a row j are contiguous.
struct VtJob {
    const bf16 *V;  // [K, r]
    bf16 *VT;       // [rpad, K]
    int K;
};

__global__ void vt_kernel(const VtJob *__restrict__ jobs, int r, int rpad)
{
    const VtJob jb = jobs[blockIdx.y];
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= jb.K) return;
    for (int j = 0; j < rpad; ++j) jb.VT[(size_t)j * jb.K + i] = j < r ? jb.V[(size_t)i * r + j] : __float2bfloat16_rn(0.f);
}

// ------------------------------------------------------------------- host
struct StackPlan {
    int device = -1;
    int L = 0, T = 0, r = 0, hidden = 0;
    int G = 0, smem = 0;
    unsigned epoch = 0;
    std::vector<StArgs> chunks;           // one launch per chunk of at most 24 layers
    std::vector<const bf16 *> chunk_x;    // input of each chunk (null: the caller's x)
    const VtJob *vt_jobs = nullptr;       // V^T jobs (device), run before each step
    int n_vt = 0, vt_maxk = 0, rpad = 0;
    void *dmem = nullptr;  // tensor maps, partial tables, partial words
};

static int cdiv_i(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

}  // namespace wl

using namespace wl;

struct wl_stack_s {
    StackPlan p;
    WidePlan *wide = nullptr;  // 5..32 tokens: the wide stack kernel (stack_wide.cu)
    std::mutex mu;
};

static wl_status check_layer_proj(const wl_proj &p, int64_t out, int64_t r, const char *what, int64_t l)
{
    if (!p.W0 || !p.s || (r > 0 && (!p.U || !p.V)))
        return fail(WL_ERR_INVALID_ARG, "wl_stack_create: layer %lld %s: NULL pointer", (long long)l, what);
    if (p.out != out)
        return fail(WL_ERR_INVALID_ARG, "wl_stack_create: layer %lld %s: out = %lld, expected %lld", (long long)l,
                    what, (long long)p.out, (long long)out);
    if ((reinterpret_cast<uintptr_t>(p.W0) & 15) || (r > 0 && (reinterpret_cast<uintptr_t>(p.V) & 15)))
        return fail(WL_ERR_INVALID_ARG, "wl_stack_create: layer %lld %s: W0 and V must be 16-byte aligned",
                    (long long)l, what);
    return WL_OK;
}

extern "C" wl_status wl_stack_create(wl_stack *out, const wl_layer *layers, const wl_layer_out *outs,
                                     int64_t L, int64_t T, int64_t hidden, int64_t r)
{
    if (!out) return fail(WL_ERR_INVALID_ARG, "wl_stack_create: out is NULL");
    *out = nullptr;
    if (!layers || !outs || L < 1 || L > 4096)
        return fail(WL_ERR_INVALID_ARG, "wl_stack_create: need 1 <= L <= 4096 layers and outputs");
    if (T < 1 || T > kStackWideMaxT)
        return fail(WL_ERR_UNSUPPORTED, "wl_stack_create: T = %lld; the stack kernels take 1..%d tokens", (long long)T,
                    kStackWideMaxT);
    if (r < 0 || r > kStMaxR)
        return fail(WL_ERR_UNSUPPORTED, "wl_stack_create: r = %lld; the stack kernel takes 0..%d", (long long)r,
                    kStMaxR);
    const int64_t qd = layers[0].q.out, kvd = layers[0].k.out, vd = layers[0].v.out, inter = layers[0].gate.out;
    if (hidden < 64 || hidden % 64 || qd < 64 || qd % 64 || inter < 64 || inter % 64 || kvd < 1 || vd < 1)
        return fail(WL_ERR_UNSUPPORTED,
                    "wl_stack_create: hidden (%lld), q.out (%lld) and gate.out (%lld) must be multiples of 64",
                    (long long)hidden, (long long)qd, (long long)inter);
    for (int64_t l = 0; l < L; ++l) {
        const wl_layer &ly = layers[l];
        wl_status s;
        if ((s = check_layer_proj(ly.q, qd, r, "q", l)) != WL_OK) return s;
        if ((s = check_layer_proj(ly.k, kvd, r, "k", l)) != WL_OK) return s;
        if ((s = check_layer_proj(ly.v, vd, r, "v", l)) != WL_OK) return s;
        if ((s = check_layer_proj(ly.o, hidden, r, "o", l)) != WL_OK) return s;
        if ((s = check_layer_proj(ly.gate, inter, r, "gate", l)) != WL_OK) return s;
        if ((s = check_layer_proj(ly.up, inter, r, "up", l)) != WL_OK) return s;
        if ((s = check_layer_proj(ly.down, hidden, r, "down", l)) != WL_OK) return s;
        const wl_layer_out &o = outs[l];
        if (!o.yq || !o.yk || !o.yv || !o.yo || !o.ym)
            return fail(WL_ERR_INVALID_ARG, "wl_stack_create: layer %lld: NULL output buffer", (long long)l);
    }
    wl_status st = WL_OK;
    const DeviceInfo *di = device_info(&st);
    if (!di) return st;
    if (T > kStMaxT) {
        WidePlan *wp = nullptr;
        st = wide_stack_create(&wp, layers, outs, L, T, hidden, r, di);
        if (st != WL_OK) return st;
        wl_stack_s *h = new (std::nothrow) wl_stack_s;
        if (!h) {
            wide_stack_destroy(wp);
            return fail(WL_ERR_INVALID_ARG, "wl_stack_create: out of host memory");
        }
        h->wide = wp;
        *out = h;
        return WL_OK;
    }

    StackPlan pl;
    pl.device = di->device;
    pl.L = (int)L;
    pl.T = (int)T;
    pl.r = (int)r;
    pl.hidden = (int)hidden;
    pl.G = di->sm_count;
    const int G = pl.G;

    // ---- phases (host copy; device pointers filled in below)
    struct HostPhase {
        StPhase P;
        const wl_proj *proj[3];
        std::vector<int> np, slot0;
        int nslots;
    };
    std::vector<HostPhase> hp(4 * L);
    for (int64_t l = 0; l < L; ++l) {
        const wl_layer &ly = layers[l];
        const wl_layer_out &o = outs[l];
        for (int k = 0; k < 4; ++k) {
            HostPhase &h = hp[4 * l + k];
            StPhase &P = h.P;
            memset(&P, 0, sizeof(P));
            P.kind = k;
            int64_t K = 0;
            if (k == kQKV) {
                K = hidden;
                P.nseg = 3;
                h.proj[0] = &ly.q;
                h.proj[1] = &ly.k;
                h.proj[2] = &ly.v;
                P.seg[0].y = static_cast<bf16 *>(o.yq);
                P.seg[1].y = static_cast<bf16 *>(o.yk);
                P.seg[2].y = static_cast<bf16 *>(o.yv);
            } else if (k == kO) {
                K = qd;
                P.nseg = 1;
                h.proj[0] = &ly.o;
                P.seg[0].y = static_cast<bf16 *>(o.yo);
            } else if (k == kGU) {
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
            P.KB = (int)(K / 64);
            int rt = 0;
            for (int j = 0; j < P.nseg; ++j) {
                P.seg[j].out = (int)h.proj[j]->out;
                P.seg[j].s = h.proj[j]->s;
                P.seg[j].U = static_cast<const bf16 *>(h.proj[j]->U);
                P.seg[j].nrt = cdiv_i(h.proj[j]->out, 64);
                P.seg[j].rt0 = (k == kGU) ? 0 : rt;
                if (k != kGU) rt += P.seg[j].nrt;
            }
            if (k == kGU) {
                P.nrt = P.seg[0].nrt;
                P.bpr = 2 * P.KB;
                P.nsub = 2;
            } else {
                P.nrt = rt;
                P.bpr = P.KB;
                P.nsub = 1;
            }
            P.nbox = P.nrt * P.bpr;
            // O is small: half the CTAs keep its row tiles' partial counts low
            const int want = (k == kO) ? (G + 1) / 2 : G;
            P.ncta = P.nbox < want ? P.nbox : want;
            // input: layer 0's QKV reads x; otherwise the previous phase
            // (row tile kb of the producer holds input block kb: q is QKV's
            // first segment and q.out is a multiple of 64)
            P.prev = (l == 0 && k == kQKV) ? -1 : (int)(4 * l + k - 1);
            if (k == kO) P.wy = static_cast<bf16 *>(o.yq);
            if (k == kGU) P.wy = static_cast<bf16 *>(o.yo);
            if (k == kQKV && l > 0) P.wy = static_cast<bf16 *>(outs[l - 1].ym);
            // outputs nobody reads: k and v (stored during O), the last ym
            if (k == kO) {
                P.xw_ph = (int)(4 * l + kQKV);
                P.xw_rt0 = cdiv_i(qd, 64);
                P.xw_n = cdiv_i(kvd, 64) + cdiv_i(vd, 64);
            }
            if (k == kD && l == L - 1) {
                P.xw_ph = (int)(4 * l + kD);
                P.xw_rt0 = 0;
                P.xw_n = cdiv_i(hidden, 64);
            }
            // partials per row tile: the CTAs whose ranges touch it
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

    // ---- work bounds per CTA: pieces, staged input blocks
    int maxp = 1, nkmax = 1;
    for (auto &h : hp) {
        const StPhase &P = h.P;
        for (int cc = 0; cc < P.ncta; ++cc) {
            const int b0 = (int)((int64_t)P.nbox * cc / P.ncta), b1 = (int)((int64_t)P.nbox * (cc + 1) / P.ncta);
            if (b0 >= b1) continue;
            int n = 0;
            for (int b = b0; b < b1;) {
                const int rt = b / P.bpr, w = b - rt * P.bpr;
                int end = (rt + 1) * P.bpr;
                if (P.kind == kGU && w < P.KB) end = rt * P.bpr + P.KB;
                if (end > b1) end = b1;
                ++n;
                b = end;
            }
            if (n > maxp) maxp = n;
            const int nk = std::min(b1 - b0, P.KB);
            if (nk > nkmax) nkmax = nk;
        }
    }

    // ---- per (phase, CTA) work records
    const int rec_ints = (kRecHead + 8 * maxp + 2 * nkmax + 3) / 4 * 4;
    auto owner = [](int b, int nbox, int n) { return (int)((((int64_t)b + 1) * n - 1) / nbox); };
    auto make_rec = [&](int gi, int cc, int *rec) {
        const StPhase &P = hp[gi].P;
        const int b0 = (int)((int64_t)P.nbox * std::min(cc, P.ncta) / P.ncta);
        const int b1 = (int)((int64_t)P.nbox * std::min(cc + 1, P.ncta) / P.ncta);
        memset(rec, 0, sizeof(int) * rec_ints);
        rec[0] = b0;
        rec[1] = b1 - b0;
        if (b1 <= b0) return;
        int n = 0;
        for (int b = b0; b < b1;) {
            const int rt = b / P.bpr, w = b - rt * P.bpr;
            const int sub = P.kind == kGU ? w / P.KB : 0;
            int end = (rt + 1) * P.bpr;
            if (P.kind == kGU && sub == 0) end = rt * P.bpr + P.KB;
            if (end > b1) end = b1;
            int si = sub;
            if (P.kind != kGU)
                while (si + 1 < P.nseg && rt >= P.seg[si + 1].rt0) ++si;
            int *pc = rec + kRecHead + 8 * n;
            pc[0] = rt;
            pc[1] = sub;
            pc[2] = si;
            pc[3] = P.kind == kGU ? rt * 64 : (rt - P.seg[si].rt0) * 64;
            pc[4] = b - b0;
            pc[5] = end - b;
            pc[6] = w - sub * P.KB;
            pc[7] = hp[gi].slot0[rt] + (cc - owner(rt * P.bpr, P.nbox, P.ncta));
            ++n;
            b = end;
        }
        rec[2] = n;
        const int kbs = (b0 % P.bpr) % P.KB, nk = std::min(b1 - b0, P.KB);
        rec[3] = kbs;
        rec[4] = nk;
        if (gi > 0) {
            // the producing phase is the previous one (a chunk's first phase
            // reads x and ignores these)
            const HostPhase &Q = hp[gi - 1];
            for (int pos = 0; pos < nk; ++pos) {
                const int kb = (kbs + pos) % P.KB;
                rec[kRecHead + 8 * maxp + pos] = Q.np[kb];
                rec[kRecHead + 8 * maxp + nkmax + pos] = Q.slot0[kb];
            }
        }
    };

    // ---- shared memory
    const int rpad = r == 0 ? 0 : (r <= 16 ? 16 : 32);
    const int us_bytes = ((int)(64 * r * 2) + 16 + 15) / 16 * 16 + (64 * 4 + 16 + 15) / 16 * 16;
    int xs32 = (nkmax * 64 + 8) / 2;  // row stride (u32); 4 mod 32 keeps the B-operand reads conflict-free
    xs32 = (xs32 + 31) / 32 * 32 + 4;
    const int wb_floats = 2 * (int)T * 64 + 2 * (int)T * (rpad > 0 ? rpad : 1);
    const int fixed = 1024 + maxp * us_bytes + 2 * (int)T * xs32 * 4 + maxp * kWarps * wb_floats * 4 +
                      maxp * kStMaxT * kStMaxR * 4 + 2 * rec_ints * 4 + 16 + 64;
    const int stage_bytes = kStBoxBytes + rpad * 128;  // W0 box + V^T box, 1024-byte multiple
    const int per_stage = stage_bytes + 16;
    int nst = (di->max_smem_optin - fixed) / per_stage;
    if (nst > 32) nst = 32;
    if (nst < kWarps)
        return fail(WL_ERR_UNSUPPORTED, "wl_stack_create: these shapes leave room for %d ring stages", nst);
    nst = round_ring_to_warps(nst, kWarps);
    pl.smem = fixed + nst * per_stage;

    // ---- device memory: maps, phases, np/slot0, partial words
    size_t off = 0;
    auto take = [&](size_t bytes, size_t align) {
        off = (off + align - 1) / align * align;
        const size_t o = off;
        off += bytes;
        return o;
    };
    const size_t o_maps = take(sizeof(CUtensorMap) * 7 * L, 128);
    const size_t o_vtmaps = take(sizeof(CUtensorMap) * 7 * L, 128);
    const size_t o_jobs = take(sizeof(VtJob) * 7 * L, 16);
    std::vector<size_t> o_np(4 * L), o_s0(4 * L), o_part(4 * L);
    for (size_t i = 0; i < hp.size(); ++i) {
        o_np[i] = take(sizeof(int) * hp[i].P.nrt, 16);
        o_s0[i] = take(sizeof(int) * hp[i].P.nrt, 16);
    }
    const size_t o_rec = take(sizeof(int) * (size_t)rec_ints * 4 * L * G, 256);
    const size_t o_tables_end = take(0, 256);
    const int64_t kin[7] = {hidden, hidden, hidden, qd, hidden, hidden, inter};
    std::vector<size_t> o_vt(7 * L);
    for (int64_t l = 0; l < L; ++l)
        for (int j = 0; j < 7; ++j) o_vt[7 * l + j] = take((size_t)rpad * kin[j] * 2, 256);
    for (size_t i = 0; i < hp.size(); ++i)
        o_part[i] = take(sizeof(unsigned long long) * (size_t)hp[i].nslots * hp[i].P.nsub * T * 64, 256);
    const size_t total = off;

    void *dmem = nullptr;
    cudaError_t e = cudaMalloc(&dmem, total);
    if (e != cudaSuccess) return cuda_fail(e, "wl_stack_create: cudaMalloc of the stack's tables and scratch");
    char *base = static_cast<char *>(dmem);
    std::vector<char> host(o_tables_end, 0);
    CUtensorMap *hmaps = reinterpret_cast<CUtensorMap *>(host.data() + o_maps);
    for (int gi = 0; gi < 4 * L; ++gi)
        for (int cc = 0; cc < G; ++cc)
            make_rec(gi, cc, reinterpret_cast<int *>(host.data() + o_rec) + ((size_t)gi * G + cc) * rec_ints);
    for (int64_t l = 0; l < L; ++l) {
        const wl_proj *pj[7] = {&layers[l].q, &layers[l].k, &layers[l].v, &layers[l].o,
                                &layers[l].gate, &layers[l].up, &layers[l].down};
        const int64_t ins[7] = {hidden, hidden, hidden, qd, hidden, hidden, inter};
        for (int j = 0; j < 7; ++j) {
            st = tmap_2d_bf16(pj[j]->W0, ins[j], pj[j]->out, ins[j], 64, 64, &hmaps[7 * l + j]);
            if (st != WL_OK) {
                cudaFree(dmem);
                return st;
            }
        }
    }
    // V^T buffers, their tensor maps and the transpose jobs
    CUtensorMap *hvt = reinterpret_cast<CUtensorMap *>(host.data() + o_vtmaps);
    VtJob *hjobs = reinterpret_cast<VtJob *>(host.data() + o_jobs);
    for (int64_t l = 0; l < L && rpad > 0; ++l) {
        const wl_proj *pj[7] = {&layers[l].q, &layers[l].k, &layers[l].v, &layers[l].o,
                                &layers[l].gate, &layers[l].up, &layers[l].down};
        for (int j = 0; j < 7; ++j) {
            bf16 *vt = reinterpret_cast<bf16 *>(base + o_vt[7 * l + j]);
            st = tmap_2d_bf16(vt, kin[j], rpad, kin[j], 64, rpad, &hvt[7 * l + j]);
            if (st != WL_OK) {
                cudaFree(dmem);
                return st;
            }
            hjobs[7 * l + j] = VtJob{static_cast<const bf16 *>(pj[j]->V), vt, (int)kin[j]};
        }
    }
    for (size_t i = 0; i < hp.size(); ++i) {
        HostPhase &h = hp[i];
        const int64_t l = (int64_t)i / 4;
        const int k = (int)(i % 4);
        const int mj[4][3] = {{0, 1, 2}, {3, -1, -1}, {4, 5, -1}, {6, -1, -1}};
        for (int j = 0; j < h.P.nseg; ++j) {
            h.P.seg[j].map = reinterpret_cast<const CUtensorMap *>(base + o_maps) + 7 * l + mj[k][j];
            h.P.seg[j].vtmap = rpad ? reinterpret_cast<const CUtensorMap *>(base + o_vtmaps) + 7 * l + mj[k][j] : nullptr;
        }
        memcpy(host.data() + o_np[i], h.np.data(), sizeof(int) * h.P.nrt);
        memcpy(host.data() + o_s0[i], h.slot0.data(), sizeof(int) * h.P.nrt);
        h.P.np = reinterpret_cast<const int *>(base + o_np[i]);
        h.P.slot0 = reinterpret_cast<const int *>(base + o_s0[i]);
        h.P.part = reinterpret_cast<unsigned long long *>(base + o_part[i]);
    }
    e = cudaMemcpy(dmem, host.data(), o_tables_end, cudaMemcpyHostToDevice);
    // partial words start at epoch 0; launches use epochs 1, 2, ...
    if (e == cudaSuccess) e = cudaMemset(base + o_tables_end, 0, total - o_tables_end);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaFree(dmem);
        return cuda_fail(e, "wl_stack_create: table upload");
    }
    e = cudaFuncSetAttribute((const void *)stack_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             di->max_smem_optin);
    if (e != cudaSuccess) {
        cudaFree(dmem);
        return cuda_fail(e, "cudaFuncSetAttribute(stack_kernel)");
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stack_kernel, kStThreads, (size_t)pl.smem);
    if (e != cudaSuccess || per_sm < 1) {
        cudaFree(dmem);
        return fail(WL_ERR_UNSUPPORTED, "wl_stack_create: the stack kernel does not fit on an SM (%d bytes)",
                    pl.smem);
    }

    // launches: chunks of at most kStMaxPh / 4 layers, of about equal size
    const int lmax = kStMaxPh / 4;
    const int nchunk = cdiv_i(L, lmax);
    StArgs a;
    memset(&a, 0, sizeof(a));
    a.T = (int)T;
    a.r = (int)r;
    a.nst = nst;
    a.maxp = maxp;
    a.xs32 = xs32;
    a.us_bytes = us_bytes;
    a.wb_floats = wb_floats;
    a.wb_zoff = 2 * (int)T * 64;
    a.rpad = rpad;
    a.stage_bytes = stage_bytes;
    a.maxnk = nkmax;
    a.rec_ints = rec_ints;
    a.status = di->status;
    for (int ch = 0; ch < nchunk; ++ch) {
        const int l0 = (int)(L * ch / nchunk), l1 = (int)(L * (ch + 1) / nchunk);
        const int base_ph = 4 * l0;
        a.nph = 4 * (l1 - l0);
        a.rec = reinterpret_cast<const int *>(base + o_rec) + (size_t)base_ph * G * rec_ints;
        for (int i = 0; i < a.nph; ++i) {
            StPhase P = hp[base_ph + i].P;
            if (i == 0) {
                // the chunk's input: x, or the previous chunk's output (stored
                // by that launch's last phase)
                P.prev = -1;
                P.wy = nullptr;
            } else {
                P.prev -= base_ph;
            }
            if (P.xw_n > 0) P.xw_ph -= base_ph;
            if (i == a.nph - 1 && P.xw_n == 0) {  // chunk end: store the last layer's output
                P.xw_ph = i;
                P.xw_rt0 = 0;
                P.xw_n = cdiv_i(hidden, 64);
            }
            a.ph[i] = P;
        }
        pl.chunks.push_back(a);
        pl.chunk_x.push_back(l0 == 0 ? nullptr : static_cast<const bf16 *>(outs[l0 - 1].ym));
    }
    pl.dmem = dmem;
    pl.rpad = rpad;
    pl.n_vt = rpad ? (int)(7 * L) : 0;
    pl.vt_maxk = (int)std::max(hidden, std::max(qd, inter));
    pl.vt_jobs = reinterpret_cast<const VtJob *>(base + o_jobs);

    wl_stack_s *h = new (std::nothrow) wl_stack_s;
    if (!h) {
        cudaFree(dmem);
        return fail(WL_ERR_INVALID_ARG, "wl_stack_create: out of host memory");
    }
    h->p = pl;
    *out = h;
    return WL_OK;
}

extern "C" wl_status wl_stack_decode(wl_stack stk, const void *x, void *stream)
{
    if (!stk || !x) return fail(WL_ERR_INVALID_ARG, "wl_stack_decode: NULL stack or x");
    if (reinterpret_cast<uintptr_t>(x) & 15) return fail(WL_ERR_INVALID_ARG, "wl_stack_decode: x must be 16-byte aligned");
    StackPlan &pl = stk->p;
    int dev = -1;
    cudaGetDevice(&dev);
    const int built_on = stk->wide ? wide_stack_device(stk->wide) : pl.device;
    if (dev != built_on)
        return fail(WL_ERR_INVALID_ARG, "wl_stack_decode: the stack was built on device %d, current is %d", built_on,
                    dev);
    if (stk->wide) return wide_stack_decode(stk->wide, x, static_cast<cudaStream_t>(stream));
    unsigned epoch;
    {
        std::lock_guard<std::mutex> lk(stk->mu);
        // epochs 1 .. 2^32-1; 0 marks words never written
        if (++pl.epoch == 0) pl.epoch = 1;
        epoch = pl.epoch;
    }
    if (pl.n_vt > 0) {
        // V^T of this step's V (read now, so later changes to V are seen)
        dim3 grid((unsigned)((pl.vt_maxk + 255) / 256), (unsigned)pl.n_vt);
        vt_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(pl.vt_jobs, pl.r, pl.rpad);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "wl_stack_decode: V^T launch");
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.G);
    cfg.blockDim = dim3(kStThreads);
    cfg.dynamicSmemBytes = (size_t)pl.smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    for (size_t ch = 0; ch < pl.chunks.size(); ++ch) {
        if (pl.chunks[ch].nst <= 0 || pl.chunks[ch].nst % kWarps != 0)
            return fail(WL_ERR_INTERNAL, "wl_stack_decode: ring of %d stages is not a multiple of the %d "
                        "consumer warps", pl.chunks[ch].nst, kWarps);
        StArgs a = pl.chunks[ch];  // a copy: calls on other threads may launch at the same time
        a.epoch = epoch;
        a.x = pl.chunk_x[ch] ? pl.chunk_x[ch] : static_cast<const bf16 *>(x);
        void *args[] = {&a};
        cudaError_t e = cudaLaunchKernelExC(&cfg, (const void *)stack_kernel, args);
        if (e != cudaSuccess) return cuda_fail(e, "wl_stack_decode: launch");
    }
    return WL_OK;
}

extern "C" void wl_stack_destroy(wl_stack stk)
{
    if (!stk) return;
    if (stk->wide) wide_stack_destroy(stk->wide);
    if (stk->p.dmem) cudaFree(stk->p.dmem);
    delete stk;
}
