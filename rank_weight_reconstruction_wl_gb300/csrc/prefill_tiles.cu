// prefill_tiles.cu -- persistent tensor-core kernel for large-T weightless
// projections: one CTA per SM walks a static list of output tiles, with the
// accumulators double-buffered in tensor memory so that the epilogue of one
// tile runs while the tensor cores work on the next.
//
// Per tile of 128 tokens x BN accumulator columns ("In-kernel
// reconstruction", formula section; "The GEMM path"):
//     acc = x W0^T                       tcgen05.mma kind::f16, fp32 in TMEM
//     z   = x V      (same K loop)       second MMA into the buffer's z columns
//     acc = s * acc                      epilogue, TMEM load / multiply / store
//     acc += z_bf16 U^T                  rank-r delta on the tensor cores (z as
//                                        bf16 hi + lo parts for fp32 outputs)
//     y   = cast(acc)                    epilogue
// z depends only on the token rows and the projection, so a CTA forms it on
// the first tile of a (rows, projection) run and keeps its bf16 split in
// shared memory for the following tiles of the run.  V is [in, r]: its rows
// are loaded by TMA as they are and serve as the MN-major B operand of the z
// MMA (r = 16, 32, 64); for other ranks warps 2-3 write V^T, the K-major
// operand, into the stage.
//
// Paired mode (fused GeGLU MLP, gate and up): a tile holds BN/2 rows of the
// gate projection and the same BN/2 rows of the up projection, and the
// epilogue writes h = gelu_tanh(g) * u directly (bf16, plus the rounding
// remainder as a second bf16 part for fp32 outputs), so g and u never leave
// the chip.
//
// Warp roles (384 threads): warp 0 = TMA producer; warp 1 = TMEM owner and MMA
// issuer (one thread; it also issues each finished tile's delta MMAs as soon
// as the epilogue has scaled the accumulator); warps 2-3 = V^T writers where
// V rows are not loaded by TMA; warps 4-11 = epilogue (warp w reads TMEM lanes 32*(w%4) .. +31; two warps per
// lane quarter split the columns).  Every wait is bounded; a wait that gives
// up sets the status word and the CTA winds down.
#include <mutex>
#include <unordered_map>

#include "dec_ptx.cuh"
#include "tc_ptx.cuh"

namespace wl {

constexpr int kTlThreads = 384;
constexpr int kTlEpiThreads = 256;  // warps 4..11
constexpr int kTlVtThreads = 64;    // warps 2..3
constexpr int kTlBM = 128;          // tokens per tile
constexpr int kTlATile = kTlBM * 128;  // x tile of one stage: 128 rows x 64 k, 16 KB
constexpr int kTlMaxStages = 6;

struct TlSeg {
    CUtensorMap mapb;  // W0 [out, in], box 64 x bh
    CUtensorMap mapv;  // V [in, r], box r x 64 (V rows as they are: the MN-major B operand of z = x V)
    const float *s;
    const bf16 *U;
    const bf16 *V;
    void *y;     // output rows of stride ldy (paired mode: h)
    int out;     // rows of W0
    int ntile0;  // first n-tile of this projection
};

struct TlArgs {
    TlSeg seg[3];
    CUtensorMap mapa;  // x [T, Ktot], box 64 x 128
    int nseg, pair;
    int T, in, Ktot, kmod, r, rpad, ydt;  // K position k meets W0 column / V row k % kmod
    int BN, bh;        // accumulator columns per tile; W0 rows per box (BN, or BN/2 paired)
    int zc, Kz;        // z columns (rpad per projection of the tile); K of the delta MMA
    int zlo;           // 1: the delta MMA takes z as bf16 hi + lo parts (fp32 outputs); 0: hi only
    int mtiles, ntiles, ktiles;
    int nst, stage_bytes;
    int vstage;        // 1: V rows of a stage arrive by bulk copy with its tiles
    int vtma;          // 1: V rows arrive by TMA in the MMA's MN-major layout (no transposition)
    int vsw;           // that layout's swizzle code in the matrix descriptor
    int ldy;           // paired: row stride of h in elements (single: rows of y are `out` long)
    int hw, hlo;       // paired: h columns written per row part; column of the remainder part (0: none)
    unsigned *status;
};

struct TlTile {
    int m0, si, n0, key;
};

__device__ __forceinline__ TlTile tl_tile(const TlArgs &a, int t)
{
    TlTile q;
    const int m = t % a.mtiles, nt = t / a.mtiles;
    int si = 0;
    if (!a.pair) {
        if (a.nseg > 1 && nt >= a.seg[1].ntile0) si = 1;
        if (a.nseg > 2 && nt >= a.seg[2].ntile0) si = 2;
    }
    q.m0 = m * kTlBM;
    q.si = si;
    q.n0 = (nt - a.seg[si].ntile0) * a.bh;
    q.key = m * 4 + si;
    return q;
}

// Contiguous global -> shared copy (16-byte aligned, size a multiple of 16)
// completing on `bar`'s transaction count.
__device__ __forceinline__ void tl_bulk(void *dst, const void *src, unsigned bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     s32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(s32(bar))
                 : "memory");
}

// Shared-memory matrix descriptor of a box of V rows (64 K rows of r bf16,
// r contiguous): an MN-major B operand whose swizzle span is the row length
// (r = 16, 32, 64 -> 32, 64, 128 bytes); 8-row groups are 8 * 2r bytes apart.
__device__ __forceinline__ uint64_t tl_vdesc(uint32_t addr, int r, int vsw)
{
    const uint64_t grp = (uint64_t)(16 * r);
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((grp >> 4) << 16) | ((grp >> 4) << 32) | ((uint64_t)1 << 46) |
           ((uint64_t)vsw << 61);
}

__device__ __forceinline__ void tl_epi_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kTlEpiThreads) : "memory"); }

// Byte offset of element (row, k) of a K-major operand tile with 128-byte
// swizzle: 8-row x 128-byte atoms (1024 B), atom columns of 64 elements, each
// `rows` x 128 bytes.
__device__ __forceinline__ uint32_t tl_swz(int row, int k, int rows)
{
    return (uint32_t)((k >> 6) * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 +
                      ((((k >> 3) & 7) ^ (row & 7)) << 4) + (k & 7) * 2);
}

__device__ __forceinline__ uint32_t tl_pack(float lo, float hi)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ uint16_t tl_ldu16(const bf16 *p) { return __ldg(reinterpret_cast<const unsigned short *>(p)); }

__device__ __forceinline__ float tl_gelu_mul(float g, float u)
{
    const float c = 0.7978845608028654f;  // sqrt(2/pi)
    return 0.5f * g * (1.0f + tanhf(c * (g + 0.044715f * g * g * g))) * u;
}

// Store 8 consecutive outputs of one row (bf16 or fp32) at element `col` of
// row `m`, keeping to the first `nvalid` of them.
__device__ __forceinline__ void tl_store8(void *y, int ydt, int64_t off, int nvalid, const float v[8])
{
    if (ydt == WL_OUT_F32) {
        float *d = static_cast<float *>(y) + off;
        if (nvalid >= 8 && (reinterpret_cast<uintptr_t>(d) & 15) == 0) {
            reinterpret_cast<float4 *>(d)[0] = make_float4(v[0], v[1], v[2], v[3]);
            reinterpret_cast<float4 *>(d)[1] = make_float4(v[4], v[5], v[6], v[7]);
        } else {
            for (int i = 0; i < 8 && i < nvalid; ++i) d[i] = v[i];
        }
    } else {
        bf16 *d = static_cast<bf16 *>(y) + off;
        if (nvalid >= 8 && (reinterpret_cast<uintptr_t>(d) & 15) == 0) {
            *reinterpret_cast<uint4 *>(d) =
                make_uint4(tl_pack(v[0], v[1]), tl_pack(v[2], v[3]), tl_pack(v[4], v[5]), tl_pack(v[6], v[7]));
        } else {
            for (int i = 0; i < 8 && i < nvalid; ++i) d[i] = __float2bfloat16_rn(v[i]);
        }
    }
}

// V rows of K position kk of stage kt for every projection slot of tile q,
// as element pairs: element e of words[0, zc/2) is V_slot[k][e - slot*rpad]
// (slot = e / rpad), zero past r.  16-byte loads where rows are aligned.
__device__ __forceinline__ void tl_load_vrow(const TlArgs &a, const TlTile &q, int kt, int kk, uint32_t w[32])
{
    const int kc = kt * 64, kg = kc + kk, kr = kc % a.kmod + kk;
    const bool valid = kg < a.Ktot && kr < a.in;
    const bf16 *V0 = a.seg[a.pair ? 0 : q.si].V, *V1 = a.seg[a.pair ? 1 : q.si].V;
    const bool vec = (a.r & 7) == 0 && ((reinterpret_cast<uintptr_t>(V0) | reinterpret_cast<uintptr_t>(V1)) & 15) == 0;
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        const int e0 = 8 * g;
        if (e0 < a.zc) {
            const int sl = e0 >= a.rpad ? 1 : 0;
            const int j0 = e0 - sl * a.rpad;
            const bf16 *row = (sl ? V1 : V0) + (int64_t)kr * a.r;
            if (vec) {
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (valid && j0 < a.r) v = __ldg(reinterpret_cast<const uint4 *>(row + j0));
                w[4 * g] = v.x;
                w[4 * g + 1] = v.y;
                w[4 * g + 2] = v.z;
                w[4 * g + 3] = v.w;
            } else {
                const unsigned short *p = reinterpret_cast<const unsigned short *>(row);
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int j = j0 + 2 * h;
                    const uint32_t lo = (valid && j < a.r) ? (uint32_t)__ldg(p + j) : 0u;
                    const uint32_t hi = (valid && j + 1 < a.r) ? (uint32_t)__ldg(p + j + 1) : 0u;
                    w[4 * g + h] = lo | (hi << 16);
                }
            }
        }
    }
}

// The same from the stage's copy of the V rows ([slot][64 rows][r] bf16).
__device__ __forceinline__ void tl_load_vrow_smem(const TlArgs &a, const char *vst, int kt, int kk, uint32_t w[32])
{
    const int kc = kt * 64, kg = kc + kk, kr = kc % a.kmod + kk;
    const bool valid = kg < a.Ktot && kr < a.in;
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        const int e0 = 8 * g;
        if (e0 < a.zc) {
            const int sl = e0 >= a.rpad ? 1 : 0;
            const int j0 = e0 - sl * a.rpad;
            const char *row = vst + (size_t)(sl * 64 + kk) * a.r * 2;
            if ((a.r & 7) == 0) {
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (valid && j0 < a.r) v = *reinterpret_cast<const uint4 *>(row + 2 * j0);
                w[4 * g] = v.x;
                w[4 * g + 1] = v.y;
                w[4 * g + 2] = v.z;
                w[4 * g + 3] = v.w;
            } else {
                const unsigned short *p = reinterpret_cast<const unsigned short *>(row);
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int j = j0 + 2 * h;
                    const uint32_t lo = (valid && j < a.r) ? (uint32_t)p[j] : 0u;
                    const uint32_t hi = (valid && j + 1 < a.r) ? (uint32_t)p[j + 1] : 0u;
                    w[4 * g + h] = lo | (hi << 16);
                }
            }
        }
    }
}

__global__ void __launch_bounds__(kTlThreads, 1) prefill_tiles_kernel(const __grid_constant__ TlArgs a)
{
    extern __shared__ __align__(1024) char smem_raw[];
    char *smem = smem_raw + ((1024u - (s32(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nkz = a.Kz / 64;  // atom columns of the delta operands

    // shared memory: stages | A_z | B_u | s tile | barriers | tmem holder, abort flag
    char *az = smem + (size_t)a.nst * a.stage_bytes;
    char *bu = az + (size_t)nkz * kTlATile;
    float *s_tile = reinterpret_cast<float *>(bu + (size_t)nkz * a.BN * 128);
    uint64_t *bars = reinterpret_cast<uint64_t *>(s_tile + a.BN);
    uint64_t *full = bars, *empty = bars + a.nst, *vfull = bars + 2 * a.nst;
    uint64_t *acc_full = bars + 3 * a.nst, *acc_empty = acc_full + 2, *dready = acc_full + 4, *dfull = acc_full + 6;
    uint64_t *drain = acc_full + 8;
    uint32_t *tmem_hold = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_hold + 1);

    const int ntall = a.mtiles * a.ntiles;
    const bool has_z = a.zc > 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < a.nst; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
            mbar_init(&vfull[i], kTlVtThreads);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kTlEpiThreads / 32);
            mbar_init(&dready[b], 1);
            mbar_init(&dfull[b], 1);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(s32(tmem_hold)),
                     "r"(512));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_hold;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.mapa)) : "memory");
            for (int j = 0; j < (a.pair ? 2 : a.nseg); ++j)
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.seg[j].mapb)) : "memory");
            int s = 0;
            unsigned ph = 0;
            int nissued = 0;
            bool ok = true;
            const unsigned tx = (unsigned)(kTlATile + a.BN * 128);
            const int nslot = a.pair ? 2 : 1;
            int prev_key = -1;
            for (int t = blockIdx.x; t < ntall && ok; t += gridDim.x) {
                const TlTile q = tl_tile(a, t);
                const bool nz = has_z && q.key != prev_key;
                prev_key = q.key;
                for (int kt = 0; kt < a.ktiles; ++kt) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, a.status, kWaitRingEmpty) || *abort_flag) {
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    char *st = smem + (size_t)s * a.stage_bytes;
                    const int kc = kt * 64, kw = kc % a.kmod;
                    const int vrows = (nz && a.vstage) ? max(0, min(64, a.in - kw)) : 0;
                    const bool vbox = nz && a.vtma;
                    mbar_expect_tx(&full[s], tx + (unsigned)(nslot * (vbox ? 64 : vrows) * a.r * 2));
                    tma_load_2d(st, &a.mapa, kc, q.m0, &full[s]);
                    if (vbox)
                        for (int sl = 0; sl < nslot; ++sl)
                            tma_load_2d(st + kTlATile + a.BN * 128 + sl * 64 * a.r * 2, &a.seg[a.pair ? sl : q.si].mapv,
                                        0, kw, &full[s]);
                    for (int sl = 0; sl < (vrows > 0 ? nslot : 0); ++sl)
                        tl_bulk(st + kTlATile + (a.BN + a.zc) * 128 + sl * 64 * a.r * 2,
                                a.seg[a.pair ? sl : q.si].V + (int64_t)kw * a.r, (unsigned)(vrows * a.r * 2), &full[s]);
                    if (a.pair) {
                        tma_load_2d(st + kTlATile, &a.seg[0].mapb, kw, q.n0, &full[s]);
                        tma_load_2d(st + kTlATile + a.bh * 128, &a.seg[1].mapb, kw, q.n0, &full[s]);
                    } else {
                        tma_load_2d(st + kTlATile, &a.seg[q.si].mapb, kw, q.n0, &full[s]);
                    }
                    ++nissued;
                    if (++s == a.nst) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // before the CTA can exit, every copy issued has landed
            for (int i = 0; i < a.nst && i < nissued; ++i) {
                const int uses = (nissued - 1 - i) / a.nst + 1;  // loads issued into stage i
                mbar_wait(&full[i], (unsigned)((uses - 1) & 1), a.status, kWaitRingFull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_main = idesc_bf16(kTlBM, a.BN);
            const uint32_t id_z = idesc_bf16(kTlBM, has_z ? a.zc : 16);
            const uint32_t id_zmn = idesc_bf16(kTlBM, a.r > 0 ? a.r : 16) | (1u << 16);  // B (V rows) MN-major
            const uint32_t saz = s32(az), sbu = s32(bu);
            int s = 0;
            unsigned ph = 0;
            int j = 0;   // tiles whose main loop has been issued
            int dn = 0;  // next tile whose delta is to be issued
            bool ok = true;
            // issue the next finished tile's delta if the epilogue has scaled its accumulator
            auto try_delta = [&]() {
                if (a.r > 0 && dn < j && mbar_test(&dready[dn & 1], (unsigned)((dn >> 1) & 1))) {
                    tc_fence_after();
                    const uint32_t dacc = tmem + (uint32_t)((dn & 1) * 256);
                    for (int kd = 0; kd < a.Kz / 16; ++kd) {
                        const int at = kd >> 2, kin = kd & 3;
                        umma(dacc, sdesc(saz + at * kTlATile + 32 * kin), sdesc(sbu + at * a.BN * 128 + 32 * kin),
                             id_main, 1u);
                    }
                    umma_commit(&dfull[dn & 1]);
                    ++dn;
                }
            };
            auto wait_poll = [&](uint64_t *bar, unsigned par, unsigned site) -> bool {
                if (mbar_test(bar, par)) return true;
                const long long t0 = wait_clock();
                while (!mbar_test(bar, par)) {
                    try_delta();
                    if (wait_clock() - t0 > kWaitLimitCycles) {
                        atomicOr(a.status, kStatusTimeout | site);
                        return false;
                    }
                }
                return true;
            };
            int prev_key = -1;
            for (int t = blockIdx.x; t < ntall; t += gridDim.x) {
                const TlTile q = tl_tile(a, t);
                const bool nz = has_z && q.key != prev_key;
                prev_key = q.key;
                const int b = j & 1;
                if (!wait_poll(&acc_empty[b], (unsigned)(((j >> 1) & 1) ^ 1), kWaitRingEmpty)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dacc = tmem + (uint32_t)(b * 256), dz = dacc + (uint32_t)a.BN;
                for (int kt = 0; kt < a.ktiles && ok; ++kt) {
                    try_delta();
                    if (!wait_poll(&full[s], ph, kWaitRingFull) ||
                        (nz && !a.vtma && !wait_poll(&vfull[s], ph, kWaitRingFull))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = s32(smem + (size_t)s * a.stage_bytes);
                    const uint32_t sb = sa + kTlATile, sv = sb + (uint32_t)a.BN * 128;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t da = sdesc(sa + 32 * k);
                        const uint32_t acc = (kt > 0 || k > 0) ? 1u : 0u;
                        umma(dacc, da, sdesc(sb + 32 * k), id_main, acc);
                        if (nz && a.vtma) {
                            for (int sl = 0; sl < (a.pair ? 2 : 1); ++sl)
                                umma(dz + (uint32_t)(sl * a.r), da,
                                     tl_vdesc(sv + (uint32_t)(sl * 64 * a.r * 2 + k * 32 * a.r), a.r, a.vsw), id_zmn, acc);
                        } else if (nz) {
                            umma(dz, da, sdesc(sv + 32 * k), id_z, acc);
                        }
                    }
                    umma_commit(&empty[s]);
                    if (++s == a.nst) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(&acc_full[b]);
                ++j;
            }
            if (!ok) *abort_flag = 1;
            if (ok && a.r > 0) {
                const long long t0 = wait_clock();
                while (dn < j) {
                    try_delta();
                    if (dn < j && wait_clock() - t0 > kWaitLimitCycles) {
                        atomicOr(a.status, kStatusTimeout | kWaitRingFull);
                        break;
                    }
                }
            }
            // every MMA issued has completed before TMEM is freed
            umma_commit(drain);
            mbar_wait(drain, 0, a.status, kWaitRingFull);
        }
    } else if (warp < 4) {
        // ------------------------------------------------ V^T writers
        // Thread kk of 64 owns K position kk of every stage: it loads the V
        // rows of that position (every projection slot of the tile) one stage
        // ahead into registers, then, once the stage is free, writes them as
        // column kk of the K-major tile V^T [zc rows, 64 k].
        if (has_z && !a.vtma) {
            const int kk = threadIdx.x - 64;
            int s = 0;
            unsigned ph = 0;
            int prev_key = -1;
            bool ok = true;
            uint32_t cur[32], nxt[32];
            for (int t = blockIdx.x; t < ntall && ok; t += gridDim.x) {
                const TlTile q = tl_tile(a, t);
                const bool nz = q.key != prev_key;
                prev_key = q.key;
                if (nz && !a.vstage) tl_load_vrow(a, q, 0, kk, cur);
                for (int kt = 0; kt < a.ktiles; ++kt) {
                    if (nz && a.vstage) {
                        // V rows came with the stage: wait for it, then transpose
                        if (!mbar_wait(&full[s], ph, a.status, kWaitRingFull) || *abort_flag) {
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        char *vtp = smem + (size_t)s * a.stage_bytes + kTlATile + a.BN * 128;
                        tl_load_vrow_smem(a, vtp + a.zc * 128, kt, kk, cur);
#pragma unroll
                        for (int w = 0; w < 32; ++w) {
                            if (2 * w < a.zc) {
                                *reinterpret_cast<uint16_t *>(vtp + tl_swz(2 * w, kk, a.zc)) = (uint16_t)(cur[w] & 0xffffu);
                                *reinterpret_cast<uint16_t *>(vtp + tl_swz(2 * w + 1, kk, a.zc)) = (uint16_t)(cur[w] >> 16);
                            }
                        }
                        fence_async_smem();
                        mbar_arrive(&vfull[s]);
                    } else if (nz) {
                        if (kt + 1 < a.ktiles) tl_load_vrow(a, q, kt + 1, kk, nxt);
                        // the stage is free once the MMAs of its previous use are done
                        if (!mbar_wait(&empty[s], ph ^ 1u, a.status, kWaitRingEmpty) || *abort_flag) {
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        char *vtp = smem + (size_t)s * a.stage_bytes + kTlATile + a.BN * 128;
#pragma unroll
                        for (int w = 0; w < 32; ++w) {
                            if (2 * w < a.zc) {
                                *reinterpret_cast<uint16_t *>(vtp + tl_swz(2 * w, kk, a.zc)) = (uint16_t)(cur[w] & 0xffffu);
                                *reinterpret_cast<uint16_t *>(vtp + tl_swz(2 * w + 1, kk, a.zc)) = (uint16_t)(cur[w] >> 16);
                            }
                        }
                        fence_async_smem();
                        mbar_arrive(&vfull[s]);
#pragma unroll
                        for (int w = 0; w < 32; ++w) cur[w] = nxt[w];
                    }
                    if (++s == a.nst) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------ epilogue
        const int e = threadIdx.x - 128;  // 0..255
        const int quarter = warp & 3;     // TMEM lane quarter
        const int half = (warp - 4) >> 2;  // which half of the columns
        const int row = quarter * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        int j = 0, prev_key = -1;
        for (int t = blockIdx.x; t < ntall; t += gridDim.x, ++j) {
            const TlTile q = tl_tile(a, t);
            const bool nz = has_z && q.key != prev_key;
            prev_key = q.key;
            const int b = j & 1;
            const unsigned par = (unsigned)((j >> 1) & 1);
            const uint32_t tacc = tmem + lane_off + (uint32_t)(b * 256);

            // (1) s and the delta's B operand [U | U] of this tile, one row
            // per thread (the previous tile's delta MMAs have completed: the
            // epilogue waited for them)
            tl_epi_bar();
            if (e < a.BN) {
                const int slot = a.pair ? (e >= a.bh) : 0;
                const TlSeg &sg = a.seg[a.pair ? slot : q.si];
                const int n = q.n0 + e - slot * a.bh;
                const bool nok = n < sg.out;
                s_tile[e] = nok ? sg.s[n] : 0.f;
                if (a.r > 0) {
                    // K positions: [hi part (zc) | lo part (zc, fp32 outputs) | zero pad]; this
                    // row's U (zero past r) sits at slot*rpad within each part
                    const bool vec = (a.r & 7) == 0 && (reinterpret_cast<uintptr_t>(sg.U) & 15) == 0;
                    const bf16 *urow = sg.U + (int64_t)n * a.r;
                    for (int p0 = 0; p0 < a.Kz; p0 += 8) {
                        const int nparts = a.zlo ? 2 : 1;
                        const int part = p0 < a.zc ? 0 : (p0 < 2 * a.zc && nparts == 2 ? 1 : 2);
                        const int j0 = p0 - part * a.zc - slot * a.rpad;
                        uint4 v = make_uint4(0u, 0u, 0u, 0u);
                        if (part < 2 && j0 >= 0 && j0 < a.r && nok) {
                            if (vec) {
                                v = __ldg(reinterpret_cast<const uint4 *>(urow + j0));
                            } else {
                                const unsigned short *pu = reinterpret_cast<const unsigned short *>(urow);
                                uint32_t w[4];
#pragma unroll
                                for (int h = 0; h < 4; ++h) {
                                    const int j = j0 + 2 * h;
                                    const uint32_t lo = j < a.r ? (uint32_t)__ldg(pu + j) : 0u;
                                    const uint32_t hi = j + 1 < a.r ? (uint32_t)__ldg(pu + j + 1) : 0u;
                                    w[h] = lo | (hi << 16);
                                }
                                v = make_uint4(w[0], w[1], w[2], w[3]);
                            }
                        }
                        *reinterpret_cast<uint4 *>(bu + tl_swz(e, p0, a.BN)) = v;
                    }
                }
            }
            fence_async_smem();
            // (2) the tile's accumulator
            {
                int ok = 1;
                if (e == 0) ok = mbar_wait(&acc_full[b], par, a.status, kWaitRingFull);
                if (e == 0 && !ok) *abort_flag = 1;
                tl_epi_bar();
                if (*abort_flag) break;
            }
            tc_fence_after();
            if (a.r > 0) {
                if (nz) {
                    // z (fp32) -> A_z = [z_hi | z_lo (fp32 outputs) | 0] for this row
                    const int zh = a.zc / 2;
                    for (int c0 = half * zh; c0 < (half + 1) * zh; c0 += 32) {
                    const int nzc = ((half + 1) * zh - c0) >= 32 ? 4 : ((half + 1) * zh - c0) / 8;
                    uint32_t zr[4][8];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (i < nzc) tmem_ld8_nw(tacc + (uint32_t)(a.BN + c0 + 8 * i), zr[i]);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (i < nzc) tmem_wait_ld8(zr[i]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (i < nzc) {
                            const int c = c0 + 8 * i;
                            uint32_t hi[4], lo[4];
#pragma unroll
                            for (int p = 0; p < 4; ++p) {
                                const float za = __uint_as_float(zr[i][2 * p]), zb = __uint_as_float(zr[i][2 * p + 1]);
                                const float ha = __bfloat162float(__float2bfloat16_rn(za));
                                const float hb = __bfloat162float(__float2bfloat16_rn(zb));
                                hi[p] = tl_pack(ha, hb);
                                lo[p] = tl_pack(za - ha, zb - hb);
                            }
                            *reinterpret_cast<uint4 *>(az + tl_swz(row, c, kTlBM)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                            if (a.zlo)
                                *reinterpret_cast<uint4 *>(az + tl_swz(row, a.zc + c, kTlBM)) =
                                    make_uint4(lo[0], lo[1], lo[2], lo[3]);
                        }
                    }
                    }
                    for (int c = (a.zlo ? 2 : 1) * a.zc + 8 * half; c < a.Kz; c += 16)
                        *reinterpret_cast<uint4 *>(az + tl_swz(row, c, kTlBM)) = make_uint4(0u, 0u, 0u, 0u);
                }
                // acc = s * acc, in place, 32 columns per TMEM round trip
                const int nc = a.pair ? a.bh / 2 : a.BN / 2;
                for (int part = 0; part < (a.pair ? 2 : 1); ++part) {
                    const int cb = part * a.bh + half * nc;
                    for (int c = cb; c < cb + nc; c += 32) {
                        const int nch = (cb + nc - c) >= 32 ? 4 : (cb + nc - c) / 8;
                        uint32_t vr[4][8];
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (i < nch) tmem_ld8_nw(tacc + (uint32_t)(c + 8 * i), vr[i]);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (i < nch) tmem_wait_ld8(vr[i]);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            if (i < nch) {
                                float v[8];
#pragma unroll
                                for (int k2 = 0; k2 < 8; ++k2) v[k2] = __uint_as_float(vr[i][k2]) * s_tile[c + 8 * i + k2];
                                tmem_st8(tacc + (uint32_t)(c + 8 * i), v);
                            }
                        }
                    }
                }
                tmem_wait_st();
                fence_async_smem();
                tc_fence_before();
                tl_epi_bar();
                if (e == 0) mbar_arrive(&dready[b]);
                int ok = 1;
                if (e == 0) ok = mbar_wait(&dfull[b], par, a.status, kWaitRingFull);
                if (e == 0 && !ok) *abort_flag = 1;
                tl_epi_bar();
                if (*abort_flag) break;
                tc_fence_after();
            }
            // (3) outputs
            const int m = q.m0 + row;
            const bool row_ok = m < a.T;
            const bool scale_here = a.r == 0;  // r == 0: s is applied here
            if (a.pair) {
                const int nc = a.bh / 2;
                const TlSeg &sg = a.seg[0];
                for (int c0 = half * nc; c0 < (half + 1) * nc; c0 += 16) {
                    const int nch = ((half + 1) * nc - c0) >= 16 ? 2 : 1;
                    uint32_t gr[2][8], ur[2][8];
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        if (i < nch) {
                            tmem_ld8_nw(tacc + (uint32_t)(c0 + 8 * i), gr[i]);
                            tmem_ld8_nw(tacc + (uint32_t)(a.bh + c0 + 8 * i), ur[i]);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        if (i < nch) {
                            tmem_wait_ld8(gr[i]);
                            tmem_wait_ld8(ur[i]);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int c = c0 + 8 * i;
                        const int n = q.n0 + c;  // h column
                        if (i < nch && row_ok && n < a.hw) {
                            float hv[8], lv[8];
#pragma unroll
                            for (int k2 = 0; k2 < 8; ++k2) {
                                float g = __uint_as_float(gr[i][k2]), u = __uint_as_float(ur[i][k2]);
                                if (scale_here) {
                                    g *= s_tile[c + k2];
                                    u *= s_tile[a.bh + c + k2];
                                }
                                const float h = (n + k2 < sg.out) ? tl_gelu_mul(g, u) : 0.f;
                                hv[k2] = h;
                                lv[k2] = h - __bfloat162float(__float2bfloat16_rn(h));
                            }
                            const int64_t off = (int64_t)m * a.ldy + n;
                            tl_store8(sg.y, WL_OUT_BF16, off, a.hw - n, hv);
                            if (a.hlo) tl_store8(sg.y, WL_OUT_BF16, off + a.hlo, a.hw - n, lv);
                        }
                    }
                }
            } else {
                const int nc = a.BN / 2;
                const TlSeg &sg = a.seg[q.si];
                for (int c0 = half * nc; c0 < (half + 1) * nc; c0 += 32) {
                    const int nch = ((half + 1) * nc - c0) >= 32 ? 4 : ((half + 1) * nc - c0) / 8;
                    uint32_t vr[4][8];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (i < nch) tmem_ld8_nw(tacc + (uint32_t)(c0 + 8 * i), vr[i]);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (i < nch) tmem_wait_ld8(vr[i]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int c = c0 + 8 * i;
                        const int n = q.n0 + c;
                        if (i < nch && row_ok && n < sg.out) {
                            float v[8];
#pragma unroll
                            for (int k2 = 0; k2 < 8; ++k2)
                                v[k2] = scale_here ? __uint_as_float(vr[i][k2]) * s_tile[c + k2] : __uint_as_float(vr[i][k2]);
                            tl_store8(sg.y, a.ydt, (int64_t)m * sg.out + n, sg.out - n, v);
                        }
                    }
                }
            }
            // (4) the buffer is free for the tile after next
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[b]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
    }
}

// ------------------------------------------------------------------ host --
static std::mutex g_tl_mu;
static std::unordered_map<int, int> g_tl_attr;

bool prefill_tiles_applicable(int64_t Ktot, int64_t r, int ydt, bool pair, bool v_aligned)
{
    const int64_t rpad = (r + 15) / 16 * 16;
    // z of a tile lives in the TMEM buffer next to the accumulator: BN + z
    // columns = 256.  Paired tiles carry z of two projections: up to rank 32,
    // or rank 64 with bf16 outputs and V rows loaded by TMA (the V^T writers
    // hold at most 64 z columns).
    if (rpad > 64) return false;
    if (pair && rpad > 32 && !(r == 64 && ydt == WL_OUT_BF16 && v_aligned)) return false;
    // fp32 outputs: the tensor cores' fp32 accumulation error grows with the
    // K chain; long chains go to the split-K kernel
    if (ydt == WL_OUT_F32 && Ktot > 4096) return false;
    return true;
}

// x [T, Ktot] (row stride Ktot); proj[0..nproj) share x.  pair: proj[0] =
// gate, proj[1] = up, y[0] = h with row stride ldy, hw columns per part
// (zeros beyond gate.out), remainder part at column hlo (0: none).
wl_status launch_prefill_tiles(const bf16 *x, const wl_proj *proj, int nproj, bool pair, void *const *y,
                               int64_t ldy, int64_t T, int64_t in, int64_t Ktot, int64_t kmod, int64_t r,
                               int ydt, int64_t hw, int64_t hlo, cudaStream_t st)
{
    wl_status s = WL_OK;
    const DeviceInfo *di = device_info(&s);
    if (!di) return s;
    bool valign = true;
    for (int jj = 0; jj < (pair ? 2 : nproj); ++jj)
        if (reinterpret_cast<uintptr_t>(proj[jj].V) & 15) valign = false;
    if (!prefill_tiles_applicable(Ktot, r, ydt, pair, valign)) return fail(WL_ERR_UNSUPPORTED, "prefill tiles: shape");
    if (kmod < in || (Ktot > kmod && kmod % 64 != 0)) return fail(WL_ERR_UNSUPPORTED, "prefill tiles: bad K period");
    TlArgs a = {};
    a.nseg = pair ? 2 : nproj;
    a.pair = pair ? 1 : 0;
    a.T = (int)T;
    a.in = (int)in;
    a.Ktot = (int)Ktot;
    a.kmod = (int)kmod;
    a.r = (int)r;
    a.rpad = r > 0 ? (int)((r + 15) / 16 * 16) : 0;
    a.ydt = ydt;
    a.zc = a.rpad * (pair ? 2 : 1);
    // z enters the delta MMA as bf16: the hi part alone moves y by about 2^-9
    // of the rank-r term (well inside the bf16 bar); fp32 outputs add the lo part
    a.zlo = ydt == WL_OUT_F32 ? 1 : 0;
    a.Kz = a.zc > 0 ? ((a.zlo ? 2 : 1) * a.zc + 63) / 64 * 64 : 0;
    a.mtiles = (int)((T + kTlBM - 1) / kTlBM);
    a.ktiles = (int)((Ktot + 63) / 64);
    a.ldy = (int)ldy;
    a.hw = (int)hw;
    a.hlo = (int)hlo;
    a.status = di->status;
    const int sm = di->sm_count;

    // Tile width: the widest that fits next to the z columns, or 128 when
    // that fills the SMs in fewer rounds (few tiles, long K).
    auto ntiles_for = [&](int BN) {
        int n = 0;
        if (pair) return (int)((hw + BN / 2 - 1) / (BN / 2));
        for (int jj = 0; jj < nproj; ++jj) n += (int)((proj[jj].out + BN - 1) / BN);
        return n;
    };
    auto grid_for = [&](int tiles) {
        int g = sm;
        if (a.mtiles <= sm && (sm / a.mtiles) * a.mtiles * 10 >= 9 * sm) g = (sm / a.mtiles) * a.mtiles;
        return tiles < g ? tiles : g;
    };
    const int bn_max = 256 - a.zc;
    int best_bn = bn_max;
    long best_cost = -1;
    const int cands[2] = {bn_max, 128};
    for (int ci = 0; ci < 2; ++ci) {
        const int BN = cands[ci];
        if (BN > bn_max || (ci == 1 && BN == bn_max)) continue;
        const int tiles = a.mtiles * ntiles_for(BN);
        const int g = grid_for(tiles);
        const long rounds = (tiles + g - 1) / g;
        const long cost = rounds * (BN + 32);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best_bn = BN;
        }
    }
    a.BN = best_bn;
    a.bh = pair ? a.BN / 2 : a.BN;
    a.ntiles = ntiles_for(a.BN);
    const int tiles = a.mtiles * a.ntiles;
    const int grid = grid_for(tiles);

    s = tmap_2d_bf16(x, Ktot, T, Ktot, 64, kTlBM, &a.mapa);
    if (s != WL_OK) return s;
    int nt = 0;
    for (int jj = 0; jj < (pair ? 2 : nproj); ++jj) {
        TlSeg &sg = a.seg[jj];
        s = tmap_2d_bf16(proj[jj].W0, in, proj[jj].out, in, 64, a.bh, &sg.mapb);
        if (s != WL_OK) return s;
        sg.s = proj[jj].s;
        sg.U = static_cast<const bf16 *>(proj[jj].U);
        sg.V = static_cast<const bf16 *>(proj[jj].V);
        sg.y = pair ? y[0] : y[jj];
        sg.out = (int)proj[jj].out;
        sg.ntile0 = pair ? 0 : nt;
        if (!pair) nt += (int)((proj[jj].out + a.BN - 1) / a.BN);
    }
    a.vstage = r > 0 ? 1 : 0;
    for (int jj = 0; jj < (pair ? 2 : nproj); ++jj)
        if (reinterpret_cast<uintptr_t>(proj[jj].V) & 15) a.vstage = 0;
    // V rows straight into the z MMA (MN-major operand) where a row is a whole
    // swizzle span: r = 16, 32, 64
    a.vtma = (a.vstage && (r == 16 || r == 32 || r == 64)) ? 1 : 0;
    a.vsw = r == 16 ? 6 : (r == 32 ? 4 : 2);  // 32-, 64-, 128-byte swizzle
    if (a.vtma) {
        a.vstage = 0;
        for (int jj = 0; jj < (pair ? 2 : nproj); ++jj) {
            s = tmap_2d_bf16_swz(proj[jj].V, r, in, r, (int)r, 64, (int)r * 2, &a.seg[jj].mapv);
            if (s != WL_OK) return s;
        }
    }
    a.stage_bytes = kTlATile + a.BN * 128 + (a.vtma ? 0 : a.zc * 128) +
                    ((a.vstage || a.vtma) ? (pair ? 2 : 1) * 64 * (int)r * 2 : 0);
    a.stage_bytes = (a.stage_bytes + 1023) / 1024 * 1024;
    const int fixed = 1024 + (a.Kz / 64) * (kTlATile + a.BN * 128) + a.BN * 4 + (3 * kTlMaxStages + 9) * 8 + 16;
    int nst = (di->max_smem_optin - fixed) / a.stage_bytes;
    if (nst > kTlMaxStages) nst = kTlMaxStages;
    if (nst < 2) return fail(WL_ERR_UNSUPPORTED, "prefill tiles: not enough shared memory");
    a.nst = nst;
    const int smem = fixed + nst * a.stage_bytes;
    {
        std::lock_guard<std::mutex> lk(g_tl_mu);
        if (!g_tl_attr.count(di->device)) {
            cudaError_t e = cudaFuncSetAttribute((const void *)prefill_tiles_kernel,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, di->max_smem_optin);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prefill tiles)");
            g_tl_attr[di->device] = 1;
        }
    }
    prefill_tiles_kernel<<<grid, kTlThreads, smem, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "prefill tiles launch");
    return WL_OK;
}

}  // namespace wl
