// prefill.cu -- large-T weightless projections on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory), fed by TMA.
//
// Computes ("In-kernel reconstruction", formula section and "The GEMM path")
//     y = s[None,:] * (x W0^T) + z U^T,   z = x V
// for a tile of 128 tokens x 256 output rows per CTA:
//   * the main product x W0^T (M = 128 tokens, N = 256 rows, K = in) runs as
//     tcgen05.mma kind::f16 (bf16 in, fp32 accumulate) into TMEM columns
//     [0, 256);
//   * z = x V is formed in the same K loop by a second MMA of the same x
//     tile against V^T (N = r rounded up to 16) into TMEM columns [256, ...);
//     V^T is written into swizzled shared memory by the epilogue warps while
//     the main loop runs (V is [in, r], so its transpose is not a TMA tile):
//     the stage's 64 V rows arrive by bulk copy with the x and W0 tiles and
//     are transposed shared-to-shared, or (r not a multiple of 8) are read
//     from global memory;
//   * the epilogue splits z into bf16 hi + lo parts (z = hi + lo to about 16
//     bits) and runs the rank-r delta [hi | lo] [U | U]^T as one more MMA into
//     TMEM columns [256, 512), then forms s * acc + delta in fp32 and casts
//     once ("The GEMM path": the final combine is done in float32).
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM owner and
// MMA issuer (one elected thread), warps 2..5 = V^T writer during the main
// loop, then the epilogue (warp w reads TMEM lanes 32*(w%4) .. +31).
// Every mbarrier wait is bounded; on a timeout the status word is set and the
// CTA winds down.
#include <mutex>
#include <unordered_map>

#include "tc_ptx.cuh"

namespace wl {

constexpr int kPfThreads = 192;
constexpr int kBM = 128;            // tokens per tile
constexpr int kBN = 256;            // output rows per tile
constexpr int kBKp = 64;            // k per stage (one 128-byte swizzle atom)
constexpr int kATile = kBM * 128;   // 16 KB
constexpr int kBTile = kBN * 128;   // 32 KB
constexpr uint32_t kTmemCols = 512;

// ------------------------------------------------------------------ PTX --

__device__ __forceinline__ void pf_mbar_init(uint64_t *bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(s32(bar)), "r"(count));
}
__device__ __forceinline__ void pf_expect_tx(uint64_t *bar, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(s32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void pf_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(s32(bar)) : "memory");
}
__device__ __forceinline__ bool pf_test(uint64_t *bar, unsigned parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(s32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __noinline__ bool pf_wait(uint64_t *bar, unsigned parity, unsigned *status, unsigned site)
{
    if (pf_test(bar, parity)) return true;
    const long long t0 = wait_clock();
    while (!pf_test(bar, parity)) {
        if (wait_clock() - t0 > kWaitLimitCycles) {
            atomicOr(status, kStatusTimeout | site);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void pf_tma_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(s32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(s32(bar))
        : "memory");
}

// Contiguous global -> shared copy (16-byte aligned addresses, size a
// multiple of 16) completing on `bar`'s transaction count.
__device__ __forceinline__ void pf_bulk(void *dst, const void *src, unsigned bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     s32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(s32(bar))
                 : "memory");
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }
__device__ __forceinline__ void pf_cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Four floats at the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ float4 ld_peer4(const float *p, uint32_t rank)
{
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(s32(p)), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(ra)
                 : "memory");
    return v;
}

// Byte offset of element (row, k) in a K-major tile with 128-byte swizzle:
// atoms of 8 rows x 128 bytes (1024 B); atom columns of 64 elements, each
// `rows` x 128 bytes.
__device__ __forceinline__ uint32_t swz(int row, int k, int rows)
{
    const int a = k >> 6, kk = k & 63;
    return (uint32_t)(a * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 + ((((kk >> 3) ^ (row & 7)) << 4)) +
                      (kk & 7) * 2);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// ---------------------------------------------------------------- kernel --
struct PfSeg {
    CUtensorMap mapb;  // W0 [out, in], box 64 x 256
    const float *s;
    const bf16 *U;
    const bf16 *V;
    void *y;
    int out;
    int ntile0;  // first n-tile of this segment
};

struct PfArgs {
    PfSeg seg[3];
    CUtensorMap mapa;  // x [T, Ktot], box 64 x 128
    int nseg;
    int T, in, Ktot, kmod, r, ydt;  // K position k maps to W0 column / V row k % kmod (< in)
    int rpad, Kz, nst, stage_bytes;
    int vstage;  // 1: V rows arrive by bulk copy with the stage (r % 8 == 0, V 16-byte aligned)
    int ns, kts;  // K splits (= cluster size along z) and k-tiles per split
    unsigned *status;
};

constexpr int kPStride = kBN + 4;  // fp32 partial tile row stride (floats)

__global__ void __launch_bounds__(kPfThreads, 1) prefill_kernel(const __grid_constant__ PfArgs a)
{
    extern __shared__ __align__(1024) char smem_raw[];
    char *smem = smem_raw + ((1024u - (s32(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = blockIdx.x, nt = blockIdx.y;
    const int si = (a.nseg > 2 && nt >= a.seg[2].ntile0) ? 2 : (a.nseg > 1 && nt >= a.seg[1].ntile0) ? 1 : 0;
    const PfSeg &sg = a.seg[si];
    const int m0 = mt * kBM, n0 = (nt - sg.ntile0) * kBN;
    const int r = a.r;
    const int ktiles_all = (a.Ktot + kBKp - 1) / kBKp;
    const int kq = (int)blockIdx.z;
    const int kt0 = kq * a.kts;
    const int ktiles = min(ktiles_all, kt0 + a.kts);  // this CTA: k-tiles [kt0, ktiles)
    const int vt_bytes = a.rpad * 128;

    // shared memory: stages | barriers | tmem holder | s tile
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)a.nst * a.stage_bytes);
    uint64_t *full = bars, *empty = bars + a.nst, *vfull = bars + 2 * a.nst;  // TMA done / V^T written / free
    uint64_t *acc_full = bars + 3 * a.nst, *z_ready = acc_full + 1, *d_ready = acc_full + 2;
    uint32_t *tmem_hold = reinterpret_cast<uint32_t *>(acc_full + 3);
    volatile int &abort_flag = *reinterpret_cast<volatile int *>(tmem_hold + 1);
    float *s_tile = reinterpret_cast<float *>(tmem_hold + 4);

    if (threadIdx.x == 0) {
        for (int i = 0; i < a.nst; ++i) {
            pf_mbar_init(&full[i], 1);
            pf_mbar_init(&empty[i], 1);
            pf_mbar_init(&vfull[i], 1);
        }
        pf_mbar_init(acc_full, 1);
        pf_mbar_init(z_ready, 1);
        pf_mbar_init(d_ready, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        abort_flag = 0;
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(s32(tmem_hold)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // zero the padding rows [r, rpad) of every stage's V^T tile once
    if (r > 0 && warp >= 2) {
        for (int st = 0; st < a.nst; ++st) {
            char *vt = smem + (size_t)st * a.stage_bytes + kATile + kBTile;
            for (int i = threadIdx.x - 64; i < vt_bytes / 16; i += 128) {
                const int row = (i * 16) / 128;
                if (row >= r) reinterpret_cast<uint4 *>(vt)[i] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        fence_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_hold;
    const uint32_t t_main = tmem, t_aux = tmem + kBN;  // columns [0,256) and [256,512)

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0;
            unsigned ph = 0;
            for (int kt = kt0; kt < ktiles; ++kt) {
                if (!pf_wait(&empty[s], ph ^ 1u, a.status, kWaitRingEmpty)) {
                    abort_flag = 1;
                    break;
                }
                char *st = smem + (size_t)s * a.stage_bytes;
                const int kc = kt * kBKp;
                const int krow0 = kc % a.kmod;  // V row of this stage's first K position
                const int vrows = a.vstage ? max(0, min(kBKp, a.in - krow0)) : 0;
                const unsigned vbytes = (unsigned)(vrows * r * 2);
                pf_expect_tx(&full[s], kATile + kBTile + vbytes);
                pf_tma_2d(st, &a.mapa, kc, m0, &full[s]);
                pf_tma_2d(st + kATile, &sg.mapb, krow0, n0, &full[s]);
                if (vbytes)
                    pf_bulk(st + kATile + kBTile + vt_bytes, sg.V + (int64_t)krow0 * r, vbytes, &full[s]);
                if (++s == a.nst) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_main = idesc_bf16(kBM, kBN);
            const uint32_t id_z = idesc_bf16(kBM, a.rpad > 0 ? a.rpad : 16);
            int s = 0;
            unsigned ph = 0;
            bool ok = true;
            for (int kt = kt0; kt < ktiles; ++kt) {
                if (!pf_wait(&full[s], ph, a.status, kWaitRingFull) ||
                    (r > 0 && !pf_wait(&vfull[s], ph, a.status, kWaitRingFull))) {
                    ok = false;
                    abort_flag = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = s32(smem + (size_t)s * a.stage_bytes);
                const uint32_t sb = sa + kATile, sv = sb + kBTile;
#pragma unroll
                for (int k = 0; k < kBKp / 16; ++k) {
                    const uint64_t da = sdesc(sa + 32 * k);
                    const uint32_t accum = (kt > kt0 || k > 0) ? 1u : 0u;
                    umma(t_main, da, sdesc(sb + 32 * k), id_main, accum);
                    if (r > 0) umma(t_aux, da, sdesc(sv + 32 * k), id_z, accum);
                }
                umma_commit(&empty[s]);  // frees the stage when these MMAs are done
                if (++s == a.nst) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            umma_commit(acc_full);
            if (ok && r > 0) {
                // rank-r delta: [z_hi | z_lo] [U | U]^T into columns [256, 512)
                if (pf_wait(z_ready, 0, a.status, kWaitRingFull)) {
                    tc_fence_after();
                    const uint32_t saz = s32(smem);                          // A_z at stage memory start
                    const uint32_t sbu = saz + (uint32_t)(a.Kz / 64) * kATile;  // B_u after it
                    const uint32_t id_d = idesc_bf16(kBM, kBN);
                    for (int kd = 0; kd < a.Kz / 16; ++kd) {
                        const int at = kd >> 2, kin = kd & 3;
                        umma(t_aux, sdesc(saz + at * kATile + 32 * kin), sdesc(sbu + at * kBTile + 32 * kin), id_d,
                             kd > 0 ? 1u : 0u);
                    }
                    umma_commit(d_ready);
                }
            }
        }
    } else {
        // ------------------------------------------------ V^T writer, then epilogue
        const int et = threadIdx.x - 64;  // 0..127
        const int erow = (warp & 3) * 32 + lane;  // TMEM lane = tile row (token)
        if (r > 0) {
            int s = 0;
            unsigned ph = 0;
            const int nch = (a.rpad < r ? a.rpad : r) * 8;  // (row j, 8-column chunk c) pairs, j < r
            for (int kt = kt0; kt < ktiles; ++kt) {
                // staged: wait for the stage's copies (V rows included);
                // otherwise only for the stage to be free
                int ok = 1;
                if (et == 0)
                    ok = a.vstage ? pf_wait(&full[s], ph, a.status, kWaitRingFull)
                                  : pf_wait(&empty[s], ph ^ 1u, a.status, kWaitRingEmpty);
                if (et == 0 && !ok) abort_flag = 1;
                epi_sync();
                if (abort_flag) break;
                char *vt = smem + (size_t)s * a.stage_bytes + kATile + kBTile;
                const bf16 *vst = reinterpret_cast<const bf16 *>(vt + vt_bytes);  // [64 rows][r]
                const int kb = kt * kBKp;
                const int krow0 = kb % a.kmod;
                for (int idx = et; idx < nch; idx += 128) {
                    const int j = idx >> 3, c = idx & 7;
                    uint16_t v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int kglob = kb + 8 * c + e;  // position along Ktot
                        const int krow = krow0 + 8 * c + e;  // V row (a tile never crosses the K period)
                        const bool in_range = kglob < a.Ktot && krow < a.in;
                        const bf16 *src = a.vstage ? vst + (8 * c + e) * r + j : sg.V + (int64_t)krow * r + j;
                        v[e] = in_range ? *reinterpret_cast<const uint16_t *>(src) : (uint16_t)0;
                    }
                    *reinterpret_cast<uint4 *>(vt + swz(j, 8 * c, a.rpad)) =
                        make_uint4(v[0] | (uint32_t)v[1] << 16, v[2] | (uint32_t)v[3] << 16,
                                   v[4] | (uint32_t)v[5] << 16, v[6] | (uint32_t)v[7] << 16);
                }
                fence_async_smem();
                epi_sync();
                if (et == 0) pf_arrive(&vfull[s]);
                if (++s == a.nst) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        // s of this tile's rows
        for (int i = et; i < kBN; i += 128) s_tile[i] = (n0 + i < sg.out) ? sg.s[n0 + i] : 0.f;

        int ok = 1;
        if (et == 0) ok = pf_wait(acc_full, 0, a.status, kWaitRingFull);
        if (et == 0 && !ok) abort_flag = 1;
        epi_sync();
        tc_fence_after();
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        if (r > 0 && !abort_flag) {
            // z (fp32) -> A_z = [hi | lo | 0] for this row; U rows -> B_u = [U | U | 0]
            char *az = smem;
            char *bu = smem + (size_t)(a.Kz / 64) * kATile;
            float z[16];
            for (int cz = 0; cz < a.rpad; cz += 16) {
                tmem_ld16(t_aux + lane_off + cz, z);
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // two 8-column groups of this 16-column load
                    const int k = cz + 8 * h;
                    if (k >= r) break;
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int ka = k + 2 * e, kb2 = ka + 1;
                        const float za = ka < r ? z[8 * h + 2 * e] : 0.f;
                        const float zb = kb2 < r ? z[8 * h + 2 * e + 1] : 0.f;
                        const float ha = __bfloat162float(__float2bfloat16_rn(za));
                        const float hb = __bfloat162float(__float2bfloat16_rn(zb));
                        hi[e] = pack_bf16(ha, hb);
                        lo[e] = pack_bf16(za - ha, zb - hb);
                    }
                    // hi part at columns [k, k+8), lo part at [r + k, r + k + 8):
                    // write element by element where r is not a multiple of 8
                    if ((r & 7) == 0) {
                        *reinterpret_cast<uint4 *>(az + swz(erow, k, kBM)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                        *reinterpret_cast<uint4 *>(az + swz(erow, r + k, kBM)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    } else {
                        const bf16 *hp = reinterpret_cast<const bf16 *>(hi);
                        const bf16 *lp = reinterpret_cast<const bf16 *>(lo);
                        for (int e = 0; e < 8 && k + e < r; ++e) {
                            *reinterpret_cast<bf16 *>(az + swz(erow, k + e, kBM)) = hp[e];
                            *reinterpret_cast<bf16 *>(az + swz(erow, r + k + e, kBM)) = lp[e];
                        }
                    }
                }
            }
            for (int k = 2 * r; k < a.Kz; ++k) *reinterpret_cast<bf16 *>(az + swz(erow, k, kBM)) = __float2bfloat16_rn(0.f);
            for (int n = et; n < kBN; n += 128) {
                const bool in_range = n0 + n < sg.out;
                const bf16 *Ur = sg.U + (int64_t)(n0 + n) * r;
                for (int kc = 0; kc < a.Kz; kc += 8) {
                    uint16_t v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int k = kc + e;
                        v[e] = (in_range && k < 2 * r) ? reinterpret_cast<const uint16_t *>(Ur)[k < r ? k : k - r] : 0;
                    }
                    *reinterpret_cast<uint4 *>(bu + swz(n, kc, kBN)) =
                        make_uint4(v[0] | (uint32_t)v[1] << 16, v[2] | (uint32_t)v[3] << 16,
                                   v[4] | (uint32_t)v[5] << 16, v[6] | (uint32_t)v[7] << 16);
                }
            }
            fence_async_smem();
            tc_fence_before();
            epi_sync();
            if (et == 0) pf_arrive(z_ready);
            int ok2 = 1;
            if (et == 0) ok2 = pf_wait(d_ready, 0, a.status, kWaitRingFull);
            if (et == 0 && !ok2) abort_flag = 1;
            epi_sync();
            tc_fence_after();
        }
        if (!abort_flag) {
            // y = s * acc + delta, one tile row per thread
            const int m = m0 + erow;
            const bool row_ok = m < a.T;
            const int es = a.ydt == WL_OUT_F32 ? 4 : 2;
            for (int c = 0; c < kBN; c += 16) {
                float acc[16], dl[16];
                tmem_ld16(t_main + lane_off + c, acc);
                if (r > 0) tmem_ld16(t_aux + lane_off + c, dl);
                else
#pragma unroll
                    for (int i = 0; i < 16; ++i) dl[i] = 0.f;
                if (!row_ok || n0 + c >= sg.out) continue;
                float yv[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) yv[i] = fmaf(s_tile[c + i], acc[i], dl[i]);
                if (a.ns > 1) {  // partial over this K split: to shared memory, added across the cluster below
                    float *prow = reinterpret_cast<float *>(smem) + erow * kPStride + c;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        reinterpret_cast<float4 *>(prow)[q] = make_float4(yv[4 * q], yv[4 * q + 1], yv[4 * q + 2], yv[4 * q + 3]);
                    continue;
                }
                const int nvalid = sg.out - (n0 + c);
                char *dst = static_cast<char *>(sg.y) + ((int64_t)m * sg.out + n0 + c) * es;
                const bool vec = nvalid >= 16 && ((reinterpret_cast<uintptr_t>(dst) & 15) == 0);
                if (a.ydt == WL_OUT_F32) {
                    if (vec) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            reinterpret_cast<float4 *>(dst)[q] =
                                make_float4(yv[4 * q], yv[4 * q + 1], yv[4 * q + 2], yv[4 * q + 3]);
                    } else {
                        for (int i = 0; i < 16 && i < nvalid; ++i) reinterpret_cast<float *>(dst)[i] = yv[i];
                    }
                } else {
                    if (vec) {
#pragma unroll
                        for (int q = 0; q < 2; ++q)
                            reinterpret_cast<uint4 *>(dst)[q] =
                                make_uint4(pack_bf16(yv[8 * q], yv[8 * q + 1]), pack_bf16(yv[8 * q + 2], yv[8 * q + 3]),
                                           pack_bf16(yv[8 * q + 4], yv[8 * q + 5]), pack_bf16(yv[8 * q + 6], yv[8 * q + 7]));
                    } else {
                        for (int i = 0; i < 16 && i < nvalid; ++i)
                            reinterpret_cast<bf16 *>(dst)[i] = __float2bfloat16_rn(yv[i]);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (a.ns > 1) {
        // Deterministic sum of the ns K-split partials (rank order), rows of
        // the tile shared out among the cluster's CTAs, then the cast.
        pf_cluster_sync();
        const uint32_t me = cluster_rank();
        const int rlo = (int)(me * kBM / a.ns), rhi = (int)((me + 1) * kBM / a.ns);
        const float *pt = reinterpret_cast<const float *>(smem);
        const int es = a.ydt == WL_OUT_F32 ? 4 : 2;
        for (int idx = threadIdx.x; idx < (rhi - rlo) * (kBN / 4); idx += kPfThreads) {
            const int row = rlo + idx / (kBN / 4), col = 4 * (idx % (kBN / 4));
            const int m = m0 + row;
            if (m >= a.T || n0 + col >= sg.out) continue;
            float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int p = 0; p < a.ns; ++p) {
                const float4 v = ld_peer4(pt + row * kPStride + col, (uint32_t)p);
                sum.x += v.x;
                sum.y += v.y;
                sum.z += v.z;
                sum.w += v.w;
            }
            const float yv[4] = {sum.x, sum.y, sum.z, sum.w};
            const int nvalid = sg.out - (n0 + col);
            char *dst = static_cast<char *>(sg.y) + ((int64_t)m * sg.out + n0 + col) * es;
            for (int i = 0; i < 4 && i < nvalid; ++i) {
                if (a.ydt == WL_OUT_F32)
                    reinterpret_cast<float *>(dst)[i] = yv[i];
                else
                    reinterpret_cast<bf16 *>(dst)[i] = __float2bfloat16_rn(yv[i]);
            }
        }
        pf_cluster_sync();  // peers are done reading this CTA's partial tile
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

// ------------------------------------------------------------------ host --
static std::mutex g_pf_mu;
static std::unordered_map<int, int> g_pf_attr;

// Whether the persistent tiles kernel would leave most SMs idle: fewer output
// tiles (128 tokens x about 224 rows) than half the SMs.  Each tile then runs
// the whole K loop on one SM, and the split-K kernel, which spreads K over a
// cluster, finishes sooner (measured on GB300: the large-set down projection at
// 64 tokens, 24 tiles of 336 k-stages; the Gemma MLP at 16 to 128 tokens).
static bool few_tiles(int64_t T, int64_t rows)
{
    wl_status s = WL_OK;
    const DeviceInfo *di = device_info(&s);
    if (!di) return false;
    const int64_t tiles = (T + 127) / 128 * ((rows + 223) / 224);
    return tiles * 2 < di->sm_count;
}

wl_status launch_prefill(const bf16 *x, const wl_proj *proj, int nproj, void *const *y, int64_t T,
                         int64_t in, int64_t Ktot, int64_t kmod, int64_t r, int ydt, cudaStream_t st)
{
    bool valign = true;
    int64_t rows = 0;
    for (int j = 0; j < nproj; ++j) {
        if (reinterpret_cast<uintptr_t>(proj[j].V) & 15) valign = false;
        rows += proj[j].out;
    }
    if (prefill_tiles_applicable(Ktot, r, ydt, false, valign) && !few_tiles(T, rows))
        return launch_prefill_tiles(x, proj, nproj, false, y, 0, T, in, Ktot, kmod, r, ydt, 0, 0, st);
    wl_status s = WL_OK;
    const DeviceInfo *di = device_info(&s);
    if (!di) return s;
    if (r > 128) return fail(WL_ERR_UNSUPPORTED, "prefill: r > 128");
    if (kmod < in || (Ktot > kmod && kmod % kBKp != 0))
        return fail(WL_ERR_UNSUPPORTED, "prefill: bad K period");
    PfArgs a = {};
    a.nseg = nproj;
    a.T = (int)T;
    a.in = (int)in;
    a.Ktot = (int)Ktot;
    a.kmod = (int)kmod;
    a.r = (int)r;
    a.ydt = ydt;
    a.rpad = r > 0 ? (int)((r + 15) / 16 * 16) : 0;
    a.Kz = r > 0 ? (int)((2 * r + 63) / 64 * 64) : 0;
    a.status = di->status;
    // V rows by bulk copy: rows of r bf16 must be a whole number of 16-byte
    // chunks, V 16-byte aligned, and the larger stage must still leave room
    // for the epilogue's A_z / B_u tiles (checked below)
    a.vstage = (r > 0 && r % 8 == 0 && (reinterpret_cast<uintptr_t>(proj[0].V) & 15) == 0) ? 1 : 0;
    for (int j = 1; j < nproj; ++j)
        if (reinterpret_cast<uintptr_t>(proj[j].V) & 15) a.vstage = 0;
    s = tmap_2d_bf16(x, Ktot, T, Ktot, kBKp, kBM, &a.mapa);
    if (s != WL_OK) return s;
    int ntile = 0;
    for (int j = 0; j < nproj; ++j) {
        PfSeg &sg = a.seg[j];
        s = tmap_2d_bf16(proj[j].W0, in, proj[j].out, in, kBKp, kBN, &sg.mapb);
        if (s != WL_OK) return s;
        sg.s = proj[j].s;
        sg.U = static_cast<const bf16 *>(proj[j].U);
        sg.V = static_cast<const bf16 *>(proj[j].V);
        sg.y = y[j];
        sg.out = (int)proj[j].out;
        sg.ntile0 = ntile;
        ntile += (int)((proj[j].out + kBN - 1) / kBN);
    }
    // stages: as many as fit; the epilogue's A_z / B_u tiles reuse the stages
    const int extra = 1024 + (3 * 8 + 3) * 8 + 16 + kBN * 4 + 64;
    const int need_epi = (a.Kz / 64) * (kATile + kBTile);
    int nst = 0;
    for (int pass = 0; pass < 2 && nst == 0; ++pass) {
        if (pass == 1) a.vstage = 0;
        a.stage_bytes = kATile + kBTile + a.rpad * 128 + (a.vstage ? kBKp * (int)r * 2 : 0);
        int n = (di->max_smem_optin - extra) / a.stage_bytes;
        if (n > 4) n = 4;
        while (n * a.stage_bytes < need_epi) ++n;
        if (n >= 2 && n * a.stage_bytes + extra <= di->max_smem_optin) nst = n;
    }
    if (nst == 0)
        return fail(WL_ERR_UNSUPPORTED, "prefill: r=%lld needs more shared memory than the device has", (long long)r);
    a.nst = nst;
    const int smem = nst * a.stage_bytes + extra;
    {
        std::lock_guard<std::mutex> lk(g_pf_mu);
        if (!g_pf_attr.count(di->device)) {
            cudaError_t e = cudaFuncSetAttribute((const void *)prefill_kernel,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, di->max_smem_optin);
            if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prefill)");
            g_pf_attr[di->device] = 1;
        }
    }
    // K splits: enough CTAs for the SMs, and (fp32 outputs) at most 4096 k
    // per accumulation chain: the tensor cores' fp32 accumulation error grows
    // with the length of the chain, and the splits meet in exact fp32.
    const int mtiles = (int)((T + kBM - 1) / kBM);
    const int ktiles = (int)((Ktot + kBKp - 1) / kBKp);
    const int ctas = mtiles * ntile;
    int ns = di->sm_count / ctas;
    if (ydt == WL_OUT_F32) {
        const int need = (ktiles + 63) / 64;
        if (ns < need) ns = need;
    }
    if (ns > 8) ns = 8;
    if (ns > ktiles / 4) ns = ktiles / 4;
    if (ns < 1) ns = 1;
    a.kts = (ktiles + ns - 1) / ns;
    a.ns = (ktiles + a.kts - 1) / a.kts;
    if (a.ns > 1 && nst * a.stage_bytes < kBM * kPStride * 4)
        return fail(WL_ERR_UNSUPPORTED, "prefill: no room for the split-K partial tile");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)mtiles, (unsigned)ntile, (unsigned)a.ns);
    cfg.blockDim = dim3(kPfThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = (unsigned)a.ns;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {&a};
    cudaError_t e = cudaLaunchKernelExC(&cfg, (const void *)prefill_kernel, args);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return WL_OK;
}

// h = gelu_tanh(g) * u as bf16 into hb[t*ld + j]; with lo_off > 0 also the
// rounding remainder (h - bf16(h)) as bf16 at column lo_off + j.  Columns
// [inter, kmod) of each part are zeroed (they meet zero-filled W0 columns, but
// garbage there could be NaN).
__global__ void mlp_gelu_kernel(const float *__restrict__ g, const float *__restrict__ u, bf16 *hb, int64_t T,
                                int inter, int kmod, int ld, int lo_off)
{
    const int64_t n = T * (int64_t)kmod;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = idx / kmod;
        const int j = (int)(idx - t * kmod);
        float hv = 0.f;
        if (j < inter) {
            const float gv = g[t * inter + j], uv = u[t * inter + j];
            const float c = 0.7978845608028654f;  // sqrt(2/pi)
            hv = 0.5f * gv * (1.0f + tanhf(c * (gv + 0.044715f * gv * gv * gv))) * uv;
        }
        const bf16 hi = __float2bfloat16_rn(hv);
        hb[t * ld + j] = hi;
        if (lo_off > 0) hb[t * ld + lo_off + j] = __float2bfloat16_rn(hv - __bfloat162float(hi));
    }
}

static inline int64_t al256(int64_t v) { return (v + 255) / 256 * 256; }

size_t prefill_mlp_workspace_bytes(int64_t T, int64_t inter, int ydt)
{
    const int64_t kmod = (inter + kBKp - 1) / kBKp * kBKp;
    const int64_t ld = ydt == WL_OUT_F32 ? 2 * kmod : kmod;
    return (size_t)(256 + 2 * al256(T * inter * 4) + al256(T * ld * 2));
}

wl_status launch_prefill_mlp(const bf16 *x, const wl_proj &gate, const wl_proj &up, const wl_proj &down,
                             void *y, int64_t T, int64_t hidden, int64_t inter, int64_t r, void *ws,
                             size_t ws_bytes, int ydt, cudaStream_t st)
{
    if (ws_bytes < prefill_mlp_workspace_bytes(T, inter, ydt))
        return fail(WL_ERR_WORKSPACE, "MLP workspace too small for %lld tokens", (long long)T);
    char *w = static_cast<char *>(ws);
    const bool gu_valign = ((reinterpret_cast<uintptr_t>(gate.V) | reinterpret_cast<uintptr_t>(up.V)) & 15) == 0;
    if (prefill_tiles_applicable(hidden, r, ydt, true, gu_valign) && !few_tiles(T, 2 * inter)) {
        // gate and up in one persistent launch whose epilogue forms h, then down
        const int64_t kmod = (inter + kBKp - 1) / kBKp * kBKp;
        const int64_t ld = ydt == WL_OUT_F32 ? 2 * kmod : kmod;
        bf16 *hb = reinterpret_cast<bf16 *>(w + 256);
        const wl_proj gu[2] = {gate, up};
        void *yh[1] = {hb};
        wl_status s = launch_prefill_tiles(x, gu, 2, true, yh, ld, T, hidden, hidden, hidden, r, ydt, kmod,
                                           ydt == WL_OUT_F32 ? kmod : 0, st);
        if (s != WL_OK) return s;
        void *yd[1] = {y};
        return launch_prefill(hb, &down, 1, yd, T, inter, ld, kmod, r, ydt, st);
    }
    float *g = reinterpret_cast<float *>(w + 256);
    float *u = reinterpret_cast<float *>(w + 256 + al256(T * inter * 4));
    bf16 *hb = reinterpret_cast<bf16 *>(w + 256 + 2 * al256(T * inter * 4));
    const int64_t kmod = (inter + kBKp - 1) / kBKp * kBKp;
    const int64_t ld = ydt == WL_OUT_F32 ? 2 * kmod : kmod;
    // gate and up: one launch, x read once, fp32 results
    const wl_proj gu[2] = {gate, up};
    void *ys[2] = {g, u};
    wl_status s = launch_prefill(x, gu, 2, ys, T, hidden, hidden, hidden, r, WL_OUT_F32, st);
    if (s != WL_OK) return s;
    const DeviceInfo *di = device_info(&s);
    if (!di) return s;
    const int64_t n = T * kmod;
    int blocks = (int)((n + 255) / 256);
    if (blocks > di->sm_count * 16) blocks = di->sm_count * 16;
    mlp_gelu_kernel<<<blocks, 256, 0, st>>>(g, u, hb, T, (int)inter, (int)kmod, (int)ld,
                                           ydt == WL_OUT_F32 ? (int)kmod : 0);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "MLP activation launch");
    // down: K walks [h_hi | h_lo] (or h_hi only for bf16 outputs)
    void *yd[1] = {y};
    return launch_prefill(hb, &down, 1, yd, T, inter, ld, kmod, r, ydt, st);
}

}  // namespace wl
