// tmap.cu -- TMA tensor maps for the kernels' 2D tile loads.
//
// A tensor map describes a row-major bf16 matrix [outer, inner] in global
// memory and the box (tile) one cp.async.bulk.tensor instruction copies into
// shared memory, with 128-byte swizzling so that tiles can be read from shared
// memory without bank conflicts.  Encoding one costs host time, so maps are
// cached: a map depends only on (address, sizes, box), so a cache hit is always
// a valid map, whatever the memory holds.
#include <cuda.h>

#include <mutex>
#include <unordered_map>

#include "wl_internal.cuh"

namespace wl {

typedef CUresult (*encode_tiled_fn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                    const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                    const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static encode_tiled_fn g_encode = nullptr;
static std::mutex g_tmap_mu;

struct TmapKey {
    uintptr_t base;
    int64_t inner, outer, ld;
    int box_inner, box_outer, swz;
    int nblk;  // 0: 2D map; > 0: 3D view of nblk consecutive 64-column blocks per box
    bool operator==(const TmapKey &o) const
    {
        return base == o.base && inner == o.inner && outer == o.outer && ld == o.ld &&
               box_inner == o.box_inner && box_outer == o.box_outer && swz == o.swz && nblk == o.nblk;
    }
};
struct TmapKeyHash {
    size_t operator()(const TmapKey &k) const
    {
        uint64_t h = k.base * 0x9E3779B97F4A7C15ull;
        h ^= (uint64_t)k.inner + 0x632BE59BD9B4E019ull + (h << 6) + (h >> 2);
        h ^= (uint64_t)k.outer + 0x85EBCA77C2B2AE63ull + (h << 6) + (h >> 2);
        h ^= (uint64_t)k.ld * 31 + (uint64_t)(k.box_inner * 1024 + k.box_outer) * 8 + (uint64_t)k.swz +
             (uint64_t)k.nblk * 0x100000001ull + (h << 6) + (h >> 2);
        return (size_t)h;
    }
};
static std::unordered_map<TmapKey, CUtensorMap, TmapKeyHash> g_tmaps;

static wl_status load_encoder()
{
    if (g_encode) return WL_OK;
    cudaDriverEntryPointQueryResult q;
    void *fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(WL_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    g_encode = reinterpret_cast<encode_tiled_fn>(fn);
    return WL_OK;
}

wl_status tmap_2d_bf16(const void *base, int64_t inner, int64_t outer, int64_t ld_elems,
                       int box_inner, int box_outer, CUtensorMap *out)
{
    return tmap_2d_bf16_swz(base, inner, outer, ld_elems, box_inner, box_outer, 128, out);
}

wl_status tmap_2d_bf16_swz(const void *base, int64_t inner, int64_t outer, int64_t ld_elems,
                           int box_inner, int box_outer, int swizzle_bytes, CUtensorMap *out)
{
    CUtensorMapSwizzle sw;
    switch (swizzle_bytes) {
    case 32: sw = CU_TENSOR_MAP_SWIZZLE_32B; break;
    case 64: sw = CU_TENSOR_MAP_SWIZZLE_64B; break;
    case 128: sw = CU_TENSOR_MAP_SWIZZLE_128B; break;
    default: return fail(WL_ERR_UNSUPPORTED, "tensor map: swizzle of %d bytes", swizzle_bytes);
    }
    std::lock_guard<std::mutex> lk(g_tmap_mu);
    const wl_status es = load_encoder();
    if (es != WL_OK) return es;
    const TmapKey key{reinterpret_cast<uintptr_t>(base), inner, outer, ld_elems, box_inner, box_outer, swizzle_bytes, 0};
    auto it = g_tmaps.find(key);
    if (it != g_tmaps.end()) {
        *out = it->second;
        return WL_OK;
    }
    if (g_tmaps.size() > 4096) g_tmaps.clear();
    CUtensorMap m;
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    const cuuint64_t strides[1] = {(cuuint64_t)ld_elems * 2};
    const cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(WL_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a [%lld, %lld] matrix", (int)r,
                    (long long)outer, (long long)inner);
    g_tmaps.emplace(key, m);
    *out = m;
    return WL_OK;
}

// A row-major bf16 matrix [rows, K] (K % 64 == 0) seen as 3D: 64 columns of
// a block, the rows, the K/64 blocks.  One box of box_rows rows and nblk
// consecutive blocks lands in shared memory as nblk standard 64-column boxes
// (128-byte swizzle) back to back, so one copy moves nblk * box_rows * 128
// bytes.  A copy costs the TMA unit a fixed time of a few hundred ns, so that
// 8 KB boxes hold a stream to about 60 % of HBM and 16 KB or larger ones do
// not (measured on GB300).  Blocks past the matrix are filled with zeros.
wl_status tmap_kblocks_bf16(const void *base, int64_t K, int64_t rows, int box_rows, int nblk, CUtensorMap *out)
{
    if (K % 64 != 0 || nblk < 1 || nblk > 8 || box_rows < 1 || box_rows > 256)
        return fail(WL_ERR_UNSUPPORTED, "k-block tensor map: K = %lld, %d blocks of %d rows", (long long)K, nblk,
                    box_rows);
    std::lock_guard<std::mutex> lk(g_tmap_mu);
    const wl_status es = load_encoder();
    if (es != WL_OK) return es;
    const TmapKey key{reinterpret_cast<uintptr_t>(base), K, rows, K, 64, box_rows, 128, nblk};
    auto it = g_tmaps.find(key);
    if (it != g_tmaps.end()) {
        *out = it->second;
        return WL_OK;
    }
    if (g_tmaps.size() > 4096) g_tmaps.clear();
    CUtensorMap m;
    const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(K / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)K * 2, 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)nblk};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(WL_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a k-block view of a [%lld, %lld] matrix", (int)r,
                    (long long)rows, (long long)K);
    g_tmaps.emplace(key, m);
    *out = m;
    return WL_OK;
}

}  // namespace wl
