// noalloc.cu -- the fused GeGLU MLP for callers that cannot allocate.
//
// wl_mlp_geglu_fused needs a device workspace from its caller.  Some callers
// cannot provide one: code running where cudaMalloc is off limits (inside a
// host callback or another library's allocator hook, under a strict memory
// budget that forbids new device allocations after start-up, or a plain C
// host with no allocator of its own).  For them this file keeps the workspace
// in a fixed, file-scope device array and exposes one more entry point that
// uses it.  The array is part of the loaded module: every GPU that loads
// libwl.so holds it until the process exits.
#include "wl_internal.cuh"

namespace wl {

// Largest workspace the built-in scratch can stand in for (4 MiB).  This
// covers the decode MLP of the Gemma-3-1B shapes (hidden 1152, inter 6912)
// and of the large set (hidden 5376, inter 21504, r = 64).
constexpr size_t kNoAllocScratchBytes = (size_t)4 << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch in the current context.  The name
// g_noalloc_scratch in host code is only a host-side stand-in; the address is
// looked up on every call (a few microseconds next to the launches), so a
// device reset or a re-created primary context, which loads the module
// again, never leaves a stale address behind.
static wl_status scratch_address(void **out)
{
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(built-in scratch)");
    *out = p;
    return WL_OK;
}

}  // namespace wl

using namespace wl;

extern "C" wl_status wl_mlp_geglu_fused_noalloc(const void *x, wl_proj gate, wl_proj up,
                                                wl_proj down, void *y, int64_t T, int64_t hidden,
                                                int64_t inter, int64_t r, wl_out_dtype ydt,
                                                void *stream)
{
    const size_t need = wl_mlp_workspace_bytes(T, hidden, inter, r, ydt);
    if (need == 0)
        return fail(WL_ERR_INVALID_ARG, "wl_mlp_geglu_fused_noalloc: invalid sizes T=%lld hidden=%lld "
                    "inter=%lld r=%lld", (long long)T, (long long)hidden, (long long)inter, (long long)r);
    if (need > kNoAllocScratchBytes)
        return fail(WL_ERR_UNSUPPORTED, "wl_mlp_geglu_fused_noalloc: these sizes need %zu bytes of "
                    "workspace; the built-in scratch holds %zu bytes (use wl_mlp_geglu_fused with a "
                    "caller workspace)", need, kNoAllocScratchBytes);
    void *scratch = nullptr;
    wl_status st = scratch_address(&scratch);
    if (st != WL_OK) return st;
    // The scratch keeps whatever the previous call left; the MLP writes every
    // part of it that it later reads, so nothing has to be cleared.
    return wl_mlp_geglu_fused(x, gate, up, down, y, T, hidden, inter, r, scratch,
                              kNoAllocScratchBytes, ydt, stream);
}
