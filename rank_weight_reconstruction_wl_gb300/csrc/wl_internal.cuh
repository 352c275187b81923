// wl_internal.cuh -- device helpers and host launch declarations shared by
// the translation units of libwl.so.  Nothing here is part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "wl.h"

namespace wl {

typedef __nv_bfloat16 bf16;

constexpr int kThreads = 256;  // CTA size of the decode and materialize kernels
constexpr int kWarps = kThreads / 32;

// ---------------------------------------------------------------- device --
// bf16 pair packed in a 32-bit word -> two fp32 values (exact).  The element
// at the lower address sits in the low half of the word.
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float bf2f(bf16 v) { return __bfloat162float(v); }

// 16-byte streaming load: read-only path, no L1 allocation (the data is used
// once; L2 still sees it).
__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// Device status bits (OR-ed into the library's status word): kStatusTimeout
// plus one bit naming the kind of wait that gave up.
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kWaitRingFull = 2u;    // consumer waiting for a loaded ring stage
constexpr unsigned kWaitRingEmpty = 4u;   // producer waiting for a free ring stage
constexpr unsigned kWaitExchange = 8u;    // waiting for cluster peers' (or other CTAs') partial sums
constexpr unsigned kWaitDrain = 16u;      // a CTA that gave up could not confirm its copies in flight had landed

// Upper bound of every spin-wait in this library, in SM clock cycles: 4e9
// cycles is 2 s at 2 GHz (longer at lower clocks).  A wait that runs longer
// sets kStatusTimeout and returns instead of waiting further.  Waits read the
// SM's cycle counter, which costs a few cycles; the global nanosecond timer
// costs far more per read and slowed every polling loop down.
constexpr long long kWaitLimitCycles = 4000000000ll;

__device__ __forceinline__ long long wait_clock() { return clock64(); }

__device__ __forceinline__ void store_out(void *y, int ydt, int64_t idx, float v)
{
    if (ydt == WL_OUT_F32)
        static_cast<float *>(y)[idx] = v;
    else
        static_cast<bf16 *>(y)[idx] = __float2bfloat16_rn(v);
}

// ------------------------------------------------------------------ host --
struct DeviceInfo {
    int device;
    int sm_count;
    int max_smem_optin;
    int l2_bytes;
    unsigned *status;  // device address of this library's status word
};

// Per-device facts of the current device, queried once per device.
const DeviceInfo *device_info(wl_status *st);

// 2D tensor map of a row-major bf16 matrix [outer, inner] with row stride
// ld_elems, box [box_outer, box_inner], 128-byte swizzle (cached).
wl_status tmap_2d_bf16(const void *base, int64_t inner, int64_t outer, int64_t ld_elems,
                       int box_inner, int box_outer, CUtensorMap *out);
// The same with a swizzle span of 32, 64 or 128 bytes (box_inner * 2 bytes
// at most the span).
wl_status tmap_2d_bf16_swz(const void *base, int64_t inner, int64_t outer, int64_t ld_elems,
                           int box_inner, int box_outer, int swizzle_bytes, CUtensorMap *out);

// 3D view of a row-major bf16 matrix [rows, K], K % 64 == 0, whose box is
// box_rows rows x nblk consecutive 64-column blocks (see tmap.cu).
wl_status tmap_kblocks_bf16(const void *base, int64_t K, int64_t rows, int box_rows, int nblk, CUtensorMap *out);

// Record a message for wl_last_error() and return the status.
wl_status fail(wl_status st, const char *fmt, ...);
void clear_error();  // empties this thread's message (after a probe that may fail)
wl_status cuda_fail(cudaError_t e, const char *what);

// Kernel launchers (arguments already validated by the C-ABI layer).
wl_status launch_decode_linear(const bf16 *x, const wl_proj *proj, int nproj,
                               void *const *y, int64_t T, int64_t in, int64_t r,
                               int ydt, cudaStream_t st);
// Whether the decode kernels have a launch plan for these shapes (shared
// memory); where not, calls of few tokens take the tensor-core path.
bool decode_linear_fits(const wl_proj *proj, int nproj, int64_t T, int64_t in, int64_t r, int ydt);
bool decode_mlp_fits(const wl_proj &gate, const wl_proj &up, const wl_proj &down, int64_t T, int64_t hidden,
                     int64_t inter, int64_t r, int ydt);
wl_status launch_decode_mlp(const bf16 *x, const wl_proj &gate, const wl_proj &up,
                            const wl_proj &down, void *y, int64_t T, int64_t hidden,
                            int64_t inter, int64_t r, void *ws, size_t ws_bytes,
                            int ydt, cudaStream_t st);
size_t decode_mlp_workspace_bytes(int64_t hidden, int64_t inter, int64_t r);
// Tensor-core path for large T.  x is [T, Ktot]; K position k meets W0
// column and V row k % kmod (zero where that is >= in), so x may hold several
// parts of each row side by side (bf16 hi and lo parts: Ktot = 2*kmod).
wl_status launch_prefill(const bf16 *x, const wl_proj *proj, int nproj, void *const *y, int64_t T,
                         int64_t in, int64_t Ktot, int64_t kmod, int64_t r, int ydt, cudaStream_t st);
size_t prefill_mlp_workspace_bytes(int64_t T, int64_t inter, int ydt);
// Persistent tensor-core kernel (double-buffered TMEM accumulators); the
// split-K kernel above takes what it does not (long K chains with fp32
// outputs, larger ranks).  pair: proj[0] = gate, proj[1] = up, and y[0] is h
// (row stride ldy) = gelu_tanh(gate) * up, hw columns per part, the bf16
// rounding remainder at column hlo (0: none).
bool prefill_tiles_applicable(int64_t Ktot, int64_t r, int ydt, bool pair, bool v_aligned);
wl_status launch_prefill_tiles(const bf16 *x, const wl_proj *proj, int nproj, bool pair, void *const *y,
                               int64_t ldy, int64_t T, int64_t in, int64_t Ktot, int64_t kmod, int64_t r,
                               int ydt, int64_t hw, int64_t hlo, cudaStream_t st);
wl_status launch_prefill_mlp(const bf16 *x, const wl_proj &gate, const wl_proj &up, const wl_proj &down,
                             void *y, int64_t T, int64_t hidden, int64_t inter, int64_t r, void *ws,
                             size_t ws_bytes, int ydt, cudaStream_t st);
// Layer stacks for 5..32 tokens (stack_wide.cu); the caller (wl_stack_create)
// has validated the layers and sizes.
struct WidePlan;
constexpr int kStackWideMaxT = 32;
wl_status wide_stack_create(WidePlan **out, const wl_layer *layers, const wl_layer_out *outs, int64_t L, int64_t T,
                            int64_t hidden, int64_t r, const DeviceInfo *di);
wl_status wide_stack_decode(WidePlan *pl, const void *x, cudaStream_t stream);
void wide_stack_destroy(WidePlan *pl);
int wide_stack_device(const WidePlan *pl);

// fp32-encoded bundles and inputs (f32_linear.cu)
wl_status launch_f32_linear(const float *x, const wl_proj_f32 *proj, int nproj, void *const *y, int64_t T,
                            int64_t in, int64_t r, int ydt, cudaStream_t st);

// Dense weights -> theta bundles, one band (decompose.cu)
constexpr int kDecompMaxLayers = 64;
constexpr int kDecompMaxK = 160;
size_t decompose_workspace_bytes(int64_t out, int64_t in, int64_t r, int64_t p);
wl_status launch_decompose(const bf16 *const *W, int n, int out, int in, int r, int p, int iters, const float *omega,
                           bf16 *W0, float *s, bf16 *U, bf16 *V, void *ws, size_t ws_bytes, cudaStream_t st);

wl_status launch_materialize(const bf16 *W0, const float *s, const bf16 *U,
                             const bf16 *V, void *W_eff, int64_t out, int64_t in,
                             int64_t r, int dt, cudaStream_t st);

}  // namespace wl
