// wl_api.cu -- the C ABI of libwl.so: argument checks, dispatch, errors.
//
// Every entry point validates all of its arguments before anything reaches
// the GPU, then hands the work to one of the kernel launchers.  No entry point
// allocates device memory; there is no CPU path.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "wl_internal.cuh"

namespace wl {

// The library's device status word (one per device context).  Kernels OR
// status bits into it; wl_device_status() reads and clears it.
__device__ unsigned g_status_word;

static thread_local char t_err[512];

void clear_error() { t_err[0] = '\0'; }

wl_status fail(wl_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof t_err, fmt, ap);
    va_end(ap);
    return st;
}

wl_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(WL_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

static constexpr int kMaxDevices = 64;
static DeviceInfo g_info[kMaxDevices];
static bool g_info_ok[kMaxDevices];
static std::mutex g_info_mu;

const DeviceInfo *device_info(wl_status *st)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *st = cuda_fail(e, "cudaGetDevice");
        return nullptr;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        *st = fail(WL_ERR_UNSUPPORTED, "device index %d out of range", dev);
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_info_mu);
    if (g_info_ok[dev]) return &g_info[dev];
    DeviceInfo di = {};
    di.device = dev;
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&di.l2_bytes, cudaDevAttrL2CacheSize, dev)) != cudaSuccess) {
        *st = cuda_fail(e, "cudaDeviceGetAttribute");
        return nullptr;
    }
    if (major != 10 || minor != 3) {
        *st = fail(WL_ERR_UNSUPPORTED, "libwl.so is built for sm_103a; device %d is sm_%d%d", dev,
                   major, minor);
        return nullptr;
    }
    e = cudaGetSymbolAddress(reinterpret_cast<void **>(&di.status), g_status_word);
    if (e != cudaSuccess) {
        *st = cuda_fail(e, "cudaGetSymbolAddress(status word)");
        return nullptr;
    }
    g_info[dev] = di;
    g_info_ok[dev] = true;
    return &g_info[dev];
}

}  // namespace wl

using namespace wl;

// ---------------------------------------------------------------- checks --
static bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static constexpr int64_t kMaxDim = (int64_t)1 << 30;

// Token counts up to this run the HBM-streaming decode kernels; larger ones
// run the tensor-core prefill kernels.  Measured on GB300 (fused Q/K/V, graph
// replay): at 16 tokens the two paths tie on the Gemma-1B shapes (18 vs 19
// us) and the tensor cores win from there on (32 tokens: 31 vs 19 us; 64:
// 73 vs 19 us; 5376 -> 4096/2048/2048 at r = 64: 934 vs 66 us at 64 tokens).
static constexpr int64_t kDecodeMaxTokens = 8;
// The fused MLP's streaming kernels take up to 8 tokens per pass; more tokens
// go to the tensor-core path (gate and up in one launch, then down).
static constexpr int64_t kMlpDecodeMaxTokens = 8;

static wl_status check_dims(int64_t T, int64_t in, int64_t out, int64_t r)
{
    if (T < 1 || T > kMaxDim) return fail(WL_ERR_INVALID_ARG, "T must be in [1, 2^30], got %lld", (long long)T);
    if (in < 8 || in > kMaxDim || in % 8 != 0)
        return fail(WL_ERR_INVALID_ARG, "in must be a positive multiple of 8 (<= 2^30), got %lld", (long long)in);
    if (out < 1 || out > kMaxDim) return fail(WL_ERR_INVALID_ARG, "out must be in [1, 2^30], got %lld", (long long)out);
    if (r < 0 || r > WL_MAX_RANK)
        return fail(WL_ERR_INVALID_ARG, "r must be in [0, %d], got %lld", WL_MAX_RANK, (long long)r);
    if (in * out > ((int64_t)1 << 40)) return fail(WL_ERR_INVALID_ARG, "in*out too large");
    return WL_OK;
}

static wl_status check_theta(const char *name, const void *W0, const float *s, const void *U,
                             const void *V, int64_t r)
{
    if (!W0 || !s) return fail(WL_ERR_INVALID_ARG, "%s: W0 and s must not be NULL", name);
    if (r > 0 && (!U || !V)) return fail(WL_ERR_INVALID_ARG, "%s: U and V must not be NULL when r > 0", name);
    if (!aligned(W0, 16)) return fail(WL_ERR_INVALID_ARG, "%s: W0 must be 16-byte aligned", name);
    if (!aligned(s, 4)) return fail(WL_ERR_INVALID_ARG, "%s: s must be 4-byte aligned", name);
    if (r > 0 && (!aligned(U, 2) || !aligned(V, 2)))
        return fail(WL_ERR_INVALID_ARG, "%s: U and V must be 2-byte aligned", name);
    return WL_OK;
}

static wl_status check_io(const void *x, const void *y, int ydt)
{
    if (!x || !y) return fail(WL_ERR_INVALID_ARG, "x and y must not be NULL");
    if (!aligned(x, 16) || !aligned(y, 16)) return fail(WL_ERR_INVALID_ARG, "x and y must be 16-byte aligned");
    if (ydt != WL_OUT_BF16 && ydt != WL_OUT_F32) return fail(WL_ERR_INVALID_ARG, "unknown output dtype %d", ydt);
    return WL_OK;
}

#define WL_TRY(expr)                    \
    do {                                \
        wl_status _s = (expr);          \
        if (_s != WL_OK) return _s;     \
    } while (0)

static wl_status begin()
{
    t_err[0] = '\0';
    wl_status st = WL_OK;
    if (!device_info(&st)) return st;
    return WL_OK;
}

// ---------------------------------------------------------------- C ABI ---
extern "C" {

wl_status wl_linear(const void *x, const void *W0, const float *s, const void *U, const void *V,
                    void *y, int64_t T, int64_t in, int64_t out, int64_t r, wl_out_dtype ydt,
                    void *stream)
{
    t_err[0] = '\0';
    WL_TRY(check_dims(T, in, out, r));
    WL_TRY(check_io(x, y, ydt));
    WL_TRY(check_theta("wl_linear", W0, s, U, V, r));
    WL_TRY(begin());
    wl_proj p = {W0, s, U, V, out};
    void *ys[1] = {y};
    if (T > kDecodeMaxTokens || !decode_linear_fits(&p, 1, T, in, r, ydt))
        return launch_prefill(static_cast<const bf16 *>(x), &p, 1, ys, T, in, in, in, r, ydt,
                              static_cast<cudaStream_t>(stream));
    return launch_decode_linear(static_cast<const bf16 *>(x), &p, 1, ys, T, in, r, ydt,
                                static_cast<cudaStream_t>(stream));
}

wl_status wl_qkv_fused(const void *x, wl_proj q, wl_proj k, wl_proj v, void *yq, void *yk,
                       void *yv, int64_t T, int64_t in, int64_t r, wl_out_dtype ydt, void *stream)
{
    t_err[0] = '\0';
    const wl_proj ps[3] = {q, k, v};
    void *ys[3] = {yq, yk, yv};
    const char *names[3] = {"q", "k", "v"};
    for (int j = 0; j < 3; ++j) {
        WL_TRY(check_dims(T, in, ps[j].out, r));
        WL_TRY(check_io(x, ys[j], ydt));
        WL_TRY(check_theta(names[j], ps[j].W0, ps[j].s, ps[j].U, ps[j].V, r));
    }
    WL_TRY(begin());
    if (T > kDecodeMaxTokens || !decode_linear_fits(ps, 3, T, in, r, ydt))
        return launch_prefill(static_cast<const bf16 *>(x), ps, 3, ys, T, in, in, in, r, ydt,
                              static_cast<cudaStream_t>(stream));
    return launch_decode_linear(static_cast<const bf16 *>(x), ps, 3, ys, T, in, r, ydt,
                                static_cast<cudaStream_t>(stream));
}

static wl_status check_theta_f32(const char *name, const float *W0, const float *s, const float *U, const float *V,
                                 int64_t r)
{
    if (!W0 || !s) return fail(WL_ERR_INVALID_ARG, "%s: W0 and s must not be NULL", name);
    if (r > 0 && (!U || !V)) return fail(WL_ERR_INVALID_ARG, "%s: U and V must not be NULL when r > 0", name);
    if (!aligned(W0, 16)) return fail(WL_ERR_INVALID_ARG, "%s: W0 must be 16-byte aligned", name);
    if (!aligned(s, 4) || (r > 0 && (!aligned(U, 4) || !aligned(V, 4))))
        return fail(WL_ERR_INVALID_ARG, "%s: s, U and V must be 4-byte aligned", name);
    return WL_OK;
}

wl_status wl_linear_f32(const float *x, const float *W0, const float *s, const float *U, const float *V,
                        void *y, int64_t T, int64_t in, int64_t out, int64_t r, wl_out_dtype ydt, void *stream)
{
    t_err[0] = '\0';
    WL_TRY(check_dims(T, in, out, r));
    WL_TRY(check_io(x, y, ydt));
    WL_TRY(check_theta_f32("wl_linear_f32", W0, s, U, V, r));
    WL_TRY(begin());
    const wl_proj_f32 p = {W0, s, U, V, out};
    void *ys[1] = {y};
    return launch_f32_linear(x, &p, 1, ys, T, in, r, ydt, static_cast<cudaStream_t>(stream));
}

wl_status wl_qkv_fused_f32(const float *x, wl_proj_f32 q, wl_proj_f32 k, wl_proj_f32 v, void *yq, void *yk,
                           void *yv, int64_t T, int64_t in, int64_t r, wl_out_dtype ydt, void *stream)
{
    t_err[0] = '\0';
    const wl_proj_f32 ps[3] = {q, k, v};
    void *ys[3] = {yq, yk, yv};
    const char *names[3] = {"q", "k", "v"};
    for (int j = 0; j < 3; ++j) {
        WL_TRY(check_dims(T, in, ps[j].out, r));
        WL_TRY(check_io(x, ys[j], ydt));
        WL_TRY(check_theta_f32(names[j], ps[j].W0, ps[j].s, ps[j].U, ps[j].V, r));
    }
    WL_TRY(begin());
    return launch_f32_linear(x, ps, 3, ys, T, in, r, ydt, static_cast<cudaStream_t>(stream));
}

size_t wl_mlp_workspace_bytes(int64_t T, int64_t hidden, int64_t inter, int64_t r, wl_out_dtype ydt)
{
    if (T < 1 || hidden < 8 || inter < 8 || hidden % 8 || inter % 8 || r < 0 || r > WL_MAX_RANK ||
        hidden > kMaxDim || inter > kMaxDim || T > kMaxDim)
        return 0;
    // few tokens run the decode kernels unless they have no plan for these
    // shapes; the workspace covers both paths
    const size_t dec = decode_mlp_workspace_bytes(hidden, inter, r);
    const size_t pre = prefill_mlp_workspace_bytes(T, inter, ydt);
    return pre > dec ? pre : dec;
}

wl_status wl_mlp_geglu_fused(const void *x, wl_proj gate, wl_proj up, wl_proj down, void *y,
                             int64_t T, int64_t hidden, int64_t inter, int64_t r, void *workspace,
                             size_t ws_bytes, wl_out_dtype ydt, void *stream)
{
    t_err[0] = '\0';
    WL_TRY(check_dims(T, hidden, inter, r));
    WL_TRY(check_dims(T, inter, hidden, r));
    WL_TRY(check_io(x, y, ydt));
    WL_TRY(check_theta("gate", gate.W0, gate.s, gate.U, gate.V, r));
    WL_TRY(check_theta("up", up.W0, up.s, up.U, up.V, r));
    WL_TRY(check_theta("down", down.W0, down.s, down.U, down.V, r));
    if (gate.out != inter || up.out != inter)
        return fail(WL_ERR_INVALID_ARG, "gate.out and up.out must equal inter (%lld)", (long long)inter);
    if (down.out != hidden)
        return fail(WL_ERR_INVALID_ARG, "down.out must equal hidden (%lld)", (long long)hidden);
    const size_t need = wl_mlp_workspace_bytes(T, hidden, inter, r, ydt);
    if (!workspace || !aligned(workspace, 256))
        return fail(WL_ERR_WORKSPACE, "workspace must be non-NULL and 256-byte aligned");
    if (ws_bytes < need)
        return fail(WL_ERR_WORKSPACE, "workspace too small: %zu bytes, need %zu", ws_bytes, need);
    WL_TRY(begin());
    if (T > kMlpDecodeMaxTokens || !decode_mlp_fits(gate, up, down, T, hidden, inter, r, ydt))
        return launch_prefill_mlp(static_cast<const bf16 *>(x), gate, up, down, y, T, hidden, inter, r,
                                  workspace, ws_bytes, ydt, static_cast<cudaStream_t>(stream));
    return launch_decode_mlp(static_cast<const bf16 *>(x), gate, up, down, y, T, hidden, inter, r,
                             workspace, ws_bytes, ydt, static_cast<cudaStream_t>(stream));
}

wl_status wl_materialize(const void *W0, const float *s, const void *U, const void *V, void *W_eff,
                         int64_t out, int64_t in, int64_t r, wl_out_dtype dt, void *stream)
{
    t_err[0] = '\0';
    WL_TRY(check_dims(1, in, out, r));
    WL_TRY(check_theta("wl_materialize", W0, s, U, V, r));
    if (!W_eff || !aligned(W_eff, 16)) return fail(WL_ERR_INVALID_ARG, "W_eff must be non-NULL and 16-byte aligned");
    if (dt != WL_OUT_BF16 && dt != WL_OUT_F32) return fail(WL_ERR_INVALID_ARG, "unknown dtype %d", dt);
    WL_TRY(begin());
    return launch_materialize(static_cast<const bf16 *>(W0), s, static_cast<const bf16 *>(U),
                              static_cast<const bf16 *>(V), W_eff, out, in, r, dt,
                              static_cast<cudaStream_t>(stream));
}

size_t wl_decompose_workspace_bytes(int64_t out, int64_t in, int64_t r, int64_t p)
{
    if (out < 1 || in < 8 || in % 8 || out > kMaxDim || in > kMaxDim || r < 0 || p < 0 || r + p > kDecompMaxK)
        return 0;
    return decompose_workspace_bytes(out, in, r, p);
}

wl_status wl_decompose_band(const void *const *W, int64_t n, int64_t out, int64_t in, int64_t r, int64_t p,
                            int64_t iters, const float *omega, void *W0, float *s, void *U, void *V,
                            void *workspace, size_t ws_bytes, void *stream)
{
    t_err[0] = '\0';
    if (!W || n < 1 || n > kDecompMaxLayers)
        return fail(WL_ERR_INVALID_ARG, "wl_decompose_band: need 1 <= n <= %d weights", kDecompMaxLayers);
    WL_TRY(check_dims(1, in, out, r));
    if (r > out || r > in) return fail(WL_ERR_INVALID_ARG, "wl_decompose_band: r = %lld exceeds min(out, in)", (long long)r);
    if (p < 0 || r + p > kDecompMaxK)
        return fail(WL_ERR_INVALID_ARG, "wl_decompose_band: need p >= 0 and r + p <= %d", kDecompMaxK);
    if (iters < 0 || iters > 64) return fail(WL_ERR_INVALID_ARG, "wl_decompose_band: need 0 <= iters <= 64");
    for (int64_t l = 0; l < n; ++l)
        if (!W[l] || !aligned(W[l], 16))
            return fail(WL_ERR_INVALID_ARG, "wl_decompose_band: weight %lld is NULL or not 16-byte aligned", (long long)l);
    if (!W0 || !aligned(W0, 16) || !s || !aligned(s, 4))
        return fail(WL_ERR_INVALID_ARG, "wl_decompose_band: W0 (16-byte aligned) and s must not be NULL");
    if (r > 0 && (!U || !V || !omega || !aligned(U, 2) || !aligned(V, 2) || !aligned(omega, 4)))
        return fail(WL_ERR_INVALID_ARG, "wl_decompose_band: U, V and omega must not be NULL when r > 0");
    if (!workspace || !aligned(workspace, 256))
        return fail(WL_ERR_WORKSPACE, "wl_decompose_band: workspace must be non-NULL and 256-byte aligned");
    const size_t need = decompose_workspace_bytes(out, in, r, p);
    if (ws_bytes < need)
        return fail(WL_ERR_WORKSPACE, "wl_decompose_band: workspace too small: %zu bytes, need %zu", ws_bytes, need);
    WL_TRY(begin());
    return launch_decompose(reinterpret_cast<const bf16 *const *>(W), (int)n, (int)out, (int)in, (int)r, (int)p,
                            (int)iters, omega, static_cast<bf16 *>(W0), s, static_cast<bf16 *>(U),
                            static_cast<bf16 *>(V), workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

int64_t wl_band_of_layer(int64_t layer, int64_t L, int64_t G)
{
    if (L < 1 || G < 1 || G > L || layer < 0 || layer >= L) return -1;
    if (L > kMaxDim) return -1;
    return (layer * G) / L;
}

wl_status wl_device_status(void *stream)
{
    t_err[0] = '\0';
    wl_status st = WL_OK;
    const DeviceInfo *di = device_info(&st);
    if (!di) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned word = 0;
    e = cudaMemcpyFromSymbol(&word, g_status_word, sizeof word);
    if (e != cudaSuccess) return cuda_fail(e, "read status word");
    if (word != 0) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero);
        if (e != cudaSuccess) return cuda_fail(e, "clear status word");
        if (word & kStatusTimeout)
            return fail(WL_ERR_TIMEOUT, "a bounded device-side wait gave up (%s%s%s)",
                        (word & kWaitRingFull) ? " ring-full" : "",
                        (word & kWaitRingEmpty) ? " ring-empty" : "",
                        (word & kWaitExchange) ? " cluster-exchange" : "");
    }
    return WL_OK;
}

const char *wl_last_error(void) { return t_err; }

const char *wl_version(void) { return "wl 0.1 (sm_103a)"; }

}  // extern "C"
