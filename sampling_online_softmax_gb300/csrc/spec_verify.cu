// spec_verify.cu -- host side of libspecverify.so: the C ABI declared in
// include/spec_verify.h (argument checks, workspace layout, cluster sizing and
// launches of the kernels in verify_kernels.cuh).
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "spec_verify.h"
#include "verify_kernels.cuh"

namespace spec {
namespace {

thread_local char g_last_error[512] = "";

spec_status fail(spec_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
spec_status fail(spec_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}

inline size_t align16(size_t n) { return (n + 15) & ~size_t(15); }
inline bool aligned(const void *ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// Shared-memory budget per CTA that still lets three CTAs share one SM.
constexpr size_t kTargetDynSmem = 70 * 1024;
constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int sms = 0;
    size_t max_dyn = 0;  // opt-in dynamic shared memory per block
};

DeviceInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];
std::mutex g_attr_mutex;

spec_status device_info(DeviceInfo *out, int *dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(SPEC_ERR_UNSUPPORTED, "device index %d", dev);
    std::call_once(g_dev_once[dev], [dev]() {
        int sms = 0, smem = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        g_dev[dev].sms = sms;
        g_dev[dev].max_dyn = static_cast<size_t>(smem) > sizeof(Ctl) + 1024
                                 ? static_cast<size_t>(smem) - sizeof(Ctl) - 1024
                                 : 0;
    });
    *out = g_dev[dev];
    *dev_out = dev;
    if (out->sms <= 0 || out->max_dyn == 0)
        return fail(SPEC_ERR_CUDA, "could not query device %d attributes", dev);
    return SPEC_OK;
}

struct Shape {
    int C;          // CTAs per cluster
    int L;          // slice length (elements)
    int row_buf;    // bytes per row buffer
    size_t dyn;     // dynamic shared memory per CTA
};

Shape shape_for(int C, int V, int eb, int rows_alloc, bool sample, int stage_ints) {
    Shape s;
    const int G = 16 / eb;
    s.C = C;
    int L = (V + C - 1) / C;
    L = ((L + G - 1) / G) * G;
    s.L = L;
    s.row_buf = ((L * eb + 32) + 127) / 128 * 128;
    size_t dyn = static_cast<size_t>(rows_alloc) * s.row_buf;
    if (sample) {
        const size_t ngmax = static_cast<size_t>(L) * eb / 16 + 2;
        dyn += (ngmax * 4 + 127) / 128 * 128;
    }
    dyn = std::max(dyn, static_cast<size_t>(stage_ints) * 4);
    s.dyn = std::max<size_t>(dyn, 128);
    return s;
}

// Cluster size: the smallest power of two whose slice fits the shared-memory
// target (else the device maximum); then doubled while the grid would not
// give every SM two CTAs.
bool choose_shape(int64_t units, int V, int eb, int rows_alloc, bool sample, int stage_ints,
                  const DeviceInfo &di, Shape *out) {
    int C = 0;
    for (int c = 1; c <= 16; c *= 2)
        if (shape_for(c, V, eb, rows_alloc, sample, stage_ints).dyn <= kTargetDynSmem) {
            C = c;
            break;
        }
    if (C == 0)
        for (int c = 1; c <= 16; c *= 2)
            if (shape_for(c, V, eb, rows_alloc, sample, stage_ints).dyn <= di.max_dyn) {
                C = c;
                break;
            }
    if (C == 0) return false;
    while (C < 16 && units * C < 2LL * di.sms) C *= 2;
    *out = shape_for(C, V, eb, rows_alloc, sample, stage_ints);
    return true;
}

// Whether at least one cluster of this shape can be resident (cached per device, kernel, shape).
bool cluster_fits(int dev, const void *kernel, const cudaLaunchConfig_t &cfg) {
    static std::mutex mu;
    static std::map<std::tuple<int, const void *, unsigned, size_t>, bool> cache;
    const auto key = std::make_tuple(dev, kernel, cfg.attrs[0].val.clusterDim.x, cfg.dynamicSmemBytes);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
    const bool ok = (e == cudaSuccess && n > 0);
    if (e != cudaSuccess) cudaGetLastError();  // clear the (non-sticky) error
    cache[key] = ok;
    return ok;
}

template <int EB, int MODE>
spec_status launch(const Params &p0, int64_t units, int rows_alloc, int stage_ints, cudaStream_t stream) {
    DeviceInfo di;
    int dev = 0;
    spec_status st = device_info(&di, &dev);
    if (st != SPEC_OK) return st;
    Shape sh;
    constexpr bool kSample = (MODE == kLinearSample || MODE == kBonusSample);
    if (!choose_shape(units, p0.V, EB, rows_alloc, kSample, stage_ints, di, &sh))
        return fail(SPEC_ERR_UNSUPPORTED, "V=%d does not fit a 16-CTA cluster's shared memory", p0.V);
    if (units * sh.C > INT_MAX) return fail(SPEC_ERR_UNSUPPORTED, "grid too large (%lld units)", (long long)units);

    auto kernel = spec_unit_kernel<EB, MODE>;
    {
        // per device and kernel, once: allow the largest dynamic shared memory and 16-CTA clusters
        static bool configured[kMaxDevices] = {};
        std::lock_guard<std::mutex> lock(g_attr_mutex);
        if (!configured[dev]) {
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(di.max_dyn));
            if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            configured[dev] = true;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // a cluster shape the GPU cannot place is replaced by the next smaller one
    for (;;) {
        attr[0].val.clusterDim.x = static_cast<unsigned>(sh.C);
        cfg.gridDim = dim3(static_cast<unsigned>(units * sh.C), 1, 1);
        cfg.dynamicSmemBytes = sh.dyn;
        if (cluster_fits(dev, reinterpret_cast<const void *>(kernel), cfg)) break;
        if (sh.C == 1) return fail(SPEC_ERR_UNSUPPORTED, "no cluster shape fits (smem=%zu)", sh.dyn);
        sh = shape_for(sh.C / 2, p0.V, EB, rows_alloc, kSample, stage_ints);
        if (sh.dyn > di.max_dyn) return fail(SPEC_ERR_UNSUPPORTED, "no cluster shape fits V=%d", p0.V);
    }
    Params p = p0;
    p.slice_len = sh.L;
    p.row_buf_bytes = sh.row_buf;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p);
    if (e != cudaSuccess)
        return fail(SPEC_ERR_CUDA, "launch (C=%d, smem=%zu): %s", sh.C, sh.dyn, cudaGetErrorString(e));
    return SPEC_OK;
}

// Workspace layout: [counter: B u32][accept bits: B*K i32][values: B*U i32], 16-byte aligned parts.
struct WsLayout {
    size_t counter, acc, val, total;
};
WsLayout ws_layout(int B, int K, int units_per_seq) {
    WsLayout w;
    w.counter = 0;
    w.acc = align16(static_cast<size_t>(B) * 4);
    w.val = w.acc + align16(static_cast<size_t>(B) * K * 4);
    w.total = w.val + align16(static_cast<size_t>(B) * units_per_seq * 4);
    return w;
}

bool valid_temperature(float T, float *c_out) {
    if (!(T >= 0.0f) || !std::isfinite(T)) return false;
    if (T == 0.0f) {
        *c_out = 0.0f;
        return true;
    }
    const double c = 1.4426950408889634 / static_cast<double>(T);  // log2(e) / T
    if (!std::isfinite(static_cast<float>(c))) return false;
    *c_out = static_cast<float>(c);
    return true;
}

}  // namespace
}  // namespace spec

using namespace spec;

extern "C" size_t spec_workspace_bytes_linear(int B, int K) {
    if (B <= 0 || K < 0) return 0;
    return ws_layout(B, K, K + 1).total;
}

extern "C" size_t spec_workspace_bytes_tree(int B, int N) {
    if (B <= 0 || N < 1) return 0;
    return ws_layout(B, 0, N).total;
}

extern "C" spec_status spec_verify_linear(const void *target_logits, const void *draft_logits,
                                          spec_dtype dtype, int B, int K, int V,
                                          const int32_t *draft_tokens, const float *u_accept,
                                          const float *u_bonus, float temperature,
                                          int32_t *accept_len, int32_t *out_tokens, int32_t *num_emitted,
                                          float *probs_out, uint32_t *dev_status, void *workspace,
                                          size_t workspace_bytes, void *stream) {
    g_last_error[0] = '\0';
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return fail(SPEC_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (B < 0 || K < 0 || V < 1) return fail(SPEC_ERR_INVALID_ARG, "need B >= 0, K >= 0, V >= 1 (B=%d K=%d V=%d)", B, K, V);
    float c = 0.f;
    if (!valid_temperature(temperature, &c)) return fail(SPEC_ERR_INVALID_ARG, "temperature must be finite and >= 0");
    if (B == 0) return SPEC_OK;
    const bool sample = temperature > 0.0f;
    const int eb = dtype == SPEC_F32 ? 4 : 2;
    if (!target_logits || !aligned(target_logits, eb)) return fail(SPEC_ERR_INVALID_ARG, "target_logits null or misaligned");
    if (K > 0 && !draft_tokens) return fail(SPEC_ERR_INVALID_ARG, "draft_tokens is null");
    if (sample && K > 0) {
        if (!draft_logits || !aligned(draft_logits, eb)) return fail(SPEC_ERR_INVALID_ARG, "draft_logits null or misaligned");
        if (!u_accept) return fail(SPEC_ERR_INVALID_ARG, "u_accept is null");
    }
    if (!accept_len || !num_emitted || !dev_status) return fail(SPEC_ERR_INVALID_ARG, "an output pointer is null");
    if (u_bonus && !out_tokens) return fail(SPEC_ERR_INVALID_ARG, "out_tokens is required with u_bonus");
    if (static_cast<int64_t>(K) + 1 > INT_MAX / 16) return fail(SPEC_ERR_UNSUPPORTED, "K too large");
    const WsLayout wl = ws_layout(B, K, K + 1);
    if (!workspace || workspace_bytes < wl.total || !aligned(workspace, 16))
        return fail(SPEC_ERR_WORKSPACE, "workspace needs %zu bytes, 16-byte aligned", wl.total);

    Params p = {};
    p.target = static_cast<const unsigned char *>(target_logits);
    p.draft = static_cast<const unsigned char *>(draft_logits);
    p.B = B;
    p.K = K;
    p.V = V;
    p.t_rows = K + 1;
    p.units_per_seq = K + 1;
    p.c = c;
    p.tokens = draft_tokens;
    p.u_accept = u_accept;
    p.u_bonus = u_bonus;
    p.accept_len = accept_len;
    p.out_tokens = out_tokens;
    p.num_emitted = num_emitted;
    p.probs = sample ? probs_out : nullptr;
    p.status = dev_status;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    p.ws_counter = reinterpret_cast<uint32_t *>(ws + wl.counter);
    p.ws_acc = reinterpret_cast<int32_t *>(ws + wl.acc);
    p.ws_val = reinterpret_cast<int32_t *>(ws + wl.val);
    const int64_t units = static_cast<int64_t>(B) * (K + 1);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (sample)
        return eb == 4 ? launch<4, kLinearSample>(p, units, 2, 0, s) : launch<2, kLinearSample>(p, units, 2, 0, s);
    return eb == 4 ? launch<4, kLinearGreedy>(p, units, 1, 0, s) : launch<2, kLinearGreedy>(p, units, 1, 0, s);
}

extern "C" spec_status spec_sample_bonus(const void *target_logits, const void *draft_logits, spec_dtype dtype,
                                         int B, int K, int V, const int32_t *accept_len, const float *u_bonus,
                                         float temperature, int32_t *bonus_token, uint32_t *dev_status,
                                         void *stream) {
    g_last_error[0] = '\0';
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return fail(SPEC_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (B < 0 || K < 0 || V < 1) return fail(SPEC_ERR_INVALID_ARG, "need B >= 0, K >= 0, V >= 1 (B=%d K=%d V=%d)", B, K, V);
    float c = 0.f;
    if (!valid_temperature(temperature, &c)) return fail(SPEC_ERR_INVALID_ARG, "temperature must be finite and >= 0");
    if (B == 0) return SPEC_OK;
    const bool sample = temperature > 0.0f;
    const int eb = dtype == SPEC_F32 ? 4 : 2;
    if (!target_logits || !aligned(target_logits, eb)) return fail(SPEC_ERR_INVALID_ARG, "target_logits null or misaligned");
    if (sample && K > 0 && (!draft_logits || !aligned(draft_logits, eb)))
        return fail(SPEC_ERR_INVALID_ARG, "draft_logits null or misaligned");
    if (sample && !u_bonus) return fail(SPEC_ERR_INVALID_ARG, "u_bonus is null");
    if (!accept_len || !bonus_token || !dev_status) return fail(SPEC_ERR_INVALID_ARG, "a pointer is null");
    Params p = {};
    p.target = static_cast<const unsigned char *>(target_logits);
    p.draft = static_cast<const unsigned char *>(draft_logits);
    p.B = B;
    p.K = K;
    p.V = V;
    p.t_rows = K + 1;
    p.units_per_seq = 1;
    p.c = c;
    p.u_bonus = u_bonus;
    p.accept_len_in = accept_len;
    p.bonus_token = bonus_token;
    p.status = dev_status;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (sample)
        return eb == 4 ? launch<4, kBonusSample>(p, B, 2, 0, s) : launch<2, kBonusSample>(p, B, 2, 0, s);
    return eb == 4 ? launch<4, kBonusGreedy>(p, B, 1, 0, s) : launch<2, kBonusGreedy>(p, B, 1, 0, s);
}

extern "C" spec_status spec_verify_tree(const void *target_logits, spec_dtype dtype, int B, int N, int V,
                                        const int32_t *parents, const int32_t *node_tokens, int max_depth,
                                        int32_t *path_nodes, int32_t *path_len, int32_t *out_tokens,
                                        uint32_t *dev_status, void *workspace, size_t workspace_bytes,
                                        void *stream) {
    g_last_error[0] = '\0';
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return fail(SPEC_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (B < 0 || N < 1 || V < 1 || max_depth < 0)
        return fail(SPEC_ERR_INVALID_ARG, "need B >= 0, N >= 1, V >= 1, max_depth >= 0");
    if (B == 0) return SPEC_OK;
    const int eb = dtype == SPEC_F32 ? 4 : 2;
    if (!target_logits || !aligned(target_logits, eb)) return fail(SPEC_ERR_INVALID_ARG, "target_logits null or misaligned");
    if (!parents || !node_tokens || !path_nodes || !path_len || !out_tokens || !dev_status)
        return fail(SPEC_ERR_INVALID_ARG, "a pointer is null");
    if (N > INT_MAX / 16) return fail(SPEC_ERR_UNSUPPORTED, "N too large");
    const WsLayout wl = ws_layout(B, 0, N);
    if (!workspace || workspace_bytes < wl.total || !aligned(workspace, 16))
        return fail(SPEC_ERR_WORKSPACE, "workspace needs %zu bytes, 16-byte aligned", wl.total);
    Params p = {};
    p.target = static_cast<const unsigned char *>(target_logits);
    p.B = B;
    p.K = N;
    p.V = V;
    p.t_rows = N;
    p.units_per_seq = N;
    p.tokens = node_tokens;
    p.parents = parents;
    p.max_depth = max_depth;
    p.accept_len = path_len;
    p.out_tokens = out_tokens;
    p.path_nodes = path_nodes;
    p.status = dev_status;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    p.ws_counter = reinterpret_cast<uint32_t *>(ws + wl.counter);
    p.ws_val = reinterpret_cast<int32_t *>(ws + wl.val);
    const int64_t units = static_cast<int64_t>(B) * N;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return eb == 4 ? launch<4, kTreeGreedy>(p, units, 1, 3 * N, s) : launch<2, kTreeGreedy>(p, units, 1, 3 * N, s);
}

extern "C" const char *spec_status_string(spec_status status) {
    switch (status) {
        case SPEC_OK: return "SPEC_OK";
        case SPEC_ERR_INVALID_ARG: return "SPEC_ERR_INVALID_ARG: invalid argument";
        case SPEC_ERR_UNSUPPORTED: return "SPEC_ERR_UNSUPPORTED: valid but not supported by this build";
        case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA: CUDA runtime error";
        case SPEC_ERR_WORKSPACE: return "SPEC_ERR_WORKSPACE: workspace missing, too small or misaligned";
    }
    return "unknown spec_status";
}

extern "C" const char *spec_last_error(void) { return g_last_error; }
