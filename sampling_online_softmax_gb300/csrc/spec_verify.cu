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

// Stage sizing: about 32 KB of logits per CTA and unit, and a ring of stages
// that lets two CTAs share an SM (the ring alone hides HBM latency).
#ifndef SPEC_STAGE_TARGET
#define SPEC_STAGE_TARGET (40 * 1024)
#endif
#ifndef SPEC_SMEM_PER_CTA
#define SPEC_SMEM_PER_CTA (110 * 1024)
#endif
constexpr size_t kStageTarget = SPEC_STAGE_TARGET;
constexpr size_t kSmemPerCta = SPEC_SMEM_PER_CTA;
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
    int stage;      // bytes per stage
    int nstage;     // stages in the ring
    size_t dyn;     // dynamic shared memory per CTA
};

size_t round128(size_t n) { return (n + 127) / 128 * 128; }

// Stage geometry for cluster size C (nstage left at 0).
Shape stage_for(int C, int V, int eb, int rows_alloc, bool sample, int stage_min) {
    Shape s;
    const int G = 16 / eb;
    s.C = C;
    int L = (V + C - 1) / C;
    L = ((L + G - 1) / G) * G;
    s.L = L;
    s.row_buf = static_cast<int>(round128(static_cast<size_t>(L) * eb + 32));
    s.stage = std::max(rows_alloc * s.row_buf, static_cast<int>(round128(static_cast<size_t>(stage_min))));
    s.nstage = 0;
    s.dyn = sample ? round128((static_cast<size_t>(L) * eb / 16 + 2) * 4) : 0;  // per-group weights
    return s;
}

// Ring depth for a stage geometry within `budget` bytes of shared memory (0 if none fits).
Shape with_stages(Shape s, size_t budget) {
    const size_t extra = s.dyn;
    int n = 0;
    while (n < kMaxStages && extra + static_cast<size_t>(n + 1) * s.stage <= budget) ++n;
    s.nstage = n;
    s.dyn = extra + static_cast<size_t>(n) * s.stage;
    return s;
}

// Cluster size: the smallest power of two whose stage holds about kStageTarget
// bytes (16 if none); the ring takes what two CTAs per SM leave, else what one does.
bool choose_shape(int V, int eb, int rows_alloc, bool sample, int stage_min, const DeviceInfo &di, Shape *out) {
    int C = 16;
    for (int c = 1; c <= 16; c *= 2)
        if (static_cast<size_t>(stage_for(c, V, eb, rows_alloc, sample, stage_min).stage) <= kStageTarget) {
            C = c;
            break;
        }
    Shape s = stage_for(C, V, eb, rows_alloc, sample, stage_min);
    Shape two = with_stages(s, std::min(kSmemPerCta, di.max_dyn));
    if (two.nstage >= 2) {
        *out = two;
        return true;
    }
    Shape one = with_stages(s, di.max_dyn);
    if (one.nstage >= 1) {
        *out = one;
        return true;
    }
    return false;
}

// Clusters of this kernel and shape that can be resident at once (cached).
int active_clusters(int dev, const void *kernel, const cudaLaunchConfig_t &cfg) {
    static std::mutex mu;
    static std::map<std::tuple<int, const void *, unsigned, size_t>, int> cache;
    const auto key = std::make_tuple(dev, kernel, cfg.attrs[0].val.clusterDim.x, cfg.dynamicSmemBytes);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();  // clear the (non-sticky) error
        n = 0;
    }
    cache[key] = n;
    return n;
}

template <int EB, int MODE>
spec_status launch(const Params &p0, int rows_alloc, int stage_min, cudaStream_t stream) {
    DeviceInfo di;
    int dev = 0;
    spec_status st = device_info(&di, &dev);
    if (st != SPEC_OK) return st;
    constexpr bool kSample = (MODE == kLinearSample || MODE == kBonusSample);
    Shape sh;
    if (!choose_shape(p0.V, EB, rows_alloc, kSample, stage_min, di, &sh))
        return fail(SPEC_ERR_UNSUPPORTED, "V=%d does not fit a 16-CTA cluster's shared memory", p0.V);

    auto kernel = spec_verify_kernel<EB, MODE>;
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
    // persistent grid: as many clusters as fit at once (a shape that cannot be
    // placed at all is replaced by the next smaller cluster)
    int nclusters = 0;
    for (;;) {
        attr[0].val.clusterDim.x = static_cast<unsigned>(sh.C);
        cfg.gridDim = dim3(static_cast<unsigned>(sh.C), 1, 1);
        cfg.dynamicSmemBytes = sh.dyn;
        nclusters = active_clusters(dev, reinterpret_cast<const void *>(kernel), cfg);
        if (nclusters > 0) break;
        if (sh.C == 1) return fail(SPEC_ERR_UNSUPPORTED, "no cluster shape fits (smem=%zu)", sh.dyn);
        Shape smaller = with_stages(stage_for(sh.C / 2, p0.V, EB, rows_alloc, kSample, stage_min), di.max_dyn);
        if (smaller.nstage < 1) return fail(SPEC_ERR_UNSUPPORTED, "no cluster shape fits V=%d", p0.V);
        sh = smaller;
    }
    nclusters = std::min(nclusters, p0.n_units);
    cfg.gridDim = dim3(static_cast<unsigned>(nclusters * sh.C), 1, 1);
    Params p = p0;
    p.slice_len = sh.L;
    p.row_buf_bytes = sh.row_buf;
    p.stage_bytes = sh.stage;
    p.nstage = sh.nstage;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p);
    if (e != cudaSuccess)
        return fail(SPEC_ERR_CUDA, "launch (C=%d, stages=%d, smem=%zu): %s", sh.C, sh.nstage, sh.dyn,
                    cudaGetErrorString(e));
    return SPEC_OK;
}

// Workspace layout (16-byte aligned parts): [counter: B u32][first rejection: B i32]
// [accept bits: B*K i32][values: B*U i32].
struct WsLayout {
    size_t counter, first, acc, val, total;
};
WsLayout ws_layout(int B, int K, int units_per_seq) {
    WsLayout w;
    w.counter = 0;
    w.first = align16(static_cast<size_t>(B) * 4);
    w.acc = w.first + align16(static_cast<size_t>(B) * 4);
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
    p.ws_first = reinterpret_cast<int32_t *>(ws + wl.first);
    p.ws_acc = reinterpret_cast<int32_t *>(ws + wl.acc);
    p.ws_val = reinterpret_cast<int32_t *>(ws + wl.val);
    if (static_cast<int64_t>(B) * (K + 1) > INT_MAX / 16) return fail(SPEC_ERR_UNSUPPORTED, "B * (K + 1) too large");
    p.n_units = B * (K + 1);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (sample) return eb == 4 ? launch<4, kLinearSample>(p, 2, 0, s) : launch<2, kLinearSample>(p, 2, 0, s);
    return eb == 4 ? launch<4, kLinearGreedy>(p, 1, 0, s) : launch<2, kLinearGreedy>(p, 1, 0, s);
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
    p.n_units = B;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (sample) return eb == 4 ? launch<4, kBonusSample>(p, 2, 0, s) : launch<2, kBonusSample>(p, 2, 0, s);
    return eb == 4 ? launch<4, kBonusGreedy>(p, 1, 0, s) : launch<2, kBonusGreedy>(p, 1, 0, s);
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
    p.ws_first = reinterpret_cast<int32_t *>(ws + wl.first);
    p.ws_val = reinterpret_cast<int32_t *>(ws + wl.val);
    if (static_cast<int64_t>(B) * N > INT_MAX / 16) return fail(SPEC_ERR_UNSUPPORTED, "B * N too large");
    p.n_units = B * N;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the last unit stages parents, node tokens and argmaxes (3 * N ints) in a stage buffer
    return eb == 4 ? launch<4, kTreeGreedy>(p, 1, 12 * N, s) : launch<2, kTreeGreedy>(p, 1, 12 * N, s);
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
