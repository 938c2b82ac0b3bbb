// spec_verify.cu -- host side of libspecverify.so: the C ABI declared in
// include/spec_verify.h (argument checks, workspace layout, tile and ring
// sizing, and the launches of the kernels in verify_kernels.cuh).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
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
inline size_t round128(size_t n) { return (n + 127) / 128 * 128; }
inline bool aligned(const void *ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// Tiling: about kSliceBytes of each row per tile; the ring of stages takes what
// two CTAs per SM leave.
#ifndef SPEC_SLICE_BYTES
#define SPEC_SLICE_BYTES (16 * 1024)
#endif
#ifndef SPEC_SMEM_PER_CTA
#define SPEC_SMEM_PER_CTA (110 * 1024)
#endif
#ifndef SPEC_GRAB
#define SPEC_GRAB 4
#endif
constexpr int kSliceBytes = SPEC_SLICE_BYTES;
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

// Slices per row and slice length: a function of V and the element size only
// (the workspace size depends on it).
struct Slicing {
    int S;  // slices (tiles) per unit
    int L;  // elements per slice, a multiple of 16 / eb
};
Slicing slicing(int V, int eb) {
    const int G = 16 / eb;
    const long long row_bytes = static_cast<long long>(V) * eb;
    int S = static_cast<int>(std::max<long long>(1, (row_bytes + kSliceBytes - 1) / kSliceBytes));
    int L = (V + S - 1) / S;
    L = (L + G - 1) / G * G;
    S = (V + L - 1) / L;  // rounding L up may leave a last slice empty: drop it
    return {S, L};
}

struct Shape {
    Slicing sl;
    int row_buf;    // bytes per row buffer
    int stage;      // bytes per stage
    int nstage;     // stages in the ring
    int cpt;        // residual chunks per tile
    size_t extra;   // bytes after the stages: residual chunk sums or tree scratch
    size_t dyn;     // dynamic shared memory per CTA
};

bool choose_shape(int V, int eb, int rows_alloc, bool sample, int tree_N, const DeviceInfo &di, Shape *out) {
    Shape s;
    s.sl = slicing(V, eb);
    s.row_buf = static_cast<int>(round128(static_cast<size_t>(s.sl.L) * eb + 32));
    s.stage = rows_alloc * s.row_buf;
    const int max_groups = s.sl.L * eb / 16 + 2;
    s.cpt = (max_groups + kChunk - 1) / kChunk;
    s.extra = sample ? round128(static_cast<size_t>(kMaxJobs) * s.sl.S * s.cpt * 8)
                     : round128(static_cast<size_t>(tree_N) * 12);
    for (size_t budget : {std::min(kSmemPerCta, di.max_dyn), di.max_dyn}) {
        int n = 0;
        while (n < kMaxStages && s.extra + static_cast<size_t>(n + 1) * s.stage <= budget) ++n;
        if (n >= 2) {
            s.nstage = n;
            s.dyn = s.extra + static_cast<size_t>(n) * s.stage;
            *out = s;
            return true;
        }
    }
    return false;
}

// Resident blocks per SM for this kernel and shared-memory size (cached).
int blocks_per_sm(int dev, const void *kernel, size_t dyn) {
    static std::mutex mu;
    static std::map<std::tuple<int, const void *, size_t>, int> cache;
    const auto key = std::make_tuple(dev, kernel, dyn);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, dyn) != cudaSuccess) {
        cudaGetLastError();  // clear the (non-sticky) error
        n = 0;
    }
    cache[key] = n;
    return n;
}

template <int EB, int MODE>
spec_status launch(const Params &p0, int rows_alloc, int tree_N, cudaStream_t stream) {
    DeviceInfo di;
    int dev = 0;
    spec_status st = device_info(&di, &dev);
    if (st != SPEC_OK) return st;
    constexpr bool kSample = (MODE == kLinearSample || MODE == kBonusSample);
    Shape sh;
    if (!choose_shape(p0.V, EB, rows_alloc, kSample, tree_N, di, &sh))
        return fail(SPEC_ERR_UNSUPPORTED, "no ring of two stages fits shared memory (V=%d)", p0.V);
    auto kernel = spec_verify_kernel<EB, MODE>;
    {
        // per device and kernel, once: allow the largest dynamic shared memory
        static bool configured[kMaxDevices] = {};
        std::lock_guard<std::mutex> lock(g_attr_mutex);
        if (!configured[dev]) {
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(di.max_dyn));
            if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
            configured[dev] = true;
        }
    }
    const int per_sm = blocks_per_sm(dev, reinterpret_cast<const void *>(kernel), sh.dyn);
    if (per_sm <= 0) return fail(SPEC_ERR_UNSUPPORTED, "kernel does not fit an SM (smem=%zu)", sh.dyn);
    const long long tiles = static_cast<long long>(p0.n_units) * sh.sl.S;
    const long long grid = std::min<long long>(tiles, static_cast<long long>(per_sm) * di.sms);
    Params p = p0;
    p.S = sh.sl.S;
    p.slice_len = sh.sl.L;
    p.row_buf_bytes = sh.row_buf;
    p.stage_bytes = sh.stage;
    p.nstage = sh.nstage;
    p.cpt = sh.cpt;
    p.grab = SPEC_GRAB;
    spec_verify_kernel<EB, MODE><<<static_cast<unsigned>(grid), kThreads, sh.dyn, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(SPEC_ERR_CUDA, "launch (grid=%lld, stages=%d, smem=%zu): %s", grid, sh.nstage, sh.dyn,
                    cudaGetErrorString(e));
    return SPEC_OK;
}

// Workspace layout (16-byte aligned parts):
//   [tile counter, CTAs finished: 2 u32][tiles done per unit: n_units u32]
//   [units done per sequence: B u32][earliest rejection: B i32]
//   [accept bits: B*K i32][candidate / argmax: B*U i32][partials: n_units*2*S uint2]
//   [t(x), d(x): n_units float2]
struct WsLayout {
    size_t ctrl, unit_cnt, seq_cnt, first, acc, val, part, tx, total;
};
WsLayout ws_layout(int B, int K, int units_per_seq, int S) {
    const size_t n_units = static_cast<size_t>(B) * units_per_seq;
    WsLayout w;
    w.ctrl = 0;
    w.unit_cnt = 16;
    w.seq_cnt = w.unit_cnt + align16(n_units * 4);
    w.first = w.seq_cnt + align16(static_cast<size_t>(B) * 4);
    w.acc = w.first + align16(static_cast<size_t>(B) * 4);
    w.val = w.acc + align16(static_cast<size_t>(B) * K * 4);
    w.part = w.val + align16(n_units * 4);
    w.tx = w.part + align16(n_units * 2 * static_cast<size_t>(S) * 8);
    w.total = w.tx + align16(n_units * 8);
    return w;
}

void bind_workspace(Params &p, unsigned char *ws, const WsLayout &wl) {
    p.ws_ctrl = reinterpret_cast<uint32_t *>(ws + wl.ctrl);
    p.ws_unit_cnt = reinterpret_cast<uint32_t *>(ws + wl.unit_cnt);
    p.ws_seq_cnt = reinterpret_cast<uint32_t *>(ws + wl.seq_cnt);
    p.ws_first = reinterpret_cast<int32_t *>(ws + wl.first);
    p.ws_acc = reinterpret_cast<int32_t *>(ws + wl.acc);
    p.ws_val = reinterpret_cast<int32_t *>(ws + wl.val);
    p.ws_part = reinterpret_cast<uint2 *>(ws + wl.part);
    p.ws_tx = reinterpret_cast<float2 *>(ws + wl.tx);
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

int elt_bytes(spec_dtype dtype) { return dtype == SPEC_F32 ? 4 : 2; }
bool valid_dtype(spec_dtype dtype) { return dtype == SPEC_F32 || dtype == SPEC_BF16; }

}  // namespace
}  // namespace spec

using namespace spec;

extern "C" size_t spec_workspace_bytes_linear(int B, int K, int V, spec_dtype dtype) {
    if (B <= 0 || K < 0 || V < 1 || !valid_dtype(dtype)) return 0;
    return ws_layout(B, K, K + 1, slicing(V, elt_bytes(dtype)).S).total;
}

extern "C" size_t spec_workspace_bytes_bonus(int B, int V, spec_dtype dtype) {
    if (B <= 0 || V < 1 || !valid_dtype(dtype)) return 0;
    return ws_layout(B, 0, 1, slicing(V, elt_bytes(dtype)).S).total;
}

extern "C" size_t spec_workspace_bytes_tree(int B, int N, int V, spec_dtype dtype) {
    if (B <= 0 || N < 1 || V < 1 || !valid_dtype(dtype)) return 0;
    return ws_layout(B, 0, N, slicing(V, elt_bytes(dtype)).S).total;
}

extern "C" spec_status spec_verify_linear(const void *target_logits, const void *draft_logits,
                                          spec_dtype dtype, int B, int K, int V,
                                          const int32_t *draft_tokens, const float *u_accept,
                                          const float *u_bonus, float temperature,
                                          int32_t *accept_len, int32_t *out_tokens, int32_t *num_emitted,
                                          float *probs_out, uint32_t *dev_status, void *workspace,
                                          size_t workspace_bytes, void *stream) {
    g_last_error[0] = '\0';
    if (!valid_dtype(dtype)) return fail(SPEC_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (B < 0 || K < 0 || V < 1) return fail(SPEC_ERR_INVALID_ARG, "need B >= 0, K >= 0, V >= 1 (B=%d K=%d V=%d)", B, K, V);
    float c = 0.f;
    if (!valid_temperature(temperature, &c)) return fail(SPEC_ERR_INVALID_ARG, "temperature must be finite and >= 0");
    if (B == 0) return SPEC_OK;
    const bool sample = temperature > 0.0f;
    const int eb = elt_bytes(dtype);
    if (!target_logits || !aligned(target_logits, eb)) return fail(SPEC_ERR_INVALID_ARG, "target_logits null or misaligned");
    if (K > 0 && !draft_tokens) return fail(SPEC_ERR_INVALID_ARG, "draft_tokens is null");
    if (sample && K > 0) {
        if (!draft_logits || !aligned(draft_logits, eb)) return fail(SPEC_ERR_INVALID_ARG, "draft_logits null or misaligned");
        if (!u_accept) return fail(SPEC_ERR_INVALID_ARG, "u_accept is null");
    }
    if (!accept_len || !num_emitted || !dev_status) return fail(SPEC_ERR_INVALID_ARG, "an output pointer is null");
    if (u_bonus && !out_tokens) return fail(SPEC_ERR_INVALID_ARG, "out_tokens is required with u_bonus");
    if (static_cast<long long>(B) * (K + 1) > INT_MAX / 64) return fail(SPEC_ERR_UNSUPPORTED, "B * (K + 1) too large");
    const WsLayout wl = ws_layout(B, K, K + 1, slicing(V, eb).S);
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
    p.n_units = B * (K + 1);
    p.c = c;
    p.tokens = draft_tokens;
    p.u_accept = u_accept;
    p.u_bonus = u_bonus;
    p.accept_len = accept_len;
    p.out_tokens = out_tokens;
    p.num_emitted = num_emitted;
    p.probs = sample ? probs_out : nullptr;
    p.status = dev_status;
    bind_workspace(p, static_cast<unsigned char *>(workspace), wl);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (sample) return eb == 4 ? launch<4, kLinearSample>(p, 2, 0, s) : launch<2, kLinearSample>(p, 2, 0, s);
    return eb == 4 ? launch<4, kLinearGreedy>(p, 1, 0, s) : launch<2, kLinearGreedy>(p, 1, 0, s);
}

extern "C" spec_status spec_sample_bonus(const void *target_logits, const void *draft_logits, spec_dtype dtype,
                                         int B, int K, int V, const int32_t *accept_len, const float *u_bonus,
                                         float temperature, int32_t *bonus_token, uint32_t *dev_status,
                                         void *workspace, size_t workspace_bytes, void *stream) {
    g_last_error[0] = '\0';
    if (!valid_dtype(dtype)) return fail(SPEC_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (B < 0 || K < 0 || V < 1) return fail(SPEC_ERR_INVALID_ARG, "need B >= 0, K >= 0, V >= 1 (B=%d K=%d V=%d)", B, K, V);
    float c = 0.f;
    if (!valid_temperature(temperature, &c)) return fail(SPEC_ERR_INVALID_ARG, "temperature must be finite and >= 0");
    if (B == 0) return SPEC_OK;
    const bool sample = temperature > 0.0f;
    const int eb = elt_bytes(dtype);
    if (!target_logits || !aligned(target_logits, eb)) return fail(SPEC_ERR_INVALID_ARG, "target_logits null or misaligned");
    if (sample && K > 0 && (!draft_logits || !aligned(draft_logits, eb)))
        return fail(SPEC_ERR_INVALID_ARG, "draft_logits null or misaligned");
    if (sample && !u_bonus) return fail(SPEC_ERR_INVALID_ARG, "u_bonus is null");
    if (!accept_len || !bonus_token || !dev_status) return fail(SPEC_ERR_INVALID_ARG, "a pointer is null");
    if (B > INT_MAX / 64) return fail(SPEC_ERR_UNSUPPORTED, "B too large");
    const WsLayout wl = ws_layout(B, 0, 1, slicing(V, eb).S);
    if (!workspace || workspace_bytes < wl.total || !aligned(workspace, 16))
        return fail(SPEC_ERR_WORKSPACE, "workspace needs %zu bytes, 16-byte aligned", wl.total);
    Params p = {};
    p.target = static_cast<const unsigned char *>(target_logits);
    p.draft = static_cast<const unsigned char *>(draft_logits);
    p.B = B;
    p.K = K;
    p.V = V;
    p.t_rows = K + 1;
    p.units_per_seq = 1;
    p.n_units = B;
    p.c = c;
    p.u_bonus = u_bonus;
    p.accept_len_in = accept_len;
    p.bonus_token = bonus_token;
    p.status = dev_status;
    bind_workspace(p, static_cast<unsigned char *>(workspace), wl);
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
    if (!valid_dtype(dtype)) return fail(SPEC_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (B < 0 || N < 1 || V < 1 || max_depth < 0)
        return fail(SPEC_ERR_INVALID_ARG, "need B >= 0, N >= 1, V >= 1, max_depth >= 0");
    if (B == 0) return SPEC_OK;
    const int eb = elt_bytes(dtype);
    if (!target_logits || !aligned(target_logits, eb)) return fail(SPEC_ERR_INVALID_ARG, "target_logits null or misaligned");
    if (!parents || !node_tokens || !path_nodes || !path_len || !out_tokens || !dev_status)
        return fail(SPEC_ERR_INVALID_ARG, "a pointer is null");
    if (static_cast<long long>(B) * N > INT_MAX / 64) return fail(SPEC_ERR_UNSUPPORTED, "B * N too large");
    const WsLayout wl = ws_layout(B, 0, N, slicing(V, eb).S);
    if (!workspace || workspace_bytes < wl.total || !aligned(workspace, 16))
        return fail(SPEC_ERR_WORKSPACE, "workspace needs %zu bytes, 16-byte aligned", wl.total);
    Params p = {};
    p.target = static_cast<const unsigned char *>(target_logits);
    p.B = B;
    p.K = N;
    p.V = V;
    p.t_rows = N;
    p.units_per_seq = N;
    p.n_units = B * N;
    p.tokens = node_tokens;
    p.parents = parents;
    p.max_depth = max_depth;
    p.accept_len = path_len;
    p.out_tokens = out_tokens;
    p.path_nodes = path_nodes;
    p.status = dev_status;
    bind_workspace(p, static_cast<unsigned char *>(workspace), wl);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the last unit of a sequence stages parents, node tokens and argmaxes (3 * N ints)
    return eb == 4 ? launch<4, kTreeGreedy>(p, 1, N, s) : launch<2, kTreeGreedy>(p, 1, N, s);
}

// ---- spec_verify_linear_static: spec_verify_linear on a workspace compiled
// into the library, one array per device, so the call allocates nothing.
namespace spec {
namespace {

static __device__ __align__(256) unsigned char g_static_ws[SPEC_STATIC_WORKSPACE_BYTES];

std::atomic<void *> g_static_addr[kMaxDevices];
std::mutex g_static_mutex;

// Device address of the current device's array; looked up once per device,
// with that device current.
spec_status static_workspace(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(SPEC_ERR_UNSUPPORTED, "device index %d", dev);
    void *a = g_static_addr[dev].load(std::memory_order_acquire);
    if (!a) {
        std::lock_guard<std::mutex> lock(g_static_mutex);
        a = g_static_addr[dev].load(std::memory_order_relaxed);
        if (!a) {
            e = cudaGetSymbolAddress(&a, g_static_ws);
            if (e != cudaSuccess || !a)
                return fail(SPEC_ERR_CUDA, "cudaGetSymbolAddress of the static workspace on device %d: %s", dev,
                            cudaGetErrorString(e));
            g_static_addr[dev].store(a, std::memory_order_release);
        }
    }
    *out = a;
    return SPEC_OK;
}

}  // namespace
}  // namespace spec

extern "C" spec_status spec_verify_linear_static(const void *target_logits, const void *draft_logits,
                                                 spec_dtype dtype, int B, int K, int V,
                                                 const int32_t *draft_tokens, const float *u_accept,
                                                 const float *u_bonus, float temperature, int32_t *accept_len,
                                                 int32_t *out_tokens, int32_t *num_emitted, float *probs_out,
                                                 uint32_t *dev_status, void *stream) {
    // Argument checks first: spec_verify_linear without a workspace enqueues
    // nothing and reports either an argument error, SPEC_OK for an empty batch,
    // or the missing workspace.
    spec_status st = spec_verify_linear(target_logits, draft_logits, dtype, B, K, V, draft_tokens, u_accept, u_bonus,
                                        temperature, accept_len, out_tokens, num_emitted, probs_out, dev_status,
                                        nullptr, 0, stream);
    if (st != SPEC_ERR_WORKSPACE) return st;
    g_last_error[0] = '\0';
    const size_t need = spec_workspace_bytes_linear(B, K, V, dtype);
    if (need == 0 || need > static_cast<size_t>(SPEC_STATIC_WORKSPACE_BYTES))
        return fail(SPEC_ERR_WORKSPACE,
                    "B=%d K=%d V=%d needs %zu workspace bytes; the static workspace holds %zu "
                    "(use spec_verify_linear with a workspace of your own)",
                    B, K, V, need, static_cast<size_t>(SPEC_STATIC_WORKSPACE_BYTES));
    void *ws = nullptr;
    st = static_workspace(&ws);
    if (st != SPEC_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(ws, 0, need, s);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaMemsetAsync of the static workspace: %s", cudaGetErrorString(e));
    return spec_verify_linear(target_logits, draft_logits, dtype, B, K, V, draft_tokens, u_accept, u_bonus,
                              temperature, accept_len, out_tokens, num_emitted, probs_out, dev_status, ws,
                              static_cast<size_t>(SPEC_STATIC_WORKSPACE_BYTES), stream);
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
