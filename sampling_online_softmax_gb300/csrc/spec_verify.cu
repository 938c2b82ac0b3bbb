// spec_verify.cu -- host side of libspecverify.so: the C ABI declared in
// include/spec_verify.h (argument checks, workspace layout, device attributes)
// and the tree-mask launch.  The verify kernel's launches go through
// launch<EB, MODE> (launch.cuh), instantiated one mode per kern_*.cu unit.
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

#include "host.h"
#include "spec_verify.h"
#include "mtp_plug.cuh"
#include "tree_mask.cuh"

namespace spec {

thread_local char g_last_error[512] = "";

spec_status fail(spec_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}

namespace {
DeviceInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];
}  // namespace

spec_status device_info(DeviceInfo *out, int *dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(SPEC_ERR_UNSUPPORTED, "device index %d", dev);
    std::call_once(g_dev_once[dev], [dev]() {
        int sms = 0, smem = 0, l2 = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
        g_dev[dev].sms = sms;
        g_dev[dev].l2 = l2 > 0 ? static_cast<size_t>(l2) : 0;
        g_dev[dev].max_dyn = static_cast<size_t>(smem);  // less each kernel's static shared memory
    });
    *out = g_dev[dev];
    *dev_out = dev;
    if (out->sms <= 0 || out->max_dyn == 0)
        return fail(SPEC_ERR_CUDA, "could not query device %d attributes", dev);
    return SPEC_OK;
}

int stats_tiles_per_row(int V, int eb) {
    return static_cast<int>((static_cast<long long>(V) * eb + 30 + kTileBytes - 1) / kTileBytes);
}
int segments_per_row(int V, int eb) { return (stats_tiles_per_row(V, eb) + kSegTiles - 1) / kSegTiles; }

Slicing resid_slicing(int V, int eb) {
    const int G = 16 / eb;
    const long long row_bytes = static_cast<long long>(V) * eb;
    int S = static_cast<int>(std::max<long long>(1, (row_bytes + kResidSliceBytes - 1) / kResidSliceBytes));
    int L = 0;
    for (;; ++S) {  // the fewest slices whose length, rounded up to whole groups, still fits
        L = (V + S - 1) / S;
        L = (L + G - 1) / G * G;
        if (static_cast<long long>(L) * eb <= kResidSliceBytes) break;
    }
    S = (V + L - 1) / L;
    return {S, L};
}

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

spec_status allow_max_dyn_smem(int dev, const void *kernel, DeviceInfo *di) {
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, size_t> done;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_pair(dev, kernel);
    auto it = done.find(key);
    if (it == done.end()) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
        if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaFuncGetAttributes: %s", cudaGetErrorString(e));
        if (fa.sharedSizeBytes >= di->max_dyn) return fail(SPEC_ERR_UNSUPPORTED, "static shared memory too large");
        const size_t m = di->max_dyn - fa.sharedSizeBytes;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(m));
        if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        it = done.emplace(key, m).first;
    }
    di->max_dyn = it->second;
    return SPEC_OK;
}

#ifdef SPEC_TEST_HOOKS
namespace {
std::atomic<int> g_test_withhold{-1};
}
int test_withhold_unit() { return g_test_withhold.load(); }
#endif

namespace {

inline size_t align16(size_t n) { return (n + 15) & ~size_t(15); }
inline bool aligned(const void *ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// Workspace layout (16-byte aligned parts):
//   [control: kCtrlWords u32][stats tiles per unit: n_units u32][units per sequence: B u32]
//   [decided / accepted masks: B u64]
//   [accept bits: B*K i32][argmax: n_units i32][run partials: n_units*2*S u64]
//   [t(x), d(x): n_units * 2 u64][draw statistics: n_units float4]
//   [draw records: entries u32][chunk sums: entries*Sr*kCpt i64]
struct WsLayout {
    size_t ctrl, unit_cnt, seq_cnt, seqmask, acc, val, part, tx, stats, draw, csum, total;
};
WsLayout ws_layout(int B, int K, int units_per_seq, int S, int Sr, size_t entries) {
    const bool draws = entries > 0;
    const size_t n_units = static_cast<size_t>(B) * units_per_seq;
    WsLayout w;
    w.ctrl = 0;
    w.unit_cnt = kCtrlWords * 4;
    w.seq_cnt = w.unit_cnt + align16(n_units * 4);
    w.seqmask = w.seq_cnt + align16(static_cast<size_t>(B) * 4);
    w.acc = w.seqmask + align16(static_cast<size_t>(B) * 8);
    w.val = w.acc + align16(static_cast<size_t>(B) * K * 4);
    w.part = w.val + align16(n_units * 4);
    w.tx = w.part + align16(n_units * 2 * static_cast<size_t>(S) * 8);
    w.stats = w.tx + align16(n_units * 16);
    w.draw = w.stats + (draws ? align16(n_units * 16) : 0);
    w.csum = w.draw + align16(entries * 4);
    w.total = w.csum + align16(entries * static_cast<size_t>(Sr) * kCpt * 8);
    return w;
}

void bind_workspace(Params &p, unsigned char *ws, const WsLayout &wl) {
    p.ws_base = ws;
    p.ws_bytes = wl.total;
    p.ws_ctrl = reinterpret_cast<uint32_t *>(ws + wl.ctrl);
    p.ws_unit_cnt = reinterpret_cast<uint32_t *>(ws + wl.unit_cnt);
    p.ws_seq_cnt = reinterpret_cast<uint32_t *>(ws + wl.seq_cnt);
    p.ws_seqmask = reinterpret_cast<unsigned long long *>(ws + wl.seqmask);
    p.ws_acc = reinterpret_cast<int32_t *>(ws + wl.acc);
    p.ws_val = reinterpret_cast<int32_t *>(ws + wl.val);
    p.ws_part = reinterpret_cast<unsigned long long *>(ws + wl.part);
    p.ws_txw = reinterpret_cast<unsigned long long *>(ws + wl.tx);
    p.ws_stats = reinterpret_cast<float4 *>(ws + wl.stats);
    p.ws_draw = reinterpret_cast<uint32_t *>(ws + wl.draw);
    p.ws_csum = reinterpret_cast<unsigned long long *>(ws + wl.csum);
}

// One draw entry per sequence (linear, extra token alone), per node (sampled
// tree), or none (greedy tree).
WsLayout layout_linear(int B, int K, int V, int eb) {
    return ws_layout(B, K, K + 1, stats_tiles_per_row(V, eb), resid_slicing(V, eb).S, static_cast<size_t>(B));
}
WsLayout layout_bonus(int B, int V, int eb) {
    return ws_layout(B, 0, 1, stats_tiles_per_row(V, eb), resid_slicing(V, eb).S, static_cast<size_t>(B));
}
WsLayout layout_tree(int B, int N, int V, int eb) {
    return ws_layout(B, 0, N, stats_tiles_per_row(V, eb), resid_slicing(V, eb).S, 0);
}
WsLayout layout_tree_sample(int B, int N, int V, int eb) {
    return ws_layout(B, 0, N, stats_tiles_per_row(V, eb), resid_slicing(V, eb).S,
                     static_cast<size_t>(B) * static_cast<size_t>(N));
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

#ifdef SPEC_TEST_HOOKS
// Test builds only: the unit whose first partial the next launches withhold (-1: none), so
// that a bounded wait runs out on purpose.
extern "C" __attribute__((visibility("default"))) void spec_test_set_withhold(int unit) {
    g_test_withhold.store(unit);
}
#endif

extern "C" size_t spec_workspace_bytes_linear(int B, int K, int V, spec_dtype dtype) {
    if (B <= 0 || K < 0 || V < 1 || !valid_dtype(dtype)) return 0;
    return layout_linear(B, K, V, elt_bytes(dtype)).total;
}

extern "C" size_t spec_workspace_bytes_bonus(int B, int V, spec_dtype dtype) {
    if (B <= 0 || V < 1 || !valid_dtype(dtype)) return 0;
    return layout_bonus(B, V, elt_bytes(dtype)).total;
}

extern "C" size_t spec_workspace_bytes_tree(int B, int N, int V, spec_dtype dtype) {
    if (B <= 0 || N < 1 || V < 1 || !valid_dtype(dtype)) return 0;
    return layout_tree(B, N, V, elt_bytes(dtype)).total;
}

extern "C" size_t spec_workspace_bytes_rows(int B, int V, spec_dtype dtype) {
    if (B <= 0 || V < 1 || !valid_dtype(dtype)) return 0;
    return layout_bonus(B, V, elt_bytes(dtype)).total;
}

extern "C" size_t spec_workspace_bytes_tree_sample(int B, int N, int V, spec_dtype dtype) {
    if (B <= 0 || N < 1 || V < 1 || !valid_dtype(dtype)) return 0;
    return layout_tree_sample(B, N, V, elt_bytes(dtype)).total;
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
    if (static_cast<long long>(B) * (2 * K + 1) > INT_MAX / 64) return fail(SPEC_ERR_UNSUPPORTED, "B * (K + 1) too large");
    const WsLayout wl = layout_linear(B, K, V, eb);
    if (!workspace || workspace_bytes < wl.total || !aligned(workspace, 16))
        return fail(SPEC_ERR_WORKSPACE, "workspace needs %zu bytes, 16-byte aligned", wl.total);

    Params p = {};
    const size_t row_bytes = static_cast<size_t>(V) * eb;
    p.target = static_cast<const unsigned char *>(target_logits);
    p.t_end = p.target + static_cast<size_t>(B) * (K + 1) * row_bytes;
    p.draft = static_cast<const unsigned char *>(draft_logits);
    p.d_end = p.draft ? p.draft + static_cast<size_t>(B) * K * row_bytes : nullptr;
    p.B = B;
    p.K = K;
    p.V = V;
    p.t_rows = K + 1;
    p.units_per_seq = K + 1;
    p.rows_per_seq = sample ? 2 * K + 1 : K + 1;
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
    const bool draws = sample && u_bonus != nullptr;
    if (sample) return eb == 4 ? launch<4, kLinearSample>(p, draws, s) : launch<2, kLinearSample>(p, draws, s);
    return eb == 4 ? launch<4, kLinearGreedy>(p, false, s) : launch<2, kLinearGreedy>(p, false, s);
}

// The extra token alone; accept_len == nullptr draws every sequence at position K.
static spec_status sample_extra(const void *target_logits, const void *draft_logits, spec_dtype dtype, int B, int K,
                                int V, const int32_t *accept_len, const float *u_bonus, float temperature,
                                int32_t *bonus_token, uint32_t *dev_status, void *workspace, size_t workspace_bytes,
                                void *stream) {
    if (!valid_dtype(dtype)) return fail(SPEC_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (B < 0 || K < 0 || V < 1) return fail(SPEC_ERR_INVALID_ARG, "need B >= 0, K >= 0, V >= 1");
    float c = 0.f;
    if (!valid_temperature(temperature, &c)) return fail(SPEC_ERR_INVALID_ARG, "temperature must be finite and >= 0");
    if (B == 0) return SPEC_OK;
    const bool sample = temperature > 0.0f;
    const int eb = elt_bytes(dtype);
    if (!target_logits || !aligned(target_logits, eb)) return fail(SPEC_ERR_INVALID_ARG, "target_logits null or misaligned");
    if (sample && K > 0 && (!draft_logits || !aligned(draft_logits, eb)))
        return fail(SPEC_ERR_INVALID_ARG, "draft_logits null or misaligned");
    if (sample && !u_bonus) return fail(SPEC_ERR_INVALID_ARG, "u_bonus is null");
    if (!bonus_token || !dev_status) return fail(SPEC_ERR_INVALID_ARG, "a pointer is null");
    if (B > INT_MAX / 64) return fail(SPEC_ERR_UNSUPPORTED, "B too large");
    const WsLayout wl = layout_bonus(B, V, eb);
    if (!workspace || workspace_bytes < wl.total || !aligned(workspace, 16))
        return fail(SPEC_ERR_WORKSPACE, "workspace needs %zu bytes, 16-byte aligned", wl.total);
    Params p = {};
    const size_t row_bytes = static_cast<size_t>(V) * eb;
    p.target = static_cast<const unsigned char *>(target_logits);
    p.t_end = p.target + static_cast<size_t>(B) * (K + 1) * row_bytes;
    p.draft = static_cast<const unsigned char *>(draft_logits);
    p.d_end = p.draft ? p.draft + static_cast<size_t>(B) * K * row_bytes : nullptr;
    p.B = B;
    p.K = K;
    p.V = V;
    p.t_rows = K + 1;
    p.units_per_seq = 1;
    p.rows_per_seq = (sample && K > 0) ? 2 : 1;  // the draft row slot exists only with a draft
    p.n_units = B;
    p.c = c;
    p.u_bonus = u_bonus;
    p.accept_len_in = accept_len;
    p.bonus_token = bonus_token;
    p.status = dev_status;
    bind_workspace(p, static_cast<unsigned char *>(workspace), wl);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (sample) return eb == 4 ? launch<4, kBonusSample>(p, true, s) : launch<2, kBonusSample>(p, true, s);
    return eb == 4 ? launch<4, kBonusGreedy>(p, false, s) : launch<2, kBonusGreedy>(p, false, s);
}

extern "C" spec_status spec_sample_bonus(const void *target_logits, const void *draft_logits, spec_dtype dtype,
                                         int B, int K, int V, const int32_t *accept_len, const float *u_bonus,
                                         float temperature, int32_t *bonus_token, uint32_t *dev_status,
                                         void *workspace, size_t workspace_bytes, void *stream) {
    g_last_error[0] = '\0';
    if (!accept_len && B > 0) return fail(SPEC_ERR_INVALID_ARG, "accept_len is null");
    return sample_extra(target_logits, draft_logits, dtype, B, K, V, accept_len, u_bonus, temperature, bonus_token,
                        dev_status, workspace, workspace_bytes, stream);
}

extern "C" spec_status spec_sample_rows(const void *logits, spec_dtype dtype, int B, int V, const float *u,
                                        float temperature, int32_t *tokens, uint32_t *dev_status, void *workspace,
                                        size_t workspace_bytes, void *stream) {
    g_last_error[0] = '\0';
    // a row per sequence is the target tail of a zero-length draft: K = 0, no draft, no lengths
    return sample_extra(logits, nullptr, dtype, B, 0, V, nullptr, u, temperature, tokens, dev_status, workspace,
                        workspace_bytes, stream);
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
    const WsLayout wl = layout_tree(B, N, V, eb);
    if (!workspace || workspace_bytes < wl.total || !aligned(workspace, 16))
        return fail(SPEC_ERR_WORKSPACE, "workspace needs %zu bytes, 16-byte aligned", wl.total);
    Params p = {};
    p.target = static_cast<const unsigned char *>(target_logits);
    p.t_end = p.target + static_cast<size_t>(B) * N * static_cast<size_t>(V) * eb;
    p.B = B;
    p.K = N;
    p.V = V;
    p.t_rows = N;
    p.units_per_seq = N;
    p.rows_per_seq = N;
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
    // the warp that finishes a sequence stages parents, node tokens and argmaxes (3 * N ints)
    return eb == 4 ? launch<4, kTreeGreedy>(p, false, s) : launch<2, kTreeGreedy>(p, false, s);
}

extern "C" spec_status spec_verify_tree_sample(const void *target_logits, spec_dtype dtype, int B, int N, int V,
                                               const int32_t *parents, const int32_t *node_tokens,
                                               const float *u_nodes, float temperature, int max_depth,
                                               int32_t *path_nodes, int32_t *path_len, int32_t *out_tokens,
                                               uint32_t *dev_status, void *workspace, size_t workspace_bytes,
                                               void *stream) {
    g_last_error[0] = '\0';
    if (!valid_dtype(dtype)) return fail(SPEC_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (B < 0 || N < 1 || V < 1 || max_depth < 0)
        return fail(SPEC_ERR_INVALID_ARG, "need B >= 0, N >= 1, V >= 1, max_depth >= 0");
    float c = 0.f;
    if (!valid_temperature(temperature, &c) || !(temperature > 0.0f))
        return fail(SPEC_ERR_INVALID_ARG, "temperature must be finite and > 0");
    if (B == 0) return SPEC_OK;
    const int eb = elt_bytes(dtype);
    if (!target_logits || !aligned(target_logits, eb)) return fail(SPEC_ERR_INVALID_ARG, "target_logits null or misaligned");
    if (!parents || !node_tokens || !u_nodes || !path_nodes || !path_len || !out_tokens || !dev_status)
        return fail(SPEC_ERR_INVALID_ARG, "a pointer is null");
    if (static_cast<long long>(B) * N > INT_MAX / 64) return fail(SPEC_ERR_UNSUPPORTED, "B * N too large");
    const WsLayout wl = layout_tree_sample(B, N, V, eb);
    if (!workspace || workspace_bytes < wl.total || !aligned(workspace, 16))
        return fail(SPEC_ERR_WORKSPACE, "workspace needs %zu bytes, 16-byte aligned", wl.total);
    Params p = {};
    p.target = static_cast<const unsigned char *>(target_logits);
    p.t_end = p.target + static_cast<size_t>(B) * N * static_cast<size_t>(V) * eb;
    p.B = B;
    p.K = N;
    p.V = V;
    p.t_rows = N;
    p.units_per_seq = N;
    p.rows_per_seq = N;
    p.n_units = B * N;
    p.c = c;
    p.tokens = node_tokens;
    p.u_bonus = u_nodes;  // one uniform per node: the draw of unit b * N + n
    p.parents = parents;
    p.max_depth = max_depth;
    p.accept_len = path_len;
    p.out_tokens = out_tokens;
    p.path_nodes = path_nodes;
    p.status = dev_status;
    bind_workspace(p, static_cast<unsigned char *>(workspace), wl);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return eb == 4 ? launch<4, kTreeSample>(p, true, s) : launch<2, kTreeSample>(p, true, s);
}

extern "C" spec_status spec_tree_mask(const int32_t *parents, int N, uint32_t *mask_words, int32_t *depth,
                                      uint32_t *dev_status, void *stream) {
    g_last_error[0] = '\0';
    if (N < 1) return fail(SPEC_ERR_INVALID_ARG, "need N >= 1");
    if (N > kMaxMaskNodes) return fail(SPEC_ERR_UNSUPPORTED, "N = %d > %d nodes", N, kMaxMaskNodes);
    if (!parents || !mask_words || !depth || !dev_status) return fail(SPEC_ERR_INVALID_ARG, "a pointer is null");
    if (!aligned(parents, 4) || !aligned(mask_words, 4) || !aligned(depth, 4) || !aligned(dev_status, 4))
        return fail(SPEC_ERR_INVALID_ARG, "a pointer is misaligned");
    DeviceInfo di;
    int dev = 0;
    spec_status st = device_info(&di, &dev);
    if (st != SPEC_OK) return st;
    const int W = (N + 31) / 32;
    const int grid = std::min((N + kMaskWarps - 1) / kMaskWarps, di.sms * 8);
    const size_t smem = static_cast<size_t>(kMaskWarps) * W * sizeof(uint32_t);
    tree_mask_kernel<<<grid, kMaskWarps * 32, smem, static_cast<cudaStream_t>(stream)>>>(parents, N, W, mask_words,
                                                                                         depth, dev_status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "tree mask launch: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

extern "C" spec_status spec_mtp_plug(const int32_t *in_tokens, int B, int K, const int32_t *out_tokens,
                                     const int32_t *num_emitted, int32_t pad, int32_t *next_tokens,
                                     int32_t *seq_lens, uint32_t *dev_status, void *stream) {
    g_last_error[0] = '\0';
    if (B < 0 || K < 0) return fail(SPEC_ERR_INVALID_ARG, "need B >= 0, K >= 0 (B=%d K=%d)", B, K);
    if (B == 0) return SPEC_OK;
    if (static_cast<long long>(B) * (K + 1) > INT_MAX) return fail(SPEC_ERR_UNSUPPORTED, "B * (K + 1) too large");
    if (!in_tokens || !out_tokens || !num_emitted || !next_tokens || !dev_status)
        return fail(SPEC_ERR_INVALID_ARG, "a pointer is null");
    if (!aligned(in_tokens, 4) || !aligned(out_tokens, 4) || !aligned(num_emitted, 4) || !aligned(next_tokens, 4) ||
        !aligned(dev_status, 4) || (seq_lens && !aligned(seq_lens, 4)))
        return fail(SPEC_ERR_INVALID_ARG, "a pointer is misaligned");
    if (next_tokens == out_tokens) return fail(SPEC_ERR_INVALID_ARG, "next_tokens must not be out_tokens");
    const int grid = (B + kPlugWarps - 1) / kPlugWarps;
    mtp_plug_kernel<<<grid, kPlugWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(
        in_tokens, B, K, out_tokens, num_emitted, pad, next_tokens, seq_lens, dev_status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "MTP plug-in launch: %s", cudaGetErrorString(e));
    return SPEC_OK;
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
        case SPEC_ERR_UNSUPPORTED: return "SPEC_ERR_UNSUPPORTED: valid but not supported by this library";
        case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA: CUDA runtime error";
        case SPEC_ERR_WORKSPACE: return "SPEC_ERR_WORKSPACE: workspace missing, too small or misaligned";
    }
    return "unknown spec_status";
}

extern "C" const char *spec_last_error(void) { return g_last_error; }
