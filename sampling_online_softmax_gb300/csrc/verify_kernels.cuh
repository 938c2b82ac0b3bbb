// verify_kernels.cuh -- device code of the speculative-decoding verify step.
//
// What is computed ("Beschleunigung von Sonar durch Spekulation", Perplexity,
// section "Spekulatives Decoding", phases "Akzeptanz" and "Zielgenerierung",
// and section "Ziel-Entwurf"; acceptance rule of the cited "Fast Inference
// from Transformers via Speculative Decoding"; tree walk of the
// "Speculative-Decoding / Medusa" blog, section 三):
//   per draft position i: p_i(x_i), q_i(x_i) under softmax(logits / T), the
//   test u_i < min(1, p_i(x_i) / q_i(x_i)) (greedy: x_i == argmax target_i),
//   the first rejected position j, and one extra token drawn by inverse CDF
//   from max(0, p_j - q_j) (j < K) or p_K (j == K), or argmax in greedy mode.
//
// How (GB300 design): a streaming reduction with no waiting between CTAs.
//   * A "unit" is one (sequence, position): target row i with draft row i for
//     linear sampling, otherwise one target row.  Each unit is cut into S
//     vocabulary slices of about 16 KB per row; a "tile" is one slice of every
//     row of one unit.  Tiles are numbered sequence-major, positions in order.
//   * Persistent CTAs (a few per SM) take tiles dynamically from a global
//     counter.  Each CTA has a control warp and eight compute warps.  The
//     control warp keeps a ring of shared-memory stages full with 1-D bulk
//     copies (cp.async.bulk, one mbarrier per stage; unaligned slice ends
//     element-wise, padding -inf); the compute warps reduce each stage (max
//     and exp2-sum per row, or max/argmax) and hand the per-warp results back
//     through a second mbarrier.
//   * The control warp writes the tile's partial to the workspace and bumps
//     the unit's tile counter (acq_rel atomic).  The CTA that completes a unit
//     merges its S partials, takes the acceptance decision, and -- for the
//     first rejection (or the tail when nothing earlier rejected) -- draws the
//     candidate extra token itself: it re-streams the unit's slices (from L2,
//     they were just read) as residual tiles whose compute warps produce exact
//     int64 fixed-point weight sums (units of 2^-52) per 64-group chunk, then
//     locates the chunk by a prefix over those sums and rescans that one chunk.
//   * The CTA that completes a sequence's last unit emits its tokens (a warp
//     ballot finds the first rejection) and zeroes its workspace entries.
//   * No tensor cores (nothing here is a contraction).  Every wait is bounded
//     and reports SPEC_DEV_TIMEOUT instead of trapping.
#pragma once

#include <climits>
#include <cstdint>

#include "ptx.cuh"
#include "spec_verify.h"

namespace spec {

constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kThreads = kComputeThreads + 32;  // warp 0 controls, warps 1..8 compute
constexpr int kMaxRows = 2;                     // rows per unit: target, draft
constexpr int kMaxStages = 4;
constexpr int kMaxJobs = kMaxStages + 1;        // pending extra-token draws per CTA
constexpr int kChunk = 64;                      // 16-byte groups per residual chunk
constexpr uint32_t kWaitLimit = 1u << 22;

enum Mode : int {
    kLinearSample = 0,
    kLinearGreedy = 1,
    kTreeGreedy = 2,
    kBonusSample = 3,
    kBonusGreedy = 4,
};

enum TileKind : int { kTileEnd = 0, kTileStats = 1, kTileResid = 2 };

struct Params {
    const unsigned char *target;   // [B, t_rows, V]
    const unsigned char *draft;    // [B, K, V] (sampling) or null
    int B, K, V;
    int t_rows;                    // target rows per sequence: K+1 (linear), N (tree)
    int units_per_seq;             // K+1 (linear), N (tree), 1 (extra token alone)
    int n_units;
    int S;                         // tiles (slices) per unit
    int slice_len;                 // elements per slice (multiple of 16/eb)
    int row_buf_bytes;             // shared bytes per row buffer in a stage
    int stage_bytes;               // shared bytes per stage
    int nstage;                    // stages in the ring (2..kMaxStages)
    int cpt;                       // residual chunks per tile
    int grab;                      // tiles taken per visit to the global counter
    float c;                       // log2(e) / T  (sampling modes)
    const int32_t *tokens;         // [B, K] draft tokens, or [B, N] node tokens
    const float *u_accept;         // [B, K]
    const float *u_bonus;          // [B] or null
    const int32_t *accept_len_in;  // [B] (extra token alone)
    const int32_t *parents;        // [N] (tree)
    int max_depth;                 // tree
    int32_t *accept_len;           // [B] accept_len / path_len
    int32_t *out_tokens;           // [B, K+1] or [B, max_depth+1]
    int32_t *num_emitted;          // [B]
    float *probs;                  // [B, K, 3] or null
    int32_t *path_nodes;           // [B, max_depth+1]
    int32_t *bonus_token;          // [B]
    uint32_t *status;              // [1]
    uint32_t *ws_ctrl;             // [0] next tile, [1] CTAs finished
    uint32_t *ws_unit_cnt;         // [n_units] tiles finished per unit
    uint32_t *ws_seq_cnt;          // [B] units finished per sequence
    int32_t *ws_first;             // [B] K + 1 - (earliest published rejection), 0 if none
    int32_t *ws_acc;               // [B*K] accept bits
    int32_t *ws_val;               // [B*units_per_seq] candidate token / argmax
    uint2 *ws_part;                // [n_units * 2 * S] per-tile partials
    float2 *ws_tx;                 // [n_units] target and draft logit of the draft token
};

struct StageMeta {
    int kind;                      // TileKind
    int unit, k, b, pos, nrows;
    int job, tailw;                // residual tiles: job slot, weights of p instead of max(0, p - q)
    float Mt, invSt, Md, invSd;    // residual tiles: row statistics
};

struct Job {                       // a pending extra-token draw, private to one CTA
    int unit, b, pos, nrows, tailw, next_k, done_k, fin;
    float Mt, invSt, Md, invSd, ub;
};

struct __align__(16) Ctl {
    unsigned long long full[kMaxStages];   // stage loaded (control -> compute)
    unsigned long long done[kMaxStages];   // stage reduced (compute -> control)
    StageMeta meta[kMaxStages];
    float wm[kMaxStages][kMaxRows][kComputeWarps];
    float wsum[kMaxStages][kMaxRows][kComputeWarps];
    int wi[kMaxStages][kMaxRows][kComputeWarps];
    float2 xval[kMaxStages];              // t(x), d(x) when the draft token lies in the stage's slice
    int xhas[kMaxStages];
    Job jobs[kMaxJobs];
    int timed_out;
};

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ unsigned atom_add_acq_rel(uint32_t *p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ int ld_relaxed(const int32_t *p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// A weight in units of 2^-52: the power-of-two scaling is exact; the
// conversion rounds only weights below 2^-29.
__device__ __forceinline__ long long fixq(float w) { return __float2ll_rn(w * 4503599627370496.0f); }

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity) {
    for (uint32_t it = 0; it < kWaitLimit; ++it)
        if (ptx::mbar_try_wait(bar, parity)) return true;
    return false;
}

// ---------------------------------------------------------------- elements
template <int EB>
struct Elt;

template <>
struct Elt<4> {
    static constexpr int G = 4;  // elements per 16-byte group
    __device__ __forceinline__ static void unpack(const uint4 &w, float (&v)[G]) {
        v[0] = __uint_as_float(w.x);
        v[1] = __uint_as_float(w.y);
        v[2] = __uint_as_float(w.z);
        v[3] = __uint_as_float(w.w);
    }
    __device__ __forceinline__ static float load(const unsigned char *p) {
        return *reinterpret_cast<const float *>(p);
    }
    __device__ __forceinline__ static float gload(const unsigned char *p) {
        return __uint_as_float(__ldg(reinterpret_cast<const unsigned int *>(p)));
    }
    __device__ __forceinline__ static void store_neg_inf(unsigned char *p) {
        *reinterpret_cast<uint32_t *>(p) = 0xff800000u;
    }
    __device__ __forceinline__ static void copy(unsigned char *dst, const unsigned char *src) {
        *reinterpret_cast<uint32_t *>(dst) = __ldg(reinterpret_cast<const uint32_t *>(src));
    }
    __device__ __forceinline__ static float group_max(const unsigned char *buf, int g0, int g1, int step) {
        float m = neg_inf();
        for (int g = g0; g < g1; g += step) {
            const uint4 w = *reinterpret_cast<const uint4 *>(buf + 16 * g);
            m = fmaxf(m, fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)),
                               fmaxf(__uint_as_float(w.z), __uint_as_float(w.w))));
        }
        return m;
    }
};

template <>
struct Elt<2> {
    static constexpr int G = 8;
    __device__ __forceinline__ static void unpack(const uint4 &w, float (&v)[G]) {
        v[0] = __uint_as_float(w.x << 16);
        v[1] = __uint_as_float(w.x & 0xffff0000u);
        v[2] = __uint_as_float(w.y << 16);
        v[3] = __uint_as_float(w.y & 0xffff0000u);
        v[4] = __uint_as_float(w.z << 16);
        v[5] = __uint_as_float(w.z & 0xffff0000u);
        v[6] = __uint_as_float(w.w << 16);
        v[7] = __uint_as_float(w.w & 0xffff0000u);
    }
    __device__ __forceinline__ static float load(const unsigned char *p) {
        return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(p)) << 16);
    }
    __device__ __forceinline__ static float gload(const unsigned char *p) {
        return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short *>(p))) << 16);
    }
    __device__ __forceinline__ static void store_neg_inf(unsigned char *p) {
        *reinterpret_cast<uint16_t *>(p) = 0xff80u;
    }
    __device__ __forceinline__ static void copy(unsigned char *dst, const unsigned char *src) {
        *reinterpret_cast<uint16_t *>(dst) = __ldg(reinterpret_cast<const unsigned short *>(src));
    }
    __device__ __forceinline__ static float group_max(const unsigned char *buf, int g0, int g1, int step) {
        uint32_t m = 0xff80ff80u;  // (-inf, -inf)
        for (int g = g0; g < g1; g += step) {
            const uint4 w = *reinterpret_cast<const uint4 *>(buf + 16 * g);
            m = ptx::bmax2(m, ptx::bmax2(ptx::bmax2(w.x, w.y), ptx::bmax2(w.z, w.w)));
        }
        return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    }
};

// ------------------------------------------------------------ row geometry
// A slice [s0, s1) of one row, mirrored in shared memory 16-byte group by
// group: buffer byte k holds global byte (glo + k), glo = 16-byte floor of the
// slice start.  Groups [hg, hg + nfull) arrive by bulk copy; partial groups at
// either end are filled element-wise, with -inf outside the slice.
struct RowGeo {
    const unsigned char *glo;  // global address of buffer byte 0
    unsigned char *buf;        // shared buffer (generic pointer)
    int ngran;                 // 16-byte groups in the buffer
    int hg;                    // 1 if group 0 is partial (and there are full groups)
    int nfull;                 // groups copied in bulk
    int vbase;                 // element index of buffer byte 0 (may be negative)
    int a0off, a1off;          // byte offsets of the slice's first / one-past-last element
};

template <int EB>
__device__ __forceinline__ RowGeo make_geo(const unsigned char *row, int s0, int s1, unsigned char *buf) {
    RowGeo g;
    const uintptr_t A = reinterpret_cast<uintptr_t>(row);
    const uintptr_t a0 = A + static_cast<uintptr_t>(s0) * EB;
    const uintptr_t a1 = A + static_cast<uintptr_t>(s1) * EB;
    const uintptr_t glo = a0 & ~uintptr_t(15);
    const uintptr_t ghi = (a1 + 15) & ~uintptr_t(15);
    const uintptr_t flo = (a0 + 15) & ~uintptr_t(15);
    const uintptr_t fhi = a1 & ~uintptr_t(15);
    g.glo = reinterpret_cast<const unsigned char *>(glo);
    g.buf = buf;
    g.ngran = static_cast<int>((ghi - glo) >> 4);
    if (flo < fhi) {
        g.hg = static_cast<int>((flo - glo) >> 4);
        g.nfull = static_cast<int>((fhi - flo) >> 4);
    } else {
        g.hg = 0;
        g.nfull = 0;
    }
    g.vbase = static_cast<int>((static_cast<long long>(glo) - static_cast<long long>(A)) / EB);
    g.a0off = static_cast<int>(a0 - glo);
    g.a1off = static_cast<int>(a1 - glo);
    return g;
}

// ------------------------------------------------------- softmax merging
// (m, s) represents sum exp2((x - m) * c) over a set; merge two such sets.
__device__ __forceinline__ void merge_ms(float &m, float &s, float m2, float s2, float c) {
    const float mm = fmaxf(m, m2);
    const float a = (m == mm) ? s : s * ptx::ex2((m - mm) * c);
    const float b = (m2 == mm) ? s2 : s2 * ptx::ex2((m2 - mm) * c);
    m = mm;
    s = a + b;
}

// (v, i): larger value wins, lower index breaks ties.
__device__ __forceinline__ void merge_vi(float &v, int &i, float v2, int i2) {
    if (v2 > v || (v2 == v && i2 < i)) {
        v = v2;
        i = i2;
    }
}

// ------------------------------------------------------ extra-token weights
// Weight of one element: pair (residual) max(0, p_v - q_v) with
// p_v = 2^((t - Mt) c) / St and q_v = 2^((d - Md) c) / Sd; tail p_v.  The
// explicit _rn intrinsics keep every evaluation of a weight bit-identical.
__device__ __forceinline__ float elem_weight(float t, float d, bool pair, float Mt, float Md, float invSt,
                                             float invSd, float c) {
    const float pv = __fmul_rn(ptx::ex2(__fmul_rn(__fsub_rn(t, Mt), c)), invSt);
    if (!pair) return pv;
    const float qv = __fmul_rn(ptx::ex2(__fmul_rn(__fsub_rn(d, Md), c)), invSd);
    return fmaxf(0.0f, __fsub_rn(pv, qv));
}

// fp32 sum of one 16-byte group's weights, in element order (the order every
// consumer of a group sum repeats).
template <int EB>
__device__ __forceinline__ float group_weight(const RowGeo &gt, const RowGeo &gd, bool pair, bool same_phase,
                                              int g, int s0, int s1, float Mt, float Md, float invSt, float invSd,
                                              float c) {
    constexpr int G = Elt<EB>::G;
    float t[G], d[G];
    Elt<EB>::unpack(*reinterpret_cast<const uint4 *>(gt.buf + 16 * g), t);
    if (pair) {
        if (same_phase) {
            Elt<EB>::unpack(*reinterpret_cast<const uint4 *>(gd.buf + 16 * g), d);
        } else {
#pragma unroll
            for (int k = 0; k < G; ++k) {
                const int v = gt.vbase + g * G + k;
                d[k] = (v >= s0 && v < s1) ? Elt<EB>::load(gd.buf + (v - gd.vbase) * EB) : neg_inf();
            }
        }
    }
    float sw = 0.f;
#pragma unroll
    for (int k = 0; k < G; ++k) sw += elem_weight(t[k], pair ? d[k] : 0.f, pair, Mt, Md, invSt, invSd, c);
    return sw;
}

// ---------------------------------------------------------- unit layout
struct UnitRows {
    int b, pos, nrows;
    const unsigned char *row[kMaxRows];
};

// Unit u: (sequence b, position pos) and its rows; pos < 0 marks an invalid
// unit of the extra-token-alone mode (no rows).
template <int EB, int MODE>
__device__ __forceinline__ UnitRows unit_rows(const Params &p, int u) {
    constexpr bool kSample = (MODE == kLinearSample || MODE == kBonusSample);
    constexpr bool kBonus = (MODE == kBonusSample || MODE == kBonusGreedy);
    UnitRows ur;
    if (kBonus) {
        ur.b = u;
        ur.pos = p.accept_len_in[u];
        if (ur.pos < 0 || ur.pos > p.K) ur.pos = -1;
    } else {
        ur.b = u / p.units_per_seq;
        ur.pos = u - ur.b * p.units_per_seq;
    }
    ur.nrows = (ur.pos < 0) ? 0 : ((kSample && ur.pos < p.K) ? 2 : 1);
    const size_t row_bytes = static_cast<size_t>(p.V) * EB;
    ur.row[0] = p.target;
    if (ur.nrows >= 1) ur.row[0] = p.target + (static_cast<size_t>(ur.b) * p.t_rows + ur.pos) * row_bytes;
    ur.row[1] = ur.row[0];
    if (ur.nrows == 2) ur.row[1] = p.draft + (static_cast<size_t>(ur.b) * p.K + ur.pos) * row_bytes;
    return ur;
}

// ====================================================== control-warp side
// The control warp fills stage s with slice k of unit u's rows (all 32 lanes call it).
template <int EB, int MODE>
__device__ void fill_stage(const Params &p, Ctl &ctl, unsigned char *dsm, int s, const StageMeta &m,
                           const UnitRows &ur, int lane) {
    unsigned char *stage = dsm + static_cast<size_t>(s) * p.stage_bytes;
    const uint32_t bar = ptx::smem_addr(&ctl.full[s]);
    const int s0 = min(p.V, m.k * p.slice_len);
    const int s1 = min(p.V, s0 + p.slice_len);
    RowGeo geo[kMaxRows];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) geo[r] = make_geo<EB>(ur.row[r], s0, s1, stage + r * p.row_buf_bytes);
    if (lane == 0) {
        ctl.meta[s] = m;
        uint32_t bytes = 0;
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r)
            if (r < ur.nrows) bytes += static_cast<uint32_t>(geo[r].nfull) * 16u;
        // the compute warps' reads of this stage are ordered before this point by
        // the stage's done-mbarrier, which the control warp waited on
        ptx::mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) {
            if (r >= ur.nrows || geo[r].nfull == 0) continue;
            const int off = 16 * geo[r].hg;
            ptx::bulk_g2s(ptx::smem_addr(geo[r].buf + off), geo[r].glo + off,
                          static_cast<uint32_t>(geo[r].nfull) * 16u, bar);
        }
    }
    // unaligned ends element-wise (at most 16 slots per row): lanes 0..15 row 0, 16..31 row 1
    {
        const int r = lane >> 4;
        const int e = lane & 15;
        if (r < ur.nrows) {
            const RowGeo g = (r == 0) ? geo[0] : geo[1];
            const int head_slots = g.hg * 16 / EB;
            const int tail_first = (g.hg + g.nfull) * 16;
            const int tail_slots = (g.ngran * 16 - tail_first) / EB;
            if (e < head_slots + tail_slots) {
                const int off = (e < head_slots) ? e * EB : tail_first + (e - head_slots) * EB;
                if (off >= g.a0off && off < g.a1off)
                    Elt<EB>::copy(g.buf + off, g.glo + off);
                else
                    Elt<EB>::store_neg_inf(g.buf + off);
            }
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);  // second arrival: the element-wise part is in place
}

// Emit sequence b (its last unit just finished) and zero its workspace entries.
template <int EB, int MODE>
__device__ void emit_sequence(const Params &p, int b, long long *stage_ints, int lane) {
    const int K = p.K;
    const int U = p.units_per_seq;
    if (MODE == kLinearSample || MODE == kLinearGreedy) {
        const bool has_bonus = p.u_bonus != nullptr;
        int j = K;
        for (int base = 0; base < K; base += 32) {
            const int i = base + lane;
            bool rej = false;
            if (i < K) {
                if (MODE == kLinearSample)
                    rej = __ldcg(&p.ws_acc[static_cast<size_t>(b) * K + i]) == 0;
                else
                    rej = p.tokens[static_cast<size_t>(b) * K + i] != __ldcg(&p.ws_val[static_cast<size_t>(b) * U + i]);
            }
            const unsigned m = __ballot_sync(0xffffffffu, rej);
            if (m) {
                j = base + __ffs(m) - 1;
                break;
            }
        }
        const int bonus = has_bonus ? __ldcg(&p.ws_val[static_cast<size_t>(b) * U + j]) : -1;
        if (p.out_tokens) {
            for (int i = lane; i <= K; i += 32)
                p.out_tokens[static_cast<size_t>(b) * (K + 1) + i] =
                    (i < j) ? p.tokens[static_cast<size_t>(b) * K + i] : ((i == j) ? bonus : -1);
        }
        if (lane == 0) {
            p.accept_len[b] = j;
            p.num_emitted[b] = j + (has_bonus ? 1 : 0);
        }
        // leave this sequence's workspace entries zero for the next call
        __syncwarp();
        if (MODE == kLinearSample)
            for (int i = lane; i < K; i += 32) p.ws_acc[static_cast<size_t>(b) * K + i] = 0;
        for (int i = lane; i < U; i += 32) p.ws_val[static_cast<size_t>(b) * U + i] = 0;
        if (lane == 0) {
            p.ws_first[b] = 0;
            p.ws_seq_cnt[b] = 0u;
        }
    } else if (MODE == kTreeGreedy) {
        // stage the tree of this sequence in the control warp's scratch area
        const int N = U;
        int *par_s = reinterpret_cast<int *>(stage_ints);
        int *tok_s = par_s + N;
        int *am_s = tok_s + N;
        for (int cidx = lane; cidx < N; cidx += 32) {
            int pc = p.parents[cidx];
            if (cidx == 0) {
                pc = -1;
            } else if (pc < 0 || pc >= cidx) {
                atomicOr(p.status, SPEC_DEV_BAD_TREE);
                pc = -2;
            }
            par_s[cidx] = pc;
            tok_s[cidx] = p.tokens[static_cast<size_t>(b) * N + cidx];
            am_s[cidx] = __ldcg(&p.ws_val[static_cast<size_t>(b) * N + cidx]);
        }
        __syncwarp();
        for (int cidx = lane; cidx < N; cidx += 32) p.ws_val[static_cast<size_t>(b) * N + cidx] = 0;
        const int D = p.max_depth;
        int32_t *pn = p.path_nodes + static_cast<size_t>(b) * (D + 1);
        int32_t *ot = p.out_tokens + static_cast<size_t>(b) * (D + 1);
        int cur = 0, depth = 0;
        while (depth < D) {
            const int want = am_s[cur];
            int next = -1;
            for (int base = cur + 1; base < N; base += 32) {
                const int cc = base + lane;
                const bool hit = cc < N && par_s[cc] == cur && tok_s[cc] == want;
                const unsigned m = __ballot_sync(0xffffffffu, hit);
                if (m) {
                    next = base + __ffs(m) - 1;
                    break;
                }
            }
            if (next < 0) break;
            if (lane == 0) {
                ot[depth] = tok_s[next];
                pn[depth + 1] = next;
            }
            ++depth;
            cur = next;
        }
        if (lane == 0) {
            pn[0] = 0;
            ot[depth] = am_s[cur];
            p.accept_len[b] = depth;
            p.ws_seq_cnt[b] = 0u;
        }
        for (int i = depth + 1 + lane; i <= D; i += 32) {
            ot[i] = -1;
            pn[i] = -1;
        }
        __syncwarp();
    }
}

// One more unit of sequence b is finished; emit the sequence if it was the last.
template <int EB, int MODE>
__device__ void unit_finished(const Params &p, int b, long long *scratch, int lane) {
    int last = 0;
    if (lane == 0)
        last = (atom_add_acq_rel(&p.ws_seq_cnt[b], 1u) == static_cast<unsigned>(p.units_per_seq - 1)) ? 1 : 0;
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
        __syncwarp();
        emit_sequence<EB, MODE>(p, b, scratch, lane);
    }
}

// Extra-token draw finished: record the token.
template <int EB, int MODE>
__device__ void token_drawn(const Params &p, const Job &jb, int token, long long *scratch, int lane) {
    constexpr bool kBonus = (MODE == kBonusSample || MODE == kBonusGreedy);
    if (kBonus) {
        if (lane == 0) p.bonus_token[jb.b] = token;
        return;
    }
    if (lane == 0) p.ws_val[static_cast<size_t>(jb.b) * p.units_per_seq + jb.pos] = token;
    __syncwarp();
    unit_finished<EB, MODE>(p, jb.b, scratch, lane);
}

// All residual tiles of job `jb` are reduced: locate the token.  Returns -1
// when the weights summed to zero (the caller then retries with p alone).
template <int EB, int MODE>
__device__ int select_token(const Params &p, const Job &jb, const long long *csum, int lane) {
    constexpr int G = Elt<EB>::G;
    const int n = p.S * p.cpt;
    const int per = (n + 31) / 32;
    const int lo = min(n, lane * per), hi = min(n, lo + per);
    long long mine = 0;
    for (int i = lo; i < hi; ++i) mine += csum[i];
    long long incl = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    const long long tot = __shfl_sync(0xffffffffu, incl, 31);
    if (tot <= 0) return -1;
    const long long target = static_cast<long long>(static_cast<double>(jb.ub) * static_cast<double>(tot));
    // the chunk holding the target: first lane, then first chunk in that lane's block
    const unsigned bl = __ballot_sync(0xffffffffu, incl > target);
    const int ol = __ffs(bl) - 1;
    long long acc = __shfl_sync(0xffffffffu, incl - mine, ol);
    int chunk = -1;
    if (lane == ol) {
        long long a = acc;
        for (int i = lo; i < hi; ++i) {
            if (a + csum[i] > target) {
                chunk = i;
                break;
            }
            a += csum[i];
        }
        acc = a;
    }
    chunk = __shfl_sync(0xffffffffu, chunk, ol);
    acc = __shfl_sync(0xffffffffu, acc, ol);
    const long long rem = target - acc;  // 0 <= rem < csum[chunk]
    // rescan that chunk from global memory, element by element, with the same weights
    const int k = chunk / p.cpt;
    const int cc = chunk - k * p.cpt;
    const int s0 = min(p.V, k * p.slice_len);
    const int s1 = min(p.V, s0 + p.slice_len);
    const UnitRows ur = unit_rows<EB, MODE>(p, jb.unit);
    const RowGeo gt = make_geo<EB>(ur.row[0], s0, s1, nullptr);
    const bool pair = !jb.tailw;
    long long q[2];
    float w[2][G];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int g = cc * kChunk + h * 32 + lane;
        float sw = 0.f;
#pragma unroll
        for (int e = 0; e < G; ++e) {
            const int v = gt.vbase + g * G + e;
            float we = 0.f;
            if (g < gt.ngran && v >= s0 && v < s1) {
                const float t = Elt<EB>::gload(ur.row[0] + static_cast<size_t>(v) * EB);
                const float d = pair ? Elt<EB>::gload(ur.row[1] + static_cast<size_t>(v) * EB) : 0.f;
                we = elem_weight(t, d, pair, jb.Mt, jb.Md, jb.invSt, jb.invSd, p.c);
            }
            w[h][e] = we;
            sw += we;
        }
        q[h] = fixq(sw);
    }
    // inclusive prefix over the chunk's 64 groups (first half, then second half)
    long long i0 = q[0], i1 = q[1];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long y0 = __shfl_up_sync(0xffffffffu, i0, off);
        const long long y1 = __shfl_up_sync(0xffffffffu, i1, off);
        if (lane >= off) {
            i0 += y0;
            i1 += y1;
        }
    }
    const long long t0 = __shfl_sync(0xffffffffu, i0, 31);
    i1 += t0;
    unsigned bh = __ballot_sync(0xffffffffu, i0 > rem);
    int half = 0;
    if (!bh) {
        bh = __ballot_sync(0xffffffffu, i1 > rem);
        half = 1;
    }
    int token = -1;
    if (bh) {
        const int gl = __ffs(bh) - 1;
        const long long excl = __shfl_sync(0xffffffffu, half ? (i1 - q[1]) : (i0 - q[0]), gl);
        if (lane == gl) {
            const int g = cc * kChunk + half * 32 + lane;
            // the same weights, summed in the same order as the group sum
            float cum = 0.f;
            int esel = -1;
#pragma unroll
            for (int e = 0; e < G; ++e) {
                cum += half ? w[1][e] : w[0][e];
                if (esel < 0 && excl + fixq(cum) > rem) esel = e;
            }
            token = gt.vbase + g * G + (esel < 0 ? G - 1 : esel);
        }
        token = __shfl_sync(0xffffffffu, token, gl);
    }
    return token < 0 ? 0 : token;
}

// ====================================================== compute-warp side
template <int EB, int MODE>
__device__ void compute_stats(const Params &p, Ctl &ctl, unsigned char *stage, const StageMeta &m, int s,
                              int ct, int cw, int lane) {
    constexpr bool kSample = (MODE == kLinearSample || MODE == kBonusSample);
    constexpr int G = Elt<EB>::G;
    const UnitRows ur = unit_rows<EB, MODE>(p, m.unit);
    const int s0 = min(p.V, m.k * p.slice_len);
    const int s1 = min(p.V, s0 + p.slice_len);
    const float c = p.c;
    // the draft token of a pair unit: its two logits are read here if this slice holds it
    int x = -1;
    if (MODE == kLinearSample && m.nrows == 2 && ct == 0) x = p.tokens[static_cast<size_t>(m.b) * p.K + m.pos];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
        if (r >= m.nrows) continue;
        const RowGeo g = make_geo<EB>(ur.row[r], s0, s1, stage + r * p.row_buf_bytes);
        if (kSample) {
            const float mp = Elt<EB>::group_max(g.buf, ct, g.ngran, kComputeThreads);
            float sa = 0.f, sb = 0.f;
            if (mp != neg_inf()) {
                int gg = ct;
                for (; gg + kComputeThreads < g.ngran; gg += 2 * kComputeThreads) {
                    float va[G], vb[G];
                    Elt<EB>::unpack(*reinterpret_cast<const uint4 *>(g.buf + 16 * gg), va);
                    Elt<EB>::unpack(*reinterpret_cast<const uint4 *>(g.buf + 16 * (gg + kComputeThreads)), vb);
#pragma unroll
                    for (int k = 0; k < G; ++k) {
                        sa += ptx::ex2((va[k] - mp) * c);
                        sb += ptx::ex2((vb[k] - mp) * c);
                    }
                }
                if (gg < g.ngran) {
                    float va[G];
                    Elt<EB>::unpack(*reinterpret_cast<const uint4 *>(g.buf + 16 * gg), va);
#pragma unroll
                    for (int k = 0; k < G; ++k) sa += ptx::ex2((va[k] - mp) * c);
                }
            }
            // warp: the max first, then one rescale per lane and a plain sum
            float wmax = mp;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, off));
            float sum = sa + sb;
            if (mp != wmax) sum *= ptx::ex2((mp - wmax) * c);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            if (lane == 0) {
                ctl.wm[s][r][cw] = wmax;
                ctl.wsum[s][r][cw] = sum;
            }
        } else {
            float bv = neg_inf();
            int bi = INT_MAX;
            for (int gg = ct; gg < g.ngran; gg += kComputeThreads) {
                float va[G];
                Elt<EB>::unpack(*reinterpret_cast<const uint4 *>(g.buf + 16 * gg), va);
#pragma unroll
                for (int k = 0; k < G; ++k)
                    if (va[k] > bv) {
                        bv = va[k];
                        bi = g.vbase + gg * G + k;
                    }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                merge_vi(bv, bi, __shfl_xor_sync(0xffffffffu, bv, off), __shfl_xor_sync(0xffffffffu, bi, off));
            if (lane == 0) {
                ctl.wm[s][r][cw] = bv;
                ctl.wi[s][r][cw] = bi;
            }
        }
    }
    if (MODE == kLinearSample && ct == 0) {
        int has = 0;
        float2 xv = make_float2(0.f, 0.f);
        if (m.nrows == 2 && x >= s0 && x < s1) {
            const RowGeo gt = make_geo<EB>(ur.row[0], s0, s1, stage);
            const RowGeo gd = make_geo<EB>(ur.row[1], s0, s1, stage + p.row_buf_bytes);
            xv = make_float2(Elt<EB>::load(gt.buf + (x - gt.vbase) * EB), Elt<EB>::load(gd.buf + (x - gd.vbase) * EB));
            has = 1;
        }
        ctl.xval[s] = xv;
        ctl.xhas[s] = has;
    }
}

// Residual tile: exact int64 weight sums per chunk of 64 groups.
template <int EB, int MODE>
__device__ void compute_resid(const Params &p, unsigned char *stage, const StageMeta &m, long long *csum, int cw,
                              int lane) {
    const UnitRows ur = unit_rows<EB, MODE>(p, m.unit);
    const int s0 = min(p.V, m.k * p.slice_len);
    const int s1 = min(p.V, s0 + p.slice_len);
    const RowGeo gt = make_geo<EB>(ur.row[0], s0, s1, stage);
    const RowGeo gd = make_geo<EB>(ur.row[1], s0, s1, stage + p.row_buf_bytes);
    const bool pair = !m.tailw;
    const bool same_phase =
        ((reinterpret_cast<uintptr_t>(ur.row[0]) - reinterpret_cast<uintptr_t>(ur.row[1])) & 15u) == 0;
    for (int ch = cw; ch < p.cpt; ch += kComputeWarps) {
        long long q = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int g = ch * kChunk + h * 32 + lane;
            if (g < gt.ngran)
                q += fixq(group_weight<EB>(gt, gd, pair, same_phase, g, s0, s1, m.Mt, m.Md, m.invSt, m.invSd, p.c));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) q += __shfl_xor_sync(0xffffffffu, q, off);
        if (lane == 0) csum[m.k * p.cpt + ch] = q;
    }
}

// ================================================================ kernel
template <int EB, int MODE>
__global__ void __maxnreg__(112) spec_verify_kernel(const Params p) {
    constexpr bool kSample = (MODE == kLinearSample || MODE == kBonusSample);
    constexpr bool kBonus = (MODE == kBonusSample || MODE == kBonusGreedy);

    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ Ctl ctl;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nstage = p.nstage;
    // after the stages: per-job residual chunk sums (sampling), or the tree-walk scratch
    long long *extra = reinterpret_cast<long long *>(dsm + static_cast<size_t>(nstage) * p.stage_bytes);
    const int job_stride = p.S * p.cpt;

    if (tid == 0) {
        for (int s = 0; s < nstage; ++s) {
            ptx::mbar_init(ptx::smem_addr(&ctl.full[s]), 2);
            ptx::mbar_init(ptx::smem_addr(&ctl.done[s]), kComputeWarps);
        }
        ptx::fence_mbar_init();
        ctl.timed_out = 0;
    }
    __syncthreads();

    if (warp != 0) {
        // ===================== compute warps: reduce the stages in ring order
        const int ct = tid - 32;
        const int cw = warp - 1;
        for (int it = 0;; ++it) {
            const int s = it % nstage;
            if (!wait_bar(ptx::smem_addr(&ctl.full[s]), static_cast<uint32_t>(it / nstage) & 1u)) {
                ctl.timed_out = 1;
                break;
            }
            const StageMeta m = ctl.meta[s];
            if (m.kind == kTileEnd) break;
            unsigned char *stage = dsm + static_cast<size_t>(s) * p.stage_bytes;
            if (m.kind == kTileStats)
                compute_stats<EB, MODE>(p, ctl, stage, m, s, ct, cw, lane);
            else if (kSample)
                compute_resid<EB, MODE>(p, stage, m, extra + static_cast<size_t>(m.job) * job_stride, cw, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(ptx::smem_addr(&ctl.done[s]));
        }
        return;
    }

    // ========================= control warp: stream tiles, publish, finalize
    const long long total = static_cast<long long>(p.n_units) * p.S;
    // tile indices from the global counter; lane 0's copies are authoritative.
    // The next batch is requested one batch ahead, so its latency is hidden.
    long long grab_next = 0, grab_end = 0;
    unsigned grab_ahead = 0;
    if (lane == 0) grab_ahead = atomicAdd(&p.ws_ctrl[0], static_cast<unsigned>(p.grab));
    bool exhausted = false;
    int job_head = 0, job_count = 0;  // FIFO of pending draws (lane 0)
    int handled = 0, filled = 0;      // tiles handled / tiles handed to the ring
    bool timed_out = false;
    // the last published run's counter increment, consumed later
    unsigned pend_old = 0;
    int pend_cnt = 0;
    bool pend_valid = false;
    StageMeta pend_m = {};
    // the run of consecutive stats tiles of one unit merged in this CTA (lane 0)
    int run_unit = -1, run_k0 = 0, run_cnt = 0, run_hasx = 0;
    uint2 run_part[kMaxRows] = {};
    float2 run_x = make_float2(0.f, 0.f);
    StageMeta run_m = {};

    // the next tile of this CTA's stream: pending draws first, then fresh tiles
    auto next_tile = [&](StageMeta &m) -> bool {
        int found = 0;
        if (lane == 0) {
            for (int q = 0; q < job_count && !found; ++q) {
                Job &jb = ctl.jobs[(job_head + q) % kMaxJobs];
                if (!jb.fin && jb.next_k < p.S) {
                    m.kind = kTileResid;
                    m.unit = jb.unit;
                    m.k = jb.next_k++;
                    m.job = (job_head + q) % kMaxJobs;
                    m.tailw = jb.tailw;
                    m.Mt = jb.Mt;
                    m.invSt = jb.invSt;
                    m.Md = jb.Md;
                    m.invSd = jb.invSd;
                    found = 1;
                }
            }
            if (!found && !exhausted) {
                if (grab_next >= grab_end) {
                    grab_next = grab_ahead;
                    grab_end = grab_next + p.grab;
                    if (grab_next < total)
                        grab_ahead = atomicAdd(&p.ws_ctrl[0], static_cast<unsigned>(p.grab));
                }
                if (grab_next < total) {
                    const long long t = grab_next++;
                    m.kind = kTileStats;
                    m.unit = static_cast<int>(t / p.S);
                    m.k = static_cast<int>(t - static_cast<long long>(m.unit) * p.S);
                    m.job = -1;
                    m.tailw = 0;
                    found = 1;
                } else {
                    exhausted = true;
                }
            }
        }
        found = __shfl_sync(0xffffffffu, found, 0);
        if (!found) return false;
        m.kind = __shfl_sync(0xffffffffu, m.kind, 0);
        m.unit = __shfl_sync(0xffffffffu, m.unit, 0);
        m.k = __shfl_sync(0xffffffffu, m.k, 0);
        m.job = __shfl_sync(0xffffffffu, m.job, 0);
        m.tailw = __shfl_sync(0xffffffffu, m.tailw, 0);
        m.Mt = __shfl_sync(0xffffffffu, m.Mt, 0);
        m.invSt = __shfl_sync(0xffffffffu, m.invSt, 0);
        m.Md = __shfl_sync(0xffffffffu, m.Md, 0);
        m.invSd = __shfl_sync(0xffffffffu, m.invSd, 0);
        return true;
    };
    auto fill_more = [&]() {
        while (filled < handled + nstage) {
            StageMeta m;
            if (!next_tile(m)) break;
            const UnitRows ur = unit_rows<EB, MODE>(p, m.unit);
            m.b = ur.b;
            m.pos = ur.pos;
            m.nrows = ur.nrows;
            fill_stage<EB, MODE>(p, ctl, dsm, filled % nstage, m, ur, lane);
            ++filled;
        }
    };
    auto push_job = [&](const Job &jb) {
        if (lane == 0) {
            if (job_count < kMaxJobs) {
                ctl.jobs[(job_head + job_count) % kMaxJobs] = jb;
                ++job_count;
            } else {
                atomicOr(p.status, SPEC_DEV_TIMEOUT);  // cannot happen: at most nstage + 1 draws pend
            }
        }
        __syncwarp();
    };

    // ---- this CTA finished unit m.unit: merge its S partials, decide, maybe queue a draw
    auto finalize_unit = [&](const StageMeta &m) {
        const int b = m.b, pos = m.pos, K = p.K;
        // one round of loads: every partial, t(x) / d(x), the draft token and uniforms
        float v0 = neg_inf(), s0_ = 0.f, v1 = neg_inf(), s1_ = 0.f;
        int i0 = INT_MAX, i1 = INT_MAX;
        for (int l = lane; l < p.S; l += 32) {
#pragma unroll
            for (int r = 0; r < kMaxRows; ++r) {
                if (r >= m.nrows) continue;
                uint2 *slot = &p.ws_part[(static_cast<size_t>(m.unit) * 2 + r) * p.S + l];
                const uint2 e = __ldcg(slot);
                if (e.y == 0u) continue;  // no run started at this slice
                *slot = make_uint2(0u, 0u);
                float &v = r ? v1 : v0;
                float &sm = r ? s1_ : s0_;
                int &ii = r ? i1 : i0;
                if (kSample)
                    merge_ms(v, sm, __uint_as_float(e.x), __uint_as_float(e.y), p.c);
                else
                    merge_vi(v, ii, __uint_as_float(e.x), static_cast<int>(e.y) - 1);
            }
        }
        int x = -1, enc = 0;
        float ua = 0.f, ub = 0.f;
        float2 txv = make_float2(0.f, 0.f);
        if (lane == 0) {
            if (MODE == kLinearSample) {
                enc = ld_relaxed(&p.ws_first[b]);
                if (p.u_bonus) ub = p.u_bonus[b];
                if (pos < K) {
                    x = p.tokens[static_cast<size_t>(b) * K + pos];
                    ua = p.u_accept[static_cast<size_t>(b) * K + pos];
                    txv = __ldcg(&p.ws_tx[m.unit]);
                    p.ws_tx[m.unit] = make_float2(0.f, 0.f);
                }
            } else if (MODE == kBonusSample) {
                if (pos >= 0) ub = p.u_bonus[b];
            }
            p.ws_unit_cnt[m.unit] = 0u;
        }
        float Mr[kMaxRows], Sr[kMaxRows];
        int Ar[kMaxRows];
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) {
            float v = r ? v1 : v0, sm = r ? s1_ : s0_;
            int ii = r ? i1 : i0;
            if (kSample) {
                float wmax = v;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, off));
                if (v != wmax) sm *= ptx::ex2((v - wmax) * p.c);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, off);
                v = wmax;
            } else {
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    merge_vi(v, ii, __shfl_xor_sync(0xffffffffu, v, off), __shfl_xor_sync(0xffffffffu, ii, off));
            }
            Mr[r] = v;
            Sr[r] = sm;
            Ar[r] = ii;
        }
        uint32_t fl = 0;
        bool finite = true;
        if (kSample) {
            for (int r = 0; r < m.nrows; ++r)
                if (!(isfinite(Mr[r]) && isfinite(Sr[r]) && Sr[r] > 0.f)) finite = false;
            if (!finite) fl |= SPEC_DEV_NONFINITE;
        } else if (m.nrows > 0 && Ar[0] == INT_MAX) {
            fl |= SPEC_DEV_NONFINITE;  // no element above -inf
            Ar[0] = 0;
        }
        Job jb;
        jb.unit = m.unit;
        jb.b = b;
        jb.pos = pos;
        jb.nrows = m.nrows;
        jb.next_k = 0;
        jb.done_k = 0;
        jb.fin = 0;
        jb.Mt = Mr[0];
        jb.invSt = 1.0f / Sr[0];
        jb.Md = Mr[1];
        jb.invSd = (m.nrows == 2) ? 1.0f / Sr[1] : 0.f;
        jb.tailw = (m.nrows == 2) ? 0 : 1;
        jb.ub = __shfl_sync(0xffffffffu, ub, 0);
        int draw = 0;
        if (lane == 0) {
            if (MODE == kLinearSample) {
                const int early = (enc != 0 && (K + 1 - enc) < pos) ? 1 : 0;
                if (pos < K) {
                    float px = 0.f, qx = 0.f, thr = 0.f;
                    int accept = 0;
                    if (x < 0 || x >= p.V) {
                        fl |= SPEC_DEV_BAD_TOKEN;
                    } else {
                        const float tx = txv.x, dx = txv.y;
                        px = ptx::ex2((tx - Mr[0]) * p.c) / Sr[0];
                        qx = ptx::ex2((dx - Mr[1]) * p.c) / Sr[1];
                        const float ratio = ptx::ex2(((tx - Mr[0]) - (dx - Mr[1])) * p.c) * (Sr[1] / Sr[0]);
                        thr = fminf(1.0f, ratio);
                        accept = (ua < thr) ? 1 : 0;
                    }
                    p.ws_acc[static_cast<size_t>(b) * K + pos] = accept;
                    if (p.probs) {
                        float *pr = p.probs + (static_cast<size_t>(b) * K + pos) * 3;
                        pr[0] = px;
                        pr[1] = qx;
                        pr[2] = thr;
                    }
                    if (!accept) atomicMax(&p.ws_first[b], K + 1 - pos);
                    draw = (!accept && p.u_bonus != nullptr && !early) ? 1 : 0;
                } else {
                    draw = (p.u_bonus != nullptr && !early) ? 1 : 0;  // tail: p_K
                }
                if (!finite) draw = 0;
            } else if (MODE == kBonusSample) {
                draw = (pos >= 0 && finite) ? 1 : 0;
                if (pos < 0) fl |= SPEC_DEV_BAD_LENGTH;
            }
            if (fl) atomicOr(p.status, fl);
        }
        draw = __shfl_sync(0xffffffffu, draw, 0);
        if (draw) {
            push_job(jb);
        } else if (MODE == kLinearGreedy || MODE == kTreeGreedy) {
            if (lane == 0) p.ws_val[static_cast<size_t>(b) * p.units_per_seq + pos] = Ar[0];
            __syncwarp();
            unit_finished<EB, MODE>(p, b, extra, lane);
        } else if (MODE == kBonusGreedy) {
            if (lane == 0) {
                if (pos < 0) atomicOr(p.status, SPEC_DEV_BAD_LENGTH);
                p.bonus_token[b] = (pos < 0) ? -1 : Ar[0];
            }
        } else if (MODE == kBonusSample) {
            if (lane == 0) p.bonus_token[b] = (pos < 0) ? -1 : 0;
        } else {  // linear sampling without a draw here
            unit_finished<EB, MODE>(p, b, extra, lane);
        }
    };
    // consume the previous stats tile's counter increment (issued a tile ago)
    auto resolve_pending = [&]() {
        if (!pend_valid) return;
        pend_valid = false;
        const int last =
            __shfl_sync(0xffffffffu, (pend_old + static_cast<unsigned>(pend_cnt) == static_cast<unsigned>(p.S)) ? 1 : 0, 0);
        if (last) {
            __syncwarp();
            finalize_unit(pend_m);
        }
    };

    // write the current run's merged partial, count its tiles (the increment is consumed later)
    auto publish_run = [&]() {
        const int have = __shfl_sync(0xffffffffu, run_unit, 0);
        if (have < 0) return;
        resolve_pending();
        const StageMeta rm = run_m;
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < kMaxRows; ++r)
                if (r < rm.nrows) p.ws_part[(static_cast<size_t>(run_unit) * 2 + r) * p.S + run_k0] = run_part[r];
            if (run_hasx) p.ws_tx[run_unit] = run_x;
            pend_old = atom_add_acq_rel(&p.ws_unit_cnt[run_unit], static_cast<unsigned>(run_cnt));
            pend_cnt = run_cnt;
            run_unit = -1;
        }
        pend_valid = true;
        pend_m = rm;
    };

    fill_more();
    for (;;) {
        if (filled == handled) {
            publish_run();
            resolve_pending();
            fill_more();
            if (filled == handled) break;  // nothing in flight and nothing left
        }
        const int s = handled % nstage;
        if (!wait_bar(ptx::smem_addr(&ctl.done[s]), static_cast<uint32_t>(handled / nstage) & 1u)) {
            timed_out = true;
            break;
        }
        const StageMeta m = ctl.meta[s];
        ++handled;
        if (m.kind != kTileStats) {
            publish_run();
            resolve_pending();
        }
        if (m.kind == kTileStats) {
            // ---- CTA partial of this tile -> workspace (the max first, then one rescale per warp)
            uint2 part[kMaxRows];
#pragma unroll
            for (int r = 0; r < kMaxRows; ++r) {
                if (r >= m.nrows) continue;
                float v = lane < kComputeWarps ? ctl.wm[s][r][lane] : neg_inf();
                if (kSample) {
                    float sum = lane < kComputeWarps ? ctl.wsum[s][r][lane] : 0.f;
                    float wmax = v;
#pragma unroll
                    for (int off = 4; off > 0; off >>= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, off));
                    if (v != wmax) sum *= ptx::ex2((v - wmax) * p.c);
#pragma unroll
                    for (int off = 4; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
                    part[r] = make_uint2(__float_as_uint(wmax), __float_as_uint(sum));
                } else {
                    int i = lane < kComputeWarps ? ctl.wi[s][r][lane] : INT_MAX;
#pragma unroll
                    for (int off = 4; off > 0; off >>= 1)
                        merge_vi(v, i, __shfl_xor_sync(0xffffffffu, v, off), __shfl_xor_sync(0xffffffffu, i, off));
                    part[r] = make_uint2(__float_as_uint(v), static_cast<unsigned>(i) + 1u);  // +1: never 0
                }
            }
            const int has_x = (MODE == kLinearSample) ? ctl.xhas[s] : 0;
            const float2 xv = ctl.xval[s];
            fill_more();  // refill first: the publication below waits on its own stores
            const int same = __shfl_sync(0xffffffffu, (run_unit == m.unit && run_k0 + run_cnt == m.k) ? 1 : 0, 0);
            if (!same) publish_run();
            if (lane == 0) {
                if (!same) {
                    run_unit = m.unit;
                    run_k0 = m.k;
                    run_cnt = 0;
                    run_hasx = 0;
#pragma unroll
                    for (int r = 0; r < kMaxRows; ++r) run_part[r] = part[r];
                } else {
#pragma unroll
                    for (int r = 0; r < kMaxRows; ++r) {
                        if (r >= m.nrows) continue;
                        float v = __uint_as_float(run_part[r].x);
                        if (kSample) {
                            float sm = __uint_as_float(run_part[r].y);
                            merge_ms(v, sm, __uint_as_float(part[r].x), __uint_as_float(part[r].y), p.c);
                            run_part[r] = make_uint2(__float_as_uint(v), __float_as_uint(sm));
                        } else {
                            int ii = static_cast<int>(run_part[r].y) - 1;
                            merge_vi(v, ii, __uint_as_float(part[r].x), static_cast<int>(part[r].y) - 1);
                            run_part[r] = make_uint2(__float_as_uint(v), static_cast<unsigned>(ii) + 1u);
                        }
                    }
                }
                run_cnt += 1;
                if (has_x) {
                    run_hasx = 1;
                    run_x = xv;
                }
            }
            if (!same) run_m = m;
        } else if (kSample) {
            // ---- a residual tile of a pending draw is reduced
            Job jb = ctl.jobs[m.job];
            __syncwarp();
            int finished = 0;
            if (lane == 0) {
                ctl.jobs[m.job].done_k += 1;
                finished = (ctl.jobs[m.job].done_k == p.S) ? 1 : 0;
            }
            finished = __shfl_sync(0xffffffffu, finished, 0);
            if (!finished) {
                fill_more();
                continue;
            }
            __syncwarp();
            const int token = select_token<EB, MODE>(p, jb, extra + static_cast<size_t>(m.job) * job_stride, lane);
            if (token < 0 && !jb.tailw) {
                // the residual vanished through rounding: draw from p_j instead
                if (lane == 0) {
                    atomicOr(p.status, SPEC_DEV_ZERO_RESIDUAL);
                    ctl.jobs[m.job].tailw = 1;
                    ctl.jobs[m.job].next_k = 0;
                    ctl.jobs[m.job].done_k = 0;
                }
                __syncwarp();
                fill_more();
                continue;
            }
            // the draw is done; drop finished draws from the head of the FIFO
            if (lane == 0) {
                ctl.jobs[m.job].fin = 1;
                while (job_count > 0 && ctl.jobs[job_head].fin) {
                    job_head = (job_head + 1) % kMaxJobs;
                    --job_count;
                }
            }
            __syncwarp();
            token_drawn<EB, MODE>(p, jb, token < 0 ? 0 : token, extra, lane);
            fill_more();
        }
    }

    // ---- end of the stream: release the compute warps, account for the CTA
    if (!timed_out) {
        const int s = filled % nstage;
        if (lane == 0) {
            StageMeta e{};
            e.kind = kTileEnd;
            ctl.meta[s] = e;
            mbar_arrive(ptx::smem_addr(&ctl.full[s]));
            mbar_arrive(ptx::smem_addr(&ctl.full[s]));
        }
    }
    if (lane == 0) {
        if (timed_out || ctl.timed_out) atomicOr(p.status, SPEC_DEV_TIMEOUT);
        if (atom_add_acq_rel(&p.ws_ctrl[1], 1u) == gridDim.x - 1) {
            p.ws_ctrl[0] = 0u;  // the last CTA leaves the tile counter zeroed
            p.ws_ctrl[1] = 0u;
        }
    }
    (void)kBonus;
}

}  // namespace spec
