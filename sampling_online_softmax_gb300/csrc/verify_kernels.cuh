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
// How (GB300 design):
//   * A "unit" is one (sequence, position): target row i together with draft
//     row i for linear sampling, otherwise one target row.  Units are numbered
//     position-major (every sequence's position 0, then position 1, ...), so
//     when a position is processed the earlier positions of its sequence have
//     usually finished.
//   * Persistent thread-block clusters of C CTAs (grid = the clusters that fit
//     at once); cluster g takes units g, g + G, g + 2G, ...  CTA r of a
//     cluster owns the vocabulary slice [r*L, (r+1)*L) of every row.
//   * Each CTA has a control warp (warp 0) and eight compute warps.  The
//     control warp keeps a ring of NSTAGE shared-memory stages full: 1-D bulk
//     copies (cp.async.bulk; one mbarrier per stage) of the CTA's slices of
//     the unit NSTAGE-1 ahead, so HBM keeps streaming while the current unit
//     is reduced and decided.  Slice ends that are not 16-byte aligned are
//     loaded element-wise; padding is -inf.
//   * Compute warps reduce their stage (max and exp2-sum per thread, or
//     max / argmax); the control warp merges the warps, and the cluster's CTAs
//     merge through distributed shared memory after one cluster barrier per
//     unit (partials double-buffered by unit parity), so every CTA holds the
//     same row statistics and takes the same decision.
//   * A rejected position -- unless an earlier rejection of its sequence has
//     already been published -- and the tail position draw their candidate
//     extra token from the rows still resident in the cluster's shared memory:
//     per-16-byte-group weights, exact int64 fixed-point sums (units of
//     2^-52) scanned across the CTA and then across the cluster, and one
//     thread walks its segment.  No second pass over HBM.
//   * The publishing CTA's control warp writes the unit's result to the
//     workspace and bumps a per-sequence counter (acq_rel atomic); the last
//     unit of a sequence to finish emits the tokens (a warp ballot finds the
//     first rejection) and zeroes the sequence's workspace entries.
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
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr int kBarStageFree = 1;                // compute warps hand a stage back to the control warp
constexpr int kBarCompute = 2;                  // barrier among the compute warps only

enum Mode : int {
    kLinearSample = 0,
    kLinearGreedy = 1,
    kTreeGreedy = 2,
    kBonusSample = 3,
    kBonusGreedy = 4,
};

struct Params {
    const unsigned char *target;   // [B, t_rows, V]
    const unsigned char *draft;    // [B, K, V] (sampling) or null
    int B, K, V;
    int t_rows;                    // target rows per sequence: K+1 (linear), N (tree)
    int units_per_seq;             // K+1 (linear), N (tree), 1 (extra token alone)
    int n_units;                   // B * units_per_seq
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
    uint32_t *ws_counter;          // [B]   units finished per sequence
    int32_t *ws_first;             // [B]   K + 1 - (earliest published rejection), 0 if none
    int32_t *ws_acc;               // [B*K] accept bits
    int32_t *ws_val;               // [B*units_per_seq] candidate token / argmax
    int slice_len;                 // elements per CTA slice (multiple of 16/eb)
    int row_buf_bytes;             // shared bytes per row buffer in a stage
    int stage_bytes;               // shared bytes per stage
    int nstage;                    // stages in the ring (1..kMaxStages)
};

struct __align__(16) Ctl {
    unsigned long long full[kMaxStages];
    long long incl[kComputeThreads];     // inclusive scan of per-thread segment weights
    long long warp_tot[kComputeWarps];
    long long part_w[2];                 // CTA weight total, by unit parity (read by the cluster)
    long long tlocal;                    // target cumulative weight inside the owner CTA
    float warp_m[kMaxRows][kComputeWarps];
    float warp_s[kMaxRows][kComputeWarps];
    int warp_i[kMaxRows][kComputeWarps];
    float part_m[2][kMaxRows];           // CTA partial statistics, by unit parity (read by the cluster)
    float part_s[2][kMaxRows];
    int part_i[2][kMaxRows];
    int part_flag[2];
    float M[kMaxRows];                   // merged statistics, identical in every CTA
    float S[kMaxRows];
    int A[kMaxRows];
    float px, qx, thr;
    int accept, do_resid, tail_weights, retry, owner_rank, publisher;
    int warp_first[kComputeWarps];
    int cand;
    int timed_out;
    uint32_t flags;
    int st_b[kMaxStages], st_pos[kMaxStages], st_nrows[kMaxStages];
};

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

__device__ __forceinline__ void bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_arrive(int id, int n) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
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

// ---------------------------------------------------------------- elements
template <int EB>
struct Elt;

template <>
struct Elt<4> {
    static constexpr int G = 4;  // elements per 16-byte granule
    __device__ __forceinline__ static void unpack(const uint4 &w, float (&v)[G]) {
        v[0] = __uint_as_float(w.x);
        v[1] = __uint_as_float(w.y);
        v[2] = __uint_as_float(w.z);
        v[3] = __uint_as_float(w.w);
    }
    __device__ __forceinline__ static float load(const unsigned char *p) {
        return *reinterpret_cast<const float *>(p);
    }
    __device__ __forceinline__ static void store_neg_inf(unsigned char *p) {
        *reinterpret_cast<uint32_t *>(p) = 0xff800000u;
    }
    __device__ __forceinline__ static void copy(unsigned char *dst, const unsigned char *src) {
        *reinterpret_cast<uint32_t *>(dst) = __ldg(reinterpret_cast<const uint32_t *>(src));
    }
    __device__ __forceinline__ static float granule_max(const unsigned char *buf, int g0, int g1, int step) {
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
    __device__ __forceinline__ static void store_neg_inf(unsigned char *p) {
        *reinterpret_cast<uint16_t *>(p) = 0xff80u;
    }
    __device__ __forceinline__ static void copy(unsigned char *dst, const unsigned char *src) {
        *reinterpret_cast<uint16_t *>(dst) = __ldg(reinterpret_cast<const unsigned short *>(src));
    }
    __device__ __forceinline__ static float granule_max(const unsigned char *buf, int g0, int g1, int step) {
        uint32_t m = 0xff80ff80u;  // (-inf, -inf)
        for (int g = g0; g < g1; g += step) {
            const uint4 w = *reinterpret_cast<const uint4 *>(buf + 16 * g);
            m = ptx::bmax2(m, ptx::bmax2(ptx::bmax2(w.x, w.y), ptx::bmax2(w.z, w.w)));
        }
        return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    }
};

// ------------------------------------------------------------ row geometry
// A CTA's slice [s0, s1) of one row, mirrored in shared memory granule by
// granule: buffer byte k holds global byte (glo + k), glo = 16-byte floor of
// the slice start.  Granules [hg, hg + nfull) arrive by bulk copy; partial
// granules at either end are filled element-wise, with -inf outside the slice.
struct RowGeo {
    const unsigned char *glo;  // global address of buffer byte 0
    unsigned char *buf;        // shared buffer (generic pointer)
    int ngran;                 // granules in the buffer
    int hg;                    // 1 if granule 0 is partial (and there are full granules)
    int nfull;                 // granules copied in bulk
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

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity) {
    for (uint32_t it = 0; it < kWaitLimit; ++it)
        if (ptx::mbar_try_wait(bar, parity)) return true;
    return false;
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
// Weights of the G elements of target granule g:
//   pair (residual):  max(0, p_v - q_v) = max(0, 2^((t-Mt)c)/St - 2^((d-Md)c)/Sd)
//   tail:             p_v = 2^((t - Mt) c) / St
// Explicit _rn intrinsics keep the two evaluations of a weight bit-identical.
template <int EB>
__device__ __forceinline__ void granule_weights(const RowGeo &gt, const RowGeo &gd, bool pair, bool same_phase,
                                                int g, int s0, int s1, float Mt, float Md, float invSt,
                                                float invSd, float c, float (&w)[Elt<EB>::G]) {
    constexpr int G = Elt<EB>::G;
    float t[G];
    Elt<EB>::unpack(*reinterpret_cast<const uint4 *>(gt.buf + 16 * g), t);
    if (!pair) {
#pragma unroll
        for (int k = 0; k < G; ++k) w[k] = __fmul_rn(ptx::ex2(__fmul_rn(__fsub_rn(t[k], Mt), c)), invSt);
        return;
    }
    float d[G];
    if (same_phase) {
        Elt<EB>::unpack(*reinterpret_cast<const uint4 *>(gd.buf + 16 * g), d);
    } else {
#pragma unroll
        for (int k = 0; k < G; ++k) {
            const int v = gt.vbase + g * G + k;
            d[k] = (v >= s0 && v < s1) ? Elt<EB>::load(gd.buf + (v - gd.vbase) * EB) : neg_inf();
        }
    }
#pragma unroll
    for (int k = 0; k < G; ++k) {
        const float pv = __fmul_rn(ptx::ex2(__fmul_rn(__fsub_rn(t[k], Mt), c)), invSt);
        const float qv = __fmul_rn(ptx::ex2(__fmul_rn(__fsub_rn(d[k], Md), c)), invSd);
        w[k] = fmaxf(0.0f, __fsub_rn(pv, qv));
    }
}

// ---------------------------------------------------------- unit layout
struct UnitRows {
    int nrows;
    const unsigned char *row[kMaxRows];
};

// Rows of unit (b, pos); pos < 0 marks an invalid unit (no rows).
template <int EB, int MODE>
__device__ __forceinline__ UnitRows unit_rows(const Params &p, int b, int pos) {
    constexpr bool kSample = (MODE == kLinearSample || MODE == kBonusSample);
    UnitRows ur;
    ur.nrows = (pos < 0) ? 0 : ((kSample && pos < p.K) ? 2 : 1);
    const size_t row_bytes = static_cast<size_t>(p.V) * EB;
    ur.row[0] = p.target;
    if (ur.nrows >= 1) ur.row[0] = p.target + (static_cast<size_t>(b) * p.t_rows + pos) * row_bytes;
    ur.row[1] = ur.row[0];
    if (ur.nrows == 2) ur.row[1] = p.draft + (static_cast<size_t>(b) * p.K + pos) * row_bytes;
    return ur;
}

// Control warp: fill stage `s` with this CTA's slices of unit u (position-major:
// u = pos * B + b; the extra-token-alone mode reads pos from accept_len).
template <int EB, int MODE>
__device__ void prefetch_unit(const Params &p, Ctl &ctl, unsigned char *dsm, int s, int u, int s0, int s1,
                              int lane) {
    constexpr bool kBonus = (MODE == kBonusSample || MODE == kBonusGreedy);
    int pos = u / p.B;
    const int b = u - pos * p.B;
    if (kBonus) {
        pos = p.accept_len_in[b];
        if (pos < 0 || pos > p.K) pos = -1;  // invalid: no rows; the publisher reports it
    }
    const UnitRows ur = unit_rows<EB, MODE>(p, b, pos);
    unsigned char *stage = dsm + static_cast<size_t>(s) * p.stage_bytes;
    const uint32_t bar = ptx::smem_addr(&ctl.full[s]);
    RowGeo geo[kMaxRows];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) geo[r] = make_geo<EB>(ur.row[r], s0, s1, stage + r * p.row_buf_bytes);
    if (lane == 0) {
        ctl.st_b[s] = b;
        ctl.st_pos[s] = pos;
        ctl.st_nrows[s] = ur.nrows;
        uint32_t bytes = 0;
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r)
            if (r < ur.nrows) bytes += static_cast<uint32_t>(geo[r].nfull) * 16u;
        fence_proxy_async();  // earlier generic reads of this stage come before the async writes
        ptx::mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) {
            if (r >= ur.nrows || geo[r].nfull == 0) continue;
            const int off = 16 * geo[r].hg;
            ptx::bulk_g2s(ptx::smem_addr(geo[r].buf + off), geo[r].glo + off,
                          static_cast<uint32_t>(geo[r].nfull) * 16u, bar);
        }
    }
    // ragged ends element-wise (at most 16 slots per row): lanes 0..15 row 0, 16..31 row 1
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

// Control warp of the publishing CTA: write the unit's result, count the unit,
// and if it was the sequence's last one, emit the sequence.
template <int EB, int MODE>
__device__ void publish(const Params &p, Ctl &ctl, int s, unsigned char *stage, int lane) {
    constexpr bool kSample = (MODE == kLinearSample || MODE == kBonusSample);
    constexpr bool kBonus = (MODE == kBonusSample || MODE == kBonusGreedy);
    const int b = ctl.st_b[s];
    const int pos = ctl.st_pos[s];
    const int K = p.K;
    const int U = p.units_per_seq;
    int last = 0;
    if (lane == 0) {
        uint32_t fl = ctl.flags;
        if (MODE == kLinearSample) {
            if (pos < K) {
                p.ws_acc[static_cast<size_t>(b) * K + pos] = ctl.accept;
                if (p.probs) {
                    float *pr = p.probs + (static_cast<size_t>(b) * K + pos) * 3;
                    pr[0] = ctl.px;
                    pr[1] = ctl.qx;
                    pr[2] = ctl.thr;
                }
            }
            if (ctl.do_resid) p.ws_val[static_cast<size_t>(b) * U + pos] = ctl.cand;
        } else if (MODE == kLinearGreedy || MODE == kTreeGreedy) {
            p.ws_val[static_cast<size_t>(b) * U + pos] = ctl.A[0];
        } else {
            if (pos < 0) fl |= SPEC_DEV_BAD_LENGTH;
            p.bonus_token[b] = (pos < 0) ? -1 : (kSample ? ctl.cand : ctl.A[0]);
        }
        if (fl) atomicOr(p.status, fl);
        if (!kBonus) last = (atom_add_acq_rel(&p.ws_counter[b], 1u) == static_cast<unsigned>(U - 1)) ? 1 : 0;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __syncwarp();
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
        // leave this sequence's workspace entries zero for the next call,
        // whatever (B, K) that call uses the workspace with
        __syncwarp();
        if (MODE == kLinearSample)
            for (int i = lane; i < K; i += 32) p.ws_acc[static_cast<size_t>(b) * K + i] = 0;
        for (int i = lane; i < U; i += 32) p.ws_val[static_cast<size_t>(b) * U + i] = 0;
        if (lane == 0) {
            p.ws_first[b] = 0;
            p.ws_counter[b] = 0u;
        }
    } else if (MODE == kTreeGreedy) {
        // stage the tree of this sequence in the current stage buffer (no longer read)
        const int N = U;
        int *par_s = reinterpret_cast<int *>(stage);
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
            p.ws_counter[b] = 0u;
        }
        for (int i = depth + 1 + lane; i <= D; i += 32) {
            ot[i] = -1;
            pn[i] = -1;
        }
        __syncwarp();
    }
}

// ================================================================ kernel
template <int EB, int MODE>
__global__ void __launch_bounds__(kThreads, 2) spec_verify_kernel(const Params p) {
    constexpr bool kSample = (MODE == kLinearSample || MODE == kBonusSample);
    constexpr int G = Elt<EB>::G;

    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ Ctl ctl;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const bool is_ctrl = (warp == 0);
    const int ct = tid - 32;  // compute-thread index (compute warps only)
    const int cw = warp - 1;  // compute-warp index
    const uint32_t crank = ptx::cluster_ctarank();
    const uint32_t csize = ptx::cluster_nctarank();
    const int cid = static_cast<int>(ptx::cluster_id_x());
    const int ncl = static_cast<int>(gridDim.x / csize);
    const int V = p.V, K = p.K;
    const float c = p.c;
    const int nstage = p.nstage;
    const int n_my = (p.n_units > cid) ? (p.n_units - cid + ncl - 1) / ncl : 0;
    const int s0 = min(V, static_cast<int>(crank) * p.slice_len);
    const int s1 = min(V, s0 + p.slice_len);
    float *wgs = reinterpret_cast<float *>(dsm + static_cast<size_t>(nstage) * p.stage_bytes);

    if (tid == 0) {
        for (int s = 0; s < nstage; ++s) ptx::mbar_init(ptx::smem_addr(&ctl.full[s]), 2);
        ptx::fence_mbar_init();
        ctl.flags = 0;
        ctl.timed_out = 0;
    }
    __syncthreads();
    if (is_ctrl)
        for (int it = 0; it < nstage - 1 && it < n_my; ++it)
            prefetch_unit<EB, MODE>(p, ctl, dsm, it % nstage, cid + it * ncl, s0, s1, lane);

    for (int it = 0; it < n_my; ++it) {
        const int s = it % nstage;
        const uint32_t ph = static_cast<uint32_t>(it / nstage) & 1u;
        const int slot = it & 1;
        unsigned char *stage = dsm + static_cast<size_t>(s) * p.stage_bytes;

        // ---- control warp: refill the ring, fetch this unit's scalars
        int x = -1;
        float tx = 0.f, dx = 0.f, ua = 0.f, ubv = 0.f;
        int early_seen = 0;
        if (is_ctrl) {
            const int ahead = it + nstage - 1;
            if (ahead < n_my) {
                if (it >= 1) bar_sync(kBarStageFree, kThreads);  // compute warps are done with that stage
                prefetch_unit<EB, MODE>(p, ctl, dsm, ahead % nstage, cid + ahead * ncl, s0, s1, lane);
            }
            if (lane == 0) {
                const int b = ctl.st_b[s];
                const int pos = ctl.st_pos[s];
                if (MODE == kLinearSample && pos < K) {
                    const UnitRows ur = unit_rows<EB, MODE>(p, b, pos);
                    x = p.tokens[static_cast<size_t>(b) * K + pos];
                    ua = p.u_accept[static_cast<size_t>(b) * K + pos];
                    if (x >= 0 && x < V) {
                        tx = Elt<EB>::load(ur.row[0] + static_cast<size_t>(x) * EB);
                        dx = Elt<EB>::load(ur.row[1] + static_cast<size_t>(x) * EB);
                    }
                }
                if (kSample && p.u_bonus && pos >= 0) ubv = p.u_bonus[b];
                if (MODE == kLinearSample) {
                    const int enc = ld_relaxed(&p.ws_first[b]);
                    early_seen = (enc != 0 && (K + 1 - enc) < pos) ? 1 : 0;
                }
            }
        }

        // ---- compute warps: row statistics of the stage
        if (!is_ctrl) {
            if (!wait_bar(ptx::smem_addr(&ctl.full[s]), ph)) ctl.timed_out = 1;
            const int nrows = ctl.st_nrows[s];
            const UnitRows ur = unit_rows<EB, MODE>(p, ctl.st_b[s], ctl.st_pos[s]);
#pragma unroll
            for (int r = 0; r < kMaxRows; ++r) {
                if (r >= nrows) continue;
                const RowGeo g = make_geo<EB>(ur.row[r], s0, s1, stage + r * p.row_buf_bytes);
                if (kSample) {
                    const float mp = Elt<EB>::granule_max(g.buf, ct, g.ngran, kComputeThreads);
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
                    float m = mp, sum = sa + sb;
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1)
                        merge_ms(m, sum, __shfl_xor_sync(0xffffffffu, m, off),
                                 __shfl_xor_sync(0xffffffffu, sum, off), c);
                    if (lane == 0) {
                        ctl.warp_m[r][cw] = m;
                        ctl.warp_s[r][cw] = sum;
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
                        ctl.warp_m[r][cw] = bv;
                        ctl.warp_i[r][cw] = bi;
                    }
                }
            }
        }
        __syncthreads();

        // ---- control warp: CTA partial; cluster merge; decision
        const int nrows_u = ctl.st_nrows[s];
        if (is_ctrl) {
#pragma unroll
            for (int r = 0; r < kMaxRows; ++r) {
                if (r >= nrows_u) continue;
                float m = lane < kComputeWarps ? ctl.warp_m[r][lane] : neg_inf();
                if (kSample) {
                    float sum = lane < kComputeWarps ? ctl.warp_s[r][lane] : 0.f;
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1)
                        merge_ms(m, sum, __shfl_xor_sync(0xffffffffu, m, off),
                                 __shfl_xor_sync(0xffffffffu, sum, off), c);
                    if (lane == 0) {
                        ctl.part_m[slot][r] = m;
                        ctl.part_s[slot][r] = sum;
                    }
                } else {
                    int i = lane < kComputeWarps ? ctl.warp_i[r][lane] : INT_MAX;
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1)
                        merge_vi(m, i, __shfl_xor_sync(0xffffffffu, m, off), __shfl_xor_sync(0xffffffffu, i, off));
                    if (lane == 0) {
                        ctl.part_m[slot][r] = m;
                        ctl.part_i[slot][r] = i;
                    }
                }
            }
            if (lane == 0) ctl.part_flag[slot] = early_seen;
        }
        ptx::cluster_sync();
        if (is_ctrl) {
            int early = 0;
            if (lane < static_cast<int>(csize))
                early = ptx::ld_dsmem_s32(ptx::mapa(ptx::smem_addr(&ctl.part_flag[slot]), lane));
            early = __any_sync(0xffffffffu, early != 0) ? 1 : 0;
#pragma unroll
            for (int r = 0; r < kMaxRows; ++r) {
                if (r >= nrows_u) continue;
                float m = neg_inf(), sum = 0.f;
                int i = INT_MAX;
                if (lane < static_cast<int>(csize)) {
                    m = ptx::ld_dsmem_f32(ptx::mapa(ptx::smem_addr(&ctl.part_m[slot][r]), lane));
                    if (kSample)
                        sum = ptx::ld_dsmem_f32(ptx::mapa(ptx::smem_addr(&ctl.part_s[slot][r]), lane));
                    else
                        i = ptx::ld_dsmem_s32(ptx::mapa(ptx::smem_addr(&ctl.part_i[slot][r]), lane));
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    if (kSample)
                        merge_ms(m, sum, __shfl_xor_sync(0xffffffffu, m, off),
                                 __shfl_xor_sync(0xffffffffu, sum, off), c);
                    else
                        merge_vi(m, i, __shfl_xor_sync(0xffffffffu, m, off), __shfl_xor_sync(0xffffffffu, i, off));
                }
                if (lane == 0) {
                    ctl.M[r] = m;
                    ctl.S[r] = sum;
                    ctl.A[r] = i;
                }
            }
            __syncwarp();
            if (lane == 0) {
                const int pos = ctl.st_pos[s];
                const int b = ctl.st_b[s];
                uint32_t fl = 0;
                int do_resid = 0, accept = 1, tailw = 0;
                bool finite = true;
                if (kSample) {
                    for (int r = 0; r < nrows_u; ++r)
                        if (!(isfinite(ctl.M[r]) && isfinite(ctl.S[r]) && ctl.S[r] > 0.f)) finite = false;
                    if (!finite) fl |= SPEC_DEV_NONFINITE;
                } else if (nrows_u > 0 && ctl.A[0] == INT_MAX) {
                    fl |= SPEC_DEV_NONFINITE;  // no element above -inf
                    ctl.A[0] = 0;
                }
                if (MODE == kLinearSample) {
                    if (pos < K) {
                        float px = 0.f, qx = 0.f, thr = 0.f;
                        if (x < 0 || x >= V) {
                            fl |= SPEC_DEV_BAD_TOKEN;
                            accept = 0;
                        } else {
                            const float Mt = ctl.M[0], St = ctl.S[0], Md = ctl.M[1], Sd = ctl.S[1];
                            px = ptx::ex2((tx - Mt) * c) / St;
                            qx = ptx::ex2((dx - Md) * c) / Sd;
                            const float ratio = ptx::ex2(((tx - Mt) - (dx - Md)) * c) * (Sd / St);
                            thr = fminf(1.0f, ratio);
                            accept = (ua < thr) ? 1 : 0;
                        }
                        ctl.px = px;
                        ctl.qx = qx;
                        ctl.thr = thr;
                        // later positions of this sequence may skip drawing a candidate
                        if (!accept && crank == 0) atomicMax(&p.ws_first[b], K + 1 - pos);
                        do_resid = (!accept && p.u_bonus != nullptr && !early) ? 1 : 0;
                    } else {
                        do_resid = (p.u_bonus != nullptr && !early) ? 1 : 0;
                        tailw = 1;
                    }
                } else if (MODE == kBonusSample) {
                    do_resid = (pos >= 0) ? 1 : 0;
                    tailw = (pos == K) ? 1 : 0;
                }
                if (!finite) do_resid = 0;
                ctl.do_resid = do_resid;
                ctl.tail_weights = tailw;
                ctl.accept = accept;
                ctl.flags = fl;
                ctl.publisher = 0;
                ctl.cand = 0;
            }
        }
        __syncthreads();

        if (kSample && ctl.do_resid) {
            // ================= extra token from the resident rows =================
            const UnitRows ur = unit_rows<EB, MODE>(p, ctl.st_b[s], ctl.st_pos[s]);
            const RowGeo gt = make_geo<EB>(ur.row[0], s0, s1, stage);
            const RowGeo gd = make_geo<EB>(ur.row[1], s0, s1, stage + p.row_buf_bytes);
            const bool same_phase =
                ((reinterpret_cast<uintptr_t>(ur.row[0]) - reinterpret_cast<uintptr_t>(ur.row[1])) & 15u) == 0;
            const float Mt = ctl.M[0], Md = ctl.M[1];
            const float invSt = 1.0f / ctl.S[0];
            const float invSd = (nrows_u == 2) ? 1.0f / ctl.S[1] : 0.f;
            const int ngran = gt.ngran;
            const int seg = (ngran + kComputeThreads - 1) / kComputeThreads;
            const int sg0 = min(ngran, max(ct, 0) * seg);
            const int sg1 = min(ngran, sg0 + seg);
            long long segq = 0, incl = 0;
            for (;;) {
                const bool pair = (ctl.tail_weights == 0);
                if (!is_ctrl) {
                    // weights per 16-byte group, then exact per-thread segment sums in element order
                    for (int g = ct; g < ngran; g += kComputeThreads) {
                        float w[G];
                        granule_weights<EB>(gt, gd, pair, same_phase, g, s0, s1, Mt, Md, invSt, invSd, c, w);
                        float sw = 0.f;
#pragma unroll
                        for (int k = 0; k < G; ++k) sw += w[k];
                        wgs[g] = sw;
                    }
                    bar_sync(kBarCompute, kComputeThreads);
                    segq = 0;
                    for (int g = sg0; g < sg1; ++g) segq += fixq(wgs[g]);
                    long long xs = segq;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const long long y = __shfl_up_sync(0xffffffffu, xs, off);
                        if (lane >= off) xs += y;
                    }
                    if (lane == 31) ctl.warp_tot[cw] = xs;
                    bar_sync(kBarCompute, kComputeThreads);
                    long long offs = 0;
                    for (int w2 = 0; w2 < cw; ++w2) offs += ctl.warp_tot[w2];
                    incl = offs + xs;
                    ctl.incl[ct] = incl;
                    if (ct == kComputeThreads - 1) ctl.part_w[slot] = incl;
                }
                __syncthreads();
                ptx::cluster_sync();
                if (is_ctrl) {
                    // cluster-wide cumulative weight, rank by rank (exact integers)
                    const long long wk = (lane < static_cast<int>(csize))
                                             ? ptx::ld_dsmem_s64(ptx::mapa(ptx::smem_addr(&ctl.part_w[slot]), lane))
                                             : 0;
                    long long tot = 0;
                    for (int k = 0; k < static_cast<int>(csize); ++k) tot += __shfl_sync(0xffffffffu, wk, k);
                    const float ub = __shfl_sync(0xffffffffu, ubv, 0);
                    const long long target = static_cast<long long>(static_cast<double>(ub) * static_cast<double>(tot));
                    long long acc = 0, pre = 0;
                    int owner = -1;
                    for (int k = 0; k < static_cast<int>(csize); ++k) {
                        const long long w = __shfl_sync(0xffffffffu, wk, k);
                        if (owner < 0 && acc + w > target) {
                            owner = k;
                            pre = acc;
                        }
                        acc += w;
                    }
                    if (lane == 0) {
                        const int retry = (tot <= 0 && ctl.tail_weights == 0) ? 1 : 0;
                        ctl.retry = retry;
                        if (retry) {  // the residual vanished through rounding: draw from p_j instead
                            ctl.tail_weights = 1;
                            ctl.flags |= SPEC_DEV_ZERO_RESIDUAL;
                        }
                        ctl.owner_rank = owner;
                        ctl.tlocal = target - pre;
                        ctl.publisher = owner < 0 ? 0 : owner;
                    }
                }
                __syncthreads();
                if (!ctl.retry) break;
                ptx::cluster_sync();  // every CTA has read this parity's part_w before it is rewritten
            }
            const bool pair = (ctl.tail_weights == 0);
            if (static_cast<int>(crank) == ctl.owner_rank) {
                if (!is_ctrl) {
                    // the first thread whose inclusive weight exceeds the target owns the token
                    const long long tl = ctl.tlocal;
                    const unsigned bal = __ballot_sync(0xffffffffu, segq > 0 && incl > tl);
                    if (lane == 0) ctl.warp_first[cw] = bal ? __ffs(bal) - 1 : 32;
                    bar_sync(kBarCompute, kComputeThreads);
                    int owner_t = -1;
                    for (int w2 = 0; w2 < kComputeWarps && owner_t < 0; ++w2)
                        if (ctl.warp_first[w2] < 32) owner_t = w2 * 32 + ctl.warp_first[w2];
                    if (ct == owner_t) {
                        long long acc = (ct == 0) ? 0 : ctl.incl[ct - 1];
                        int gsel = -1;
                        for (int g = sg0; g < sg1; ++g) {
                            const long long q = fixq(wgs[g]);
                            if (q > 0 && acc + q > tl) {
                                gsel = g;
                                break;
                            }
                            acc += q;
                        }
                        int token = 0;
                        if (gsel >= 0) {
                            // same weights, same fp32 summation order as the group sum
                            float w[G];
                            granule_weights<EB>(gt, gd, pair, same_phase, gsel, s0, s1, Mt, Md, invSt, invSd, c, w);
                            float cum = 0.f;
                            int ksel = G - 1;
                            for (int k = 0; k < G; ++k) {
                                cum += w[k];
                                if (acc + fixq(cum) > tl) {
                                    ksel = k;
                                    break;
                                }
                            }
                            token = gt.vbase + gsel * G + ksel;
                        }
                        ctl.cand = token;
                    }
                }
                __syncthreads();
            }
        }

        // ---- the compute warps are done with this stage; publish
        if (!is_ctrl && it + nstage < n_my) bar_arrive(kBarStageFree, kThreads);
        if (is_ctrl && static_cast<int>(crank) == ctl.publisher) publish<EB, MODE>(p, ctl, s, stage, lane);
    }

    // no CTA leaves while a peer may still read its control block
    ptx::cluster_sync();
    if (tid == 0 && ctl.timed_out) {
        atomicOr(p.status, SPEC_DEV_TIMEOUT);
        // wait (bounded) for copies that may still be in flight into any stage
        for (int s = 0; s < nstage && s < n_my; ++s) {
            const int last_it = s + ((n_my - 1 - s) / nstage) * nstage;
            wait_bar(ptx::smem_addr(&ctl.full[s]), static_cast<uint32_t>(last_it / nstage) & 1u);
        }
    }
}

}  // namespace spec
