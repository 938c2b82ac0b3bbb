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
//   * A "unit" is one (sequence, position) -- for linear sampling the target
//     row i together with the draft row i, otherwise one target row.  Each unit
//     is one thread-block cluster of C CTAs; CTA r of the cluster owns the
//     contiguous vocabulary slice [r*L, (r+1)*L) of every row of the unit.
//   * A CTA streams its slices from HBM exactly once with 1-D bulk copies
//     (cp.async.bulk, in four pieces per row with one mbarrier each) into its
//     own shared memory, and reduces them as the pieces land: a max pass and
//     an exp2-sum pass per piece (online-softmax merge across pieces), or a
//     max/argmax pass in greedy mode.  Ragged ends that are not 16-byte
//     aligned are loaded element by element; padding is -inf.
//   * Warp shuffles, then shared memory, reduce the CTA; the cluster merges
//     the CTAs' (max, exp-sum) or (max, index) over distributed shared memory
//     in rank order, so every CTA holds identical row statistics.
//   * A rejected position (and the tail position) draws its candidate extra
//     token right away from the rows still resident in the cluster's shared
//     memory -- no second HBM pass: per-16-byte-group weights, an fp64 scan of
//     per-thread segments, an fp64 scan across the cluster, then one thread
//     walks its segment.  The token is written into the leader CTA over DSMEM.
//   * The leader CTA of each unit publishes its result and bumps a
//     per-sequence counter; the last unit of a sequence to finish (no waiting
//     anywhere) finds the first rejection with a warp ballot, writes the
//     emitted tokens, and zeroes the sequence's counter and entries, so the
//     workspace is all zero again after every call.
//   * No tensor cores (nothing here is a contraction); every wait is bounded
//     and reports SPEC_DEV_TIMEOUT instead of trapping.
#pragma once

#include <climits>
#include <cstdint>

#include "ptx.cuh"
#include "spec_verify.h"

namespace spec {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPieces = 4;            // bulk copies (and mbarriers) per row slice
constexpr int kMaxRows = 2;           // rows per unit: target, draft
constexpr uint32_t kWaitLimit = 1u << 22;

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
    int32_t *ws_acc;               // [B*K] accept bits
    int32_t *ws_val;               // [B*units_per_seq] candidate token / argmax
    int slice_len;                 // elements per CTA slice (multiple of 16/eb)
    int row_buf_bytes;             // dynamic shared bytes per row buffer
};

struct __align__(16) Ctl {
    unsigned long long mbar[kMaxRows][kPieces];
    double incl[kThreads];         // inclusive scan of per-thread segment weights
    double warp_tot[kWarps];
    double part_w;                 // this CTA's total weight (read by the cluster)
    double tlocal;                 // target cumulative weight inside the owner CTA
    float warp_m[kMaxRows][kWarps];
    float warp_s[kMaxRows][kWarps];
    int warp_i[kMaxRows][kWarps];
    float part_m[kMaxRows];        // this CTA's partial statistics (read by the cluster)
    float part_s[kMaxRows];
    int part_i[kMaxRows];
    float M[kMaxRows];             // merged statistics, identical in every CTA
    float S[kMaxRows];
    int A[kMaxRows];
    float px, qx, thr, ub;
    int warp_first[kWarps];
    int warp_last[kWarps];
    int owner_rank;
    int fallback;
    int do_resid;
    int accept;
    int cand;                      // extra-token candidate, written into rank 0 over DSMEM
    int is_last;
    uint32_t flags;
};

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

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
    // max over the thread's granules g = gstart, gstart + kThreads, ... < gend
    __device__ __forceinline__ static float granule_max(const unsigned char *buf, int gstart, int gend) {
        float m = neg_inf();
        for (int g = gstart; g < gend; g += kThreads) {
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
    __device__ __forceinline__ static float granule_max(const unsigned char *buf, int gstart, int gend) {
        uint32_t m = 0xff80ff80u;  // (-inf, -inf)
        for (int g = gstart; g < gend; g += kThreads) {
            const uint4 w = *reinterpret_cast<const uint4 *>(buf + 16 * g);
            m = ptx::bmax2(m, ptx::bmax2(ptx::bmax2(w.x, w.y), ptx::bmax2(w.z, w.w)));
        }
        return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    }
};

// ------------------------------------------------------------ row geometry
// A CTA's slice [s0, s1) of one row, mirrored in shared memory granule by
// granule: buffer byte k holds global byte (glo + k), glo = 16-byte floor of
// the slice start.  Granules [hg, hg + nfull) arrive by bulk copy; the partial
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

// First granule of piece q (q = kPieces gives the end).
__device__ __forceinline__ int piece_begin(const RowGeo &g, int q) {
    if (q == 0) return 0;
    if (q == kPieces) return g.ngran;
    return g.hg + static_cast<int>((static_cast<long long>(g.nfull) * q) / kPieces);
}

__device__ __forceinline__ bool wait_bar(uint32_t bar) {
    for (uint32_t it = 0; it < kWaitLimit; ++it)
        if (ptx::mbar_try_wait(bar, 0)) return true;
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
//   tail:             2^((t - Mt) c)    (unnormalised p_v)
// Explicit _rn intrinsics keep the two evaluations of a weight bit-identical.
template <int EB>
__device__ __forceinline__ void granule_weights(const RowGeo &gt, const RowGeo &gd, bool pair,
                                                bool same_phase, int g, int s0, int s1, float Mt,
                                                float Md, float invSt, float invSd, float c,
                                                float (&w)[Elt<EB>::G]) {
    constexpr int G = Elt<EB>::G;
    float t[G];
    Elt<EB>::unpack(*reinterpret_cast<const uint4 *>(gt.buf + 16 * g), t);
    if (!pair) {
#pragma unroll
        for (int k = 0; k < G; ++k) w[k] = ptx::ex2(__fmul_rn(__fsub_rn(t[k], Mt), c));
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

// ================================================================ kernel
template <int EB, int MODE>
__global__ void __launch_bounds__(kThreads, 3) spec_unit_kernel(const Params p) {
    constexpr bool kSample = (MODE == kLinearSample || MODE == kBonusSample);
    constexpr bool kBonus = (MODE == kBonusSample || MODE == kBonusGreedy);
    constexpr int G = Elt<EB>::G;
    constexpr int kRowsAlloc = kSample ? 2 : 1;

    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ Ctl ctl;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint32_t crank = ptx::cluster_ctarank();
    const uint32_t csize = ptx::cluster_nctarank();
    const int unit = static_cast<int>(ptx::cluster_id_x());
    const int V = p.V;
    const int K = p.K;
    const float c = p.c;

    // ---- which sequence / position this cluster handles
    int b, pos;
    if (kBonus) {
        b = unit;
        pos = p.accept_len_in[b];
        if (pos < 0 || pos > K) {  // same value in every CTA: the cluster leaves together
            if (crank == 0 && tid == 0) {
                p.bonus_token[b] = -1;
                atomicOr(p.status, SPEC_DEV_BAD_LENGTH);
            }
            return;
        }
    } else {
        b = unit / p.units_per_seq;
        pos = unit - b * p.units_per_seq;
    }
    const int nrows = (kSample && pos < K) ? 2 : 1;
    const size_t row_bytes = static_cast<size_t>(V) * EB;
    const unsigned char *rowp[kMaxRows];
    rowp[0] = p.target + (static_cast<size_t>(b) * p.t_rows + pos) * row_bytes;
    rowp[1] = (nrows == 2) ? p.draft + (static_cast<size_t>(b) * K + pos) * row_bytes : rowp[0];

    const int s0 = min(V, static_cast<int>(crank) * p.slice_len);
    const int s1 = min(V, s0 + p.slice_len);
    RowGeo geo[kMaxRows];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) geo[r] = make_geo<EB>(rowp[r], s0, s1, dsm + r * p.row_buf_bytes);

    // ---- start the bulk copies
    if (tid == 0) {
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r)
            if (r < nrows)
                for (int q = 0; q < kPieces; ++q) ptx::mbar_init(ptx::smem_addr(&ctl.mbar[r][q]), 1);
        ptx::fence_mbar_init();
        ctl.cand = 0;
        ctl.flags = 0;
    }
    __syncthreads();
    if (tid == 0) {
        for (int q = 0; q < kPieces; ++q) {
#pragma unroll
            for (int r = 0; r < kMaxRows; ++r) {
                if (r >= nrows) continue;
                const RowGeo &g = geo[r];
                const int f0 = g.hg + static_cast<int>((static_cast<long long>(g.nfull) * q) / kPieces);
                const int f1 = g.hg + static_cast<int>((static_cast<long long>(g.nfull) * (q + 1)) / kPieces);
                const uint32_t bytes = static_cast<uint32_t>(f1 - f0) * 16u;
                const uint32_t bar = ptx::smem_addr(&ctl.mbar[r][q]);
                ptx::mbar_arrive_expect_tx(bar, bytes);
                if (bytes) ptx::bulk_g2s(ptx::smem_addr(g.buf + 16 * f0), g.glo + 16 * f0, bytes, bar);
            }
        }
    }
    // ragged ends (element-wise) and padding (-inf); <= 16 slots per row
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
        if (r >= nrows) continue;
        const RowGeo &g = geo[r];
        const int head_slots = g.hg * 16 / EB;
        const int tail_first = (g.hg + g.nfull) * 16;
        const int tail_slots = (g.ngran * 16 - tail_first) / EB;
        const int e = tid - 32 * (r + 1);
        if (e >= 0 && e < head_slots + tail_slots) {
            const int off = (e < head_slots) ? e * EB : tail_first + (e - head_slots) * EB;
            if (off >= g.a0off && off < g.a1off)
                Elt<EB>::copy(g.buf + off, g.glo + off);
            else
                Elt<EB>::store_neg_inf(g.buf + off);
        }
    }
    // operands of the acceptance test, fetched while the rows stream in
    int x = -1;
    float tx = 0.f, dx = 0.f, ua = 0.f, ubv = 0.f;
    if (tid == 0) {
        if (MODE == kLinearSample && pos < K) {
            x = p.tokens[static_cast<size_t>(b) * K + pos];
            ua = p.u_accept[static_cast<size_t>(b) * K + pos];
            if (x >= 0 && x < V) {
                tx = Elt<EB>::load(rowp[0] + static_cast<size_t>(x) * EB);
                dx = Elt<EB>::load(rowp[1] + static_cast<size_t>(x) * EB);
            }
        }
        if (kSample && p.u_bonus) ubv = p.u_bonus[b];
    }
    __syncthreads();

    // ---- pass over the pieces as they land
    bool timed_out = false;
    float rm[kMaxRows], rs[kMaxRows];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
        rm[r] = neg_inf();
        rs[r] = 0.f;
    }
    float bv = neg_inf();
    int bi = INT_MAX;
    for (int q = 0; q < kPieces; ++q) {
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) {
            if (r >= nrows) continue;
            if (!wait_bar(ptx::smem_addr(&ctl.mbar[r][q]))) timed_out = true;
            const RowGeo &g = geo[r];
            const int g0 = piece_begin(g, q) + tid;
            const int g1 = piece_begin(g, q + 1);
            if (kSample) {
                const float mp = Elt<EB>::granule_max(g.buf, g0, g1);
                if (mp != neg_inf()) {
                    float sa = 0.f, sb = 0.f;
                    int gg = g0;
                    for (; gg + kThreads < g1; gg += 2 * kThreads) {
                        float va[G], vb[G];
                        Elt<EB>::unpack(*reinterpret_cast<const uint4 *>(g.buf + 16 * gg), va);
                        Elt<EB>::unpack(*reinterpret_cast<const uint4 *>(g.buf + 16 * (gg + kThreads)), vb);
#pragma unroll
                        for (int k = 0; k < G; ++k) {
                            sa += ptx::ex2((va[k] - mp) * c);
                            sb += ptx::ex2((vb[k] - mp) * c);
                        }
                    }
                    if (gg < g1) {
                        float va[G];
                        Elt<EB>::unpack(*reinterpret_cast<const uint4 *>(g.buf + 16 * gg), va);
#pragma unroll
                        for (int k = 0; k < G; ++k) sa += ptx::ex2((va[k] - mp) * c);
                    }
                    merge_ms(rm[r], rs[r], mp, sa + sb, c);
                }
            } else {
                for (int gg = g0; gg < g1; gg += kThreads) {
                    float va[G];
                    Elt<EB>::unpack(*reinterpret_cast<const uint4 *>(g.buf + 16 * gg), va);
#pragma unroll
                    for (int k = 0; k < G; ++k)
                        if (va[k] > bv) {
                            bv = va[k];
                            bi = g.vbase + gg * G + k;
                        }
                }
            }
        }
    }

    // ---- reduce the CTA: warps, then warp 0 over the warps
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
        if (r >= nrows) continue;
        if (kSample) {
            float m = rm[r], s = rs[r];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                merge_ms(m, s, __shfl_xor_sync(0xffffffffu, m, off), __shfl_xor_sync(0xffffffffu, s, off), c);
            if (lane == 0) {
                ctl.warp_m[r][warp] = m;
                ctl.warp_s[r][warp] = s;
            }
        } else {
            float v = bv;
            int i = bi;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                merge_vi(v, i, __shfl_xor_sync(0xffffffffu, v, off), __shfl_xor_sync(0xffffffffu, i, off));
            if (lane == 0) {
                ctl.warp_m[r][warp] = v;
                ctl.warp_i[r][warp] = i;
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) {
            if (r >= nrows) continue;
            if (kSample) {
                float m = lane < kWarps ? ctl.warp_m[r][lane] : neg_inf();
                float s = lane < kWarps ? ctl.warp_s[r][lane] : 0.f;
#pragma unroll
                for (int off = kWarps / 2; off > 0; off >>= 1)
                    merge_ms(m, s, __shfl_xor_sync(0xffffffffu, m, off), __shfl_xor_sync(0xffffffffu, s, off), c);
                if (lane == 0) {
                    ctl.part_m[r] = m;
                    ctl.part_s[r] = s;
                }
            } else {
                float v = lane < kWarps ? ctl.warp_m[r][lane] : neg_inf();
                int i = lane < kWarps ? ctl.warp_i[r][lane] : INT_MAX;
#pragma unroll
                for (int off = kWarps / 2; off > 0; off >>= 1)
                    merge_vi(v, i, __shfl_xor_sync(0xffffffffu, v, off), __shfl_xor_sync(0xffffffffu, i, off));
                if (lane == 0) {
                    ctl.part_m[r] = v;
                    ctl.part_i[r] = i;
                }
            }
        }
    }

    // ---- merge the cluster's partials in rank order (identical in every CTA)
    ptx::cluster_sync();
    if (warp == 0) {
#pragma unroll
        for (int r = 0; r < kMaxRows; ++r) {
            if (r >= nrows) continue;
            float m = neg_inf(), s = 0.f;
            int i = INT_MAX;
            if (lane < static_cast<int>(csize)) {
                m = ptx::ld_dsmem_f32(ptx::mapa(ptx::smem_addr(&ctl.part_m[r]), lane));
                if (kSample)
                    s = ptx::ld_dsmem_f32(ptx::mapa(ptx::smem_addr(&ctl.part_s[r]), lane));
                else
                    i = ptx::ld_dsmem_s32(ptx::mapa(ptx::smem_addr(&ctl.part_i[r]), lane));
            }
            float Mr = neg_inf(), Sr = 0.f;
            int Ar = INT_MAX;
            for (int k = 0; k < static_cast<int>(csize); ++k) {
                const float mk = __shfl_sync(0xffffffffu, m, k);
                if (kSample)
                    merge_ms(Mr, Sr, mk, __shfl_sync(0xffffffffu, s, k), c);
                else
                    merge_vi(Mr, Ar, mk, __shfl_sync(0xffffffffu, i, k));
            }
            if (lane == 0) {
                ctl.M[r] = Mr;
                ctl.S[r] = Sr;
                ctl.A[r] = Ar;
            }
        }
    }
    __syncthreads();

    // ---- per-unit decision (every CTA computes it identically)
    if (tid == 0) {
        uint32_t fl = 0;
        int do_resid = 0, accept = 1;
        if (kSample) {
            for (int r = 0; r < nrows; ++r)
                if (!(isfinite(ctl.M[r]) && isfinite(ctl.S[r]) && ctl.S[r] > 0.f)) fl |= SPEC_DEV_NONFINITE;
        } else if (ctl.A[0] == INT_MAX) {
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
                do_resid = (!accept && p.u_bonus != nullptr) ? 1 : 0;
            } else {
                do_resid = (p.u_bonus != nullptr) ? 1 : 0;
            }
        } else if (MODE == kBonusSample) {
            do_resid = 1;
        }
        ctl.do_resid = do_resid;
        ctl.accept = accept;
        ctl.ub = ubv;
        ctl.flags = fl;
    }
    __syncthreads();

    if (kSample && ctl.do_resid) {
        // ================= extra token from the resident rows =================
        const RowGeo &gt = geo[0];
        const RowGeo &gd = geo[1];
        bool pair = (nrows == 2);
        const bool same_phase =
            ((reinterpret_cast<uintptr_t>(rowp[0]) - reinterpret_cast<uintptr_t>(rowp[1])) & 15u) == 0;
        const float Mt = ctl.M[0], Md = ctl.M[1];
        const float invSt = 1.0f / ctl.S[0];
        const float invSd = pair ? 1.0f / ctl.S[1] : 0.f;
        float *wgs = reinterpret_cast<float *>(dsm + kRowsAlloc * p.row_buf_bytes);
        const int ngran = gt.ngran;
        const int seg = (ngran + kThreads - 1) / kThreads;
        const int sg0 = min(ngran, tid * seg), sg1 = min(ngran, sg0 + seg);
        double segsum = 0.0, incl = 0.0;
        for (int attempt = 0; attempt < 2; ++attempt) {
            // weights per granule, then per-thread segment sums in element order
            for (int g = tid; g < ngran; g += kThreads) {
                float w[G];
                granule_weights<EB>(gt, gd, pair, same_phase, g, s0, s1, Mt, Md, invSt, invSd, c, w);
                float s = 0.f;
#pragma unroll
                for (int k = 0; k < G; ++k) s += w[k];
                wgs[g] = s;
            }
            __syncthreads();
            segsum = 0.0;
            for (int g = sg0; g < sg1; ++g) segsum += static_cast<double>(wgs[g]);
            double xs = segsum;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const double y = __shfl_up_sync(0xffffffffu, xs, off);
                if (lane >= off) xs += y;
            }
            if (lane == 31) ctl.warp_tot[warp] = xs;
            __syncthreads();
            double offs = 0.0;
            for (int w2 = 0; w2 < warp; ++w2) offs += ctl.warp_tot[w2];
            incl = offs + xs;
            ctl.incl[tid] = incl;
            if (tid == kThreads - 1) ctl.part_w = incl;
            ptx::cluster_sync();
            // cluster-wide cumulative weight, rank by rank
            if (warp == 0) {
                const double wk = (lane < static_cast<int>(csize))
                                      ? ptx::ld_dsmem_f64(ptx::mapa(ptx::smem_addr(&ctl.part_w), lane))
                                      : 0.0;
                double tot = 0.0;
                for (int k = 0; k < static_cast<int>(csize); ++k) tot += __shfl_sync(0xffffffffu, wk, k);
                const double target = static_cast<double>(ctl.ub) * tot;
                double acc = 0.0, pre_owner = 0.0, pre_last = 0.0;
                int owner = -1, last = -1;
                for (int k = 0; k < static_cast<int>(csize); ++k) {
                    const double w = __shfl_sync(0xffffffffu, wk, k);
                    if (owner < 0 && acc + w > target) {
                        owner = k;
                        pre_owner = acc;
                    }
                    if (w > 0.0) {
                        last = k;
                        pre_last = acc;
                    }
                    acc += w;
                }
                if (lane == 0) {
                    ctl.fallback = (owner < 0) ? 1 : 0;
                    if (owner < 0) {
                        owner = last;
                        pre_owner = pre_last;
                    }
                    ctl.owner_rank = owner;
                    ctl.tlocal = target - pre_owner;
                    ctl.warp_tot[0] = tot;  // reused: cluster total
                }
            }
            __syncthreads();
            if (!(ctl.warp_tot[0] > 0.0) && pair && attempt == 0) {
                // residual vanished through rounding: draw from p_j instead
                if (tid == 0) ctl.flags |= SPEC_DEV_ZERO_RESIDUAL;
                pair = false;
                ptx::cluster_sync();  // peers may still read this CTA's part_w
                continue;
            }
            break;
        }
        // the owner CTA finds the token
        if (static_cast<int>(crank) == ctl.owner_rank) {
            const double tl = ctl.tlocal;
            const bool fb = ctl.fallback != 0;
            const bool pred = !fb && segsum > 0.0 && incl > tl;
            const unsigned bal = __ballot_sync(0xffffffffu, pred);
            const unsigned bal_last = __ballot_sync(0xffffffffu, segsum > 0.0);
            if (lane == 0) {
                ctl.warp_first[warp] = bal ? __ffs(bal) - 1 : 32;
                ctl.warp_last[warp] = bal_last ? 31 - __clz(bal_last) : -1;
            }
            __syncthreads();
            int owner_t = -1;
            bool lastmode = fb;
            for (int w2 = 0; w2 < kWarps && owner_t < 0; ++w2)
                if (ctl.warp_first[w2] < 32) owner_t = w2 * 32 + ctl.warp_first[w2];
            if (owner_t < 0) {
                lastmode = true;
                for (int w2 = kWarps - 1; w2 >= 0 && owner_t < 0; --w2)
                    if (ctl.warp_last[w2] >= 0) owner_t = w2 * 32 + ctl.warp_last[w2];
            }
            if (tid == owner_t) {
                double acc = (tid == 0) ? 0.0 : ctl.incl[tid - 1];
                int gsel = -1;
                if (!lastmode) {
                    for (int g = sg0; g < sg1; ++g) {
                        const double wg = static_cast<double>(wgs[g]);
                        if (wg > 0.0 && acc + wg > tl) {
                            gsel = g;
                            break;
                        }
                        acc += wg;
                    }
                }
                if (gsel < 0) {
                    lastmode = true;
                    for (int g = sg1 - 1; g >= sg0 && gsel < 0; --g)
                        if (wgs[g] > 0.f) gsel = g;
                }
                int ksel = -1;
                if (gsel >= 0) {
                    float w[G];
                    granule_weights<EB>(gt, gd, pair, same_phase, gsel, s0, s1, Mt, Md, invSt, invSd, c, w);
                    if (!lastmode) {
#pragma unroll
                        for (int k = 0; k < G; ++k) {
                            if (ksel < 0 && w[k] > 0.f && acc + static_cast<double>(w[k]) > tl) ksel = k;
                            acc += static_cast<double>(w[k]);
                        }
                    }
                    if (ksel < 0)
                        for (int k = G - 1; k >= 0 && ksel < 0; --k)
                            if (w[k] > 0.f) ksel = k;
                }
                const int token = (gsel >= 0 && ksel >= 0) ? gt.vbase + gsel * G + ksel : 0;
                ptx::st_dsmem_s32(ptx::mapa(ptx::smem_addr(&ctl.cand), 0), token);
            }
        }
        ptx::cluster_sync();  // the candidate is in rank 0; no DSMEM access after this point
    } else {
        ptx::cluster_arrive();  // done reading the peers' partials
    }

    // ---- leader: publish the unit's result; the last unit of a sequence emits
    if (crank == 0) {
        if (tid == 0) {
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
                if (ctl.do_resid) p.ws_val[static_cast<size_t>(b) * p.units_per_seq + pos] = ctl.cand;
            } else if (MODE == kLinearGreedy || MODE == kTreeGreedy) {
                p.ws_val[static_cast<size_t>(b) * p.units_per_seq + pos] = ctl.A[0];
            } else {  // extra token alone
                p.bonus_token[b] = kSample ? ctl.cand : ctl.A[0];
            }
            uint32_t fl = ctl.flags | (timed_out ? SPEC_DEV_TIMEOUT : 0u);
            if (fl) atomicOr(p.status, fl);
            int last = 0;
            if (!kBonus) {
                __threadfence();
                const unsigned old = atomicAdd(&p.ws_counter[b], 1u);
                last = (old == static_cast<unsigned>(p.units_per_seq - 1)) ? 1 : 0;
                if (last) __threadfence();
            }
            ctl.is_last = last;
        }
        __syncthreads();
        if (!kBonus && ctl.is_last) {
            if (timed_out) {  // never reuse shared memory a copy may still write
                for (int r = 0; r < nrows; ++r)
                    for (int q = 0; q < kPieces; ++q) wait_bar(ptx::smem_addr(&ctl.mbar[r][q]));
                __syncthreads();
            }
            if (MODE == kLinearSample || MODE == kLinearGreedy) {
                if (warp == 0) {
                    const bool has_bonus = p.u_bonus != nullptr;
                    int j = K;
                    for (int base = 0; base < K; base += 32) {
                        const int i = base + lane;
                        bool rej = false;
                        if (i < K) {
                            if (MODE == kLinearSample)
                                rej = __ldcg(&p.ws_acc[static_cast<size_t>(b) * K + i]) == 0;
                            else
                                rej = p.tokens[static_cast<size_t>(b) * K + i] !=
                                      __ldcg(&p.ws_val[static_cast<size_t>(b) * (K + 1) + i]);
                        }
                        const unsigned m = __ballot_sync(0xffffffffu, rej);
                        if (m) {
                            j = base + __ffs(m) - 1;
                            break;
                        }
                    }
                    const int bonus = has_bonus ? __ldcg(&p.ws_val[static_cast<size_t>(b) * (K + 1) + j]) : -1;
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
                    for (int i = lane; i <= K; i += 32) p.ws_val[static_cast<size_t>(b) * (K + 1) + i] = 0;
                    if (lane == 0) p.ws_counter[b] = 0u;
                }
            } else {  // tree walk
                const int N = p.units_per_seq;
                int *par_s = reinterpret_cast<int *>(dsm);
                int *tok_s = par_s + N;
                int *am_s = tok_s + N;
                for (int cidx = tid; cidx < N; cidx += kThreads) {
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
                __syncthreads();
                for (int cidx = tid; cidx < N; cidx += kThreads) p.ws_val[static_cast<size_t>(b) * N + cidx] = 0;
                if (warp == 0) {
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
                }
            }
        }
    }
    if (timed_out) {  // drain any copy still in flight before the CTA retires
        for (int r = 0; r < nrows; ++r)
            for (int q = 0; q < kPieces; ++q) wait_bar(ptx::smem_addr(&ctl.mbar[r][q]));
    }
    if (!(kSample && ctl.do_resid)) ptx::cluster_wait();
}

}  // namespace spec
