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
// How (GB300 design): a streaming reduction in which every warp runs its own
// pipeline and no warp waits on another while it holds unfinished work.
//   * A "unit" is one (sequence, position): target row i with draft row i for
//     linear sampling, otherwise one target row (a tree node, or the one row
//     of an extra-token-alone call).  Every row is read as S tiles, 8 KB
//     windows on the 16-byte grid of global memory (only a row's first and
//     last window can hold bytes of a neighbouring row).  Linear rows are
//     ordered position-major, tail rows last.
//   * Persistent CTAs of twelve warps, one per SM.  Small problems (at most
//     kStaticTilesPerWarp tiles per resident warp) split the tiles statically:
//     warp w reduces tiles [T*w/W, T*(w+1)/W) as runs cut at row boundaries,
//     with no counter on the issue side.  Large problems take ranges of
//     kSegTiles-tile segments from a global counter (requested one range
//     ahead; ranges shrink as the work runs out).  Every warp keeps a ring of
//     two stages filled with 1-D bulk copies (cp.async.bulk, one mbarrier and
//     one descriptor per stage).
//   * Row statistics live in the log2-scaled domain: every lane keeps a running
//     (mc, s), s = sum 2^(fma(l, c, -mc)), c = log2(e) / T, with packed fp32x2
//     FMA/ADD and one MUFU ex2 per logit; mc is only an offset, re-based on the
//     lane's max when a tile's terms grow past 2^64.  Greedy lanes keep (max,
//     lowest argmax), a tile's best group found first by a max tree.  One warp
//     reduces each whole run (or segment) and
//     publishes one partial; the runs depend only on the shape, so results do
//     not depend on timing.
//   * Publishing costs no fence: a partial (or the draft token's logit) is
//     written once per call as a non-zero 64-bit value with a relaxed store and
//     counted with a relaxed atomic.  The warp whose count completes a unit
//     reads the values, waiting for any that still read zero, decides the
//     unit, and records it in the sequence's decided/accepted mask; the update
//     that makes the first rejection known records the sequence's draw in the
//     sequence's own slot (or emits the sequence).  For a linear draw that
//     update is relaxed: its readers come after a grid barrier.
//   * The extra token is drawn in three more phases separated by grid-wide
//     barriers (the launch is cooperative, so every CTA is resident):
//       C. the B * Sr residual tiles -- slices of at most 4 KB of each drawn
//          row pair (or row: the tail, a tree node, a row to sample) -- are
//          split statically over all warps; a tile sums the fp32 weights
//          max(0, p - q) (or p) of every 16-byte group exactly in int64 fixed
//          point (units of 2^-52) per 64-group chunk, in code specialised at
//          compile time on the row kind, with the slice's geometry carried by
//          its stage from the issue;
//       D. one warp per draw locates the token: a prefix over the chunk sums,
//          then a rescan of one chunk with bit-identical weights;
//       E. (sampled tree) one warp per sequence walks the tree.
//     No counter, claim or record is polled after the stream: each phase's
//     inputs are complete when its barrier opens.
//   * L2 policy: the rows a residual pass is likely to re-read (the first
//     positions' row pairs in stream order, up to 1/kKeepDiv of L2) load at
//     normal priority, everything else evict-first, so the re-reads mostly
//     hit L2 and no high-priority line outlives the call.
//   * No tensor cores (nothing here is a contraction).  Every wait is bounded
//     and reports SPEC_DEV_TIMEOUT instead of trapping.
#pragma once

#include <climits>
#include <cstdint>

#include "params.cuh"
#include "ptx.cuh"
#include "spec_verify.h"

namespace spec {

// One stage's tile: {kTileStats, row, tile, run's last tile} or {kTileResid, draw, entry record,
// slice}; a residual stage also carries the geometry its issue computed: {target window's groups,
// target vbase, draft vbase, 1 if an edge group needs fixing}.
struct __align__(16) WarpCtl {
    unsigned long long full[kMaxStages];
    int4 desc[kMaxStages];
    int4 cgeo[kMaxStages];
};

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

__device__ __forceinline__ unsigned atom_add_acq_rel(uint32_t *p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
// Release only: the returned count is looked at later, and only the thread
// that completes a count takes an acquire fence before reading what it guards.
__device__ __forceinline__ unsigned atom_add_release(uint32_t *p, unsigned v) {
    unsigned old;
    asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ unsigned long long atom_or_acq_rel64(unsigned long long *p, unsigned long long v) {
    unsigned long long old;
    asm volatile("atom.acq_rel.gpu.global.or.b64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
    return old;
}
__device__ __forceinline__ unsigned long long atom_or_relaxed64(unsigned long long *p, unsigned long long v) {
    unsigned long long old;
    asm volatile("atom.relaxed.gpu.global.or.b64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
    return old;
}
// floor(u * tot) for a uniform u in [0, 1), exactly, in integer arithmetic: u = m * 2^-s
// with a 24-bit m, so u * tot is the 88-bit product m * tot shifted right by s.  A NaN or
// negative u counts as 0, u >= 1 as the largest target, tot - 1.
__device__ __forceinline__ long long cdf_target(float u, long long tot) {
    if (!(u > 0.f)) return 0;
    if (u >= 1.f) return tot - 1;
    const uint32_t bits = __float_as_uint(u);
    const uint32_t ex = bits >> 23;  // 1..126 (normal) or 0 (subnormal)
    const unsigned long long m = ex ? ((bits & 0x7fffffu) | 0x800000u) : (bits & 0x7fffffu);
    const int sh = ex ? 150 - static_cast<int>(ex) : 149;  // u = m * 2^-sh, sh >= 24
    const unsigned long long t = static_cast<unsigned long long>(tot);
    const unsigned long long lo = m * t, hi = __umul64hi(m, t);
    unsigned long long r;
    if (sh >= 128)
        r = 0;
    else if (sh >= 64)
        r = hi >> (sh - 64);
    else
        r = (hi << (64 - sh)) | (lo >> sh);
    return static_cast<long long>(r);  // < tot, since u < 1
}
// First rejected position of a sequence once it is known from a decided /
// accepted mask (every earlier position decided and accepted), K when every
// position 0..K is decided and none rejected, else -1.  K < 32.
__device__ __forceinline__ int first_rejection(unsigned long long m, int K) {
    const unsigned dec = static_cast<unsigned>(m);
    const unsigned acc = static_cast<unsigned>(m >> 32);
    const unsigned rej = dec & ~acc & ((1u << K) - 1u);
    const int f = __ffs(~dec) - 1;  // first undecided position, -1 if none
    if (rej) {
        const int j = __ffs(rej) - 1;
        return (f < 0 || j < f) ? j : -1;
    }
    const unsigned all = (K + 1 == 32) ? 0xffffffffu : ((1u << (K + 1)) - 1u);
    return ((dec & all) == all) ? K : -1;
}
__device__ __forceinline__ void fence_acquire() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
// Values another warp writes exactly once per call, never as zero: a relaxed
// 64-bit store is seen whole, so a reader that finds zero simply looks again.
// This spares the writers a release fence on the hot path.
__device__ __forceinline__ void st_relaxed64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long await64(const unsigned long long *p, bool &late) {
    unsigned long long v = ld_relaxed64(p);
    for (uint32_t i = 0; v == 0ull && i < kSpinLimit; ++i) {
        __nanosleep(32);
        v = ld_relaxed64(p);
    }
    if (v == 0ull) late = true;
    return v;
}
__device__ __forceinline__ unsigned ld_relaxed(const uint32_t *p) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned ld_acquire(const uint32_t *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(uint32_t *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// A weight in units of 2^-52: the power-of-two scaling is exact; the
// conversion rounds only weights below 2^-29.
__device__ __forceinline__ long long fixq(float w) { return __float2ll_rn(w * 4503599627370496.0f); }

// Every lane waits for the stage's copy; the answer is the warp's, so a wait
// that gives up leaves the warp converged.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity) {
    bool ok = false;
    for (uint32_t it = 0; it < kWaitLimit && !ok; ++it) ok = ptx::mbar_try_wait(bar, parity);
    return __all_sync(kFull, ok);
}

// ---- packed fp32 pairs (sm_100+ fma/add .f32x2)
__device__ __forceinline__ unsigned long long f2pack(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2unpack(unsigned long long v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2fma(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long f2add(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long f2mul(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long f2ex2(unsigned long long v) {
    float a, b;
    f2unpack(v, a, b);
    return f2pack(ptx::ex2(a), ptx::ex2(b));
}
// sum + (2^x.lo, 2^x.hi) with x = fma(v, c, -mc)
__device__ __forceinline__ unsigned long long exp_acc(unsigned long long sum, unsigned long long v,
                                                      unsigned long long c2, unsigned long long nmc2) {
    float a, b;
    f2unpack(f2fma(v, c2, nmc2), a, b);
    return f2add(sum, f2pack(ptx::ex2(a), ptx::ex2(b)));
}

// ---------------------------------------------------------------- elements
template <int EB>
struct Elt;

template <>
struct Elt<4> {
    static constexpr int G = 4;  // elements per 16-byte group
    static constexpr int P = 2;  // packed pairs per group
    __device__ __forceinline__ static void unpack(const uint4 &w, float (&v)[G]) {
        v[0] = __uint_as_float(w.x);
        v[1] = __uint_as_float(w.y);
        v[2] = __uint_as_float(w.z);
        v[3] = __uint_as_float(w.w);
    }
    __device__ __forceinline__ static void pairs(const uint4 &w, unsigned long long (&q)[P]) {
        q[0] = f2pack(__uint_as_float(w.x), __uint_as_float(w.y));
        q[1] = f2pack(__uint_as_float(w.z), __uint_as_float(w.w));
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
    // max of one group's elements (NaN only if all are NaN)
    __device__ __forceinline__ static float max16(const uint4 &w) {
        return fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)), fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
    }
    __device__ __forceinline__ static float group_max(const unsigned char *buf, int g0, int g1) {
        float m = neg_inf();
#pragma unroll 4
        for (int g = g0; g < g1; g += 32) {
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
    static constexpr int P = 4;
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
    __device__ __forceinline__ static void pairs(const uint4 &w, unsigned long long (&q)[P]) {
        q[0] = f2pack(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u));
        q[1] = f2pack(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
        q[2] = f2pack(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u));
        q[3] = f2pack(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u));
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
    // max of one group's elements (NaN only if all are NaN)
    __device__ __forceinline__ static float max16(const uint4 &w) {
        const uint32_t m = ptx::bmax2(ptx::bmax2(w.x, w.y), ptx::bmax2(w.z, w.w));
        return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    }
    __device__ __forceinline__ static float group_max(const unsigned char *buf, int g0, int g1) {
        uint32_t m = 0xff80ff80u;  // (-inf, -inf)
#pragma unroll 4
        for (int g = g0; g < g1; g += 32) {
            const uint4 w = *reinterpret_cast<const uint4 *>(buf + 16 * g);
            m = ptx::bmax2(m, ptx::bmax2(ptx::bmax2(w.x, w.y), ptx::bmax2(w.z, w.w)));
        }
        return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    }
};

// ------------------------------------------------------------ row geometry
// A slice [s0, s1) of one row is mirrored in a shared buffer 16-byte group by
// group: buffer byte k holds global byte glo + k, glo = 16-byte floor of the
// slice start.  The bulk copy covers [c0, c1) (offsets from glo), the part of
// the window inside the tensor's 16-byte-aligned interior; window bytes
// outside the slice, or slice bytes outside [c0, c1), are fixed afterwards.
struct Geo {
    const unsigned char *glo;
    int ngran;   // 16-byte groups in the window
    int c0, c1;  // bulk-copied bytes
    int a0, a1;  // the slice's bytes
    int vbase;   // element index of buffer byte 0 (may be negative)
    bool patch;  // some window byte needs fixing
};

template <int EB>
__device__ __forceinline__ Geo make_geo(const unsigned char *row, int s0, int s1, const unsigned char *lo,
                                        const unsigned char *hi) {
    Geo g;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(row) + static_cast<uintptr_t>(s0) * EB;
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(row) + static_cast<uintptr_t>(s1) * EB;
    const uintptr_t glo = a0 & ~uintptr_t(15);
    const uintptr_t ghi = (a1 + 15) & ~uintptr_t(15);
    const uintptr_t safe_lo = (reinterpret_cast<uintptr_t>(lo) + 15) & ~uintptr_t(15);
    const uintptr_t safe_hi = reinterpret_cast<uintptr_t>(hi) & ~uintptr_t(15);
    uintptr_t c0 = glo > safe_lo ? glo : safe_lo;
    uintptr_t c1 = ghi < safe_hi ? ghi : safe_hi;
    if (c0 > ghi) c0 = ghi;
    if (c1 < c0) c1 = c0;
    g.glo = reinterpret_cast<const unsigned char *>(glo);
    g.ngran = static_cast<int>((ghi - glo) >> 4);
    g.c0 = static_cast<int>(c0 - glo);
    g.c1 = static_cast<int>(c1 - glo);
    g.a0 = static_cast<int>(a0 - glo);
    g.a1 = static_cast<int>(a1 - glo);
    g.vbase = s0 - g.a0 / EB;
    g.patch = (a0 != glo) || (a1 != ghi) || (c0 != glo) || (c1 != ghi);
    return g;
}

// Fix the edge groups of one row buffer after its bulk copy has landed:
// window bytes outside the slice become -inf, slice bytes outside the copied
// range are loaded element by element.  16 lanes: 0..7 the first group,
// 8..15 the last group.
template <int EB>
__device__ __forceinline__ void patch_row(unsigned char *buf, const Geo &g, int l16) {
    constexpr int G = 16 / EB;
    const int e = l16 & 7;
    if (e >= G) return;
    const int grp = (l16 < 8) ? 0 : g.ngran - 1;
    const int off = grp * 16 + e * EB;
    if (off < g.a0 || off >= g.a1)
        Elt<EB>::store_neg_inf(buf + off);
    else if (off < g.c0 || off >= g.c1)
        Elt<EB>::copy(buf + off, g.glo + off);
}

// ------------------------------------------------------- partial merging
// (mc, s) represents sum 2^(l*c - mc) over a set of logits l (scaled domain).
__device__ __forceinline__ void merge_sc(float &m, float &s, float m2, float s2) {
    const float mm = fmaxf(m, m2);
    const float a = (m == mm) ? s : s * ptx::ex2(m - mm);
    const float b = (m2 == mm) ? s2 : s2 * ptx::ex2(m2 - mm);
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

// Warp-wide merge of the lanes' (mc, s): the max first, then one rescale per
// lane and a plain sum.  Every lane ends with the result.
__device__ __forceinline__ void warp_merge_sc(float &m, float &s) {
    float mm = m;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mm = fmaxf(mm, __shfl_xor_sync(kFull, mm, off));
    if (m != mm) s *= ptx::ex2(m - mm);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(kFull, s, off);
    m = mm;
}

__device__ __forceinline__ void warp_merge_vi(float &v, int &i) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        merge_vi(v, i, __shfl_xor_sync(kFull, v, off), __shfl_xor_sync(kFull, i, off));
}

// The warp sums of N (2 or 4) per-lane values at once: lanes trade halves of
// what they hold (xor 16, then 8 when N is 4), then sum the one value left.
// Lane l returns the sum over all lanes of q[l / (32 / N)].  Integer sums are
// exact, so the order does not matter.
template <int N>
__device__ __forceinline__ long long warp_sum64xN(const long long (&q)[N], int lane) {
    static_assert(N == 2 || N == 4, "two or four values");
    const bool hi16 = (lane & 16) != 0;
    long long b;
    if (N == 4) {
        const bool hi8 = (lane & 8) != 0;
        const long long a0 = (hi16 ? q[2 % N] : q[0]) + __shfl_xor_sync(kFull, hi16 ? q[0] : q[2 % N], 16);
        const long long a1 = (hi16 ? q[3 % N] : q[1]) + __shfl_xor_sync(kFull, hi16 ? q[1] : q[3 % N], 16);
        b = (hi8 ? a1 : a0) + __shfl_xor_sync(kFull, hi8 ? a0 : a1, 8);
    } else {
        b = (hi16 ? q[1] : q[0]) + __shfl_xor_sync(kFull, hi16 ? q[0] : q[1], 16);
    }
#pragma unroll
    for (int off = (N == 4) ? 4 : 8; off > 0; off >>= 1) b += __shfl_xor_sync(kFull, b, off);
    return b;
}
constexpr int kSumLanes = 32 / kCpt;  // lanes l with l % kSumLanes == 0 hold chunk l / kSumLanes

#ifndef SPEC_RESID_UNROLL
#define SPEC_RESID_UNROLL 4
#endif
constexpr int kResidUnroll = SPEC_RESID_UNROLL;  // group iterations of a residual tile unrolled together

// ------------------------------------------------------ extra-token weights
// The weights of a 16-byte group are summed by group_sum's order (below); the
// packed tile pass and the element-wise rescans all follow it.
// Weight of one element: pair (residual) max(0, p_v - q_v) with
// p_v = 2^(t c - MCt) / St and q_v = 2^(d c - MCd) / Sd; tail p_v.
// js = (MCt, 1/St, MCd, 1/Sd).  The pair weight is one fused multiply-add,
// 2^(t c - MCt) * (1/St) + (-q_v), so p_v is never rounded on its own.  The
// explicit _rn intrinsics keep every evaluation of a weight bit-identical.
__device__ __forceinline__ float elem_weight(float t, float d, bool pair, const float4 &js, float c) {
    const float et = ptx::ex2(__fmaf_rn(t, c, -js.x));
    if (!pair) return __fmul_rn(et, js.y);
    const float nqv = __fmul_rn(ptx::ex2(__fmaf_rn(d, c, -js.z)), -js.w);  // -q_v, exactly
    return fmaxf(0.0f, __fmaf_rn(et, js.y, nqv));
}

// The sum of one 16-byte group's weights: the even and the odd elements apart,
// each as a pairwise tree, then the two.  The packed tile pass (pairs of
// adjacent elements) forms exactly these sums, so every pass agrees bit for bit.
template <int G>
__device__ __forceinline__ float group_sum(const float (&w)[G]) {
    static_assert(G == 4 || G == 8, "16-byte groups of fp32 or bf16");
    if (G == 8) {
        const float se = (w[0] + w[2]) + (w[4] + w[6]);
        const float so = (w[1] + w[3]) + (w[5] + w[7]);
        return se + so;
    }
    return (w[0] + w[2]) + (w[1] + w[3]);
}

// ---------------------------------------------------------- tile reductions
// Sum of 2^(fma(l, c, -mc)) over this lane's logits of one stats tile (the
// 16-byte groups lane, lane + 32, ...): packed FMA/ADD, one ex2 per logit.
template <int EB>
__device__ __forceinline__ float lane_tile_sum(const unsigned char *buf, int ngran, int lane, float c, float mc) {
    constexpr int P = Elt<EB>::P;
    const unsigned long long c2 = f2pack(c, c), nmc2 = f2pack(-mc, -mc);
    unsigned long long acc[P];
#pragma unroll
    for (int q = 0; q < P; ++q) acc[q] = 0ull;
#pragma unroll 4
    for (int g = lane; g < ngran; g += 32) {
        unsigned long long v[P];
        Elt<EB>::pairs(*reinterpret_cast<const uint4 *>(buf + 16 * g), v);
#pragma unroll
        for (int q = 0; q < P; ++q) acc[q] = exp_acc(acc[q], v[q], c2, nmc2);
    }
#pragma unroll
    for (int q = 1; q < P; ++q) acc[0] = f2add(acc[0], acc[q]);
    float a, b;
    f2unpack(acc[0], a, b);
    return a + b;
}

// Add one stats tile to this lane's running (mc, sum), sum = sum 2^(l c - mc).
// The offset mc need not be the max: the lane's max is taken only to start,
// or when a tile's terms grow past 2^64 (a new, much larger max); so every
// term stays below 2^64 and nothing overflows.
template <int EB>
__device__ __forceinline__ void lane_sum(const unsigned char *buf, int ngran, float c, int lane, float &mc,
                                         float &sum) {
    if (mc > neg_inf()) {
        const float t = lane_tile_sum<EB>(buf, ngran, lane, c, mc);
        if (t < 18446744073709551616.0f) {  // 2^64 (false for NaN and inf: redone below)
            sum += t;
            return;
        }
    }
    const float mx = Elt<EB>::group_max(buf, lane, ngran);
    if (!(mx > neg_inf())) {        // no logit above -inf in this lane's part
        if (mx != mx) sum = mx;     // all NaN: poison the sum so the row is flagged
        return;
    }
    const float mn = mx * c;        // fl(max * c): the largest fl(l * c) of these logits
    if (mn > mc) {
        sum *= ptx::ex2(mc - mn);   // 0 while mc is still -inf
        mc = mn;
    }
    sum += lane_tile_sum<EB>(buf, ngran, lane, c, mc);
}

// Add one stats tile to this lane's running (max, lowest index of the max).
// The lane's best group comes first (its elements' max, a tree with no index), then the
// lowest element of that group holding it: the lane's elements run in index order, so a
// strictly greater max is needed to move (ties keep the lowest index; NaN never wins).
template <int EB>
__device__ __forceinline__ void lane_argmax(const unsigned char *buf, int ngran, int vbase, int lane, float &bv,
                                            int &bi) {
    constexpr int G = Elt<EB>::G;
    float tm = neg_inf();
    int tg = -1;
#pragma unroll 4
    for (int g = lane; g < ngran; g += 32) {
        const float gm = Elt<EB>::max16(*reinterpret_cast<const uint4 *>(buf + 16 * g));
        if (gm > tm) {
            tm = gm;
            tg = g;
        }
    }
    if (tm > bv) {
        float va[G];
        Elt<EB>::unpack(*reinterpret_cast<const uint4 *>(buf + 16 * tg), va);
        int k0 = G - 1;
#pragma unroll
        for (int k = G - 1; k >= 0; --k)
            if (va[k] == tm) k0 = k;
        bv = tm;
        bi = vbase + tg * G + k0;
    }
}

// Exact weight sums of one residual tile per chunk of 64 groups: this lane's
// share of each (warp_sum64xN adds the shares up).  Groups follow the target
// row's window.  Packed fp32x2 arithmetic on element
// pairs; every weight is the same as elem_weight's.  All 2 * kCpt groups of a
// lane are reduced without a branch (they lie inside the row buffers); groups
// past the window hold stale bytes and are given no weight, so the iterations
// are independent and overlap.
// KIND (fixed at compile time, so the unrolled groups carry no branch): kResidTail, a target
// row alone; kResidPair, a row pair whose buffers share the 16-byte phase; kResidPairShifted,
// a row pair whose draft row is read element by element.
constexpr int kResidTail = 0, kResidPair = 1, kResidPairShifted = 2;
template <int EB, int KIND>
__device__ __forceinline__ void tile_resid(const unsigned char *buf, int ngran, int vbase0, int vbase1, int s0,
                                           int s1, const float4 &js, float c, int lane, long long (&q)[kCpt]) {
    constexpr bool pair = KIND != kResidTail;
    constexpr bool same = KIND == kResidPair;
    constexpr int G = Elt<EB>::G;
    constexpr int P = Elt<EB>::P;
    const unsigned char *bt = buf;
    const unsigned char *bd = buf + kRowBuf;
    const unsigned long long c2 = f2pack(c, c);
    const unsigned long long nmt = f2pack(-js.x, -js.x), ist = f2pack(js.y, js.y);
    const unsigned long long nmd = f2pack(-js.z, -js.z), nisd = f2pack(-js.w, -js.w);
    static_assert(kChunk == 64 && 2 * kCpt * 32 * 16 == kRowBuf, "two groups per lane and chunk, covering the buffer");
    // Chunk ch's two groups are summed into `cs`, which then enters q[kCpt - 1] as the
    // earlier chunks shift down (after kCpt chunks q[c] is chunk c): every index stays a
    // compile-time constant under a partial unroll, so q lives in registers.
#pragma unroll (KIND == kResidPairShifted ? 1 : kResidUnroll / 2)
    for (int ch = 0; ch < kCpt; ++ch) {
        long long cs = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int g = (2 * ch + h) * 32 + lane;
            unsigned long long t2[P], d2[P];
            Elt<EB>::pairs(*reinterpret_cast<const uint4 *>(bt + 16 * g), t2);
            if (pair) {
                if (same) {
                    Elt<EB>::pairs(*reinterpret_cast<const uint4 *>(bd + 16 * g), d2);
                } else {
                    float d[G];
#pragma unroll
                    for (int k = 0; k < G; ++k) {
                        const int v = vbase0 + g * G + k;
                        d[k] = (v >= s0 && v < s1) ? Elt<EB>::load(bd + (v - vbase1) * EB) : neg_inf();
                    }
#pragma unroll
                    for (int k = 0; k < P; ++k) d2[k] = f2pack(d[2 * k], d[2 * k + 1]);
                }
            }
            unsigned long long w2[P];  // the weights of element pairs (2k, 2k + 1)
#pragma unroll
            for (int k = 0; k < P; ++k) {
                const unsigned long long et = f2ex2(f2fma(t2[k], c2, nmt));
                if (pair) {
                    const unsigned long long nq2 = f2mul(f2ex2(f2fma(d2[k], c2, nmd)), nisd);  // -q of two elements
                    float a, b;
                    f2unpack(f2fma(et, ist, nq2), a, b);
                    w2[k] = f2pack(fmaxf(0.0f, a), fmaxf(0.0f, b));
                } else {
                    w2[k] = f2mul(et, ist);  // p of two elements
                }
            }
            // (even sum, odd sum), each a pairwise tree: group_sum's order
            const unsigned long long acc =
                (P == 4) ? f2add(f2add(w2[0], w2[1]), f2add(w2[2 % P], w2[3 % P])) : f2add(w2[0], w2[1 % P]);
            float se, so;
            f2unpack(acc, se, so);
            cs += fixq(g < ngran ? se + so : 0.0f);
        }
#pragma unroll
        for (int c = 0; c + 1 < kCpt; ++c) q[c] = q[c + 1];
        q[kCpt - 1] = cs;
    }
}

// ---------------------------------------------------------- unit layout
template <int MODE>
struct Traits {
    static constexpr bool kSample = (MODE == kLinearSample || MODE == kBonusSample || MODE == kTreeSample);
    static constexpr bool kBonus = (MODE == kBonusSample || MODE == kBonusGreedy);
};

template <int EB>
__device__ __forceinline__ const unsigned char *row_ptr(const Params &p, int b, int pos, int r) {
    const size_t rb = static_cast<size_t>(p.V) * EB;
    if (r == 0) return p.target + (static_cast<size_t>(b) * p.t_rows + pos) * rb;
    return p.draft + (static_cast<size_t>(b) * p.K + pos) * rb;
}

// Position of sequence b's unit in the extra-token-alone modes; -1 if invalid.
// Without lengths every sequence draws at position K (one row per sequence).
__device__ __forceinline__ int bonus_pos(const Params &p, int b) {
    if (p.accept_len_in == nullptr) return p.K;
    const int j = __ldg(&p.accept_len_in[b]);
    return (j < 0 || j > p.K) ? -1 : j;
}

// Rows of the unit at position pos (-1: an invalid length, one unused row).
template <int MODE>
__device__ __forceinline__ int unit_nrows(const Params &p, int pos) {
    return (Traits<MODE>::kSample && MODE != kTreeSample && pos >= 0 && pos < p.K) ? 2 : 1;
}

// Row slot rs of a sequence in the stats tiling: its position, its row within
// the unit, and whether it exists (bpos: the extra-token position, if any).
template <int MODE>
__device__ __forceinline__ bool row_slot(const Params &p, int rs, int bpos, int &pos, int &r) {
    if (MODE == kLinearSample) {
        pos = rs >> 1;
        r = rs & 1;
        return true;
    }
    if (MODE == kBonusSample || MODE == kBonusGreedy) {
        pos = bpos < 0 ? 0 : bpos;  // an invalid length still reads one row, so its unit completes
        r = rs;
        return r == 0 || (MODE == kBonusSample && bpos >= 0 && bpos < p.K);
    }
    pos = rs;
    r = 0;
    return true;
}

// Row id (index in the stats tiling) of row r of unit (b, pos); the inverse of
// the kernel's row decoding.  pos < 0 (an invalid length) reads row 0.
template <int MODE>
__device__ __forceinline__ int row_id_of(const Params &p, int b, int pos, int r) {
    if (MODE == kLinearSample) return (pos < p.K) ? (pos * p.B + b) * 2 + r : 2 * p.K * p.B + b;
    if (MODE == kLinearGreedy) return pos * p.B + b;
    if (MODE == kTreeGreedy || MODE == kTreeSample) return b * p.rows_per_seq + pos;
    if (MODE == kBonusSample) return b * p.rows_per_seq + r;  // rows_per_seq is 1 when K == 0
    return b;  // kBonusGreedy
}

// Does a run of stats tiles start at global tile t?  Static split: at every
// warp's first tile and at every row start; dynamic: at every segment start.
__device__ __forceinline__ bool run_starts_at(const Params &p, long long t, int k) {
    if (!p.static_split) return (k % kSegTiles) == 0;
    if (k == 0) return true;
    const long long T = p.stats_tiles, W = p.nwarps;
    const long long w = (t * W + T - 1) / T;  // the first warp whose range starts at or after t
    return (T * w) / W == t;
}

// One grid-wide barrier (the target-th arrival in all): every CTA's writes
// before it are visible to every CTA after it.  The launch is cooperative, so
// every CTA is resident and the barrier completes; the wait is bounded all the
// same, and a wait that gives up answers false.  All threads of the CTA call it.
__device__ __forceinline__ bool grid_barrier(uint32_t *ctr, unsigned target, int *s_flag) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        (void)atom_add_release(ctr, 1u);
        unsigned v = ld_acquire(ctr);
        for (uint32_t i = 0; v < target && i < kSpinLimit; ++i) {
            __nanosleep(32);
            v = ld_acquire(ctr);
        }
        *s_flag = (v >= target) ? 1 : 0;
    }
    __syncthreads();
    return *s_flag != 0;
}

// =================================================================== kernel
template <int EB, int MODE>
__global__ void __launch_bounds__(kThreads, kMinCtas) spec_verify_kernel(const Params p) {
    using T = Traits<MODE>;
    constexpr int G = Elt<EB>::G;

    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ WarpCtl wctl[kWarps];
    __shared__ int s_flag;             // a CTA-wide answer: a grid barrier's, then "last CTA"

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    WarpCtl &wc = wctl[warp];
    const int NS = p.nstage;  // stats stages of the ring; the residual phase splits the same bytes finer
    static_assert(kCWarps == kWarps, "every warp reduces residual tiles in its own ring");
    const int NSC = min(kMaxStages, NS * kStageBytes / kCStageBytes);  // residual stages of a warp's ring
    unsigned char *ring = dsm + static_cast<size_t>(warp) * NS * kStageBytes;
    int *tscratch = reinterpret_cast<int *>(dsm + static_cast<size_t>(kWarps) * NS * kStageBytes) +
                    static_cast<size_t>(warp) * 3 * p.units_per_seq;

    if (lane == 0) {
        for (int s = 0; s < kMaxStages; ++s) ptx::mbar_init(ptx::smem_addr(&wc.full[s]), 1);
        ptx::fence_mbar_init();
    }
    __syncwarp();

    const long long NSEG = p.stats_segs;
    const long long RT = p.res_tiles;
    const int S = p.S;
    const size_t row_bytes = static_cast<size_t>(p.V) * EB;
    const bool draws = T::kSample && (T::kBonus || p.u_bonus != nullptr);
    const long long nwarps = static_cast<long long>(gridDim.x) * kWarps;
    const long long gw = static_cast<long long>(blockIdx.x) * kWarps + warp;  // this warp's index in the grid
    bool timed_out = false;
    // Linear sampling with an extra token and K < 32: a draw record carries no skip bit; the
    // residual and select phases test the drawn unit's statistics (1/St = 0 when non-finite)
    // and the select clears the sequence's mask and statistics.
    const bool late_skip = MODE == kLinearSample && draws && p.K < 32;

    // A row of the stats tiling: row slot rs of sequence b.
    struct Row {
        int id;                        // b * rows_per_seq + rs
        int b, pos, r, unit;
        bool present;
        uintptr_t R0, A, E, lo, hi;    // row start, window grid start / end, tensor's aligned interior
    };
    auto decode_row = [&](int id) -> Row {
        Row t;
        t.id = id;
        int rs;
        if (MODE == kLinearSample) {
            // position-major: (target i, draft i) of every sequence for i = 0..K-1, then every tail row
            const int twoB = 2 * p.B;
            if (id < p.K * twoB) {
                const int i = id / twoB;
                const int rem = id - i * twoB;
                t.b = rem >> 1;
                rs = 2 * i + (rem & 1);
            } else {
                t.b = id - p.K * twoB;
                rs = 2 * p.K;
            }
        } else if (MODE == kLinearGreedy) {
            const int i = id / p.B;  // position-major
            t.b = id - i * p.B;
            rs = i;
        } else {
            t.b = id / p.rows_per_seq;
            rs = id - t.b * p.rows_per_seq;
        }
        const int bpos = T::kBonus ? bonus_pos(p, t.b) : 0;
        t.present = row_slot<MODE>(p, rs, bpos, t.pos, t.r);
        t.unit = T::kBonus ? t.b : t.b * p.units_per_seq + t.pos;
        if (T::kBonus) t.pos = bpos;  // -1 for an invalid length (its row 0 is read all the same)
        const unsigned char *row = row_ptr<EB>(p, t.b, t.pos < 0 ? 0 : t.pos, t.r);
        t.R0 = reinterpret_cast<uintptr_t>(row);
        t.A = t.R0 & ~uintptr_t(15);
        t.E = (t.R0 + row_bytes + 15) & ~uintptr_t(15);
        t.lo = (reinterpret_cast<uintptr_t>(t.r ? p.draft : p.target) + 15) & ~uintptr_t(15);
        t.hi = reinterpret_cast<uintptr_t>(t.r ? p.d_end : p.t_end) & ~uintptr_t(15);
        return t;
    };
    // window [w0, w1) of tile k of a row, and its bulk-copied part [c0, c1)
    auto tile_window = [&](const Row &t, int k, uintptr_t &w0, uintptr_t &w1, uintptr_t &c0, uintptr_t &c1) {
        w0 = t.A + static_cast<uintptr_t>(k) * kTileBytes;
        w1 = w0 + kTileBytes < t.E ? w0 + kTileBytes : t.E;
        if (w1 < w0) w1 = w0;  // past the row's end: an empty tile
        c0 = w0 > t.lo ? w0 : t.lo;
        c1 = w1 < t.hi ? w1 : t.hi;
        if (c0 > w1) c0 = w1;
        if (c1 < c0) c1 = c0;
    };
    // unit (b, pos) of a draw entry record
    auto entry_unit = [&](uint32_t rec, int &u, int &b, int &pos) {
        u = static_cast<int>(rec & kRecUnit) - 1;
        if (T::kBonus) {
            b = u;
            pos = max(0, bonus_pos(p, b));
        } else {
            b = u / p.units_per_seq;
            pos = u - b * p.units_per_seq;
        }
    };
    // tiles to take at once: shrinks as the space runs out, so the last grabs are short
    auto guided = [&](long long left, int most) -> int {
        const long long g = left / (nwarps * kGuidedDiv);
        return static_cast<int>(g < 1 ? 1 : (g > most ? most : g));
    };

    // ---------------------------------------------------------- issue side
    const uint64_t pol_first = ptx::policy_evict_first();
    // dynamic: stats segments [sc, se) grabbed, not yet begun; static: this warp's tiles [sc, se)
    long long sc = 0, se = 0;
    Row irow = {};                     // the row of the run being issued
    irow.id = -1;
    int ik = 0, ik1 = 0;               // that run's tiles [ik, ik1) still to issue (within the row)
    int irun_last = 0;                 // the run's last tile
    unsigned s_ahead = 0;              // lane 0: start of the next stats grab
    int s_ahead_n = 0;                 // its size
    bool ahead_issued = false;         // the next grab was requested ahead (away from the end)
    bool stats_done = (NSEG == 0);
    if (p.static_split) {
        sc = p.stats_tiles * gw / p.nwarps;
        se = p.stats_tiles * (gw + 1) / p.nwarps;
        stats_done = sc >= se;
    } else if (!stats_done) {
        s_ahead_n = guided(NSEG, kMaxGrab);
        if (lane == 0) s_ahead = atomicAdd(&p.ws_ctrl[0], static_cast<unsigned>(s_ahead_n));
        ahead_issued = true;
    }
    int issued = 0, handled = 0;
    int nst = NS;                      // stages in use: NS of kStageBytes, then NSC of kCStageBytes
    int islot = 0;                     // stage of the next issue
    auto next_islot = [&]() {
        const int s = islot;
        islot = (islot + 1 == nst) ? 0 : islot + 1;
        return s;
    };

    // begin segment sg: its row and tiles; false if the row slot holds no row
    auto begin_segment = [&](long long sg) -> bool {
        const int id = static_cast<int>(static_cast<unsigned>(sg) / static_cast<unsigned>(p.nseg));
        const int j = static_cast<int>(sg) - id * p.nseg;
        if (id != irow.id) irow = decode_row(id);
        ik = j * kSegTiles;
        ik1 = min(S, ik + kSegTiles);
        irun_last = ik1 - 1;
        return irow.present;
    };
    // static split: begin the next run of this warp's tiles (up to the row's end)
    auto begin_static_run = [&]() -> bool {
        const int id = static_cast<int>(static_cast<unsigned long long>(sc) / static_cast<unsigned>(S));
        const int k = static_cast<int>(sc - static_cast<long long>(id) * S);
        const int n = static_cast<int>(min(static_cast<long long>(S - k), se - sc));
        if (id != irow.id) irow = decode_row(id);
        ik = k;
        ik1 = k + n;
        irun_last = ik1 - 1;
        sc += n;
        return irow.present;
    };
    // issue tile ik of the current segment
    auto issue_stats = [&]() {
        const int s = next_islot();
        unsigned char *buf = ring + static_cast<size_t>(s) * kStageBytes;
        uintptr_t w0, w1, c0, c1;
        tile_window(irow, ik, w0, w1, c0, c1);
        if (lane == 0) {
            wc.desc[s] = make_int4(kTileStats, irow.id, ik, irun_last);
            const uint32_t bar = ptx::smem_addr(&wc.full[s]);
            const uint32_t bytes = static_cast<uint32_t>(c1 - c0);
            ptx::mbar_arrive_expect_tx(bar, bytes);
            if (bytes) {
                // rows a residual pass is likely to re-read stay in L2 at normal priority; the rest
                // of the stream is marked first to go
                if (irow.id < p.keep_rows)
                    ptx::bulk_g2s(ptx::smem_addr(buf + (c0 - w0)), reinterpret_cast<const void *>(c0), bytes, bar);
                else
                    ptx::bulk_g2s_hint(ptx::smem_addr(buf + (c0 - w0)), reinterpret_cast<const void *>(c0), bytes,
                                       bar, pol_first);
            }
        }
        ++ik;
        ++issued;
    };

    // Residual stage s of this warp: the ring re-cut into stages of kCStageBytes.
    auto cstage = [&](int s) -> unsigned char * { return ring + static_cast<size_t>(s) * kCStageBytes; };
    // issue residual slice k of draw e: record rec, rows rt (target) and rd (draft, pairs only)
    auto issue_resid = [&](int e, int k, uint32_t rec, const unsigned char *rt, const unsigned char *rd) {
        const bool pair = (rec & kRecPair) != 0;
        const bool skip = (rec & kRecSkip) != 0;
        const int s = next_islot();
        unsigned char *buf = cstage(s);
        const int s0 = k * p.Lr;
        const int s1 = min(p.V, s0 + p.Lr);
        const Geo g0 = make_geo<EB>(rt, s0, s1, p.target, p.t_end);
        Geo g1 = g0;
        if (pair) g1 = make_geo<EB>(rd, s0, s1, p.draft, p.d_end);
        if (lane == 0) {
            wc.desc[s] = make_int4(kTileResid, e, static_cast<int>(rec), k);
            wc.cgeo[s] = make_int4(g0.ngran, g0.vbase, g1.vbase, (g0.patch || (pair && g1.patch)) ? 1 : 0);
            const uint32_t bar = ptx::smem_addr(&wc.full[s]);
            uint32_t bytes = 0;
            if (!skip)
                bytes = static_cast<uint32_t>(g0.c1 - g0.c0) + (pair ? static_cast<uint32_t>(g1.c1 - g1.c0) : 0u);
            ptx::mbar_arrive_expect_tx(bar, bytes);
            if (!skip) {
                // the last read of these rows: they may leave L2 first
                if (g0.c1 > g0.c0)
                    ptx::bulk_g2s_hint(ptx::smem_addr(buf + g0.c0), g0.glo + g0.c0,
                                       static_cast<uint32_t>(g0.c1 - g0.c0), bar, pol_first);
                if (pair && g1.c1 > g1.c0)
                    ptx::bulk_g2s_hint(ptx::smem_addr(buf + kRowBuf + g1.c0), g1.glo + g1.c0,
                                       static_cast<uint32_t>(g1.c1 - g1.c0), bar, pol_first);
            }
        }
        ++issued;
    };

    // Hand the next stats tile to the ring.  Returns false when nothing was issued:
    // nothing is ready now (blocking == false), or no stats work is left at all.
    auto try_issue = [&](bool blocking) -> bool {
        for (int guard = 0; guard < (1 << 20); ++guard) {
            if (!stats_done && p.static_split) {
                if (ik >= ik1) {
                    if (sc >= se) {
                        stats_done = true;
                    } else if (!begin_static_run()) {  // a row slot with no row
                        ik = ik1 = 0;
                        continue;
                    }
                }
                if (!stats_done) {
                    issue_stats();
                    return true;
                }
            }
            if (!stats_done && !p.static_split) {
                if (ik >= ik1) {
                    if (sc >= se) {
                        // near the end a grab is made only when needed, so no warp holds work in reserve
                        if (!ahead_issued && lane == 0)
                            s_ahead = atomicAdd(&p.ws_ctrl[0], static_cast<unsigned>(s_ahead_n));
                        const unsigned a = __shfl_sync(kFull, s_ahead, 0);
                        if (static_cast<long long>(a) >= NSEG) {
                            stats_done = true;
                        } else {
                            sc = a;
                            se = min(NSEG, static_cast<long long>(a) + s_ahead_n);
                            s_ahead_n = guided(NSEG - se, kMaxGrab);
                            ahead_issued = NSEG - se >= kTailZone * nwarps;
                            if (ahead_issued && lane == 0)
                                s_ahead = atomicAdd(&p.ws_ctrl[0], static_cast<unsigned>(s_ahead_n));
                        }
                    }
                    if (!stats_done) {
                        if (!begin_segment(sc++)) {  // a row slot with no row (the draft row at the tail)
                            ik = ik1 = 0;
                            continue;
                        }
                    }
                }
                if (!stats_done) {
                    issue_stats();
                    return true;
                }
            }
            return false;
        }
        timed_out = true;
        return false;
    };
    auto fill_ring = [&]() {
        while (issued - handled < nst) {
            if (ik < ik1) {  // the next tile of the segment
                issue_stats();
                continue;
            }
            if (!try_issue(false)) break;
        }
        __syncwarp();
    };

    // ----------------------------------------------------- processing side
    // the stats segment being reduced (one row, tiles [k0, k1))
    bool srun = false;
    int run_k0 = 0, run_last = 0, run_len = 0;
    Row prow = {};
    prow.id = -1;
    int px = -1;                       // the draft token whose logit this row holds, or -1
    float am = neg_inf(), as = 0.f;    // lane: running (mc, s), or (max, -) in greedy mode
    int ai = INT_MAX;                  // lane: index of the max (greedy)
    int hasx = 0;
    float xval = 0.f;
    // a unit-tile count whose result is consumed later
    bool pend = false;
    int pend_unit = 0, pend_b = 0, pend_pos = 0, pend_add = 0;
    unsigned pend_old = 0;             // lane 0

    // ----------------------------------------------------- finishing side
    // Draft token `lane` of sequence b when lane < j (else -1): loaded ahead of an emission.
    auto lane_draft_token = [&](int b, int j) -> int {
        return (lane < j && lane < p.K && p.out_tokens) ? ptx::ld_nc_early(&p.tokens[static_cast<size_t>(b) * p.K + lane])
                                                       : -1;
    };
    // Emit the sequence: the first j draft tokens, then `extra` (if any), then -1.  `pre` is
    // lane_draft_token(b, j).
    auto emit_linear = [&](int b, int j, int extra, bool has_extra, int pre) {
        const int K = p.K;
        if (p.out_tokens) {
            for (int i = lane; i <= K; i += 32)
                p.out_tokens[static_cast<size_t>(b) * (K + 1) + i] =
                    (i < j) ? (i < 32 ? pre : __ldg(&p.tokens[static_cast<size_t>(b) * K + i]))
                            : ((i == j && has_extra) ? extra : -1);
        }
        if (lane == 0) {
            p.accept_len[b] = j;
            p.num_emitted[b] = j + (has_extra ? 1 : 0);
        }
    };

    // Greedy tree walk of sequence b (every node's choice is in ws_val).
    auto emit_tree = [&](int b) {
        const int N = p.units_per_seq;
        int *par_s = tscratch;
        int *tok_s = par_s + N;
        int *am_s = tok_s + N;
        for (int cidx = lane; cidx < N; cidx += 32) {
            int pc = __ldg(&p.parents[cidx]);
            if (cidx == 0) {
                pc = -1;
            } else if (pc < 0 || pc >= cidx) {
                atomicOr(p.status, SPEC_DEV_BAD_TREE);
                pc = -2;
            }
            par_s[cidx] = pc;
            tok_s[cidx] = __ldg(&p.tokens[static_cast<size_t>(b) * N + cidx]);
            am_s[cidx] = __ldcg(&p.ws_val[static_cast<size_t>(b) * N + cidx]);
            p.ws_val[static_cast<size_t>(b) * N + cidx] = 0;
        }
        __syncwarp();
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
                const unsigned m = __ballot_sync(kFull, hit);
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
        }
        for (int i = depth + 1 + lane; i <= D; i += 32) {
            ot[i] = -1;
            pn[i] = -1;
        }
        __syncwarp();
    };

    // Record the draw of unit u in slot e (the sequence's, or the node's own).
    auto set_draw = [&](int e, int u, bool pair, bool skip) {
        if (lane == 0)
            p.ws_draw[e] = (static_cast<uint32_t>(u) + 1u) | (pair ? kRecPair : 0u) | (skip ? kRecSkip : 0u);
        __syncwarp();
    };

    // The first rejection j of linear sequence b is known: record its draw of the
    // extra token, or emit the sequence; unit j's scratch is ours.
    // skip: 1 / 0 when the caller knows whether unit j is non-finite, -1 if not.  own: unit
    // j's argmax when the caller has just found it (greedy), else INT_MIN.  pre: this lane's
    // draft token, lane_draft_token(b, K) (valid wherever lane < j).
    auto draw_or_emit = [&](int b, int j, int skip, int own, int pre) {
        const int U = p.units_per_seq;
        const int u = b * U + j;
        if (MODE == kLinearSample) {
            if (draws) {
                if (skip < 0) skip = (__ldcg(&p.ws_stats[u]).y > 0.f) ? 0 : 1;  // a non-finite unit recorded 1/St = 0
                set_draw(b, u, j < p.K, skip != 0);
            } else {
                emit_linear(b, j, -1, false, pre);
            }
        } else if (MODE == kLinearGreedy) {
            const int extra = (p.u_bonus == nullptr) ? -1 : (own != INT_MIN ? own : __ldcg(&p.ws_val[u]));
            __syncwarp();
            if (lane == 0) p.ws_val[u] = 0;
            emit_linear(b, j, extra, p.u_bonus != nullptr, pre);
        }
        __syncwarp();
    };

    // Every unit of linear sequence b is decided: zero its scratch except unit j's.
    auto cleanup_seq = [&](int b, int j, bool masked) {
        const int U = p.units_per_seq;
        if (masked) {
            if (lane == 0) p.ws_seqmask[b] = 0ull;
        } else {
            if (MODE == kLinearSample)
                for (int i = lane; i < p.K; i += 32) p.ws_acc[static_cast<size_t>(b) * p.K + i] = 0;
            if (lane == 0) p.ws_seq_cnt[b] = 0u;
        }
        for (int i = lane; i < U; i += 32) {
            if (i == j) continue;
            if (MODE == kLinearSample && draws) p.ws_stats[static_cast<size_t>(b) * U + i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (MODE == kLinearGreedy) p.ws_val[static_cast<size_t>(b) * U + i] = 0;
        }
        __syncwarp();
    };

    // Every unit of sequence b is decided (trees, and linear sequences with K >= 32).
    auto finish_sequence = [&](int b) {
        const int K = p.K;
        const int U = p.units_per_seq;
        if (MODE == kTreeGreedy) {
            emit_tree(b);
            if (lane == 0) p.ws_seq_cnt[b] = 0u;
            __syncwarp();
            return;
        }
        int j = K;
        for (int base = 0; base < K; base += 32) {
            const int i = base + lane;
            bool rej = false;
            if (i < K) {
                if (MODE == kLinearSample)
                    rej = __ldcg(&p.ws_acc[static_cast<size_t>(b) * K + i]) == 0;
                else
                    rej = __ldg(&p.tokens[static_cast<size_t>(b) * K + i]) !=
                          __ldcg(&p.ws_val[static_cast<size_t>(b) * U + i]);
            }
            const unsigned m = __ballot_sync(kFull, rej);
            if (m) {
                j = base + __ffs(m) - 1;
                break;
            }
        }
        draw_or_emit(b, j, -1, INT_MIN, lane_draft_token(b, j));
        cleanup_seq(b, j, false);
    };

    // Every stats tile of unit u is published: merge, decide, record.
    auto finish_unit = [&](int u, int b, int pos) {
        const int K = p.K;
        const int nrows = unit_nrows<MODE>(p, pos);
        // the decision's inputs, loaded while the partials are merged (and the draft tokens, for
        // an emission at the end)
        int x = -1;
        float ua = 0.f;
        const int pre = ((MODE == kLinearSample && !draws) || MODE == kLinearGreedy) ? lane_draft_token(b, K) : -1;
        if ((MODE == kLinearSample || MODE == kLinearGreedy) && pos >= 0 && pos < K) {
            x = __ldg(&p.tokens[static_cast<size_t>(b) * K + pos]);
            if (MODE == kLinearSample) ua = __ldg(&p.u_accept[static_cast<size_t>(b) * K + pos]);
        }
        // t(x), d(x): lane 0 loads them with its first partials and waits for them after the merge
        const bool want_tx = MODE == kLinearSample && pos >= 0 && pos < K && x >= 0 && x < p.V;
        unsigned long long *txs = p.ws_txw + static_cast<size_t>(u) * 2;
        unsigned long long txw[2] = {0ull, 0ull};
        long long t0[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) t0[r] = static_cast<long long>(row_id_of<MODE>(p, b, pos, r < nrows ? r : 0)) * S;
        float Mr[2], Sm[2];
        int Ar[2];
        float v[2] = {neg_inf(), neg_inf()}, sm[2] = {0.f, 0.f};
        int ii[2] = {INT_MAX, INT_MAX};
        // every run publishes one partial at its first tile; both rows' loads are issued before any wait
        for (int k = lane; k < S; k += 32) {
            unsigned long long *slot[2];
            unsigned long long w[2];
            bool has[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                slot[r] = &p.ws_part[(static_cast<size_t>(u) * 2 + r) * S + k];
                has[r] = r < nrows && run_starts_at(p, t0[r] + k, k);
                w[r] = has[r] ? ld_relaxed64(slot[r]) : 0ull;
            }
            if (want_tx && k == 0) {  // lane 0's first slot
                txw[0] = ld_relaxed64(&txs[0]);
                txw[1] = ld_relaxed64(&txs[1]);
            }
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                if (!has[r]) continue;
                bool late = false;
                if (w[r] == 0ull) w[r] = await64(slot[r], late);  // every run publishes once
                if (late) {  // reported (and the workspace cleared) at the end of the kernel
                    timed_out = true;
                    continue;
                }
                *slot[r] = 0ull;
                const uint2 e = make_uint2(static_cast<unsigned>(w[r]), static_cast<unsigned>(w[r] >> 32));
                if (T::kSample)
                    merge_sc(v[r], sm[r], __uint_as_float(e.x), __uint_as_float(e.y));
                else
                    merge_vi(v[r], ii[r], __uint_as_float(e.x), static_cast<int>(e.y - 1u));
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            if (T::kSample)
                warp_merge_sc(v[r], sm[r]);
            else
                warp_merge_vi(v[r], ii[r]);
            Mr[r] = v[r];
            Sm[r] = sm[r];
            Ar[r] = ii[r];
        }
        uint32_t fl = 0;
        bool finite = true;
        int accept = 0;  // lane 0
        if (T::kSample) {
            for (int r = 0; r < nrows; ++r)
                if (!(isfinite(Mr[r]) && isfinite(Sm[r]) && Sm[r] > 0.f)) finite = false;
            if (!finite) fl |= SPEC_DEV_NONFINITE;
        } else if (Ar[0] == INT_MAX) {
            fl |= SPEC_DEV_NONFINITE;  // no element above -inf
            Ar[0] = 0;
        }
        if (lane == 0) {
            p.ws_unit_cnt[u] = 0u;
            if (MODE == kLinearSample && pos < K) {
                float2 txv = make_float2(0.f, 0.f);
                if (want_tx) {  // the runs holding x published its logits
                    bool late = false;
                    if (txw[0] == 0ull) txw[0] = await64(&txs[0], late);
                    if (txw[1] == 0ull) txw[1] = await64(&txs[1], late);
                    if (late) timed_out = true;
                    txs[0] = 0ull;
                    txs[1] = 0ull;
                    txv = make_float2(__uint_as_float(static_cast<unsigned>(txw[0])),
                                      __uint_as_float(static_cast<unsigned>(txw[1])));
                }
                float px = 0.f, qx = 0.f, thr = 0.f;
                if (x < 0 || x >= p.V) {
                    fl |= SPEC_DEV_BAD_TOKEN;
                } else {
                    const float lt = __fmaf_rn(txv.x, p.c, -Mr[0]);  // log2 of p(x) * S_t
                    const float ld = __fmaf_rn(txv.y, p.c, -Mr[1]);
                    px = ptx::ex2(lt) / Sm[0];
                    qx = ptx::ex2(ld) / Sm[1];
                    thr = fminf(1.0f, ptx::ex2(lt - ld) * (Sm[1] / Sm[0]));
                    accept = (ua < thr) ? 1 : 0;
                }
                if (K >= 32) p.ws_acc[static_cast<size_t>(b) * K + pos] = accept;
                if (p.probs) {
                    float *pr = p.probs + (static_cast<size_t>(b) * K + pos) * 3;
                    pr[0] = px;
                    pr[1] = qx;
                    pr[2] = thr;
                }
            }
            if (draws) {
                // a non-finite unit records 1/St = 0, which marks its draw as skipped
                p.ws_stats[u] = finite ? make_float4(Mr[0], 1.0f / Sm[0], Mr[1], nrows == 2 ? 1.0f / Sm[1] : 0.f)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (!T::kSample) {
                if (T::kBonus)
                    p.bonus_token[b] = (pos < 0) ? -1 : Ar[0];
                else
                    p.ws_val[static_cast<size_t>(b) * p.units_per_seq + pos] = Ar[0];
                if (MODE == kLinearGreedy && pos < K) accept = (x == Ar[0]) ? 1 : 0;
            }
            if (T::kBonus && pos < 0) fl |= SPEC_DEV_BAD_LENGTH;
            if (fl) atomicOr(p.status, fl);
        }
        __syncwarp();
        if (T::kBonus || MODE == kTreeSample) {  // every unit draws, in a slot of its own
            if (T::kSample) set_draw(u, u, nrows == 2, pos < 0 || !finite);
            return;
        }
        if ((MODE == kLinearSample || MODE == kLinearGreedy) && K < 32) {
            // the first rejection is known as soon as every earlier position is decided
            unsigned long long bits = 1ull << pos;
            if (pos < K && __shfl_sync(kFull, accept, 0)) bits |= 1ull << (32 + pos);
            // Linear sampling with an extra token: the draw's readers (residual tiles, selects)
            // run after a grid barrier, so the mask update orders nothing here; whether the drawn
            // unit is non-finite, and the sequence's cleanup, are left to them (late_skip).
            unsigned long long old = 0;
            if (lane == 0)
                old = late_skip ? atom_or_relaxed64(&p.ws_seqmask[b], bits) : atom_or_acq_rel64(&p.ws_seqmask[b], bits);
            old = __shfl_sync(kFull, old, 0);
            __syncwarp();
            const unsigned long long now = old | bits;
            const int jn = first_rejection(now, K);
            if (first_rejection(old, K) < 0 && jn >= 0) {
                if (late_skip)
                    set_draw(b, b * p.units_per_seq + jn, jn < K, false);
                else
                    draw_or_emit(b, jn, jn == pos ? (finite ? 0 : 1) : -1, (!T::kSample && jn == pos) ? Ar[0] : INT_MIN,
                                 pre);
            }
            if (!late_skip && __popc(static_cast<unsigned>(now)) == K + 1) cleanup_seq(b, jn, true);
            return;
        }
        int last = 0;
        if (lane == 0)
            last = (atom_add_acq_rel(&p.ws_seq_cnt[b], 1u) == static_cast<unsigned>(p.units_per_seq - 1)) ? 1 : 0;
        last = __shfl_sync(kFull, last, 0);
        __syncwarp();
        if (last) finish_sequence(b);
    };

    // Chunk sums of every residual slice of unit (b, pos) with weights p
    // alone, read from global memory (the rare redraw after a vanished residual).
    auto resid_from_global = [&](int e, int b, int pos, const float4 &js) {
        const unsigned char *rt = row_ptr<EB>(p, b, pos, 0);
        unsigned long long *cs = p.ws_csum + static_cast<size_t>(e) * p.Sr * kCpt;
        for (int k = 0; k < p.Sr; ++k) {
            const int s0 = k * p.Lr;
            const int s1 = min(p.V, s0 + p.Lr);
            const Geo g = make_geo<EB>(rt, s0, s1, p.target, p.t_end);
            long long q[kCpt];
#pragma unroll
            for (int c = 0; c < kCpt; ++c) q[c] = 0;
#pragma unroll
            for (int h = 0; h < (kCpt * kChunk) / 32; ++h) {
                const int gi = h * 32 + lane;
                float w[G];
#pragma unroll
                for (int k2 = 0; k2 < G; ++k2) {
                    const int v = g.vbase + gi * G + k2;
                    w[k2] = 0.f;
                    if (gi < g.ngran && v >= s0 && v < s1)
                        w[k2] = elem_weight(Elt<EB>::gload(rt + static_cast<size_t>(v) * EB), 0.f, false, js, p.c);
                }
                q[h / 2] += fixq(group_sum<G>(w));
            }
            const long long t = warp_sum64xN<kCpt>(q, lane);
            if (lane % kSumLanes == 0) cs[k * kCpt + lane / kSumLanes] = static_cast<unsigned long long>(t);
        }
        __syncwarp();
    };

    // Locate the extra token of draw e from its chunk sums; -1 when the weights sum to zero.
    auto select_token = [&](int e, int b, int pos, bool pair, const float4 &js, float ub) -> int {
        const int n = p.Sr * kCpt;
        const unsigned long long *cs = p.ws_csum + static_cast<size_t>(e) * n;
        // lane l owns the chunk sums [l0, l0 + m), l0 = lane * m; the first kHold stay in registers
        const int m = (n + 31) / 32;
        const int l0 = lane * m;
        long long v[kHold];
#pragma unroll
        for (int r = 0; r < kHold; ++r)
            v[r] = (r < m && l0 + r < n) ? static_cast<long long>(__ldcg(&cs[l0 + r])) : 0;
        long long mine = 0;
#pragma unroll
        for (int r = 0; r < kHold; ++r) mine += v[r];
        for (int j = kHold; j < m && l0 + j < n; ++j)  // long rows only
            mine += static_cast<long long>(__ldcg(&cs[l0 + j]));
        long long incl = mine;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long y = __shfl_up_sync(kFull, incl, off);
            if (lane >= off) incl += y;
        }
        const long long tot = __shfl_sync(kFull, incl, 31);
        if (tot <= 0) return -1;
        const long long target = cdf_target(ub, tot);
        // the first chunk whose cumulative sum exceeds the target: its lane, then its place there
        const unsigned bl = __ballot_sync(kFull, incl > target);
        const int ol = __ffs(bl) - 1;  // bl != 0: lane 31 holds tot > target
        int ch = -1;
        long long a = incl - mine;
        if (lane == ol) {
#pragma unroll
            for (int r = 0; r < kHold; ++r) {
                if (ch < 0 && r < m && l0 + r < n) {
                    if (a + v[r] > target)
                        ch = l0 + r;
                    else
                        a += v[r];
                }
            }
            for (int j = kHold; ch < 0 && j < m && l0 + j < n; ++j) {
                const long long w = static_cast<long long>(__ldcg(&cs[l0 + j]));
                if (a + w > target)
                    ch = l0 + j;
                else
                    a += w;
            }
        }
        const int chunk = __shfl_sync(kFull, ch, ol);
        const long long acc = __shfl_sync(kFull, a, ol);
        if (chunk < 0) return -1;  // (not reached: target < tot)
        const long long rem = target - acc;  // 0 <= rem < cs[chunk]
        // rescan that chunk from global memory with the same weights and order
        const int k = chunk / kCpt;
        const int cc = chunk - k * kCpt;
        const int s0 = k * p.Lr;
        const int s1 = min(p.V, s0 + p.Lr);
        const unsigned char *rt = row_ptr<EB>(p, b, pos, 0);
        const unsigned char *rd = pair ? row_ptr<EB>(p, b, pos, 1) : rt;
        const Geo gt = make_geo<EB>(rt, s0, s1, p.target, p.t_end);
        long long q[2];
        float w[2][G];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int g = cc * kChunk + h * 32 + lane;
#pragma unroll
            for (int k2 = 0; k2 < G; ++k2) {
                const int v = gt.vbase + g * G + k2;
                float we = 0.f;
                if (g < gt.ngran && v >= s0 && v < s1) {
                    const float t = Elt<EB>::gload(rt + static_cast<size_t>(v) * EB);
                    const float d = pair ? Elt<EB>::gload(rd + static_cast<size_t>(v) * EB) : 0.f;
                    we = elem_weight(t, d, pair, js, p.c);
                }
                w[h][k2] = we;
            }
            q[h] = fixq(group_sum<G>(w[h]));  // the group's sum, as the tile pass forms it
        }
        long long i0 = q[0], i1 = q[1];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long y0 = __shfl_up_sync(kFull, i0, off);
            const long long y1 = __shfl_up_sync(kFull, i1, off);
            if (lane >= off) {
                i0 += y0;
                i1 += y1;
            }
        }
        i1 += __shfl_sync(kFull, i0, 31);
        unsigned bh = __ballot_sync(kFull, i0 > rem);
        int half = 0;
        if (!bh) {
            bh = __ballot_sync(kFull, i1 > rem);
            half = 1;
        }
        int token = -1;
        if (bh) {
            const int gl = __ffs(bh) - 1;
            const long long excl = __shfl_sync(kFull, half ? (i1 - q[1]) : (i0 - q[0]), gl);
            if (lane == gl) {
                const int g = cc * kChunk + half * 32 + lane;
                float cum = 0.f;
                int esel = -1;
#pragma unroll
                for (int k2 = 0; k2 < G; ++k2) {
                    cum += half ? w[1][k2] : w[0][k2];
                    if (esel < 0 && excl + fixq(cum) > rem) esel = k2;
                }
                token = gt.vbase + g * G + (esel < 0 ? G - 1 : esel);
            }
            token = __shfl_sync(kFull, token, gl);
        }
        return token < 0 ? 0 : token;
    };

    // Draw e's chunk sums are all in: select its token, emit it, clear its scratch.
    // rec, js and ub were loaded once the draws were recorded (see phase C).
    auto finish_entry = [&](int e, uint32_t rec, const float4 &js, float ub) {
        if (rec == 0u) {  // never recorded: only after a wait upstream gave up
            timed_out = true;
            return;
        }
        const int u = static_cast<int>(rec & kRecUnit) - 1;
        const bool pair = (rec & kRecPair) != 0;
        const bool skip = (rec & kRecSkip) != 0 || (late_skip && !(js.y > 0.f));
        int b, pos;
        if (T::kBonus) {
            b = u;
            pos = bonus_pos(p, b);
        } else {
            b = u / p.units_per_seq;
            pos = u - b * p.units_per_seq;
        }
        // the draft tokens to emit, loaded while the token is located
        const int pre = (T::kBonus || MODE == kTreeSample) ? -1 : lane_draft_token(b, pos);
        int token = 0;
        if (!skip) {
            token = select_token(e, b, pos, pair, js, ub);
            if (token < 0 && pair) {
                // the residual vanished through rounding: draw from p_j instead
                if (lane == 0) atomicOr(p.status, SPEC_DEV_ZERO_RESIDUAL);
                resid_from_global(e, b, pos, js);
                token = select_token(e, b, pos, false, js, ub);
            }
            if (token < 0) token = 0;
        }
        if (T::kBonus) {
            if (lane == 0) p.bonus_token[b] = (pos < 0) ? -1 : token;
        } else if (MODE == kTreeSample) {
            if (lane == 0) p.ws_val[u] = token;  // the target's choice at node pos
        } else {
            emit_linear(b, pos, token, true, pre);
        }
        // leave the workspace zeroed (late_skip: the sequence's mask and every unit's statistics too)
        uint4 *cs = reinterpret_cast<uint4 *>(p.ws_csum + static_cast<size_t>(e) * p.Sr * kCpt);
        for (int i = lane; i < p.Sr * kCpt / 2; i += 32) cs[i] = make_uint4(0u, 0u, 0u, 0u);
        if (late_skip) {
            for (int i = lane; i < p.units_per_seq; i += 32)
                p.ws_stats[static_cast<size_t>(b) * p.units_per_seq + i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (lane == 0) p.ws_seqmask[b] = 0ull;
        }
        if (lane == 0) {
            p.ws_stats[u] = make_float4(0.f, 0.f, 0.f, 0.f);  // the other units' by their sequence
            p.ws_draw[e] = 0u;
        }
        __syncwarp();
    };

    // consume the pending unit-tile count: the warp that completes a unit finishes it
    auto resolve_pending = [&]() {
        if (!pend) return;
        pend = false;
        int last = 0;
        if (lane == 0)
            last = (pend_old + static_cast<unsigned>(pend_add) == static_cast<unsigned>(unit_nrows<MODE>(p, pend_pos) * S))
                       ? 1 : 0;
        last = __shfl_sync(kFull, last, 0);
        if (!last) return;
        __syncwarp();  // (the partials are validated as they are read: no fence needed)
        finish_unit(pend_unit, pend_b, pend_pos);
    };

    // the segment's last tile is reduced: merge the lanes, publish, count its tiles
    auto close_stats = [&]() {
        if (T::kSample)
            warp_merge_sc(am, as);
        else
            warp_merge_vi(am, ai);
        resolve_pending();
        if (lane == 0) {
            const uint2 part = T::kSample ? make_uint2(__float_as_uint(am), __float_as_uint(as))
                                          : make_uint2(__float_as_uint(am), static_cast<unsigned>(ai) + 1u);
#ifdef SPEC_TEST_HOOKS
            if (!(prow.unit == p.test_withhold && prow.r == 0 && run_k0 == 0))
#endif
            st_relaxed64(&p.ws_part[(static_cast<size_t>(prow.unit) * 2 + prow.r) * S + run_k0],
                         static_cast<unsigned long long>(part.x) | (static_cast<unsigned long long>(part.y) << 32));
            if (hasx)
                st_relaxed64(&p.ws_txw[static_cast<size_t>(prow.unit) * 2 + prow.r],
                             static_cast<unsigned long long>(__float_as_uint(xval)) | (1ull << 32));
            pend_old = atomicAdd(&p.ws_unit_cnt[prow.unit], static_cast<unsigned>(run_len));
        }
        pend = true;
        pend_unit = prow.unit;
        pend_b = prow.b;
        pend_pos = prow.pos;
        pend_add = run_len;
        srun = false;
    };

    int hslot = 0;                     // stage of the next tile to reduce
    uint32_t bar_par = 0;              // bit s: the phase parity stage s's mbarrier completes next
    auto advance_slot = [&]() {
        ++handled;
        bar_par ^= 1u << hslot;
        if (++hslot == nst) hslot = 0;
    };
    // A wait that gave up can leave bulk copies in flight into this warp's ring:
    // let them land (each wait bounded again) before the ring is used again or the CTA exits.
    auto drain = [&]() {
        while (handled < issued) {
            (void)wait_bar(ptx::smem_addr(&wc.full[hslot]), (bar_par >> hslot) & 1u);
            advance_slot();
        }
    };

    // ======================================================= phase A: statistics
    // Every row is streamed once; the warp that completes a unit decides it, and the
    // update that fixes a sequence's first rejection records its draw (or emits it).
    fill_ring();
    for (;;) {
        if (issued == handled) {
            resolve_pending();  // settle before anything that may wait
            if (!try_issue(true)) break;
            fill_ring();
        }
        const int s = hslot;
        const int4 d = wc.desc[s];
        unsigned char *buf = ring + static_cast<size_t>(s) * kStageBytes;
        const uint32_t bar = ptx::smem_addr(&wc.full[s]);
        const uint32_t parity = (bar_par >> s) & 1u;
        const int k = d.z;
        if (!srun) {
            // a new run: its row, and fresh lane statistics
            if (d.y != prow.id) prow = decode_row(d.y);
            srun = true;
            run_k0 = k;
            run_last = d.w;
            run_len = 0;
            am = neg_inf();
            as = 0.f;
            ai = INT_MAX;
            hasx = 0;
            xval = 0.f;
            px = -1;
            if (MODE == kLinearSample && prow.pos < p.K) {
                const int x = __ldg(&p.tokens[static_cast<size_t>(prow.b) * p.K + prow.pos]);
                px = (x >= 0 && x < p.V) ? x : -1;
            }
        }
        if (!wait_bar(bar, parity)) {
            timed_out = true;
            break;
        }
        uintptr_t w0, w1, c0, c1;
        tile_window(prow, k, w0, w1, c0, c1);
        const int ngran = static_cast<int>((w1 - w0) >> 4);
        const int vbase = static_cast<int>((static_cast<long long>(w0) - static_cast<long long>(prow.R0)) / EB);
        const uintptr_t R1 = prow.R0 + row_bytes;
        const bool patch = ngran > 0 && (w0 < prow.R0 || w1 > R1 || c0 > w0 || c1 < w1);
        if (patch) {
            if (lane < 16) {
                Geo g;
                g.glo = reinterpret_cast<const unsigned char *>(w0);
                g.ngran = ngran;
                g.c0 = static_cast<int>(c0 - w0);
                g.c1 = static_cast<int>(c1 - w0);
                g.a0 = w0 < prow.R0 ? static_cast<int>(prow.R0 - w0) : 0;
                g.a1 = static_cast<int>((R1 < w1 ? R1 : w1) - w0);
                g.vbase = vbase;
                g.patch = true;
                patch_row<EB>(buf, g, lane);
            }
            __syncwarp();
        }
        if (T::kSample)
            lane_sum<EB>(buf, ngran, p.c, lane, am, as);
        else
            lane_argmax<EB>(buf, ngran, vbase, lane, am, ai);
        if (px >= 0) {
            const int off = px - vbase;
            if (off >= 0 && off < ngran * G) {
                hasx = 1;
                xval = Elt<EB>::load(buf + off * EB);
            }
        }
        __syncwarp();
        if (patch) fence_proxy_async();  // generic writes to this stage precede its next bulk copy
        ++run_len;
        advance_slot();
        fill_ring();
        resolve_pending();
        if (k == run_last) close_stats();
    }

    if (draws) {
        drain();
        // ================================================= phase C: residual tiles
        // Every draw is recorded once every CTA is here.  Warp gw then takes the
        // residual tiles [RT * gw / W, RT * (gw + 1) / W): slices of the drawn row
        // pairs (or rows), each reduced to exact chunk sums of its weights.
        if (!grid_barrier(&p.ws_ctrl[5], gridDim.x, &s_flag)) timed_out = true;
        nst = NSC;  // nothing is in flight: re-cut the ring(s) into NSC residual stages
        islot = hslot = 0;
        const long long q1 = RT * (gw + 1) / nwarps;
        long long qi = RT * gw / nwarps;   // the next tile to issue
        // it is slice ik of draw ie (tracked as qi advances: no division per tile)
        int ie = static_cast<int>(qi / p.Sr);
        int ik = static_cast<int>(qi - static_cast<long long>(ie) * p.Sr);
        // The selects of phase D are spread over the grid (consecutive draws on different SMs):
        // warp gw selects draws [n * gw / W, n * (gw + 1) / W).  Every record is complete now:
        // the first one this warp issues and the first one it selects load together.
        const long long nd = p.n_draws;
        const int d0 = static_cast<int>(nd * gw / nwarps), d1 = static_cast<int>(nd * (gw + 1) / nwarps);
        uint32_t irec = (qi < q1) ? __ldcg(&p.ws_draw[ie]) : 0u;
        uint32_t drec = (d0 < d1) ? __ldcg(&p.ws_draw[d0]) : 0u;
        bool irec_ok = true;
        // the record of the next draw this warp issues, loaded one draw ahead
        uint32_t nrec = (qi < q1 && ie + 1 < nd && static_cast<long long>(ie + 1) * p.Sr < q1) ? __ldcg(&p.ws_draw[ie + 1]) : 0u;
        // The draw being issued, decoded once: its rows; its statistics are loaded for the
        // reducing side (hand_e / hand_js), which reaches the draw a tile or two later.
        const unsigned char *irt = nullptr, *ird = nullptr;
        int hand_e = -1;
        float4 hand_js = make_float4(0.f, 0.f, 0.f, 0.f);
        auto begin_draw = [&]() {
            if (irec == 0u) {          // never recorded (only after a timed-out wait): read nothing
                timed_out = true;
                irec = 1u | kRecSkip;
            }
            int u, b, pos;
            entry_unit(irec, u, b, pos);
            irt = row_ptr<EB>(p, b, pos, 0);
            ird = (irec & kRecPair) ? row_ptr<EB>(p, b, pos, 1) : irt;
            if (!(irec & kRecSkip)) {
                hand_e = ie;
                hand_js = __ldcg(&p.ws_stats[u]);
            }
        };
        auto issue_next = [&]() {
            if (!irec_ok) {
                irec_ok = true;
                irec = nrec;
                nrec = (ie + 1 < nd && static_cast<long long>(ie + 1) * p.Sr < q1) ? __ldcg(&p.ws_draw[ie + 1]) : 0u;
                begin_draw();
            }
            issue_resid(ie, ik, irec, irt, ird);
            ++qi;
            if (++ik == p.Sr) {
                ik = 0;
                ++ie;
                irec_ok = false;
            }
        };
        if (qi < q1) begin_draw();
        while (qi < q1 && issued - handled < nst) issue_next();
        __syncwarp();
        // phase D's statistics and uniform for its first draw: not needed before then
        float4 djs = make_float4(0.f, 0.f, 0.f, 0.f);
        float dub = 0.f;
        if (d0 < d1 && drec != 0u && !(drec & kRecSkip)) {
            const int u = static_cast<int>(drec & kRecUnit) - 1;
            djs = __ldcg(&p.ws_stats[u]);
            dub = __ldg(&p.u_bonus[(MODE == kTreeSample || T::kBonus) ? u : u / p.units_per_seq]);
        }
        int ce = -1, cu = 0;
        bool cpair = false, cskip = true;
        float4 js = make_float4(0.f, 0.f, 0.f, 0.f);
        while (handled < issued) {
            const int s = hslot;
            const int4 d = wc.desc[s];
            const int4 cg = wc.cgeo[s];
            unsigned char *buf = cstage(s);
            const uint32_t rec = static_cast<uint32_t>(d.z);
            const int e = d.y;
            const int k = d.w;
            if (e != ce) {
                ce = e;
                cpair = (rec & kRecPair) != 0;
                cskip = (rec & kRecSkip) != 0;
                cu = static_cast<int>(rec & kRecUnit) - 1;
                if (!cskip) js = (e == hand_e) ? hand_js : __ldcg(&p.ws_stats[cu]);
            }
            if (!wait_bar(ptx::smem_addr(&wc.full[s]), (bar_par >> s) & 1u)) {
                timed_out = true;
                break;
            }
            long long q[kCpt];
#pragma unroll
            for (int c = 0; c < kCpt; ++c) q[c] = 0;
            const bool tskip = cskip || (late_skip && !(js.y > 0.f));  // a non-finite unit: its bytes are ignored
            const bool patched = !tskip && cg.w != 0;
            if (!tskip) {
                const int s0 = k * p.Lr;
                const int s1 = min(p.V, s0 + p.Lr);
                if (patched) {  // an edge group to fix (rows off the 16-byte grid, tensor ends)
                    int cuu, cb, cpos;
                    entry_unit(rec, cuu, cb, cpos);
                    const Geo g0 = make_geo<EB>(row_ptr<EB>(p, cb, cpos, 0), s0, s1, p.target, p.t_end);
                    Geo g1 = g0;
                    if (cpair) g1 = make_geo<EB>(row_ptr<EB>(p, cb, cpos, 1), s0, s1, p.draft, p.d_end);
                    if (lane < 16) {
                        if (g0.patch) patch_row<EB>(buf, g0, lane);
                    } else if (cpair && g1.patch) {
                        patch_row<EB>(buf + kRowBuf, g1, lane - 16);
                    }
                    __syncwarp();
                }
                if (!cpair)
                    tile_resid<EB, kResidTail>(buf, cg.x, cg.y, cg.z, s0, s1, js, p.c, lane, q);
                else if (cg.y == cg.z)
                    tile_resid<EB, kResidPair>(buf, cg.x, cg.y, cg.z, s0, s1, js, p.c, lane, q);
                else
                    tile_resid<EB, kResidPairShifted>(buf, cg.x, cg.y, cg.z, s0, s1, js, p.c, lane, q);
            }
            __syncwarp();
            if (patched) fence_proxy_async();
            {
                const long long t = warp_sum64xN<kCpt>(q, lane);
                if (lane % kSumLanes == 0)
                    p.ws_csum[(static_cast<size_t>(e) * p.Sr + k) * kCpt + lane / kSumLanes] =
                        static_cast<unsigned long long>(t);
            }
            advance_slot();
            while (qi < q1 && issued - handled < nst) issue_next();
            __syncwarp();
        }
        drain();
        // ================================================= phase D: one select per draw
        if (!grid_barrier(&p.ws_ctrl[5], 2 * gridDim.x, &s_flag)) timed_out = true;
        for (int e = d0; e < d1; ++e) {
            if (e > d0) {  // more draws than warps: the later ones load here
                drec = __ldcg(&p.ws_draw[e]);
                if (drec != 0u && !(drec & kRecSkip)) {
                    const int u = static_cast<int>(drec & kRecUnit) - 1;
                    djs = __ldcg(&p.ws_stats[u]);
                    dub = __ldg(&p.u_bonus[(MODE == kTreeSample || T::kBonus) ? u : u / p.units_per_seq]);
                }
            }
            finish_entry(e, drec, djs, dub);
        }
        if (MODE == kTreeSample) {
            // ============================================= phase E: the walks
            if (!grid_barrier(&p.ws_ctrl[5], 3 * gridDim.x, &s_flag)) timed_out = true;
            const int b0 = static_cast<int>(static_cast<long long>(p.B) * gw / nwarps);
            const int b1 = static_cast<int>(static_cast<long long>(p.B) * (gw + 1) / nwarps);
            for (int b = b0; b < b1; ++b) emit_tree(b);
        }
    }

    drain();
    timed_out = __any_sync(kFull, timed_out);
    if (lane == 0 && timed_out) {
        atomicOr(p.status, SPEC_DEV_TIMEOUT);
        atomicOr(&p.ws_ctrl[4], 1u);  // leftovers anywhere: the last CTA clears the whole workspace
    }
    // ---- the last CTA to finish leaves the workspace zeroed: the control words always,
    //      everything else after a timed-out wait (whose values may have landed late,
    //      or never been consumed)
    __threadfence();  // this CTA's workspace writes precede its count
    __syncthreads();
    if (threadIdx.x == 0) s_flag = (atom_add_acq_rel(&p.ws_ctrl[1], 1u) == gridDim.x - 1) ? 1 : 0;
    __syncthreads();
    if (s_flag) {
        if (__ldcg(&p.ws_ctrl[4]) != 0u) {
            uint4 *w = reinterpret_cast<uint4 *>(p.ws_base + kCtrlWords * 4);
            const unsigned long long n = (p.ws_bytes - kCtrlWords * 4) / 16;
            for (unsigned long long i = threadIdx.x; i < n; i += blockDim.x) w[i] = make_uint4(0u, 0u, 0u, 0u);
            __threadfence();
        }
        __syncthreads();
        if (threadIdx.x < kCtrlWords) p.ws_ctrl[threadIdx.x] = 0u;
    }
}

}  // namespace spec
