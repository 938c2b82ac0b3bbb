// launch.cuh -- the launcher of spec_verify_kernel<EB, MODE>.  Each kern_*.cu
// unit includes this and instantiates it for one mode, so the kernel's
// instantiations compile as separate translation units in parallel.
#pragma once

#include <algorithm>

#include "host.h"
#include "verify_kernels.cuh"

#ifndef SPEC_MAX_STAGES
#define SPEC_MAX_STAGES 2
#endif

namespace spec {

#ifdef SPEC_TEST_HOOKS
int test_withhold_unit();  // test builds only
#endif

template <int EB, int MODE>
spec_status launch(const Params &p0, bool draws, cudaStream_t stream) {
    DeviceInfo di;
    int dev = 0;
    spec_status st = device_info(&di, &dev);
    if (st != SPEC_OK) return st;
    auto kernel = spec_verify_kernel<EB, MODE>;
    st = allow_max_dyn_smem(dev, reinterpret_cast<const void *>(kernel), &di);
    if (st != SPEC_OK) return st;
    Params p = p0;
    const Slicing rs = resid_slicing(p.V, EB);
    p.S = stats_tiles_per_row(p.V, EB);
    p.nseg = segments_per_row(p.V, EB);
    p.Sr = rs.S;
    p.Lr = rs.L;
    p.stats_segs = static_cast<long long>(p.B) * p.rows_per_seq * p.nseg;
    p.n_draws = draws ? (MODE == kTreeSample ? p.n_units : p.B) : 0;
    p.res_tiles = static_cast<long long>(p.n_draws) * p.Sr;
#ifdef SPEC_TEST_HOOKS
    p.test_withhold = test_withhold_unit();
#endif
    // ring depth: the deepest ring that keeps kMinCtas CTAs on an SM
    const size_t scratch =
        (MODE == kTreeGreedy || MODE == kTreeSample) ? static_cast<size_t>(kWarps) * 3 * p.units_per_seq * 4 : 0;
    int ns = 0, per_sm = 0;
    size_t dyn = 0;
    for (int cand : {SPEC_MAX_STAGES, 2}) {
        const size_t d = static_cast<size_t>(kWarps) * cand * kStageBytes + scratch;
        if (d > di.max_dyn) continue;
        const int b = blocks_per_sm(dev, reinterpret_cast<const void *>(kernel), d);
        if (b >= kMinCtas || (cand == 2 && b >= 1)) {
            ns = cand;
            per_sm = b;
            dyn = d;
            break;
        }
    }
    if (per_sm <= 0) return fail(SPEC_ERR_UNSUPPORTED, "kernel does not fit an SM (N=%d)", p.units_per_seq);
    p.nstage = ns;
    // Small problems (up to kStaticTilesPerWarp tiles per resident warp): a static split of the tiles,
    // balanced to one tile, over enough CTAs for every warp to get a tile.  Large ones: dynamic
    // segments, over enough CTAs for every warp to get a segment.  Never more than is resident.
    const long long resident = static_cast<long long>(per_sm) * di.sms;
    p.stats_tiles = static_cast<long long>(p.B) * p.rows_per_seq * p.S;
    p.static_split = p.stats_tiles <= kStaticTilesPerWarp * resident * kWarps ? 1 : 0;
    const long long units = p.static_split ? p.stats_tiles : p.stats_segs;
    const long long grid = std::min<long long>(std::max<long long>(1, (units + kWarps - 1) / kWarps), resident);
    const long long warps = grid * kWarps;
    p.nwarps = static_cast<int>(warps);
    // Rows a residual pass may re-read, in stream order, up to 1/kKeepDiv of L2, are read at normal
    // L2 priority and everything else first-to-evict, so the first draws find their rows in L2:
    // the row pairs of the first positions (linear), or every row (extra token alone).
    p.keep_rows = 0;
    if (draws) {
        const long long budget = static_cast<long long>(di.l2 / kKeepDiv) / (static_cast<long long>(p.V) * EB);
        const long long cand = (MODE == kLinearSample) ? 2ll * p.K * p.B : static_cast<long long>(p.B) * p.rows_per_seq;
        p.keep_rows = static_cast<int>(std::min(budget, cand));
    }
    if (p.stats_segs + (warps + 1) * kMaxGrab >= (1ll << 31) || p.res_tiles >= (1ll << 31))
        return fail(SPEC_ERR_UNSUPPORTED, "too many tiles (B=%d, V=%d)", p.B, p.V);
    // Warps wait on values that warps of other CTAs publish, so every CTA must be resident at once: a
    // cooperative launch guarantees that, or fails here (e.g. when other work holds part of the GPU).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(SPEC_ERR_CUDA, "cooperative launch (grid=%lld, stages=%d, smem=%zu): %s", grid, ns, dyn,
                    cudaGetErrorString(e));
    return SPEC_OK;
}

}  // namespace spec
