// tree_mask.cuh -- the tree attention mask of a candidate tree, and its depths.
//
// "Speculative-Decoding / Medusa" blog, section 三 (Attention Tree): the tree is
// flattened into one sequence and verified in one target pass, under a mask
// modelled on the causal mask, so that no token attends to a token of another
// path.  Row i of the mask therefore holds node i and every ancestor of node i
// (its root path); depth[i], the number of edges from the root, is the token's
// position offset.
//
// One warp per row: lane 0 walks from node i up to the root, which takes at
// most i steps because every parent precedes its child (a parent that does
// not stops the walk and sets SPEC_DEV_BAD_TREE), setting the row's bits in
// shared memory; the warp then writes the row out coalesced.  Nothing waits on
// anything, so nothing here can hang.
#pragma once

#include <cstdint>

#include "spec_verify.h"

namespace spec {

constexpr int kMaskWarps = 8;          // rows in flight per CTA
constexpr int kMaxMaskNodes = 16384;   // W <= 512 words a row: 16 KB of shared memory per CTA

__global__ void __launch_bounds__(kMaskWarps * 32)
    tree_mask_kernel(const int32_t *parents, int N, int W, uint32_t *mask, int32_t *depth, uint32_t *status) {
    extern __shared__ uint32_t srow[];  // kMaskWarps rows of W words
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint32_t *row = srow + static_cast<size_t>(warp) * W;
    for (int i = blockIdx.x * kMaskWarps + warp; i < N; i += gridDim.x * kMaskWarps) {
        for (int w = lane; w < W; w += 32) row[w] = 0u;
        __syncwarp();
        if (lane == 0) {
            int cur = i;
            int d = 0;
            bool bad = false;
            row[cur >> 5] |= 1u << (cur & 31);
            while (cur != 0) {
                const int par = __ldg(&parents[cur]);
                if (par < 0 || par >= cur) {
                    bad = true;
                    break;
                }
                cur = par;
                ++d;
                row[cur >> 5] |= 1u << (cur & 31);
            }
            depth[i] = d;
            if (bad) atomicOr(status, SPEC_DEV_BAD_TREE);
        }
        __syncwarp();
        uint32_t *out = mask + static_cast<size_t>(i) * W;
        for (int w = lane; w < W; w += 32) out[w] = row[w];
        __syncwarp();
    }
}

}  // namespace spec
