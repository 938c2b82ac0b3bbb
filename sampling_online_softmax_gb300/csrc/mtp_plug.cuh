// mtp_plug.cuh -- the MTP token plug-in: the draft layer's next input tokens,
// written on the device from a linear verify's outputs.
//
// "Beschleunigung von Sonar durch Spekulation" (Perplexity), section "MTP":
// the draft layer predicts the token after position i from the target's hidden
// state H_i together with the token that follows position i, so its input
// token buffer is the target's shifted left by one step.  Section
// "MTP-Zeitplan für ein einzelnes Token": after the target's input tokens are
// shifted, a kernel inserts the target's next tokens at their places, so that
// no CPU-GPU synchronisation follows acceptance; the draft then runs over the
// same positions (redundant work past the accepted prefix).
//
// Row b: next[i] = in[i + 1] for i < K, next[K] = pad; then the n = num_emitted[b]
// emitted tokens (the accepted draft tokens, then the extra token) overwrite
// positions 0 .. n - 1; seq_lens[b] += n.  A count outside [0, K + 1] leaves the
// row shifted and the length unchanged, and sets SPEC_DEV_BAD_LENGTH.
//
// One warp per sequence, 32 positions at a time in increasing order: every
// lane reads its chunk before any lane writes it, and a chunk reads only
// positions the later chunks write, so next may be in itself.  Nothing waits
// on anything.
#pragma once

#include <cstdint>

#include "spec_verify.h"

namespace spec {

constexpr int kPlugWarps = 8;  // sequences per CTA

__global__ void __launch_bounds__(kPlugWarps * 32)
    mtp_plug_kernel(const int32_t *in, int B, int K, const int32_t *__restrict__ emitted,
                    const int32_t *__restrict__ num_emitted, int32_t pad, int32_t *next, int32_t *seq_lens,
                    uint32_t *status) {
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * kPlugWarps + (threadIdx.x >> 5);
    if (b >= B) return;  // the whole warp
    const int W = K + 1;
    const int n = __ldg(&num_emitted[b]);
    const bool ok = n >= 0 && n <= W;
    const int32_t *ir = in + static_cast<size_t>(b) * W;
    const int32_t *er = emitted + static_cast<size_t>(b) * W;
    int32_t *nr = next + static_cast<size_t>(b) * W;
    for (int base = 0; base < W; base += 32) {
        const int i = base + lane;
        int32_t v = 0;
        if (i < W) {
            if (ok && i < n)
                v = __ldg(&er[i]);       // the target's next token at position i
            else
                v = (i < K) ? ir[i + 1] : pad;  // the shift (plain load: next may alias in)
        }
        __syncwarp();
        if (i < W) nr[i] = v;
        __syncwarp();
    }
    if (lane == 0) {
        if (!ok)
            atomicOr(status, SPEC_DEV_BAD_LENGTH);
        else if (seq_lens)
            seq_lens[b] += n;
    }
}

}  // namespace spec
