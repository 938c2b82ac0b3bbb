// host.h -- host-side helpers shared by the C ABI (spec_verify.cu) and the
// per-mode launch units (kern_*.cu): error text, device attributes, the
// tiling of a row, and the declaration of the kernel launcher.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>

#include "params.cuh"
#include "spec_verify.h"

namespace spec {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int sms = 0;
    size_t max_dyn = 0;  // opt-in dynamic shared memory per block
    size_t l2 = 0;       // L2 cache bytes
};

// Record a printf-style message as the calling thread's last error and return s.
spec_status fail(spec_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));

// Attributes of the current device (cached per device) and its index.
spec_status device_info(DeviceInfo *out, int *dev_out);

// Resident blocks per SM of a kernel at kThreads threads and `dyn` bytes of
// dynamic shared memory (cached).
int blocks_per_sm(int dev, const void *kernel, size_t dyn);

// Once per device and kernel: allow the kernel the largest dynamic shared
// memory next to its static part; di->max_dyn becomes that amount.  (The
// record of what was set lives in this library's host code, not in a
// function-local static of the launch template, which the dynamic linker
// would share with any other copy of the library in the process.)
spec_status allow_max_dyn_smem(int dev, const void *kernel, DeviceInfo *di);

// Stats tiles per row: kTileBytes windows on the 16-byte grid of global
// memory, the count for the worst alignment (a spare last window is empty).
int stats_tiles_per_row(int V, int eb);
int segments_per_row(int V, int eb);

// Residual slices of a row: at most kResidSliceBytes each, a whole number of
// 16-byte groups long, none empty.  A function of V and the element size only.
struct Slicing {
    int S;  // slices per row
    int L;  // elements per slice
};
Slicing resid_slicing(int V, int eb);

// Fill in the tiling of p0 (rows_per_seq and the problem sizes already set),
// choose the ring depth and grid, and launch spec_verify_kernel<EB, MODE> on
// `stream` as a cooperative launch (every CTA resident at once, or an error).
template <int EB, int MODE>
spec_status launch(const Params &p0, bool draws, cudaStream_t stream);

}  // namespace spec
