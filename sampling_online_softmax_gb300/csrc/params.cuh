// params.cuh -- what the host and the verify kernel share: tile and workspace
// constants, the kernel's modes, and its parameter block.  Included by the
// host-side launch code and by the device code in verify_kernels.cuh.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace spec {

#ifndef SPEC_WARPS
#define SPEC_WARPS 12
#endif
constexpr int kWarps = SPEC_WARPS;  // streaming warps per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kMaxStages = 4;             // mbarriers per warp: the residual phase may use more stages
#ifndef SPEC_TILE_KB
#define SPEC_TILE_KB 8
#endif
#ifndef SPEC_MIN_CTAS
#define SPEC_MIN_CTAS 1
#endif
constexpr int kMinCtas = SPEC_MIN_CTAS;              // CTAs resident per SM
constexpr int kTileBytes = SPEC_TILE_KB * 1024;      // stats tile: a window of one row on the 16-byte grid
constexpr int kStageBytes = kTileBytes;              // a stats stage of a warp's ring
#ifndef SPEC_ROW_BUF
#define SPEC_ROW_BUF 4096
#endif
constexpr int kRowBuf = SPEC_ROW_BUF;                // residual row buffer: a slice plus its two ragged groups
constexpr int kResidSliceBytes = kRowBuf - 32;       // at most this many bytes of each row per residual tile
constexpr int kCStageBytes = 2 * kRowBuf;            // a residual stage: the slice of a row pair
constexpr int kChunk = 64;                           // 16-byte groups per residual chunk
constexpr int kCpt = kRowBuf / 16 / kChunk;          // residual chunks per tile (the whole row buffer)
static_assert(kResidSliceBytes % 16 == 0 && kResidSliceBytes + 32 <= kRowBuf, "a slice's window fits its buffer");
static_assert(kRowBuf % (16 * kChunk) == 0 && (kCpt == 2 || kCpt == 4), "two or four chunks per residual tile");
static_assert(kStageBytes % kCStageBytes == 0 && kStageBytes % 128 == 0, "stage layout");
// Warps of a CTA that reduce residual tiles (all of them: the reduction is bound by each warp's
// dependent arithmetic, so fewer warps with deeper rings measured slower).
constexpr int kCWarps = kWarps;
#ifndef SPEC_SEG_TILES
#define SPEC_SEG_TILES 4
#endif
constexpr int kSegTiles = SPEC_SEG_TILES;  // stats tiles per segment: one partial each, never split between warps
#ifndef SPEC_MAX_GRAB
#define SPEC_MAX_GRAB 4
#endif
constexpr int kMaxGrab = SPEC_MAX_GRAB;  // stats segments taken from the global counter at once (at most)
#ifndef SPEC_TAIL_ZONE
#define SPEC_TAIL_ZONE 16
#endif
#ifndef SPEC_GUIDED_DIV
#define SPEC_GUIDED_DIV 2
#endif
constexpr int kTailZone = SPEC_TAIL_ZONE;    // below this many segments per warp left, grab without reserve
constexpr int kGuidedDiv = SPEC_GUIDED_DIV;  // a grab takes 1/kGuidedDiv of a fair share of what is left
#ifndef SPEC_KEEP_DIV
#define SPEC_KEEP_DIV 4
#endif
constexpr int kKeepDiv = SPEC_KEEP_DIV;  // rows kept in L2 for a residual pass: at most 1/kKeepDiv of L2
constexpr int kHold = 12;               // chunk sums per lane held in registers while an extra token is located
#ifndef SPEC_STATIC_TILES_PER_WARP
#define SPEC_STATIC_TILES_PER_WARP 32
#endif
constexpr long long kStaticTilesPerWarp = SPEC_STATIC_TILES_PER_WARP;  // up to this many stats tiles per warp: a static split
#ifndef SPEC_WAIT_LIMIT
#define SPEC_WAIT_LIMIT (1u << 22)
#endif
#ifndef SPEC_SPIN_LIMIT
#define SPEC_SPIN_LIMIT (1u << 21)
#endif
constexpr uint32_t kWaitLimit = SPEC_WAIT_LIMIT;  // mbarrier polls before a copy counts as lost
constexpr uint32_t kSpinLimit = SPEC_SPIN_LIMIT;  // polls (with a short sleep) of a value another warp publishes
constexpr int kCtrlWords = 8;                     // workspace control words (32 bytes)
constexpr unsigned kFull = 0xffffffffu;

enum Mode : int {
    kLinearSample = 0,
    kLinearGreedy = 1,
    kTreeGreedy = 2,
    kBonusSample = 3,
    kBonusGreedy = 4,
    kTreeSample = 5,  // tree walk with the target's choice drawn at every node
};

enum TileKind : int { kTileNone = 0, kTileStats = 1, kTileResid = 2 };

// A draw record: (unit + 1) | pair | skip.
constexpr uint32_t kRecUnit = (1u << 30) - 1;
constexpr uint32_t kRecPair = 1u << 30;  // weights max(0, p - q); else p
constexpr uint32_t kRecSkip = 1u << 31;  // nothing to draw (non-finite row, bad length)

struct Params {
    const unsigned char *target;   // [B, t_rows, V]
    const unsigned char *draft;    // [B, K, V] (sampling) or null
    const unsigned char *t_end;    // one past the last byte of target
    const unsigned char *d_end;    // one past the last byte of draft
    int B, K, V;
    int t_rows;                    // target rows per sequence: K+1 (linear), N (tree)
    int rows_per_seq;              // row slots per sequence in the stats tiling
    int units_per_seq;             // K+1 (linear), N (tree), 1 (extra token alone)
    int n_units;
    int S;                         // stats tiles per row (windows of kTileBytes on the 16-byte grid)
    int nseg;                      // segments per row: ceil(S / kSegTiles) (dynamic mode)
    int static_split;              // 1: warp w reduces stats tiles [T*w/W, T*(w+1)/W) (small problems)
    long long stats_tiles;         // T = rows * S
    int nwarps;                    // W = grid * kWarps
    int keep_rows;                 // stats rows with id < keep_rows are read at normal L2 priority (the
                                   // rest first-to-evict), so that a residual pass finds them in L2
    int Sr, Lr;                    // residual slices per entry, elements per slice
    int nstage;                    // stages per warp ring (2..kMaxStages)
    long long stats_segs;          // B * rows_per_seq * nseg
    int n_draws;                   // draws recorded: B (linear, extra token alone), B * N (sampled tree) or 0
    long long res_tiles;           // n_draws * Sr
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
    uint32_t *ws_ctrl;             // [0] stats segments taken, [1] CTAs finished, [4] some wait gave up
                                   // (clear everything), [5] grid-barrier arrivals; [2], [3], [6], [7] unused
    unsigned char *ws_base;        // the workspace: ws_bytes bytes, 16-byte aligned
    unsigned long long ws_bytes;
#ifdef SPEC_TEST_HOOKS
    int test_withhold;             // test builds only: the unit whose row-0 partial at tile 0 is never published
#endif
    uint32_t *ws_unit_cnt;         // [n_units] stats tiles published per unit
    uint32_t *ws_seq_cnt;          // [B] units decided per sequence (K >= 32 and trees)
    unsigned long long *ws_seqmask;  // [B] decided bits 0..31, accepted bits 32..63 (linear, K < 32)
    int32_t *ws_acc;               // [B*K] accept bits
    int32_t *ws_val;               // [B*units_per_seq] argmax per unit (greedy)
    unsigned long long *ws_part;   // [n_units * 2 * S] run partials at the run's first tile: (mc | s << 32) or (max | (index + 1) << 32)
    unsigned long long *ws_txw;    // [n_units * 2] the draft token's logit in each row: bits | 1 << 32
    float4 *ws_stats;              // [n_units] (MCt, 1/St, MCd, 1/Sd) of units that may draw
    uint32_t *ws_draw;             // [n_draws] draw records: (unit + 1) | pair | skip
    unsigned long long *ws_csum;   // [n_draws * Sr * kCpt] residual chunk sums (int64, units of 2^-52)
};

}  // namespace spec
