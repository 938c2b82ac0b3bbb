/*
 * spec_verify.h -- C ABI of libspecverify.so, the verify-and-sample step of
 * speculative decoding on NVIDIA GB300 (sm_103a).
 *
 * The operation ("Beschleunigung von Sonar durch Spekulation", Perplexity,
 * section "Spekulatives Decoding", phases "Akzeptanz" and "Zielgenerierung";
 * section "Ziel-Entwurf"): after the target model has scored a draft of K
 * tokens, find the longest prefix of the draft the target accepts, and draw
 * one extra token from the target at the first mismatch or after the last
 * draft token, so that at most K + 1 tokens leave one step.  Acceptance
 * compares the full draft and target distributions; the rule used is that of
 * the method the page cites ("Fast Inference from Transformers via
 * Speculative Decoding"):
 *
 *   p_i = softmax(target_i / T), q_i = softmax(draft_i / T)      (over V)
 *   accept draft token x_i  iff  u_i < min(1, p_i(x_i) / q_i(x_i)), in order i = 0..K-1
 *   j = first rejected position, or K if none
 *   extra token ~ max(0, p_j - q_j) / W  if j < K,   ~ p_K  if j == K
 *   (inverse CDF: first v with cumulative weight C_v > u_b * W)
 *
 * With T == 0 (greedy): accept iff x_i == argmax target_i (lowest index on
 * ties) and the extra token is argmax target_j.  The tree variant ("Speculative-
 * Decoding / Medusa" blog, section 三 Attention Tree) follows, from the root,
 * the child whose token equals the target's argmax at the current node.
 *
 * Conventions shared by every entry point
 *   - Every pointer except `stream` is DEVICE memory owned by the caller; the
 *     library allocates nothing and keeps no pointer after the call returns.
 *   - Logits are row-major with the vocabulary contiguous (row stride V
 *     elements), fp32 or bf16, aligned to their element size.
 *   - Calls are stream-ordered and asynchronous: they enqueue kernels on
 *     `stream` (a cudaStream_t; NULL means the legacy default stream) and
 *     return without synchronising.  Outputs are valid once the stream has
 *     reached that point.
 *   - Argument errors are found on the host before anything is enqueued and
 *     return a status (nothing is written).  A failed launch returns
 *     SPEC_ERR_CUDA.  Errors that depend on device data are OR-ed as
 *     SPEC_DEV_* bits into *dev_status (which the caller zeroes); kernels never
 *     trap and never abort.
 *   - All arithmetic on the device is fp32 (bf16 inputs are widened exactly);
 *     cumulative sums for the inverse CDF are exact int64 sums of the fp32
 *     weights of 16-byte groups of logits, in units of 2^-52.
 *   - Workspace: every entry point except spec_verify_linear_static and
 *     spec_tree_mask needs a caller-owned device workspace of
 *     spec_workspace_bytes_*() bytes, 16-byte aligned and zero-filled before
 *     its first use.  Every call leaves it zero-filled again -- also a call
 *     that reports SPEC_DEV_TIMEOUT: its last CTA then clears every byte the
 *     call used -- so one zeroing suffices for any number of calls, but one
 *     workspace must not be shared by calls that may run at the same time.
 *   - Residency: the verify kernel's warps wait (bounded) on values that
 *     warps of other CTAs publish, so it is launched cooperatively: all its
 *     CTAs (at most one per SM) are resident at once, or the launch fails and
 *     the call returns SPEC_ERR_CUDA.  A launch can fail that way when other
 *     work holds SMs (an MPS client limited to part of the GPU, a green
 *     context); it never deadlocks waiting for a CTA that cannot start.
 *   - Apart from a per-thread copy of the last error message, the library keeps
 *     only caches filled once per device and guarded by locks (a kernel's
 *     occupancy and shared-memory limit, the static workspace's address); the
 *     functions may be called from several host threads.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

/* Exported symbols: the library is built with hidden visibility, and only the
 * functions declared here are exported from it. */
#if defined(__GNUC__)
#define SPEC_API __attribute__((visibility("default")))
#else
#define SPEC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum spec_status {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1, /* a null, misaligned or out-of-range argument */
    SPEC_ERR_UNSUPPORTED = 2, /* valid, but beyond what this library handles (e.g. V too large) */
    SPEC_ERR_CUDA = 3,        /* the CUDA runtime reported an error; see spec_last_error() */
    SPEC_ERR_WORKSPACE = 4    /* workspace missing, too small or misaligned */
} spec_status;

typedef enum spec_dtype {
    SPEC_F32 = 0,  /* IEEE binary32 logits */
    SPEC_BF16 = 1  /* bfloat16 logits (upper half of an IEEE binary32) */
} spec_dtype;

/* Bits OR-ed into *dev_status by the kernels. */
#define SPEC_DEV_BAD_TOKEN     1u  /* a draft token outside [0, V): treated as rejected */
#define SPEC_DEV_NONFINITE     2u  /* a row whose max or exp-sum is not finite; outputs unspecified */
#define SPEC_DEV_TIMEOUT       4u  /* a bounded wait (a copy, or a value another warp publishes) gave up; outputs unspecified, workspace cleared */
#define SPEC_DEV_ZERO_RESIDUAL 8u  /* residual weight W == 0 at a rejection: drew from p_j instead */
#define SPEC_DEV_BAD_TREE     16u  /* parents[] not topological (0 <= parents[c] < c): edge ignored */
#define SPEC_DEV_BAD_LENGTH   32u  /* spec_sample_bonus: accept_len[b] outside [0, K] (token -1);
                                      spec_mtp_plug: num_emitted[b] outside [0, K+1] */

/* Bytes of workspace spec_verify_linear needs for B sequences of K draft
 * tokens over a vocabulary of V logits of `dtype` (0 for invalid sizes). */
SPEC_API size_t spec_workspace_bytes_linear(int B, int K, int V, spec_dtype dtype);

/* Bytes of workspace spec_sample_bonus needs for B sequences. */
SPEC_API size_t spec_workspace_bytes_bonus(int B, int V, spec_dtype dtype);

/* Bytes of workspace spec_sample_rows needs for B rows of V logits. */
SPEC_API size_t spec_workspace_bytes_rows(int B, int V, spec_dtype dtype);

/* Bytes of workspace spec_verify_tree needs for B sequences of N tree nodes. */
SPEC_API size_t spec_workspace_bytes_tree(int B, int N, int V, spec_dtype dtype);

/* Bytes of workspace spec_verify_tree_sample needs (one draw per node: grows
 * with B * N * V). */
SPEC_API size_t spec_workspace_bytes_tree_sample(int B, int N, int V, spec_dtype dtype);

/*
 * Linear verify and (optionally) the extra token, in one launch.
 *
 *   target_logits [B, K+1, V]  row i scores draft token i; row K is the tail.
 *   draft_logits  [B, K, V]    the draft's logits for the same positions; may be
 *                              NULL when temperature == 0 (greedy) or K == 0.
 *   dtype, B >= 0, K >= 0, V >= 1.
 *   draft_tokens  [B, K] int32 the drafted tokens x_i (may be NULL when K == 0).
 *   u_accept      [B, K] fp32  uniforms in [0, 1) for the acceptance tests;
 *                              ignored (may be NULL) when greedy or K == 0.
 *   u_bonus       [B]    fp32  uniform in [0, 1) for the extra token, or NULL to
 *                              emit no extra token (spec_sample_bonus can draw it
 *                              later); ignored when greedy except as the switch.
 *   temperature   T >= 0, finite; T == 0 selects greedy mode.
 * Outputs (device, caller-owned):
 *   accept_len    [B]      j = number of accepted draft tokens, 0 <= j <= K.
 *   out_tokens    [B, K+1] x_0..x_{j-1}, then the extra token (if u_bonus), then -1.
 *                          Required when u_bonus != NULL, else may be NULL.
 *   num_emitted   [B]      j + 1 with an extra token, j without.
 *   probs_out     [B, K, 3] or NULL: p_i(x_i), q_i(x_i), min(1, p_i/q_i) for every
 *                          position (computed for all K, not only up to j); sampling only.
 *   dev_status    [1]      SPEC_DEV_* bits OR-ed in.
 *   workspace, workspace_bytes: see the conventions above.
 */
SPEC_API spec_status spec_verify_linear(const void *target_logits, const void *draft_logits,
                               spec_dtype dtype, int B, int K, int V,
                               const int32_t *draft_tokens, const float *u_accept,
                               const float *u_bonus, float temperature,
                               int32_t *accept_len, int32_t *out_tokens, int32_t *num_emitted,
                               float *probs_out, uint32_t *dev_status,
                               void *workspace, size_t workspace_bytes, void *stream);

/*
 * The extra token alone, for callers that already hold accept_len: draws from
 * max(0, p_j - q_j) / W at j = accept_len[b] < K, or from p_K when j == K
 * (argmax of target row j when temperature == 0).  Same layouts as above.
 *   accept_len  [B] int32 (device, input); u_bonus [B] (ignored when greedy).
 *   bonus_token [B] int32 (device, output); -1 where accept_len[b] is out of
 *               range (and SPEC_DEV_BAD_LENGTH is set).
 *   workspace, workspace_bytes: spec_workspace_bytes_bonus(B, V, dtype) bytes.
 */
SPEC_API spec_status spec_sample_bonus(const void *target_logits, const void *draft_logits,
                              spec_dtype dtype, int B, int K, int V,
                              const int32_t *accept_len, const float *u_bonus, float temperature,
                              int32_t *bonus_token, uint32_t *dev_status,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * One token per row: the draft side's choice of its next draft token (the
 * draft proposes tokens drawn from its own distribution q in the cited
 * speculative-sampling method), or any row a caller wants sampled.
 *   logits [B, V] (device, row-major, fp32 or bf16), u [B] fp32 in [0, 1)
 *   (ignored, may be NULL, when temperature == 0), temperature T >= 0.
 *   tokens [B] int32 (device, output): the first v whose cumulative weight of
 *   softmax(l / T) exceeds u[b] * W (exact int64 sums, as in the extra token),
 *   or the lowest-index argmax when T == 0.
 *   workspace, workspace_bytes: spec_workspace_bytes_rows(B, V, dtype) bytes.
 * It runs the extra-token path with no draft (K = 0).
 */
SPEC_API spec_status spec_sample_rows(const void *logits, spec_dtype dtype, int B, int V, const float *u, float temperature,
                             int32_t *tokens, uint32_t *dev_status, void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * Greedy verify of a candidate tree ("Speculative-Decoding / Medusa" blog,
 * section 三): at the current node take argmax of its target row; move to the
 * lowest-index child whose token equals it; stop when none does or max_depth
 * nodes were accepted; the extra token is argmax at the last accepted node.
 *
 *   target_logits [B, N, V]  row n holds the target logits after node n;
 *                            node 0 is the root (the last accepted token).
 *   parents       [N] int32  parents[0] ignored; 0 <= parents[c] < c for c >= 1.
 *   node_tokens   [B, N]     candidate token of each node (column 0 ignored).
 *   max_depth >= 0, N >= 1, V >= 1.
 * Outputs (max_depth + 1 columns, -1 padded):
 *   path_nodes [B, max_depth+1]  0, n_1, n_2, ... (node ids of the accepted path)
 *   path_len   [B]               number of accepted non-root nodes
 *   out_tokens [B, max_depth+1]  tokens of n_1..n_len, then the extra token
 */
SPEC_API spec_status spec_verify_tree(const void *target_logits, spec_dtype dtype, int B, int N, int V,
                             const int32_t *parents, const int32_t *node_tokens, int max_depth,
                             int32_t *path_nodes, int32_t *path_len, int32_t *out_tokens,
                             uint32_t *dev_status, void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * Tree verify in sampling mode ("Speculative-Decoding / Medusa" blog, section
 * 三: the target's choice at a node may be greedy or sampled).  At every node n
 * the target's choice is a draw from softmax(target_n / T) by inverse CDF with
 * the caller's uniform u_nodes[b, n] (the first v whose cumulative weight
 * exceeds u * W, over exact int64 sums as in the linear draw).  The walk is that
 * of spec_verify_tree with the draw in place of the argmax: from the root, move
 * to the lowest-index child whose token equals the draw at the current node;
 * stop when none does or max_depth nodes were accepted.  The extra token is
 * the draw at the last accepted node.  Every node is drawn, visited or not
 * (a data-parallel pass: two reads of every row, the second mostly from L2).
 *
 *   target_logits [B, N, V], parents [N], node_tokens [B, N]: as spec_verify_tree.
 *   u_nodes       [B, N] fp32 in [0, 1): one uniform per node (device).
 *   temperature   T > 0, finite.
 *   max_depth, path_nodes, path_len, out_tokens, dev_status: as spec_verify_tree.
 *   workspace, workspace_bytes: spec_workspace_bytes_tree_sample(B, N, V, dtype).
 */
SPEC_API spec_status spec_verify_tree_sample(const void *target_logits, spec_dtype dtype, int B, int N, int V,
                                    const int32_t *parents, const int32_t *node_tokens, const float *u_nodes,
                                    float temperature, int max_depth, int32_t *path_nodes, int32_t *path_len,
                                    int32_t *out_tokens, uint32_t *dev_status, void *workspace,
                                    size_t workspace_bytes, void *stream);

/*
 * The tree attention mask of a candidate tree ("Speculative-Decoding / Medusa"
 * blog, section 三: the tree is flattened into one sequence and a mask modelled
 * on the causal mask keeps tokens of different paths apart).  Row i holds node
 * i and every ancestor of node i; depth[i] is the number of edges from the
 * root (the token's position offset).
 *   parents    [N] int32 (device): parents[0] ignored, 0 <= parents[c] < c.
 *   mask_words [N, ceil(N/32)] uint32 (device, output): bit (j % 32) of word
 *              j / 32 of row i is set iff node j is node i or its ancestor.
 *   depth      [N] int32 (device, output).
 *   dev_status [1]: SPEC_DEV_BAD_TREE when a parent breaks the rule; that
 *              node's row and depth then hold the path up to the bad edge.
 * 1 <= N <= 16384.  No workspace; one small launch.
 */
SPEC_API spec_status spec_tree_mask(const int32_t *parents, int N, uint32_t *mask_words, int32_t *depth, uint32_t *dev_status,
                           void *stream);

/*
 * Sparse candidate tree ("Speculative-Decoding / Medusa" blog, section 四,
 * optimized tree construction).  With a_k^(i) the accuracy of head k's i-th
 * ranked token (taken as independent), the node reached by the rank path
 * [i_1 .. i_m] is accepted with probability prod_j a_j^(i_j), and E[L] is the
 * sum of that product over the tree's non-root nodes.  The tree grows from
 * the root one node at a time by the candidate (a child of a node already in
 * the tree) of largest product, until it holds n_nodes nodes or no candidate
 * is left.  Equal products go to the smaller depth, then to the
 * lexicographically smaller rank path.  Nodes are numbered by (depth, rank
 * path), so 0 <= parents[c] < c and the result feeds spec_tree_mask and
 * spec_verify_tree / spec_verify_tree_sample as it is.
 *
 * Unlike every other entry point this one runs on the HOST (all pointers are
 * host memory, no stream): the tree has a few dozen nodes and is built once
 * per accuracy table, not per decode step.
 *   accuracy     [K * S] double: accuracy[(k-1) * S + (i-1)] = a_k^(i), in [0, 1].
 *   K            heads (the tree's depth limit), 1 <= K <= 64.
 *   S            ranked tokens per head, 1 <= S <= 4096.
 *   n_nodes      nodes wanted, the root included, 1 <= n_nodes <= 16384.
 * Outputs (n_nodes entries each; the first *n_built are written):
 *   parents      parents[0] = -1, else the parent's number.
 *   depth        the node's depth (0 for the root).
 *   rank         the rank i of the node's token among its head's candidates
 *                (1-based; 0 for the root).
 *   n_built      min(n_nodes, the full tree's size).
 *   expected_len E[L] of the tree, or NULL.
 * Errors: SPEC_ERR_INVALID_ARG for sizes out of range, a null pointer, or an
 * accuracy that is not a finite value in [0, 1].
 */
SPEC_API spec_status spec_build_sparse_tree(const double *accuracy, int K, int S, int n_nodes, int32_t *parents,
                                            int32_t *depth, int32_t *rank, int *n_built, double *expected_len);

/*
 * MTP token plug-in ("Beschleunigung von Sonar durch Spekulation", sections
 * "MTP" and "MTP-Zeitplan für ein einzelnes Token"): the draft layer at
 * position i reads the target's hidden state H_i with the token that follows
 * position i, so its input is the target's input shifted left by one; after
 * verification the target's next tokens go into their places on the device,
 * and the sequence lengths advance, with no host round trip.
 *
 *   in_tokens   [B, K+1] int32  the target's input tokens of the step: row b is
 *                               (the token the step started from, x_0 .. x_{K-1});
 *                               for single-token MTP (K = 1) these are the 2 * B
 *                               tokens the target scored.
 *   out_tokens  [B, K+1] int32  spec_verify_linear's out_tokens (accepted draft
 *                               tokens, then the extra token).
 *   num_emitted [B] int32       spec_verify_linear's num_emitted.
 *   pad                         the token written at position K when nothing is
 *                               shifted into it (only when fewer than K + 1 tokens
 *                               were emitted).
 * Outputs (device, caller-owned):
 *   next_tokens [B, K+1] int32  next[b, i] = out_tokens[b, i] for i < n_b, else
 *                               in_tokens[b, i + 1] for i < K, else pad; it may be
 *                               in_tokens itself (in place), but not out_tokens.
 *   seq_lens    [B] int32       incremented by num_emitted[b] in place; NULL to skip.
 *   dev_status  [1]             SPEC_DEV_BAD_LENGTH when num_emitted[b] is outside
 *                               [0, K+1] (that row is only shifted, its length unchanged).
 * B >= 0, K >= 0, every pointer 4-byte aligned.  No workspace; one small launch
 * (one warp per sequence), ordered after the verify on the same stream.
 */
SPEC_API spec_status spec_mtp_plug(const int32_t *in_tokens, int B, int K, const int32_t *out_tokens,
                                   const int32_t *num_emitted, int32_t pad, int32_t *next_tokens,
                                   int32_t *seq_lens, uint32_t *dev_status, void *stream);

/*
 * spec_verify_linear with the library's own workspace.  The pages describe no
 * such call: it exists for callers that cannot allocate device memory at the
 * point where they verify -- e.g. a host program embedded in an inference
 * engine whose memory pool already owns the device, or a decode loop that must
 * not call cudaMalloc / cudaFree between steps because cudaFree synchronises
 * the whole device.  It allocates nothing (no cudaMalloc, no cudaFree, no
 * allocating library routine).
 *
 * The workspace is one statically sized array per device, compiled into the
 * library: SPEC_STATIC_WORKSPACE_BYTES bytes.  Shapes whose
 * spec_workspace_bytes_linear(B, K, V, dtype) exceeds that are rejected with
 * SPEC_ERR_WORKSPACE (spec_last_error() gives both sizes); use
 * spec_verify_linear with a workspace of your own for those.
 *
 * First call on each device: it looks up the array's device address
 * (cudaGetSymbolAddress, with that device current; this may also load the
 * library's kernels onto the device) and keeps it for the life of the
 * process.  Make one call on every device you will use before you begin any
 * stream capture on it.  Resetting a device (cudaDeviceReset) after that
 * first call is not supported: the kept address would name memory of the
 * destroyed context.
 *
 * Every call clears the part of the array it uses with cudaMemsetAsync on
 * `stream` before its kernel, so no earlier call's leftovers matter.  There is
 * ONE array per device and process: calls that may overlap in time (different
 * streams, or host threads without ordering) race on it and give wrong
 * results.  Issue them on one stream, or use spec_verify_linear.
 *
 * Arguments, outputs and errors are those of spec_verify_linear, without
 * `workspace` and `workspace_bytes`.
 */
#define SPEC_STATIC_WORKSPACE_BYTES (16u << 20)

SPEC_API spec_status spec_verify_linear_static(const void *target_logits, const void *draft_logits,
                                      spec_dtype dtype, int B, int K, int V,
                                      const int32_t *draft_tokens, const float *u_accept,
                                      const float *u_bonus, float temperature,
                                      int32_t *accept_len, int32_t *out_tokens, int32_t *num_emitted,
                                      float *probs_out, uint32_t *dev_status, void *stream);

/* Static text for a status code. */
SPEC_API const char *spec_status_string(spec_status status);

/* Detail of the last error returned on the calling host thread ("" if none). */
SPEC_API const char *spec_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
