/*
 * spec_verify.h -- C ABI of libspecverify: batched draft-token verification
 * for speculative decoding on one NVIDIA GB300 (sm_103a).
 *
 * What is computed (sources are web pages, cited by title and section):
 *   [REVIEW] "EAGLE-3 speculative decoding review" (6unoyunr.github.io)
 *   [MATH]   "EAGLE math" (aicassindra.com, tm_eagle_math)
 *   [WIKI]   "Speculative decoding" (addictedtoai.net wiki)
 *
 * Conventions shared by every entry point
 *   - All array arguments are DEVICE pointers (cudaMalloc / torch CUDA
 *     memory), row-major and contiguous.  The caller owns all memory; the
 *     library allocates nothing.  State kept across calls: the launch counter
 *     read by spec_verify_launch_count(); per device context, the kernels'
 *     shared-memory opt-ins and launch shapes; and the fixed scratch array of
 *     spec_verify_greedy_noalloc (resident on every device that loads the
 *     library) with its device address.  Each per-context entry records the
 *     context's unique id and is redone when it changes (after
 *     cudaDeviceReset, for example).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call only enqueues work on that stream and returns; it
 *     never synchronises.  Outputs are valid once the stream reaches them.
 *   - Logits are fp32 (SPEC_DTYPE_F32) or bf16 (SPEC_DTYPE_BF16, raw 16-bit
 *     patterns).  Logit pointers must be aligned to the element size; rows
 *     whose byte length is a multiple of 16 starting at a 16-byte aligned base
 *     take the vectorised path, others a scalar path with identical results.
 *   - Logits must be finite with |logit / T| < 2^23; other values give
 *     unspecified (but memory-safe) outputs.
 *   - `workspace`: device scratch of at least spec_verify_workspace_bytes()
 *     bytes, 256-byte aligned.  Its contents on entry do not matter: every
 *     record a kernel reads is written earlier in the same call, so one
 *     workspace serves calls of any shape.  Its first 4 bytes hold the sticky
 *     flag word (see spec_verify_read_flags): zero the workspace once, or
 *     read the flags with clear != 0, before relying on them.  Two calls that
 *     share a workspace must not run concurrently (issue them on one stream,
 *     or order them with events).
 *   - Errors found on the host (NULL pointer, bad size, bad temperature,
 *     misalignment, workspace too small) return before anything is enqueued.
 *     A failed kernel launch returns SPEC_ERR_CUDA.  Bad DEVICE data (a token
 *     id outside [0, V), a malformed tree) is never trapped: the kernels clamp
 *     every access, treat the item as not matching, and set a bit of the
 *     workspace's flag word (spec_verify_read_flags).
 *   - B = 0 is a no-op that returns SPEC_OK.
 *   - Every call's kernels are programmatic dependent launches:
 *     the first kernel of a call waits for the kernel before it in the
 *     stream to finish (and its writes to be visible) before it writes
 *     memory or reads anything but its logits, and the last kernel of a call
 *     lets the next kernel in the stream be scheduled early.  The streaming
 *     kernels of spec_verify_greedy, spec_verify_tree_greedy and (for short
 *     per-CTA ranges) spec_verify_sample start reading their logits (and
 *     sampling its draft tokens) before that wait, while the call before
 *     them on the stream is finishing.  So the inputs of a call must not be
 *     written by the library call issued just before it on the same stream
 *     (a kernel of the caller's own, issued between two calls, has always
 *     finished before the next call's kernels start).
 */
#ifndef SPEC_VERIFY_H_
#define SPEC_VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_VERIFY_ABI_VERSION 1

#if defined(__GNUC__)
#define SPEC_API __attribute__((visibility("default")))
#else
#define SPEC_API
#endif

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = 1, /* NULL pointer, size out of range, T <= 0 or NaN */
  SPEC_ERR_ALIGNMENT = 2,   /* pointer not aligned as documented */
  SPEC_ERR_WORKSPACE = 3,   /* workspace NULL or smaller than required */
  SPEC_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
  SPEC_ERR_TOO_LARGE = 5    /* the call needs more scratch than the fixed
                               array of spec_verify_greedy_noalloc holds */
} spec_status_t;

typedef enum { SPEC_DTYPE_F32 = 0, SPEC_DTYPE_BF16 = 1 } spec_dtype_t;

typedef enum {
  SPEC_MODE_SAMPLE = 0,
  SPEC_MODE_GREEDY = 1,
  SPEC_MODE_TREE_GREEDY = 2,
  SPEC_MODE_TREE_MASK = 3, /* spec_tree_attention_mask: the flag header only */
  SPEC_MODE_KV_COMMIT = 4, /* spec_kv_commit_path: the flag header only */
  SPEC_MODE_LM_HEAD_GREEDY = 5, /* spec_lm_head_verify_greedy (k_or_N = k) */
  SPEC_MODE_TREE_GROW = 6,      /* spec_tree_grow (k_or_N = K children per node) */
  SPEC_MODE_LM_HEAD_SAMPLE = 7  /* spec_lm_head_verify_sample (k_or_N = k, d <= SPEC_LM_MAX_D) */
} spec_mode_t;

/* Bits of the workspace flag word (sticky until read with clear != 0). */
#define SPEC_FLAG_TOKEN_RANGE 1u       /* a draft/node token was outside [0, V) */
#define SPEC_FLAG_BAD_PARENT 2u        /* parents[v] outside [0, v) for some v >= 1 */
#define SPEC_FLAG_DEPTH 4u             /* a node deeper than max_depth */
#define SPEC_FLAG_RESIDUAL_FALLBACK 8u /* residual mass was 0 after a rejection;
                                          that position was sampled from p */
#define SPEC_FLAG_TIMEOUT 16u          /* a kernel gave up waiting for its own
                                          bulk copies (outputs of that call are
                                          unspecified); never expected */
#define SPEC_FLAG_BAD_PATH 32u         /* spec_kv_commit_path: a path that does
                                          not start at node 0, names a node
                                          outside [1, N), is longer than
                                          max_depth, or a tree that does not fit
                                          the cache; that sequence is untouched */

/* Limits checked on the host. */
#define SPEC_MAX_V (1 << 26)
#define SPEC_MAX_K 256
#define SPEC_MAX_TREE_NODES 65536
#define SPEC_MAX_TREE_DEPTH 1024

/*
 * Bytes of workspace needed by one call.  mode: spec_mode_t; k_or_N: k draft
 * tokens (chain modes) or N tree nodes (tree mode).  Returns 0 for arguments
 * outside the limits above or whose scratch index space exceeds 2^31 records.
 */
SPEC_API size_t spec_verify_workspace_bytes(int mode, int B, int k_or_N, int V, int dtype);

/*
 * Rejection-sampling verification of B chains of k draft tokens.
 *
 * Computes, per sequence b ([REVIEW] "Speculative Decoding" step 3 "Accept or
 * Reject"; "Does Using a Small Model's Answer Reduce Quality?", eqs. A(x) and
 * p_residual; [MATH] "Vanilla speculative decoding"; [WIKI] "The mechanism"):
 *   p_i = softmax(target[b,i,:] / T),  q_i = softmax(draft[b,i,:] / T)
 *   accept draft i iff u_accept[b,i] * q_i(x_i) < p_i(x_i)  (strict; left to
 *   right); n = index of the first rejection, or k if none;
 *   if n < k: token ~ norm(max(0, p_n - q_n)) by inverse CDF with u_sample[b]
 *   else:     bonus token ~ p_k by inverse CDF with u_sample[b].
 * Inverse CDF: the smallest vocabulary index j with u * R < C_j, C_j the
 * inclusive prefix sum of the weights and R their total.
 *
 *   target_logits [B, k+1, V]  row i scores draft position i; row k = bonus row
 *   draft_logits  [B, k, V]    row i = the distribution draft i was drawn from
 *   draft_tokens  int32 [B, k]
 *   u_accept      float [B, k] in [0, 1);   u_sample float [B] in [0, 1)
 *   temperature   > 0, finite; the same T scales target and draft rows
 * Outputs (device, written in full):
 *   accepted_len  int32 [B]       n in [0, k]
 *   out_tokens    int32 [B, k+1]  x_0..x_{n-1}, the resampled/bonus token, then -1
 *   p_out, q_out  float [B, k]    p_i(x_i), q_i(x_i) for EVERY i (also i > n)
 *   resid_mass    float [B]       R = sum_j max(0, p_n - q_n) when n < k, else 0
 * With k = 0, draft_logits, draft_tokens, u_accept, p_out and q_out may be
 * NULL and the call samples one token from softmax(target[b,0,:] / T).
 * Launches two kernels: the softmax statistics, then one thread-block cluster
 * per sequence for row merge, accept test, residual/bonus prefix sums and the
 * inverse-CDF walk (three kernels when a row spans more than 16 32-KB chunks:
 * V > 262144 bf16 or 131072 fp32).
 */
SPEC_API spec_status_t spec_verify_sample(const void* target_logits, const void* draft_logits,
                                 int dtype, const int32_t* draft_tokens,
                                 const float* u_accept, const float* u_sample,
                                 float temperature, int B, int k, int V,
                                 int32_t* accepted_len, int32_t* out_tokens,
                                 float* p_out, float* q_out, float* resid_mass,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Greedy verification ([REVIEW] "Does Using a Small Model's Answer Reduce
 * Quality?", greedy bullets): g_i = argmax_j target[b,i,j] on raw logits,
 * lowest index among ties; n = first i < k with draft_tokens[b,i] != g_i, or
 * k; emits x_0..x_{n-1}, g_n.  Temperature plays no part.
 *   target_logits [B, k+1, V]; draft_tokens int32 [B, k] (NULL allowed if k = 0)
 *   accepted_len  int32 [B];   out_tokens int32 [B, k+1] (unused slots -1)
 * Launches two kernels (argmax partials; row merge + accept).
 */
SPEC_API spec_status_t spec_verify_greedy(const void* target_logits, int dtype,
                                 const int32_t* draft_tokens, int B, int k, int V,
                                 int32_t* accepted_len, int32_t* out_tokens,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Draft-tree greedy verification (EAGLE-2 style trees; [REVIEW] "EAGLE-2",
 * "The Complete EAGLE-3 Inference Process" steps 3-4; [MATH] "EAGLE-2:
 * dynamic draft trees").  Node 0 is the root (the last committed token); row v
 * of target_logits is the target's next-token logits after the path root..v.
 * Node v >= 1 is accepted iff every node w on the path root..v has
 * node_tokens[w] == argmax(target row of parent(w)).  The deepest accepted
 * node v* wins (lowest node index among equally deep ones); the bonus token
 * is argmax(target row v*).
 *   target_logits [B, N, V]
 *   node_tokens   int32 [B, N]   (node 0's entry is ignored)
 *   parents       int32 [B, N]   parents[b,0] ignored; 0 <= parents[b,v] < v
 *   max_depth     depth limit of the trees, 0..SPEC_MAX_TREE_DEPTH
 * Outputs:
 *   accepted_len  int32 [B]                depth of v*
 *   path_nodes    int32 [B, max_depth+1]   0, ..., v*, then -1
 *   out_tokens    int32 [B, max_depth+1]   tokens of path nodes 1..depth, the
 *                                          bonus token, then -1
 * Launches two kernels (argmax partials; row merge + tree walk).
 */
SPEC_API spec_status_t spec_verify_tree_greedy(const void* target_logits, int dtype,
                                      const int32_t* node_tokens, const int32_t* parents,
                                      int B, int N, int V, int max_depth,
                                      int32_t* accepted_len, int32_t* path_nodes,
                                      int32_t* out_tokens, void* workspace,
                                      size_t workspace_bytes, void* stream);

/*
 * Tree attention mask of B draft trees ("EAGLE-3 speculative decoding
 * review", "EAGLE-2: Does Every Context Need the Same Draft Tree?" and "Must
 * the Feature Be Predicted Exactly?": each node sees the shared prefix and
 * only its own ancestors; "The Complete EAGLE-3 Inference Process" step 3).
 * The prefix columns are visible to every node and are not written; this
 * call writes the tree block.
 *   parents  int32 [B, N]  parents[b,0] ignored (node 0 is the root, the
 *                          last committed token); 0 <= parents[b,v] < v
 * Outputs:
 *   mask     uint32 [B, N, W], W = (N + 31) / 32: bit (u % 32) of word u / 32
 *            of row (b, v) is set iff u == v or u is an ancestor of v; the
 *            bits past N in the last word are 0
 *   depth    int32 [B, N] or NULL: edges from v to the root
 * A node whose ancestor chain meets a parent outside [0, child) keeps the
 * nodes walked so far, gets depth -1 and raises SPEC_FLAG_BAD_PARENT.
 * Pointers: device memory, 4-byte aligned; workspace of at least
 * spec_verify_workspace_bytes(SPEC_MODE_TREE_MASK, ...) bytes (the flag
 * header), 256-byte aligned.  One kernel launch; N <= SPEC_MAX_TREE_NODES.
 */
SPEC_API spec_status_t spec_tree_attention_mask(const int32_t* parents, int B, int N,
                                                uint32_t* mask, int32_t* depth, void* workspace,
                                                size_t workspace_bytes, void* stream);

/*
 * KV commit of the accepted path ("EAGLE-3 speculative decoding review",
 * "The Complete EAGLE-3 Inference Process" step 5: keep only the accepted
 * path's cache entries, discard the rejected branches, resume drafting from
 * the committed prefix).  Tree node v >= 1 of sequence b holds its entries at
 * cache position base_len[b] + v - 1 (the tree follows the committed prefix,
 * whose last token is the root).  For the path 0, v_1, ..., v_d written by
 * spec_verify_tree_greedy (d = accepted_len[b]), node v_i's entry moves to
 * position base_len[b] + i - 1 in every plane, in place; every other
 * position keeps its contents; new_len[b] = base_len[b] + d (the bonus token
 * has no cache entry yet).
 *   cache        device bytes; entry (plane p, sequence b, position t) starts
 *                at p * plane_stride + b * seq_stride + t * entry_bytes (a
 *                plane is one layer's K or V); 16-byte aligned, entry_bytes
 *                and both strides multiples of 16; entries must not overlap
 *   L            positions per sequence; N tree nodes; base_len[b] >= 1 and
 *                base_len[b] + N - 1 <= L
 *   base_len, accepted_len  int32 [B]; path_nodes int32 [B, max_depth + 1]
 *   new_len      int32 [B] out
 * A malformed sequence (see SPEC_FLAG_BAD_PATH) is left untouched with
 * new_len = base_len.  Workspace: spec_verify_workspace_bytes(
 * SPEC_MODE_KV_COMMIT, ...) bytes (the flag header).  One kernel launch (one
 * CTA per sequence and plane; the moved entries are staged in shared memory
 * before any is stored); planes <= 65535.
 */
SPEC_API spec_status_t spec_kv_commit_path(void* cache, int B, int planes, long long plane_stride,
                                           long long seq_stride, int entry_bytes, int L, int N,
                                           const int32_t* base_len, const int32_t* accepted_len,
                                           const int32_t* path_nodes, int max_depth,
                                           int32_t* new_len, void* workspace,
                                           size_t workspace_bytes, void* stream);

/*
 * The target's LM head fused with greedy verification ("EAGLE math", "Why
 * feature drafting lands a higher acceptance rate": the target's logits are
 * its LM head applied to the hidden state, z = W_LM h; "EAGLE-3 speculative
 * decoding review", "Does Using a Small Model's Answer Reduce Quality?"
 * greedy bullets).  Computes every target row's argmax of z = W_LM h on the
 * tensor cores without writing the logits, then the same acceptance as
 * spec_verify_greedy.
 *   hidden       bf16 [B*(k+1), d]  row b*(k+1)+i: the target's hidden state
 *                                   at draft position i of sequence b
 *   w_lm         bf16 [V, d]        the LM head, row j = vocabulary entry j
 *   draft_tokens int32 [B, k]
 *   d            multiple of 8; hidden and w_lm 16-byte aligned
 * Outputs as spec_verify_greedy.  The argmax is of the float32-accumulated
 * products (lowest index among equal values); rows whose top two logits lie
 * closer than the accumulation error may pick either.  Two kernel launches
 * (tcgen05 GEMM with an argmax epilogue; record merge + chain resolve).  The
 * GEMM runs on clusters of two CTAs, one per SM, that share each 256-entry
 * vocabulary tile through two-CTA MMAs; it occupies every SM it can hold a
 * pair on (most of each SM's shared and tensor memory) until it ends.
 * Workspace: spec_verify_workspace_bytes(SPEC_MODE_LM_HEAD_GREEDY, B, k, V,
 * SPEC_DTYPE_BF16).
 */
SPEC_API spec_status_t spec_lm_head_verify_greedy(const void* hidden, const void* w_lm,
                                                  const int32_t* draft_tokens, int B, int k,
                                                  int d, int V, int32_t* accepted_len,
                                                  int32_t* out_tokens, void* workspace,
                                                  size_t workspace_bytes, void* stream);

/*
 * The target's LM head fused with sampling verification ("EAGLE math",
 * "EAGLE's move": p = softmax(LM_head(f)), the drafted features going through
 * the target's own LM head; "EAGLE-3 speculative decoding review", "Does
 * Using a Small Model's Answer Reduce Quality?" eqs. A(x), p_residual).
 * The target rows' logits W_LM h_t and the draft rows' logits W_LM h_d are
 * reduced on the tensor cores to their softmax statistics and draft-token
 * logits without being written; the accept test follows, and only the rows
 * a sequence draws from (the target and draft rows of its first rejection,
 * or its bonus row) are recomputed as fp32 logits in the workspace for the
 * residual or bonus draw.  Same decisions and outputs as spec_verify_sample
 * on the float32-accumulated logits.
 *   hidden_target bf16 [B*(k+1), d]  row b*(k+1)+i: the target's hidden state
 *                                    at position i of sequence b
 *   hidden_draft  bf16 [B*k, d]      row b*k+i: the drafted feature of
 *                                    position i (NULL when k = 0)
 *   w_lm          bf16 [V, d]        the LM head, row j = vocabulary entry j
 *   draft_tokens, u_accept, u_sample, temperature, outputs: as
 *                 spec_verify_sample
 *   d             multiple of 8, at most SPEC_LM_MAX_D; the matrices 16-byte
 *                 aligned
 * Four kernel launches: the statistics GEMM (tcgen05, softmax epilogue), the
 * accept test with the gather of the drawn rows' hidden states, the GEMM
 * that writes those rows' logits, and the draw (as spec_verify_sample's).
 * Workspace: spec_verify_workspace_bytes(SPEC_MODE_LM_HEAD_SAMPLE, B, k, V,
 * SPEC_DTYPE_BF16).
 */
#define SPEC_LM_MAX_D 8192
SPEC_API spec_status_t spec_lm_head_verify_sample(
    const void* hidden_target, const void* hidden_draft, const void* w_lm,
    const int32_t* draft_tokens, const float* u_accept, const float* u_sample, float temperature,
    int B, int k, int d, int V, int32_t* accepted_len, int32_t* out_tokens, float* p_out,
    float* q_out, float* resid_mass, void* workspace, size_t workspace_bytes, void* stream);

/*
 * EAGLE-2 dynamic draft-tree growth ("EAGLE math", "EAGLE-2: dynamic draft
 * trees": expand the nodes with the highest cumulative draft probability,
 * prune low-probability paths, re-rank under an unchanged node budget;
 * "EAGLE-3 speculative decoding review", "EAGLE-2: Does Every Context Need
 * the Same Draft Tree?").  Layer l expands the frontier (slot j holds a node;
 * layer 0: the root in slot 0) with the draft row draft_logits[b, l, j]:
 * q = softmax(z / T); the node's children are its K most probable tokens
 * (ties: lower token), valued parent + ln q(token) (root 0); the next
 * frontier is the layer's K best children (ties: creation order).  After D
 * layers the tree is the root plus the M best nodes (ties: creation order),
 * listed in creation order (parents before children) with parents
 * renumbered, ready for spec_verify_tree_greedy and spec_tree_attention_mask.
 *   draft_logits  [B, D, K, V] dtype (slot j of layer 0 is read for j = 0 only)
 *   K             1..16 children per node and frontier size; D 1..16 layers
 *   M             node budget, 0 <= M <= K + (D-1) K^2
 * Outputs [B, M+1]: tokens (root -1), parents (root -1), depth, values
 * (float32 cumulative ln probability; computed in float64).  Token choices
 * compare raw logits (exact); node values near a selection boundary may
 * order differently from a float64 reference when within ~1e-12.
 * Workspace: spec_verify_workspace_bytes(SPEC_MODE_TREE_GROW, B, K, V, dtype)
 * (sized for up to 16 layers); requires ceil(V / chunk) * K <= 2048 (chunk =
 * 16384 bf16 / 8192 fp32 elements).  Two kernel launches: the K best tokens
 * and softmax normaliser of every draft row read (B (1 + (D-1) K) rows, one
 * streaming pass), then a cluster of two CTAs per tree for the rows' merge,
 * the layer-by-layer expansion and the selection of the M best nodes.
 */
SPEC_API spec_status_t spec_tree_grow(const void* draft_logits, int dtype, float temperature,
                                      int B, int D, int K, int V, int M, int32_t* tokens,
                                      int32_t* parents, int32_t* depth, float* values,
                                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * Copy the workspace's flag word to *host_flags (synchronises `stream`); with
 * clear != 0 the word is then reset to 0 on the stream.
 */
SPEC_API spec_status_t spec_verify_read_flags(void* workspace, uint32_t* host_flags, int clear,
                                     void* stream);

/*
 * Self-test of the two 2^x evaluations the kernels use (no counterpart in the
 * pages): y_fma[i] = the FMA-pipe polynomial (Cody-Waite reduction, degree-5
 * minimax; relative error below 2e-7 for -126 <= x <= 0.5), y_sfu[i] = the
 * special-function unit's ex2.approx.ftz.  x, y_fma, y_sfu: device float [n].
 */
SPEC_API spec_status_t spec_verify_selftest_exp2(const float* x, float* y_fma, float* y_sfu,
                                                 int n, void* stream);

/* Number of kernels this library has launched in this process. */
SPEC_API uint64_t spec_verify_launch_count(void);

/*
 * Diagnostic control of the bounded waits (no counterpart in the pages).
 *
 * Every wait of the verification kernels on their own bulk copies gives up
 * after a limit (0.2 s by default): the CTA then sets SPEC_FLAG_TIMEOUT,
 * stops copying, waits (with the default limit) for the copies it has in
 * flight and finishes its control flow, so the call completes with
 * unspecified outputs and the flag raised instead of hanging.  This sets the
 * limit used by calls of spec_verify_sample, spec_verify_greedy,
 * spec_verify_tree_greedy and spec_verify_greedy_noalloc enqueued afterwards,
 * process-wide; limit_ns = 0 restores the default.  limit_ns = 1 gives up
 * whenever a copy has not landed at the first look, which is how a test
 * exercises that path (other limits below a microsecond are rounded up by
 * the resolution of the GPU's global timer).  Not for production use.
 */
SPEC_API void spec_verify_set_wait_limit_ns(uint64_t limit_ns);

/*
 * Greedy verification without any allocation (no counterpart in the pages:
 * this is a deployment convenience, not part of the method).
 *
 * Same computation, arguments and outputs as spec_verify_greedy, minus the
 * workspace: its scratch is a fixed array of SPEC_NOALLOC_SCRATCH_BYTES in
 * the library's own device memory, resident on every GPU that loads the
 * library until the process exits.  It is for callers that cannot allocate
 * device memory at the point of the call: for example a plugin inside a
 * serving framework that owns every device allocation, or a decode loop that
 * must not allocate once it is running.  The library itself calls no
 * cudaMalloc, cudaFree or other allocating routine on this path.
 *
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it for the
 *     device's current context; make that first call before any stream
 *     capture begins on the device, and again after a cudaDeviceReset.
 *   - Calls whose scratch would exceed SPEC_NOALLOC_SCRATCH_BYTES return
 *     SPEC_ERR_TOO_LARGE before anything is enqueued (B=64 sequences of k=4
 *     drafts over V=128256 bf16 need about 0.66 MB).
 *   - Every call uses the same array, which keeps what the previous call left
 *     there.  Nothing the kernels read needs to start at zero; the flag word is
 *     cleared on entry and device-side input errors are not reported.  Calls
 *     that overlap on the GPU (different streams without ordering, or
 *     concurrent host threads) race on the array: serialise them.
 */
#define SPEC_NOALLOC_SCRATCH_BYTES (4u << 20)
SPEC_API spec_status_t spec_verify_greedy_noalloc(const void* target_logits, int dtype,
                                                  const int32_t* draft_tokens, int B, int k, int V,
                                                  int32_t* accepted_len, int32_t* out_tokens,
                                                  void* stream);

/* Static description of a status code. */
SPEC_API const char* spec_status_string(int status);

/* SPEC_VERIFY_ABI_VERSION of the loaded library. */
SPEC_API int spec_verify_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H_ */
