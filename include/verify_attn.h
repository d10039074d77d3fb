/*
 * verify_attn.h -- C ABI of the GB300 (sm_103a) MLA tree-verify attention library.
 *
 * The operation (The Milestone Commit, "Input Knowledge Required"): in tree
 * speculative decoding the target model verifies T draft-tree tokens in one
 * pass; each token's H absorbed query heads attend over the request's whole
 * cached KV.  The cache is the MLA latent cache (The Milestone Commit,
 * "Context"): one row per token, shared by every head, addressed through a
 * page_size=1 slot table.  A row holds 576 bf16: 512 latent columns, which
 * are also the value, followed by 64 rotary columns.  The Checkpoint Report,
 * "Mistakes and Incorrect Assumptions": the request's keys are its prefix
 * followed by the draft tokens' own keys, and draft node i sees every prefix
 * key plus the draft keys of itself and its ancestors.
 *
 * For request b, node i, head h (row r = (b*T + i)*H + h):
 *   s_j   = sm_scale * <q[r, 0:576], kv[slot(b, j), 0:576]>   for visible j
 *   lse_r = ln sum_j exp(s_j)                 (natural log, scale included)
 *   out_r = sum_j exp(s_j - lse_r) * kv[slot(b, j), 0:512]
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never allocates, frees or synchronises inside a call, and launches only
 *    on the caller's stream, so every call can be captured into a CUDA graph
 *    (The Commit That Locked In 6x Decode, "1. Capture-Safe Design": no
 *    cudaMalloc and no host sync inside the call; a workspace allocated once
 *    by the caller).
 *  - Step-varying data (prefix lengths, slot tables, tree parents) is read on
 *    the device, so one captured graph replays across decode steps.
 *  - Stream order holds as for any launch.  The first kernel of the attention
 *    calls and of the placement calls (va_kv_append_contiguous,
 *    va_kv_compact_accepted) is a programmatic dependent of the stream's
 *    previous kernel: its CTAs may become resident while that kernel
 *    finishes, but read no input until it has completed (griddepcontrol.wait).
 *    Their last kernel lets the stream's next kernel do the same once it has
 *    itself passed that point,
 *    so a caller's next kernel launched as a programmatic dependent must wait
 *    (griddepcontrol.wait / cudaGridDependencySynchronize) before it reads the
 *    call's outputs; a plainly launched one is ordered as usual.
 *  - Host-checkable argument errors return a negative VA_ERR_* code before any
 *    device work is enqueued.  Device-data errors (a slot outside the pool, a
 *    parent that is not an earlier node, a slot list shorter than
 *    prefix_len + T, a dense mask shorter than its rows) set bits in the
 *    workspace status word; the offending key or entry is skipped and the
 *    call still returns VA_OK.  Kernels never trap.
 *  - bf16 tensors are passed as `const void*` holding IEEE bfloat16 values.
 *  - Calls on distinct workspaces are thread-safe.
 */
#ifndef VERIFY_ATTN_H
#define VERIFY_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st *va_stream_t;

/* Return codes of every entry point. */
#define VA_OK               0
#define VA_ERR_NULL        -1  /* a required pointer is NULL                        */
#define VA_ERR_SHAPE       -2  /* B, T, H, num_slots, stride or nsplit out of range */
#define VA_ERR_ALIGN       -3  /* pointer or stride misaligned (see each argument)  */
#define VA_ERR_WORKSPACE   -4  /* workspace smaller than va_workspace_bytes()       */
#define VA_ERR_UNSUPPORTED -5  /* no va_init() for the current device, device is
                                  not sm_103, or the requested path is unavailable */
#define VA_ERR_LAUNCH      -6  /* a kernel launch failed (cudaGetLastError)         */
#define VA_ERR_CUDA        -7  /* another CUDA runtime call failed                  */

/* Bits of the device status word (first 4 bytes of the workspace). */
#define VA_STATUS_BAD_SLOT    0x1u  /* a slot index outside [0, num_slots)           */
#define VA_STATUS_BAD_PARENT  0x2u  /* parent[i] not in [-1, i); node treated as a
                                       child of the prefix                          */
#define VA_STATUS_BAD_INDPTR  0x4u  /* slot list of a request shorter than
                                       prefix_len + T, or prefix_len < 0; the
                                       request's prefix is clamped to what exists  */
#define VA_STATUS_TIMEOUT     0x8u  /* a bounded device-side wait gave up            */
#define VA_STATUS_BAD_DST     0x10u /* defrag destination outside the pool           */
#define VA_STATUS_BAD_MASK    0x20u /* a dense mask row past custom_mask_len; the
                                       node's missing draft columns read as 0      */

/* Fixed widths of the MLA latent row. */
#define VA_D_QK 576   /* key / query width: 512 latent + 64 rotary */
#define VA_D_V  512   /* value / output width: the first 512 columns */
#define VA_T_MAX 64   /* draft nodes per request (one 64-bit mask word per node) */
#define VA_NSPLIT_MAX 1024

/* Compute-path selection for the verify entry points (`flags`). */
#define VA_PATH_AUTO 0  /* library's choice                                     */
#define VA_PATH_FMA  1  /* CUDA-core FMA path (any shape)                       */
#define VA_PATH_TC   2  /* tcgen05 tensor-core path (two-SM products, M = 256,
                           once a request has more than 128 rows)            */
#define VA_PATH_TC_1SM 3 /* tensor-core path with one-SM products (M = 128) at
                           every row count                                   */

/* Library ABI version (major * 100 + minor). */
int va_version(void);

/*
 * Caches the device's SM count and checks that it is an sm_103 part.  Call
 * once per device, outside stream capture, before the first verify call on
 * that device.  It also places the scratch array of
 * verify_attn_paged_noalloc on the device (VA_NOALLOC_SCRATCH_BYTES; see
 * there).  Returns VA_OK, VA_ERR_UNSUPPORTED or VA_ERR_CUDA.
 */
int va_init(int device);

/*
 * Split count the library picks for nsplit = 0 on the current device (after
 * va_init): enough (request, row-block, split) work items to cover the SMs.
 * Pure host arithmetic.  Returns >= 1, or a VA_ERR_* code.
 */
int va_auto_nsplit(int B, int T, int H, int flags);

/*
 * Bytes of workspace a verify call with these sizes needs (nsplit >= 1; pass
 * the value from va_auto_nsplit for automatic splitting).  Pure host
 * arithmetic, no CUDA call.  Layout (each region 256-byte aligned):
 *   [0, 256)        status word (uint32) and reserved header
 *   tree masks      uint64 [B*T]
 *   CTA status      uint32 [B][2*ceil(T*H/256)][nsplit][2] (tensor-core
 *                   path: each split-K CTA's status bits, OR-ed into the
 *                   status word by the merge)
 *   partial lse     float  [nsplit][B*T*H]
 *   partial out     bf16   [nsplit][B*T*H][512] (normalised by the split's
 *                   row sum; merged in fp32)
 * The Commit That Locked In 6x Decode, "Input Knowledge Required" (NSPLIT and
 * partial-reduce: each split writes a partial result that a reduction merges).
 */
size_t va_workspace_bytes(int B, int T, int H, int nsplit);

/*
 * Paged verify attention: keys gathered through a page_size=1 slot table.
 *   q             bf16 [B*T, H, 576], contiguous, 16-byte aligned.
 *   kv_pool       bf16 [num_slots, kv_row_stride]; row stride in elements,
 *                 >= 576 and a multiple of 8; base 16-byte aligned.  Only the
 *                 first 576 columns of a row are read.
 *   slot_idx      int32, request b's N_b = prefix_len[b] + T slots start at
 *                 slot_idx[kv_indptr[b]]: the prefix slots in order, then the
 *                 slots of draft nodes 0..T-1 (The Checkpoint Report,
 *                 "Mistakes and Incorrect Assumptions": prefix in kv_indices,
 *                 draft tokens at out_cache_loc -- concatenated here).
 *   kv_indptr     int32 [B+1] device offsets into slot_idx.
 *   prefix_len    int32 [B] device, keys before the draft nodes (>= 0).
 *   tree_parent   int32 [B, T] device, parent[i] in [-1, i); -1 = the node
 *                 hangs off the prefix.  May be NULL when tree_bits is given.
 *   tree_bits     uint64 [B, T] device, bit k of tree_bits[b*T+i] set when
 *                 draft node k is node i or one of its ancestors.  When
 *                 non-NULL it is used and tree_parent is ignored.
 *   B, T, H       1 <= B, 1 <= T <= 64, 1 <= H.
 *   sm_scale      scale applied to the 576-wide dot product.
 *   nsplit        key-range splits per (request, row unit: 128 rows, or 256
 *                 with two-SM products); 0 = automatic
 *                 (The Commit That Locked In 6x Decode, "2. NSPLIT=64 for TP8
 *                 Occupancy").  Splits that would hold fewer than 64 keys are
 *                 dropped on the device from the actual prefix length.
 *   flags         VA_PATH_*.
 *   workspace     device buffer of workspace_bytes >= va_workspace_bytes(B, T,
 *                 H, nsplit or the automatic value), 256-byte aligned, owned
 *                 by the caller; reused across calls; calls that overlap on
 *                 the device must not share one.
 *   out           bf16 [B*T, H, 512], 16-byte aligned (round-to-nearest-even).
 *   lse           float [B*T, H]; -inf for a row that sees no key.
 *   stream        stream the kernels are launched on.
 * The status word describes this call only: every call rewrites it (no
 * clearing by the caller), and it is complete once the call's work is.
 */
int verify_attn_paged(const void *q, const void *kv_pool, int64_t num_slots,
                      int64_t kv_row_stride, const int32_t *slot_idx, const int32_t *kv_indptr,
                      const int32_t *prefix_len, const int32_t *tree_parent,
                      const uint64_t *tree_bits, int B, int T, int H, float sm_scale, int nsplit,
                      int flags, void *workspace, size_t workspace_bytes, void *out, float *lse,
                      va_stream_t stream);

/*
 * Contiguous verify attention: request b's N_b = prefix_len[b] + T keys are
 * the pool rows kv_start[b] + j, j < N_b (prefix rows first, then the draft
 * nodes' rows) -- the layout after defragmentation (The Checkpoint Report,
 * "Input Knowledge Required": defragmentation keeps per-request KV
 * contiguous; The Milestone Commit, "What the Commit Captures": the first
 * kernel read contiguous KV).  kv_start is int64 [B] on the device; rows
 * outside [0, num_slots) are skipped and flagged VA_STATUS_BAD_SLOT.  Every
 * other argument is as for verify_attn_paged.
 */
int verify_attn_contiguous(const void *q, const void *kv_pool, int64_t num_slots,
                           int64_t kv_row_stride, const int64_t *kv_start,
                           const int32_t *prefix_len, const int32_t *tree_parent,
                           const uint64_t *tree_bits, int B, int T, int H, float sm_scale,
                           int nsplit, int flags, void *workspace, size_t workspace_bytes,
                           void *out, float *lse, va_stream_t stream);

/*
 * Segmented verify attention: the prefix and the draft nodes' keys come as two
 * slot lists, and the tree may come as a dense mask (The Checkpoint Report,
 * "Mistakes and Incorrect Assumptions": the extend call takes the prefix in
 * kv_indices and the draft tokens' own keys at out_cache_loc, and its custom
 * mask holds one row per draft token with stride prefix + q_len).  Computes
 * exactly what verify_attn_paged computes on the concatenated list.
 *   kv_indices     int32 device; request b's prefix slots are
 *                  kv_indices[kv_indptr[b] .. kv_indptr[b+1]), so its prefix
 *                  length is P_b = kv_indptr[b+1] - kv_indptr[b] (no
 *                  prefix_len argument).
 *   kv_indptr      int32 [B+1] device, non-decreasing.
 *   out_cache_loc  int32 [B*T] device; out_cache_loc[b*T + i] is the slot of
 *                  request b's draft node i.
 *   draft_kv       bf16 [B*T, 576] device (contiguous rows, 16-byte aligned),
 *                  or NULL.  When given, the call first writes row b*T + i
 *                  into the first 576 columns of pool row out_cache_loc[b*T +
 *                  i] (the draft tokens' new latents), then verifies against
 *                  the pool with those rows in place.  The draft slots must be
 *                  distinct and must not hold any request's prefix key; a slot
 *                  outside the pool is skipped (and flagged when read).
 *   custom_mask    uint8 device (0 = hidden, non-zero = visible), or NULL.
 *                  Request b's T rows of P_b + T entries each start at entry
 *                  T * (kv_indptr[b] - kv_indptr[0] + b*T); row i, column
 *                  P_b + k says whether node i sees draft node k.  Only those
 *                  last T columns are read: every prefix key is visible to
 *                  every draft node.  Entries at or past custom_mask_len are
 *                  read as 0 and flag VA_STATUS_BAD_MASK.
 *   custom_mask_len entries in custom_mask (ignored when it is NULL).
 *   tree_parent, tree_bits  as for verify_attn_paged; exactly one of
 *                  custom_mask, tree_bits, tree_parent is used, in that order
 *                  of precedence.
 * Every other argument is as for verify_attn_paged.
 */
int verify_attn_segmented(const void *q, const void *kv_pool, int64_t num_slots,
                          int64_t kv_row_stride, const int32_t *kv_indices,
                          const int32_t *kv_indptr, const int32_t *out_cache_loc,
                          const void *draft_kv, const uint8_t *custom_mask,
                          int64_t custom_mask_len,
                          const int32_t *tree_parent, const uint64_t *tree_bits, int B, int T,
                          int H, float sm_scale, int nsplit, int flags, void *workspace,
                          size_t workspace_bytes, void *out, float *lse, va_stream_t stream);

/*
 * Greedy tree acceptance after verify (The Milestone Commit, "Input Knowledge
 * Required": the verify step checks whether the draft predictions are
 * correct; The Checkpoint Report, "Input Knowledge Required to Understand
 * This Message": a drafter proposes a tree of candidate tokens, the target
 * model checks them in one parallel pass).  For request b:
 *   t = argmax(root_logits[b]); cur = the prefix; n = 0
 *   repeat: among the draft nodes whose parent is cur (parent -1: the
 *     prefix), take the lowest-numbered one whose draft token is t; if there
 *     is none, stop; else accept it (accept_nodes[b*T + n++] = it), cur = it,
 *     t = argmax(logits[b, it]).
 *   accept_len[b] = n; bonus_token[b] = t (the target's token after the
 *   accepted path); accept_nodes past n = -1.
 * argmax = the lowest index among the largest non-NaN values (0 when a row is
 * all NaN).  A node whose parent is not an earlier node counts as a child of
 * the prefix and sets VA_STATUS_BAD_PARENT in the workspace status word.
 *   root_logits   float [B, V] device: the target's logits at the last prefix
 *                 position (the token after the prefix).
 *   logits        float [B, T, V] device: its logits at each draft node.
 *   draft_tokens  int32 [B, T] device: the token each draft node carries.
 *   tree_parent   int32 [B, T] device, as for the verify calls.
 *   draft_slots   int32 [B, T] device or NULL: each node's pool slot (e.g.
 *                 out_cache_loc); accept_slots[b*T + m] = the slot of
 *                 accept_nodes[b*T + m] (-1 past n, and everywhere when
 *                 draft_slots is NULL).  accept_slots may be NULL.
 *   workspace     device, >= va_tree_accept_workspace_bytes(B, T, V) bytes,
 *                 256-byte aligned; first 4 bytes: the status word.
 *   accept_len, bonus_token  int32 [B]; accept_nodes  int32 [B, T].
 * 1 <= T <= 64, 1 <= V < 2^31 - 1.  Reads every logit once (HBM-bound).
 */
size_t va_tree_accept_workspace_bytes(int B, int T, int64_t V);
int va_tree_accept(const float *root_logits, const float *logits, int64_t V,
                   const int32_t *draft_tokens, const int32_t *tree_parent,
                   const int32_t *draft_slots, int B, int T, void *workspace,
                   size_t workspace_bytes, int32_t *accept_len, int32_t *accept_nodes,
                   int32_t *accept_slots, int32_t *bonus_token, va_stream_t stream);

/*
 * Draft tree and draft KV slots, built on the device from the drafter's
 * output (The Checkpoint Report, "Input Knowledge Required to Understand
 * This Message": a drafter proposes candidate tokens and DDTree builds a tree
 * of draft tokens from them; The Commit That Locked In 6x Decode, "4. The
 * Marshaling Realization": this per-step tree build ran on the host).  The
 * pages give no selection rule; the drafter's output is read as K candidate
 * tokens with log-probabilities at each of D draft positions, and the tree is
 * grown best first:
 *   - at each depth the candidates are ranked by log-probability, highest
 *     first, ties by lower index (NaN and +inf count as -inf);
 *   - a node is a path of one candidate per depth from depth 0 down; its
 *     score is the float32 running sum of its log-probabilities, root first;
 *   - T times, the highest-scoring node whose parent is already in the tree is
 *     added (depth-0 nodes hang off the prefix); equal scores go to the
 *     shallower node, then to the lexicographically smaller path of ranks.
 * With log-probabilities (<= 0) this is the T best nodes of the whole
 * candidate tree.  Node i of request b is the i-th node added, so parents
 * precede children, as every verify call requires.
 *   cand_tokens   int32 [B, D, K] device; cand_logp float [B, D, K] device.
 *   1 <= D <= VA_TREE_MAX_DEPTH, 1 <= K <= VA_TREE_MAX_CAND,
 *   1 <= T <= VA_T_MAX and T <= K + K^2 + ... + K^D.
 *   tree_parent   int32 [B, T]: parent node, -1 for depth 0 (the layout
 *                 every verify call and va_tree_accept take).
 *   draft_tokens  int32 [B, T]: the candidate token of each node.
 *   node_depth    int32 [B, T] or NULL: 0-based depth (the node's position
 *                 after the prefix is prefix_len + depth).
 *   free_slots    int32 [free_capacity] device, or NULL (no slots taken):
 *                 pool slots available for new KV rows.  Node i of request b
 *                 takes free_slots[*free_head + b*T + i] into
 *                 out_cache_loc[b*T + i] (int32 [B*T]), -1 where the list has
 *                 run out (and VA_STATUS_BAD_SLOT is set); then *free_head
 *                 (int32, device) advances by B*T.  out_cache_loc is the list
 *                 verify_attn_segmented takes.
 *   status        uint32 device word or NULL: set to this call's status bits.
 * One kernel launch, one CTA (a warp per request, eight at a time); no host
 * sync, capture-safe: the free-list head is device state.  Returns VA_OK or a
 * VA_ERR_* code.
 */
#define VA_TREE_MAX_DEPTH 15
#define VA_TREE_MAX_CAND  16
int va_tree_build(const int32_t *cand_tokens, const float *cand_logp, int B, int D, int K, int T,
                  const int32_t *free_slots, int64_t free_capacity, int32_t *free_head,
                  int32_t *tree_parent, int32_t *draft_tokens, int32_t *node_depth,
                  int32_t *out_cache_loc, uint32_t *status, va_stream_t stream);

/*
 * KV defragmentation (The Checkpoint Report, "Input Knowledge Required" and
 * "The Architecture of the Report": the deferred defragmentation phase).
 * For every request b and i < n_b = src_indptr[b+1] - src_indptr[b]:
 *   kv_pool[dst_base[b] + i, :] <- kv_pool[src_slots[src_indptr[b] + i], :]
 * copying whole rows (kv_row_stride elements), and, when slot_idx_out is not
 * NULL, slot_idx_out[src_indptr[b] + i] <- dst_base[b] + i.
 *   src_slots    int32 device; src_indptr int32 [B+1] device; dst_base int64
 *                [B] device.  slot_idx_out may alias src_slots.
 *   max_rows     host upper bound on sum_b n_b, used only to size the grid
 *                (any value >= 1 is correct; larger gives more parallelism).
 *   status       optional device uint32 word; bits VA_STATUS_BAD_SLOT /
 *                VA_STATUS_BAD_DST are OR-ed in for rows that are skipped.
 * The destination ranges must not overlap any source row of the same call;
 * rows are copied by independent threads, so an overlap gives an undefined
 * result (never a fault: every address is range-checked).
 */
int verify_attn_defrag(void *kv_pool, int64_t num_slots, int64_t kv_row_stride,
                       const int32_t *src_slots, const int32_t *src_indptr,
                       const int64_t *dst_base, int32_t *slot_idx_out, int B, int64_t max_rows,
                       uint32_t *status, va_stream_t stream);

/*
 * Contiguous placement of the draft latents, and compaction of the accepted
 * path: the defragmentation policy the pages name but defer (The Checkpoint
 * Report, "Input Knowledge Required": defragmentation keeps per-request KV
 * contiguous; "The Architecture of the Report": the deferred defragmentation
 * phase).  Read here as: request b owns the pool rows [kv_start[b],
 * kv_start[b] + kv_capacity[b]); its prefix occupies the first prefix_len[b]
 * of them; before verify, its T draft latents go to the next T rows (so
 * verify_attn_contiguous reads prefix and draft keys as one run of rows);
 * after acceptance, the accepted path's rows move to directly after the
 * prefix and the prefix grows by the accepted count, so the request stays
 * contiguous from step to step.
 *
 * va_kv_append_contiguous: for every request b and node i < T, writes draft
 * row b*T + i into the first 576 columns of pool row
 *   kv_start[b] + prefix_len[b] + i
 * and sets out_cache_loc[b*T + i] to that row; a node gets no row (-1, row
 * not written, VA_STATUS_BAD_DST OR-ed into *status) when prefix_len[b] < 0,
 * prefix_len[b] + T > kv_capacity[b], or the row lies outside [0, num_slots)
 * or above 2^31 - 1.
 *   kv_pool        bf16 [num_slots, kv_row_stride] device, 16-byte aligned,
 *                  kv_row_stride >= 576 and a multiple of 8.
 *   kv_start       int64 [B] device; prefix_len, kv_capacity int32 [B] device.
 *   draft_kv       bf16 [B*T, 576] device, contiguous, 16-byte aligned.
 *   out_cache_loc  int32 [B*T] device or NULL.
 *   status         uint32 device word or NULL; bits are OR-ed in (the caller
 *                  clears it).
 * One warp per draft row; capture-safe, no host sync.  Returns VA_OK or a
 * VA_ERR_* code before any launch.
 */
int va_kv_append_contiguous(void *kv_pool, int64_t num_slots, int64_t kv_row_stride,
                            const int64_t *kv_start, const int32_t *prefix_len,
                            const int32_t *kv_capacity, const void *draft_kv, int B, int T,
                            int32_t *out_cache_loc, uint32_t *status, va_stream_t stream);

/*
 * va_kv_compact_accepted: for every request b, with P = prefix_len[b] and
 * n = accept_len[b], copies the first 576 columns of row
 *   kv_start[b] + P + accept_nodes[b*T + k]   to   kv_start[b] + P + k,
 * k < n, reading all n rows before writing any (a path may list its nodes in
 * any order), then sets prefix_len[b] = P + n.  accept_len and accept_nodes
 * are va_tree_accept's outputs.  A request with n outside [0, T], an accepted
 * node outside [0, T), P < 0, P + T > kv_capacity[b], or rows outside the
 * pool is left unchanged (pool and prefix_len) and sets VA_STATUS_BAD_DST in
 * *status (OR-ed in; NULL: not reported).
 *   accept_len    int32 [B] device; accept_nodes int32 [B, T] device.
 *   prefix_len    int32 [B] device, read and advanced in place.
 *   other arguments as for va_kv_append_contiguous.
 * One CTA per request, the rows staged in shared memory (T * 1152 bytes);
 * capture-safe, no host sync.  Returns VA_OK or a VA_ERR_* code before any
 * launch.
 */
int va_kv_compact_accepted(void *kv_pool, int64_t num_slots, int64_t kv_row_stride,
                           const int64_t *kv_start, int32_t *prefix_len,
                           const int32_t *kv_capacity, const int32_t *accept_len,
                           const int32_t *accept_nodes, int B, int T, uint32_t *status,
                           va_stream_t stream);

/*
 * Paged verify attention that allocates nothing and takes no workspace.
 * The pages have no counterpart; this entry point exists for callers that
 * cannot call cudaMalloc: a plugin inside a serving engine whose allocator
 * owns all device memory (the engine reserves nearly every byte for its KV
 * pool and gives plugins no allocation hook), or a caller on a latency path
 * where cudaMalloc / cudaFree would synchronise the device.
 *
 * Arguments are those of verify_attn_paged without workspace and
 * workspace_bytes; the caller still provides every input and out / lse.  The
 * scratch is a fixed device array of VA_NOALLOC_SCRATCH_BYTES inside the
 * library.  va_init(device) places it on that device (the driver loads the
 * library's device code lazily, so the array's memory is taken then) and
 * resolves its device address with cudaGetSymbolAddress; from then on each
 * GPU that was initialised holds the array until the process exits.  Call
 * va_init before reserving the rest of device memory.
 *  - Sizes: with nsplit = 0 the split count is lowered until the scratch
 *    layout fits; an explicit nsplit whose layout does not fit, or sizes for
 *    which even one split does not fit, return VA_ERR_WORKSPACE.
 *  - If va_init could not place the array (no device memory left for it),
 *    the first call on that device tries again and returns VA_ERR_CUDA if it
 *    still cannot; such a first call must come before any stream capture and
 *    is not thread-safe.
 *  - Every call shares the one array and leaves its contents behind; the call
 *    clears its status word itself.  Calls that overlap on the GPU (other
 *    streams, other threads) race on the array and must be serialised by the
 *    caller.  The status word sits in that array; it cannot be read with
 *    va_read_status.
 */
#define VA_NOALLOC_SCRATCH_BYTES (16u << 20)
int verify_attn_paged_noalloc(const void *q, const void *kv_pool, int64_t num_slots,
                              int64_t kv_row_stride, const int32_t *slot_idx,
                              const int32_t *kv_indptr, const int32_t *prefix_len,
                              const int32_t *tree_parent, const uint64_t *tree_bits, int B, int T,
                              int H, float sm_scale, int nsplit, int flags, void *out, float *lse,
                              va_stream_t stream);

/*
 * Benchmark helper: while both handles are non-NULL, every verify call on this
 * process records cudaEvent_t `before` on its stream immediately before it
 * launches the split-K partial kernel and `after` immediately after, so the
 * caller can time that kernel alone with cudaEventElapsedTime.  Pass NULLs to
 * stop.  Process-wide setting, not thread-safe; the events must belong to the
 * device of the calls.  Recording is a stream operation, so it is captured
 * into a graph like the kernels are.  Returns VA_OK.
 */
int va_set_partial_events(void *before, void *after);

/*
 * Test helper: waits for `stream`, then copies the workspace status word to
 * *status_host.  This one call synchronises; do not use it inside capture.
 */
int va_read_status(const void *workspace, uint32_t *status_host, va_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* VERIFY_ATTN_H */
