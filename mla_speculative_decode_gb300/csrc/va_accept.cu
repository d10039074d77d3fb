// va_accept.cu -- greedy tree acceptance after verify.
//
// The Milestone Commit, "Input Knowledge Required": the verify step checks
// whether the draft predictions are correct.  The Checkpoint Report, "Input
// Knowledge Required to Understand This Message": a drafter proposes a tree
// of candidate tokens and the target model checks them in one parallel pass.
// Greedy acceptance walks that tree: from the prefix, the target's most
// likely next token selects the child that carries it; the walk ends at the
// first position where no child does, and the target's token there is the
// bonus token emitted after the accepted path.
//
// Two kernels, chained by programmatic dependent launch:
//  - argmax_partial_kernel: the logits rows (per request the last prefix
//    position, then its T draft nodes) cut into chunks, one CTA per chunk,
//    each writing its best (value, index) to the workspace.  Every logit is
//    read once: HBM-bound.
//  - accept_walk_kernel: one warp per request merges its rows' chunks (a
//    lane per row) and walks the tree, a vote of the lanes per step (lane
//    c % 32 holding node c's parent, token and slot).
// The argmax is the lowest index among the largest non-NaN values (0 for a
// row of NaN only); both kernels compare with the same rule, so the result
// does not depend on the chunking.
#include <string.h>

#include "va_common.cuh"

#ifndef VA_API
#define VA_API extern "C" __attribute__((visibility("default")))
#endif

namespace va {
namespace {

constexpr int kArgThreads = 256;
constexpr int kWalkWarps = 8;
constexpr int kTargetCtas = 1024;   // argmax CTAs aimed for (several per SM)
constexpr int64_t kMinChunk = 4096; // logits per CTA at least

struct AcceptParams {
  const float* root_logits;   // [B, V]
  const float* logits;        // [B, T, V]
  int64_t V;
  const int32_t* tokens;      // [B, T]
  const int32_t* parent;      // [B, T]
  const int32_t* slots;       // [B, T] or NULL
  int B, T, chunks;
  int64_t chunk_len;
  float* part_val;            // [B*(T+1)][chunks]
  int32_t* part_idx;          // [B*(T+1)][chunks]
  uint32_t* status;
  int32_t* accept_len;        // [B]
  int32_t* accept_nodes;      // [B, T]
  int32_t* accept_slots;      // [B, T] or NULL
  int32_t* bonus;             // [B]
};

// (v, i) ranks above (bv, bi): a larger value, or the same value at a lower
// index.  NaN compares false both ways, so it never ranks above anything.
__device__ __forceinline__ bool ranks_above(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void warp_best(float& bv, int& bi) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ranks_above(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
}

__global__ void __launch_bounds__(kArgThreads) argmax_partial_kernel(AcceptParams a) {
  griddep_launch_dependents();   // the walk kernel may be scheduled now
  __shared__ float sv[kArgThreads / 32];
  __shared__ int si[kArgThreads / 32];
  const int r = blockIdx.x, c = blockIdx.y;   // logits row, chunk of it
  if (c == 0 && r == 0 && threadIdx.x == 0) *a.status = 0u;
  const int b = r / (a.T + 1), k = r - b * (a.T + 1);
  const float* row = k == 0 ? a.root_logits + size_t(b) * a.V
                            : a.logits + (size_t(b) * a.T + (k - 1)) * a.V;
  const int64_t i0 = int64_t(c) * a.chunk_len;
  const int64_t i1 = i0 + a.chunk_len < a.V ? i0 + a.chunk_len : a.V;
  float bv = -INFINITY;
  int bi = int(a.V);   // past every index: any non-NaN value ranks above it
  if ((a.V & 3) == 0 && (reinterpret_cast<uintptr_t>(row) & 15) == 0) {
    // 16-byte loads (chunks start at multiples of 4 elements)
    const float4* row4 = reinterpret_cast<const float4*>(row);
#pragma unroll 4
    for (int64_t i4 = i0 / 4 + threadIdx.x; i4 < i1 / 4; i4 += kArgThreads) {
      const float4 v = __ldg(row4 + i4);
      const int i = int(i4 * 4);
      if (ranks_above(v.x, i, bv, bi)) { bv = v.x; bi = i; }
      if (ranks_above(v.y, i + 1, bv, bi)) { bv = v.y; bi = i + 1; }
      if (ranks_above(v.z, i + 2, bv, bi)) { bv = v.z; bi = i + 2; }
      if (ranks_above(v.w, i + 3, bv, bi)) { bv = v.w; bi = i + 3; }
    }
  } else {
#pragma unroll 8
    for (int64_t i = i0 + threadIdx.x; i < i1; i += kArgThreads) {
      const float v = __ldg(row + i);
      if (ranks_above(v, int(i), bv, bi)) {
        bv = v;
        bi = int(i);
      }
    }
  }
  warp_best(bv, bi);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[warp] = bv;
    si[warp] = bi;
  }
  __syncthreads();
  if (warp == 0) {
    bv = lane < kArgThreads / 32 ? sv[lane] : -INFINITY;
    bi = lane < kArgThreads / 32 ? si[lane] : int(a.V);
    warp_best(bv, bi);
    if (lane == 0) {
      a.part_val[size_t(r) * a.chunks + c] = bv;
      a.part_idx[size_t(r) * a.chunks + c] = bi;
    }
  }
}

__global__ void __launch_bounds__(kWalkWarps * 32) accept_walk_kernel(AcceptParams a) {
  __shared__ int tok[kWalkWarps][kTmax + 1];
  griddep_wait();   // the argmax kernel's partials are complete and visible
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kWalkWarps + warp;
  if (b >= a.B) return;
  const int T = a.T;
  // lane l merges the chunks of rows l, l + 32, ...: the loads of every row
  // are independent, so they are all in flight together
  for (int k = lane; k <= T; k += 32) {
    const size_t r = size_t(b) * (T + 1) + k;
    float bv = -INFINITY;
    int bi = int(a.V);
    for (int c = 0; c < a.chunks; ++c) {
      const float v = a.part_val[r * a.chunks + c];
      const int i = a.part_idx[r * a.chunks + c];
      if (ranks_above(v, i, bv, bi)) {
        bv = v;
        bi = i;
      }
    }
    tok[warp][k] = bi < a.V ? bi : 0;   // a row of NaN only: token 0
  }
  __syncwarp();
  // Node c = lane + 32h (h = 0, 1; T <= 64) in registers of lane c % 32: its
  // parent (one that is not an earlier node counts as the prefix, and is
  // flagged), its draft token and its slot; -2 marks "no node".
  const int32_t* par = a.parent + size_t(b) * T;
  const int32_t* tk = a.tokens + size_t(b) * T;
  const int32_t* sl = a.slots ? a.slots + size_t(b) * T : nullptr;
  int pc[2], tc[2], sc[2];
  bool bad = false;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c = lane + 32 * h;
    pc[h] = -2;
    tc[h] = 0;
    sc[h] = -1;
    if (c < T) {
      const int q = par[c];
      const bool ok = q >= -1 && q < c;
      bad |= !ok;
      pc[h] = ok ? q : -1;
      tc[h] = tk[c];
      if (sl) sc[h] = sl[c];
    }
  }
  bad = __any_sync(0xffffffffu, bad);
  // Each accepted node is a child of the previous one, so has a larger index:
  // at most T steps, each one vote of the lanes (the lowest-numbered child of
  // `cur` whose draft token is the target's token `t`).
  int cur = -1, n = 0, t = tok[warp][0];
  for (;;) {
    const uint32_t m0 = __ballot_sync(0xffffffffu, lane > cur && pc[0] == cur && tc[0] == t);
    const uint32_t m1 = __ballot_sync(0xffffffffu, lane + 32 > cur && pc[1] == cur && tc[1] == t);
    const int pick = m0 ? __ffs(m0) - 1 : (m1 ? 32 + __ffs(m1) - 1 : -1);
    if (pick < 0) break;
    const int ps = __shfl_sync(0xffffffffu, pick < 32 ? sc[0] : sc[1], pick & 31);
    if (lane == 0) {
      a.accept_nodes[size_t(b) * T + n] = pick;
      if (a.accept_slots) a.accept_slots[size_t(b) * T + n] = ps;
    }
    ++n;
    cur = pick;
    t = tok[warp][pick + 1];
  }
  for (int m = n + lane; m < T; m += 32) {
    a.accept_nodes[size_t(b) * T + m] = -1;
    if (a.accept_slots) a.accept_slots[size_t(b) * T + m] = -1;
  }
  if (lane == 0) {
    a.accept_len[b] = n;
    a.bonus[b] = t;
    if (bad) atomicOr(a.status, VA_STATUS_BAD_PARENT);
  }
}

struct AcceptLayout {
  int chunks;
  int64_t chunk_len;
  size_t val, idx, total;
};

AcceptLayout accept_layout(int B, int T, int64_t V) {
  AcceptLayout L;
  const int rows = B * (T + 1);
  int64_t c = (kTargetCtas + rows - 1) / rows;
  const int64_t cmax = V / kMinChunk > 1 ? V / kMinChunk : 1;
  if (c > cmax) c = cmax;
  if (c < 1) c = 1;
  L.chunk_len = ((V + c - 1) / c + 3) & ~int64_t(3);   // a multiple of 4 elements
  L.chunks = int((V + L.chunk_len - 1) / L.chunk_len);
  L.val = kHeaderBytes;
  L.idx = L.val + align256(size_t(rows) * L.chunks * sizeof(float));
  L.total = L.idx + align256(size_t(rows) * L.chunks * sizeof(int32_t));
  return L;
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace va

VA_API size_t va_tree_accept_workspace_bytes(int B, int T, int64_t V) {
  if (B < 1 || B > 65535 || T < 1 || T > VA_T_MAX || V < 1 || V > 0x7ffffffe) return 0;
  return va::accept_layout(B, T, V).total;
}

VA_API int va_tree_accept(const float* root_logits, const float* logits, int64_t V,
                          const int32_t* draft_tokens, const int32_t* tree_parent,
                          const int32_t* draft_slots, int B, int T, void* workspace,
                          size_t workspace_bytes, int32_t* accept_len, int32_t* accept_nodes,
                          int32_t* accept_slots, int32_t* bonus_token, va_stream_t stream) {
  using namespace va;
  if (!root_logits || !logits || !draft_tokens || !tree_parent || !workspace || !accept_len ||
      !accept_nodes || !bonus_token)
    return VA_ERR_NULL;
  if (B < 1 || B > 65535 || T < 1 || T > VA_T_MAX || V < 1 || V > 0x7ffffffe) return VA_ERR_SHAPE;
  if (!aligned_to(root_logits, 4) || !aligned_to(logits, 4) || !aligned_to(draft_tokens, 4) ||
      !aligned_to(tree_parent, 4) || !aligned_to(workspace, 256) || !aligned_to(accept_len, 4) ||
      !aligned_to(accept_nodes, 4) || !aligned_to(bonus_token, 4) ||
      (draft_slots && !aligned_to(draft_slots, 4)) || (accept_slots && !aligned_to(accept_slots, 4)))
    return VA_ERR_ALIGN;
  const AcceptLayout L = accept_layout(B, T, V);
  if (workspace_bytes < L.total) return VA_ERR_WORKSPACE;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  AcceptParams a;
  memset(&a, 0, sizeof a);
  a.root_logits = root_logits;
  a.logits = logits;
  a.V = V;
  a.tokens = draft_tokens;
  a.parent = tree_parent;
  a.slots = draft_slots;
  a.B = B;
  a.T = T;
  a.chunks = L.chunks;
  a.chunk_len = L.chunk_len;
  a.part_val = reinterpret_cast<float*>(w + L.val);
  a.part_idx = reinterpret_cast<int32_t*>(w + L.idx);
  a.status = reinterpret_cast<uint32_t*>(w);
  a.accept_len = accept_len;
  a.accept_nodes = accept_nodes;
  a.accept_slots = accept_slots;
  a.bonus = bonus_token;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  argmax_partial_kernel<<<dim3(unsigned(B * (T + 1)), unsigned(L.chunks), 1u), kArgThreads, 0,
                          st>>>(a);
  if (cudaGetLastError() != cudaSuccess) return VA_ERR_LAUNCH;
  // the walk kernel may be scheduled while the argmax CTAs run; it waits
  // (griddepcontrol.wait) before reading their partials
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(unsigned((B + kWalkWarps - 1) / kWalkWarps), 1u, 1u);
  cfg.blockDim = dim3(kWalkWarps * 32, 1u, 1u);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, accept_walk_kernel, a) != cudaSuccess) return VA_ERR_LAUNCH;
  return VA_OK;
}
