// va_mask.cu -- tree-mask evaluator (K0).
//
// Turns each request's draft-tree parent list into one 64-bit ancestor-or-self
// mask per node (The Checkpoint Report, "Mistakes and Incorrect Assumptions":
// the draft rows of the extend mask; "Input Knowledge Required": DDTree
// verifies a tree of draft tokens in one pass).  For segmented calls it reads
// the same sets out of the dense extend mask instead (the last T columns of
// each draft row, stride prefix + q_len).  It also opens every verify call by
// clearing the workspace status word, so it runs even when the caller
// supplies the masks itself.
//
// One CTA; a warp per request.  The request's parents are staged in shared
// memory and each lane builds its own node's set by walking up the tree
// (indices strictly decrease, so at most T steps).  A node whose parent is
// not an earlier node is flagged and treated as hanging off the prefix; the
// walk stops there too, which is the same as taking node i's set as its own
// bit plus its parent's set.
#include "va_common.cuh"

namespace va {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32) tree_bits_kernel(Params p, uint64_t* bits_out) {
  __shared__ int par[kWarps][kTmax];
  griddep_launch_dependents();   // the split-K kernel may start its set-up now
  if (threadIdx.x == 0) *p.status = 0u;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (p.dense_mask) {
    // Dense extend-mask rows (segmented calls): request b's T rows of P_b + T
    // entries follow the rows of the requests before it; node i's set is the
    // last T entries of its row.  Entries outside the mask read as 0.
    const int64_t first = p.kv_indptr[0];
    for (int b = warp; b < p.B; b += kWarps) {
      const int i0 = p.kv_indptr[b], i1 = p.kv_indptr[b + 1];
      const int64_t P = i1 > i0 ? int64_t(i1) - i0 : 0;
      const int64_t off = int64_t(p.T) * ((int64_t(i0) - first) + int64_t(b) * p.T);
      bool bad = false;
      for (int i = lane; i < p.T; i += 32) {
        const int64_t row = off + int64_t(i) * (P + p.T) + P;
        uint64_t m = 0;
        for (int k = 0; k < p.T; ++k) {
          const int64_t e = row + k;
          if (e >= 0 && e < p.dense_mask_len) {
            if (p.dense_mask[e]) m |= 1ull << k;
          } else {
            bad = true;
          }
        }
        bits_out[size_t(b) * p.T + i] = m;
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.status, VA_STATUS_BAD_MASK);
      __syncwarp();
    }
    return;
  }
  if (p.tree_parent == nullptr) return;
  for (int b = warp; b < p.B; b += kWarps) {
    for (int i = lane; i < p.T; i += 32) par[warp][i] = p.tree_parent[size_t(b) * p.T + i];
    __syncwarp();
    bool bad = false;
    for (int i = lane; i < p.T; i += 32) {
      uint64_t m = 1ull << i;
      int q = par[warp][i];
      if (q < -1 || q >= i) {
        bad = true;
      } else {
        while (q >= 0) {
          m |= 1ull << q;
          const int up = par[warp][q];
          if (up < -1 || up >= q) break;
          q = up;
        }
      }
      bits_out[size_t(b) * p.T + i] = m;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.status, VA_STATUS_BAD_PARENT);
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_tree_bits(const Params& p, uint64_t* bits_out, cudaStream_t st) {
  tree_bits_kernel<<<1, kWarps * 32, 0, st>>>(p, bits_out);
  return cudaGetLastError();
}

}  // namespace va
