// va_mask.cu -- tree-mask evaluator (K0).
//
// Turns each request's draft-tree parent list into one 64-bit ancestor-or-self
// mask per node (The Checkpoint Report, "Mistakes and Incorrect Assumptions":
// the draft rows of the extend mask; "Input Knowledge Required": DDTree
// verifies a tree of draft tokens in one pass).  It also opens every verify
// call by clearing the workspace status word, so it runs even when the caller
// supplies the masks itself.
//
// One CTA; a warp per request, one lane walking the nodes in order.  Since
// parent[i] < i, node i's mask is its parent's mask plus its own bit.  A node
// whose parent is not an earlier node is flagged and treated as a child of the
// prefix.
#include "va_common.cuh"

namespace va {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32) tree_bits_kernel(Params p, uint64_t* bits_out) {
  __shared__ uint64_t masks[kWarps][kTmax];
  if (threadIdx.x == 0) *p.status = 0u;
  __syncthreads();
  if (p.tree_parent == nullptr) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int b = warp; b < p.B; b += kWarps) {
    if (lane == 0) {
      bool bad = false;
      for (int i = 0; i < p.T; ++i) {
        int par = p.tree_parent[size_t(b) * p.T + i];
        uint64_t m = 1ull << i;
        if (par < -1 || par >= i) bad = true;
        else if (par >= 0) m |= masks[warp][par];
        masks[warp][i] = m;
        bits_out[size_t(b) * p.T + i] = m;
      }
      if (bad) atomicOr(p.status, VA_STATUS_BAD_PARENT);
    }
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_tree_bits(const Params& p, uint64_t* bits_out, cudaStream_t st) {
  tree_bits_kernel<<<1, kWarps * 32, 0, st>>>(p, bits_out);
  return cudaGetLastError();
}

}  // namespace va
