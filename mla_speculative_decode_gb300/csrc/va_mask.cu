// va_mask.cu -- tree-mask evaluator (K0).
//
// Turns each request's draft-tree parent list into one 64-bit ancestor-or-self
// mask per node (The Checkpoint Report, "Mistakes and Incorrect Assumptions":
// the draft rows of the extend mask; "Input Knowledge Required": DDTree
// verifies a tree of draft tokens in one pass).  For segmented calls it reads
// the same sets out of the dense extend mask instead (the last T columns of
// each draft row, stride prefix + q_len).  On the FMA path it also opens
// every verify call by clearing the workspace status word, so it runs even
// when the caller supplies the masks itself.  On the tensor-core path the
// split-K kernel computes the masks itself and this kernel runs only to
// append draft rows (its extra CTAs).
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

constexpr int kAppendRowsPerCta = 32;

__global__ void __launch_bounds__(kWarps * 32) tree_bits_kernel(Params p, uint64_t* bits_out) {
  __shared__ int par[kWarps][kTmax];
  griddep_launch_dependents();   // the split-K kernel may start its set-up now
  if (blockIdx.x > 0) {
    // Draft-row append (segmented calls with draft_kv): row b*T + i of
    // draft_kv goes to the pool row of request b's draft key P_b + i, one
    // warp per row, 16-byte chunks.  Rows without a valid pool row are
    // skipped (the split-K kernel flags them when it reads the key).  The
    // split-K kernel reads draft keys only after griddepcontrol.wait, that
    // is after this grid has completed.
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = (blockIdx.x - 1) * kAppendRowsPerCta;
    const int nrows = p.B * p.T;
    for (int r = r0 + warp; r < r0 + kAppendRowsPerCta && r < nrows; r += kWarps) {
      const int b = r / p.T, i = r - b * p.T;
      const ReqInfo ri = req_info(p, b, false);
      const int64_t row = key_row(p, ri, ri.P + i);
      if (row < 0) continue;
      const uint4* src = reinterpret_cast<const uint4*>(p.draft_kv + size_t(r) * kDqk);
      uint4* dst = reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(p.kv) + row * p.kv_stride);
      for (int c = lane; c < kDqk / 8; c += 32) dst[c] = src[c];
    }
    return;
  }
  // tensor-core path: the split-K kernel computes the masks and the merge
  // kernel writes the status word; this kernel only appends draft rows there
  if (p.cta_flags) return;
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
  // one CTA for the masks and the status word, and with draft rows to append,
  // one more per kAppendRowsPerCta rows
  const int rows = p.draft_kv ? p.B * p.T : 0;
  const int grid = 1 + (rows + kAppendRowsPerCta - 1) / kAppendRowsPerCta;
  tree_bits_kernel<<<grid, kWarps * 32, 0, st>>>(p, bits_out);
  return cudaGetLastError();
}

}  // namespace va
