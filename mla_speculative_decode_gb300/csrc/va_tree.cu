// va_tree.cu -- the draft tree and its KV slots, built on the device.
//
// The Checkpoint Report, "Input Knowledge Required to Understand This
// Message": a drafter proposes candidate tokens and DDTree builds a tree of
// draft tokens from them, which the target model verifies in one pass.  The
// Commit That Locked In 6x Decode, "4. The Marshaling Realization": that tree
// build (1.8 ms) and the mask build ran on the host every step.  Here they
// run in one small kernel that a CUDA graph can hold next to the verify call,
// and the draft tokens' KV slots (out_cache_loc, The Checkpoint Report,
// "Mistakes and Incorrect Assumptions") are taken from a device free list.
//
// The pages give no selection rule.  The drafter's output is read as K
// candidate tokens with log-probabilities for each of D draft positions, and
// the tree is grown best first: a node is a path of one candidate per depth
// from depth 0 down, scored by the float32 running sum of its log-
// probabilities; T times, the highest-scoring node whose parent is already in
// the tree is added (ties: the shallower node, then the lexicographically
// smaller path of candidate ranks).  Candidates of a depth are ranked by
// log-probability, highest first, ties by lower index; NaN and +inf are not
// log-probabilities and count as -inf.
//
// One warp grows one request's tree.  The frontier -- for every node added,
// its first child and its next sibling by rank -- always holds the best node
// that can be attached, and at most T + 1 entries; it lives in registers,
// entry e in lane e % 32.  A node's identity is a 64-bit key: depth in bits
// 60-63, candidate rank r_i at depth i in bits 56 - 4i .. 59 - 4i, so that
// comparing keys compares depth first, then the rank path lexicographically.
#include <math.h>
#include <string.h>

#include "va_common.cuh"

#ifndef VA_API
#define VA_API extern "C" __attribute__((visibility("default")))
#endif

namespace va {
namespace {

constexpr int kTreeWarps = 8;                 // requests per CTA at a time
constexpr int kMaxDepth = VA_TREE_MAX_DEPTH;  // 15: the rank path fits 60 bits
constexpr int kMaxCand = VA_TREE_MAX_CAND;    // 16: a rank fits 4 bits
constexpr int kSlotsPerLane = (VA_T_MAX + 1 + 31) / 32;   // frontier capacity 96

struct TreeParams {
  const int32_t* cand_tokens;   // [B, D, K]
  const float* cand_logp;       // [B, D, K]
  int B, D, K, T;
  const int32_t* free_slots;    // [free_capacity] or NULL
  int64_t free_capacity;
  int32_t* free_head;           // device int32, or NULL with free_slots
  int32_t* parent;              // [B, T]
  int32_t* tokens;              // [B, T]
  int32_t* depth;               // [B, T] or NULL
  int32_t* out_cache_loc;       // [B*T] or NULL with free_slots
  uint32_t* status;             // or NULL
};

// a ranks above b: higher score, else (equal score) smaller key
__device__ __forceinline__ bool better(float sa, uint64_t ka, float sb, uint64_t kb) {
  return sa > sb || (sa == sb && ka < kb);
}

// Unsigned key with the order of the scores (which are never NaN: the
// candidates' NaN and +inf count as -inf); -0 counts as +0, as it compares
// equal to it.  Every score maps above 0.
__device__ __forceinline__ uint32_t score_order(float sc) {
  const uint32_t u = __float_as_uint(sc == 0.f ? 0.f : sc);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int key_depth(uint64_t key) { return int(key >> 60); }
__device__ __forceinline__ int key_rank(uint64_t key, int d) {
  return int((key >> (56 - 4 * d)) & 15u);
}

__global__ void __launch_bounds__(kTreeWarps * 32) tree_build_kernel(TreeParams p) {
  __shared__ float s_lp[kTreeWarps][kMaxDepth][kMaxCand];     // ranked log-probabilities
  __shared__ int32_t s_tok[kTreeWarps][kMaxDepth][kMaxCand];  // ranked tokens
  __shared__ float s_rlp[kTreeWarps][kMaxDepth * kMaxCand];   // as drafted
  __shared__ int32_t s_rtok[kTreeWarps][kMaxDepth * kMaxCand];
  __shared__ int64_t s_head;
  __shared__ uint32_t s_flags;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    s_head = p.free_head ? int64_t(*p.free_head) : 0;
    s_flags = 0u;
  }
  __syncthreads();
  const int64_t head = s_head;
  for (int b = warp; b < p.B; b += kTreeWarps) {
    // 1. the request's D*K candidates, all loads in flight at once (one
    // memory round trip, not one per depth), then each depth ranked: lane
    // k < K finds how many candidates beat its own and stores itself at that
    // rank
    {
      constexpr int kLoads = (kMaxDepth * kMaxCand + 31) / 32;
      const int dk = p.D * p.K;
      const size_t base = size_t(b) * dk;
      float lv[kLoads];
      int32_t lt[kLoads];
#pragma unroll
      for (int j = 0; j < kLoads; ++j) {
        const int e = lane + 32 * j;
        if (e < dk) {
          lv[j] = p.cand_logp[base + e];
          lt[j] = p.cand_tokens[base + e];
        }
      }
#pragma unroll
      for (int j = 0; j < kLoads; ++j) {
        const int e = lane + 32 * j;
        if (e < dk) {
          s_rlp[warp][e] = lv[j];
          s_rtok[warp][e] = lt[j];
        }
      }
      __syncwarp();
    }
    for (int d = 0; d < p.D; ++d) {
      float v = -INFINITY;
      int32_t tk = 0;
      if (lane < p.K) {
        v = s_rlp[warp][d * p.K + lane];
        tk = s_rtok[warp][d * p.K + lane];
        if (!(v < INFINITY)) v = -INFINITY;    // NaN, +inf
      }
      int rank = 0;
      for (int k = 0; k < p.K; ++k) {
        const float o = __shfl_sync(0xffffffffu, v, k);
        rank += (o > v || (o == v && k < lane)) ? 1 : 0;
      }
      if (lane < p.K) {
        s_lp[warp][d][rank] = v;
        s_tok[warp][d][rank] = tk;
      }
    }
    __syncwarp();
    // 2. grow the tree best first
    float f_score[kSlotsPerLane], f_pscore[kSlotsPerLane];
    uint64_t f_key[kSlotsPerLane];
    int f_parent[kSlotsPerLane];
#pragma unroll
    for (int j = 0; j < kSlotsPerLane; ++j) {
      f_score[j] = -INFINITY;
      f_pscore[j] = 0.f;
      f_key[j] = ~0ull;
      f_parent[j] = -1;
    }
    // the first node: rank 0 at depth 0, parent score 0
    if (lane == 0) {
      f_score[0] = __fadd_rn(0.f, s_lp[warp][0][0]);
      f_key[0] = 0ull;
      f_pscore[0] = 0.f;
      f_parent[0] = -1;
    }
    int n = 1;
    for (int i = 0; i < p.T; ++i) {
      // best entry of this lane, then of the warp
      float bs = -INFINITY;
      uint64_t bk = ~0ull;
      int bj = -1;
#pragma unroll
      for (int j = 0; j < kSlotsPerLane; ++j) {
        const int e = j * 32 + lane;
        if (e < n && (bj < 0 || better(f_score[j], f_key[j], bs, bk))) {
          bs = f_score[j];
          bk = f_key[j];
          bj = j;
        }
      }
      int be = bj < 0 ? -1 : bj * 32 + lane;   // frontier index of the lane's best
      // The warp's best with three reductions instead of a shuffle tree: the
      // highest score (as an order-preserving unsigned key; a lane without an
      // entry offers 0, below every score), then among the lanes holding it
      // the smallest node key, high word then low word.  Node keys are
      // unique, so exactly one lane wins.
      {
        const uint32_t sk = be < 0 ? 0u : score_order(bs);
        const uint32_t smax = __reduce_max_sync(0xffffffffu, sk);
        const bool top = be >= 0 && sk == smax;
        const uint32_t hi = uint32_t(bk >> 32), lo = uint32_t(bk);
        const uint32_t hmin = __reduce_min_sync(0xffffffffu, top ? hi : 0xffffffffu);
        const bool top2 = top && hi == hmin;
        const uint32_t lmin = __reduce_min_sync(0xffffffffu, top2 ? lo : 0xffffffffu);
        const int src = __ffs(__ballot_sync(0xffffffffu, top2 && lo == lmin)) - 1;
        bs = __shfl_sync(0xffffffffu, bs, src);
        bk = (uint64_t(hmin) << 32) | lmin;
        be = __shfl_sync(0xffffffffu, be, src);
      }
      // the winner's parent fields, from the lane that holds it
      const int wl = be & 31, wj = be >> 5;
      float my_ps = 0.f;
      int my_par = -1;
#pragma unroll
      for (int j = 0; j < kSlotsPerLane; ++j)
        if (j == wj) {
          my_ps = f_pscore[j];
          my_par = f_parent[j];
        }
      const float wps = __shfl_sync(0xffffffffu, my_ps, wl);
      const int wpar = __shfl_sync(0xffffffffu, my_par, wl);
      const int d = key_depth(bk);
      const int r = key_rank(bk, d);
      if (lane == 0) {
        const size_t o = size_t(b) * p.T + i;
        p.parent[o] = wpar;
        p.tokens[o] = s_tok[warp][d][r];
        if (p.depth) p.depth[o] = d;
      }
      // remove the winner: the last entry moves into its place
      const int last = n - 1;
      const int ll = last & 31, lj = last >> 5;
      float l_s = 0.f, l_ps = 0.f;
      uint64_t l_k = 0ull;
      int l_par = -1;
#pragma unroll
      for (int j = 0; j < kSlotsPerLane; ++j)
        if (j == lj) {
          l_s = f_score[j];
          l_ps = f_pscore[j];
          l_k = f_key[j];
          l_par = f_parent[j];
        }
      l_s = __shfl_sync(0xffffffffu, l_s, ll);
      l_ps = __shfl_sync(0xffffffffu, l_ps, ll);
      l_k = __shfl_sync(0xffffffffu, l_k, ll);
      l_par = __shfl_sync(0xffffffffu, l_par, ll);
      if (lane == wl) {
#pragma unroll
        for (int j = 0; j < kSlotsPerLane; ++j)
          if (j == wj) {
            f_score[j] = l_s;
            f_pscore[j] = l_ps;
            f_key[j] = l_k;
            f_parent[j] = l_par;
          }
      }
      n = last;
      // add its first child and its next sibling
      auto push = [&](float sc, float ps, uint64_t key, int par) {
        const int pl = n & 31, pj = n >> 5;
        if (lane == pl) {
#pragma unroll
          for (int j = 0; j < kSlotsPerLane; ++j)
            if (j == pj) {
              f_score[j] = sc;
              f_pscore[j] = ps;
              f_key[j] = key;
              f_parent[j] = par;
            }
        }
        ++n;
      };
      if (d + 1 < p.D) push(__fadd_rn(bs, s_lp[warp][d + 1][0]), bs, bk + (1ull << 60), i);
      if (r + 1 < p.K)
        push(__fadd_rn(wps, s_lp[warp][d][r + 1]), wps, bk + (1ull << (56 - 4 * d)), wpar);
    }
    // 3. the draft nodes' KV slots, in request order from the free list
    if (p.free_slots) {
      bool ran_out = false;
      for (int i = lane; i < p.T; i += 32) {
        const int64_t e = head + int64_t(b) * p.T + i;
        const bool in = e >= 0 && e < p.free_capacity;
        p.out_cache_loc[size_t(b) * p.T + i] = in ? p.free_slots[e] : -1;
        ran_out |= !in;
      }
      if (__any_sync(0xffffffffu, ran_out) && lane == 0) atomicOr(&s_flags, VA_STATUS_BAD_SLOT);
    }
    __syncwarp();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (p.free_head) *p.free_head = int32_t(head + int64_t(p.B) * p.T);
    if (p.status) *p.status = s_flags;
  }
}

bool aligned4(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; }

}  // namespace
}  // namespace va

VA_API int va_tree_build(const int32_t* cand_tokens, const float* cand_logp, int B, int D, int K,
                         int T, const int32_t* free_slots, int64_t free_capacity,
                         int32_t* free_head, int32_t* tree_parent, int32_t* draft_tokens,
                         int32_t* node_depth, int32_t* out_cache_loc, uint32_t* status,
                         va_stream_t stream) {
  using namespace va;
  if (!cand_tokens || !cand_logp || !tree_parent || !draft_tokens) return VA_ERR_NULL;
  if (free_slots && (!free_head || !out_cache_loc)) return VA_ERR_NULL;
  if (B < 1 || B > 65535 || D < 1 || D > VA_TREE_MAX_DEPTH || K < 1 || K > VA_TREE_MAX_CAND ||
      T < 1 || T > VA_T_MAX || (free_slots && free_capacity < 0))
    return VA_ERR_SHAPE;
  // the candidate tree must hold at least T nodes: K + K^2 + ... + K^D
  int64_t nodes = 0, level = 1;
  for (int d = 0; d < D && nodes < T; ++d) {
    level *= K;
    nodes += level;
  }
  if (nodes < T) return VA_ERR_SHAPE;
  if (!aligned4(cand_tokens) || !aligned4(cand_logp) || !aligned4(tree_parent) ||
      !aligned4(draft_tokens) || (node_depth && !aligned4(node_depth)) ||
      (free_slots && !aligned4(free_slots)) || (free_head && !aligned4(free_head)) ||
      (out_cache_loc && !aligned4(out_cache_loc)) || (status && !aligned4(status)))
    return VA_ERR_ALIGN;
  TreeParams p;
  memset(&p, 0, sizeof p);
  p.cand_tokens = cand_tokens;
  p.cand_logp = cand_logp;
  p.B = B;
  p.D = D;
  p.K = K;
  p.T = T;
  p.free_slots = free_slots;
  p.free_capacity = free_capacity;
  p.free_head = free_slots ? free_head : nullptr;
  p.parent = tree_parent;
  p.tokens = draft_tokens;
  p.depth = node_depth;
  p.out_cache_loc = free_slots ? out_cache_loc : nullptr;
  p.status = status;
  // one CTA: every request's slots are taken at the free-list head read at
  // its start, and the head is advanced once, after all of them
  tree_build_kernel<<<1, kTreeWarps * 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? VA_OK : VA_ERR_LAUNCH;
}
