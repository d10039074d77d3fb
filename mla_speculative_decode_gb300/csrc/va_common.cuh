// va_common.cuh -- definitions shared by the verify-attention kernels and the
// host launcher: launch parameters, workspace layout, the split schedule and
// small device helpers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "verify_attn.h"

namespace va {

constexpr int kDqk = VA_D_QK;   // 576: latent 512 + rotary 64
constexpr int kDv = VA_D_V;     // 512
constexpr int kTmax = VA_T_MAX;
// Splits are cut on multiples of this many keys, so a split never holds a
// ragged tile except at the request's end.
constexpr int kSplitGrain = 64;
constexpr size_t kHeaderBytes = 256;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__host__ __device__ constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Workspace regions (byte offsets from the workspace base).
struct WsLayout {
  size_t bits;   // uint64 [B*T]
  size_t flags;  // uint32 [B][2 x row units of 256][nsplit][2]: status bits of each split-K CTA
  size_t plse;   // float  [nsplit][rows]
  size_t po;     // bf16   [nsplit][rows][512]
  size_t total;
};

__host__ __device__ inline WsLayout ws_layout(int B, int T, int H, int nsplit) {
  WsLayout L;
  const size_t rows = size_t(B) * T * H;
  L.bits = kHeaderBytes;
  L.flags = L.bits + align256(size_t(B) * T * sizeof(uint64_t));
  const size_t rbs = 2 * ((size_t(T) * H + 255) / 256);   // 128-row blocks, rounded to pairs
  L.plse = L.flags + align256(size_t(B) * rbs * nsplit * 2 * sizeof(uint32_t));
  L.po = L.plse + align256(size_t(nsplit) * rows * sizeof(float));
  L.total = L.po + align256(size_t(nsplit) * rows * kDv * sizeof(__nv_bfloat16));
  return L;
}

// Everything a verify launch needs (passed by value to every kernel).
struct Params {
  const __nv_bfloat16* q;      // [B*T, H, 576]
  const __nv_bfloat16* kv;     // [num_slots, kv_stride]
  int64_t num_slots;
  int64_t kv_stride;           // elements
  const int32_t* slot_idx;     // paged: concatenated slot lists; segmented: prefix lists
  const int32_t* kv_indptr;    // paged, segmented: [B+1]
  const int64_t* kv_start;     // contiguous: [B] (NULL when paged)
  const int32_t* draft_slots;  // segmented: [B*T] slots of the draft nodes (else NULL)
  const __nv_bfloat16* draft_kv;  // segmented: [B*T, 576] rows written to those slots first, or NULL
  const int32_t* prefix_len;   // [B] (NULL when segmented: the prefix list's length)
  const uint8_t* dense_mask;   // segmented: dense extend mask rows, or NULL
  int64_t dense_mask_len;      // entries in dense_mask
  const int32_t* tree_parent;  // [B, T] or NULL
  const uint64_t* bits;        // [B, T] ancestor-or-self masks (caller's or workspace)
  int B, T, H;
  int rows_per_req;            // T * H
  int nsplit;                  // splits per (request, row block) grid slot
  float sm_scale;
  float scale_log2;            // sm_scale * log2(e)
  float* part_lse;             // [nsplit][rows]
  __nv_bfloat16* part_o;       // [nsplit][rows][512], normalised by the split's row sum
  uint32_t* status;
  // Tensor-core path: each split-K CTA stores its status bits to its own word
  // here ([B][row blocks][nsplit][2]) and the merge kernel writes their OR to
  // *status, so no kernel has to clear *status first.  NULL on the FMA path,
  // where the mask kernel clears *status and the kernels OR into it.
  uint32_t* cta_flags;
  int flag_blocks;             // 128-row blocks of status words per request
  int tc_pair;                 // tensor-core path: two-SM products (clusters of 4)
  __nv_bfloat16* out;          // [rows, 512]
  float* lse;                  // [rows]
};

// Key range of one split.  A request has N = prefix + T keys; it is cut into
// at most `nsplit` pieces of a whole number of 64-key grains, so a short
// request uses fewer splits (empty splits exit at once and the merge reads
// only the first `nsplit_eff`).
struct SplitRange {
  int k0, k1, nsplit_eff;
};

__host__ __device__ inline SplitRange split_range(int N, int nsplit, int s) {
  SplitRange r;
  int grains = ceil_div(N > 0 ? N : 1, kSplitGrain);
  int ne = nsplit < grains ? nsplit : grains;
  if (ne < 1) ne = 1;
  int chunk = ceil_div(grains, ne) * kSplitGrain;
  ne = ceil_div(N > 0 ? N : 1, chunk);
  r.nsplit_eff = ne;
  r.k0 = s * chunk;
  r.k1 = r.k0 + chunk < N ? r.k0 + chunk : N;
  return r;
}

// Per-request key bookkeeping read on the device.
struct ReqInfo {
  int P;         // effective prefix length
  int N;         // P + T
  int nlist;     // keys that have a slot (paged: slot list length; contiguous: N)
  int64_t base;  // paged, segmented: offset into slot_idx; contiguous: first pool row
  int64_t dbase; // segmented: draft key j >= P is draft_slots[dbase + j]
};

__device__ inline ReqInfo req_info(const Params& p, int b, bool flag, bool* bad_out = nullptr) {
  ReqInfo r;
  r.dbase = 0;
  bool bad = false;
  if (p.draft_slots) {
    // segmented: the prefix is the whole prefix list, the draft nodes' slots
    // are a list of their own
    const int i0 = p.kv_indptr[b], i1 = p.kv_indptr[b + 1];
    int P = i1 - i0;
    if (P < 0) { P = 0; bad = true; }
    r.P = P;
    r.N = P + p.T;
    r.nlist = r.N;
    r.base = i0;
    r.dbase = int64_t(b) * p.T - P;
    if (bad && flag) atomicOr(p.status, VA_STATUS_BAD_INDPTR);
    if (bad_out) *bad_out = bad;
    return r;
  }
  int P = p.prefix_len[b];
  if (P < 0) { P = 0; bad = true; }
  if (p.kv_start == nullptr) {
    int i0 = p.kv_indptr[b], i1 = p.kv_indptr[b + 1];
    int nl = i1 - i0;
    if (nl < 0) nl = 0;
    if (nl < P + p.T) {
      bad = true;
      P = nl - p.T > 0 ? (nl - p.T < P ? nl - p.T : P) : 0;
    }
    r.nlist = nl;
    r.base = i0;
  } else {
    r.base = p.kv_start[b];
    r.nlist = P + p.T;
  }
  r.P = P;
  r.N = P + p.T;
  if (bad && flag) atomicOr(p.status, VA_STATUS_BAD_INDPTR);
  if (bad_out) *bad_out = bad;
  return r;
}

// Pool row of key j of a request, or -1 when the key has no valid row.
__device__ inline int64_t key_row(const Params& p, const ReqInfo& r, int j) {
  if (j >= r.nlist) return -1;
  int64_t s = p.kv_start ? r.base + j
              : (p.draft_slots && j >= r.P) ? int64_t(p.draft_slots[r.dbase + j])
                                             : int64_t(p.slot_idx[r.base + j]);
  return (s >= 0 && s < p.num_slots) ? s : -1;
}

// Is key j visible to draft node i of request b?  (prefix: always; draft key
// k = j - P: when bit k of node i's ancestor-or-self mask is set.)
__device__ inline bool key_visible(const Params& p, const ReqInfo& r, int b, int i, int j) {
  if (j < r.P) return true;
  int k = j - r.P;
  if (k >= p.T) return false;
  return (p.bits[size_t(b) * p.T + i] >> k) & 1ull;
}

__device__ inline float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ inline float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ inline uint32_t smem_u32(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

// Event tracing for pipeline analysis.  Compiled out unless VA_TRACE is
// defined; a traced build records %globaltimer per (role, event, tile) for the
// first cluster of the grid into the device buffer `g_va_trace`, which the
// translation unit that uses the macro defines.
// Programmatic dependent launch.  The kernels of a step run back to back on
// one stream; a kernel launched with programmatic stream serialization may
// start while its predecessor still runs, and griddep_wait() holds the calling
// thread until the predecessor has completed and its writes are visible (for a
// kernel launched the ordinary way it returns at once).  A kernel calls
// griddep_launch_dependents() to let its successor start early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

#ifdef VA_TRACE
// Trace build only.  The buffer g_va_trace holds 18 roles x 8 slots x 512
// entries; only the grid's first (row unit, request) column is traced:
//   roles 0-4   per-tile events of cluster 0: key producers, QK products,
//               softmax, value producers, PV products (the first CTA of each
//               role: cluster ranks 0 and 1, or 0 and 2 in a pair);
//   role 5      write-out marks; roles 6-7 and 16-17 per-CTA marks by
//               cluster rank (0-1, 2-3);
//   roles 8-12  phase clock sums per cluster: softmax, QK products, PV
//               products, key producers, value producers (13-15: softmax
//               and producers of a pair's odd ranks).
__device__ __forceinline__ unsigned va_trace_cluster() {
  unsigned n;
  asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return blockIdx.x / n;
}
__device__ __forceinline__ bool va_trace_first_of_role() {
  unsigned r, n;
  asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  asm("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return r == 0 || 2 * r == n;
}
#ifdef VA_TRACE_NO_EVENTS
#define VA_TRACE_EVENT(role, ev, t) ((void)0)
#else
#define VA_TRACE_EVENT(role, ev, t)                                                        \
  do {                                                                                     \
    if (g_va_trace && blockIdx.y == 0 && blockIdx.z == 0 && va_trace_cluster() == 0 &&       \
        va_trace_first_of_role() && (t) < 512) {                                           \
      unsigned long long _ts;                                                              \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(_ts));                               \
      g_va_trace[((role) * 8 + (ev)) * 512 + (t)] = _ts;                                   \
    }                                                                                      \
  } while (0)
#endif
// Per-cluster marks of the partial kernel: slot (role, ev, cluster index).
#define VA_TRACE_CTA(role, ev)                                                             \
  do {                                                                                     \
    if (g_va_trace && blockIdx.y == 0 && blockIdx.z == 0 && va_trace_cluster() < 512) {     \
      unsigned long long _ts;                                                              \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(_ts));                               \
      g_va_trace[((role) * 8 + (ev)) * 512 + va_trace_cluster()] = _ts;                    \
    }                                                                                      \
  } while (0)
// Phase clocks: a role accumulates clock64 deltas per phase over all tiles
// in registers and stores the sums once.
#define VA_PH_DECL long long _ph[8] = {0, 0, 0, 0, 0, 0, 0, 0}; long long _pt = clock64()
#define VA_PH(i)                                                                           \
  do {                                                                                     \
    const long long _n = clock64();                                                        \
    _ph[i] += _n - _pt;                                                                    \
    _pt = _n;                                                                              \
  } while (0)
#define VA_PH_STORE(role)                                                                  \
  do {                                                                                     \
    if (g_va_trace && blockIdx.y == 0 && blockIdx.z == 0 && va_trace_cluster() < 512)       \
      for (int _i = 0; _i < 8; ++_i)                                                       \
        g_va_trace[((role) * 8 + _i) * 512 + va_trace_cluster()] = (unsigned long long)_ph[_i]; \
  } while (0)
#else
#define VA_TRACE_EVENT(role, ev, t) ((void)0)
#define VA_TRACE_CTA(role, ev) ((void)0)
#define VA_PH_DECL ((void)0)
#define VA_PH(i) ((void)0)
#define VA_PH_STORE(role) ((void)0)
#endif

// Launchers (defined in the kernel translation units).
cudaError_t launch_tree_bits(const Params& p, uint64_t* bits_out, cudaStream_t st);
cudaError_t launch_partial_fma(const Params& p, int num_sms, cudaStream_t st);
cudaError_t launch_combine(const Params& p, cudaStream_t st);
cudaError_t launch_defrag(void* pool, int64_t num_slots, int64_t stride, const int32_t* src,
                          const int32_t* indptr, const int64_t* dst_base, int32_t* slots_out,
                          int B, int64_t max_rows, uint32_t* status, cudaStream_t st);

// Rows handled by one CTA of the FMA partial kernel.
constexpr int kFmaRows = 16;

}  // namespace va
