// va_place.cu -- contiguous placement of draft latents and compaction of the
// accepted path (the defragmentation policy the pages defer: The Checkpoint
// Report, "Input Knowledge Required": defragmentation keeps per-request KV
// contiguous; "The Architecture of the Report": the deferred phase).
//
// A request owns a reserved range of pool rows [kv_start, kv_start +
// capacity).  Before verify, its T draft latents are written right after its
// prefix, so verify_attn_contiguous reads prefix and draft keys as one run of
// rows (TMA boxes); after acceptance, the accepted path's rows are moved to
// directly after the prefix, which grows by the accepted count -- the request
// stays contiguous from step to step and never needs a separate
// defragmentation pass.
#include <string.h>

#include "va_common.cuh"

#ifndef VA_API
#define VA_API extern "C" __attribute__((visibility("default")))
#endif

namespace va {
namespace {

constexpr int kPlaceWarps = 8;
constexpr int kRowChunks = kDqk / 8;   // 16-byte chunks of a 576-column row

struct PlaceParams {
  __nv_bfloat16* pool;
  int64_t num_slots;
  int64_t stride;              // elements
  const int64_t* kv_start;
  int32_t* prefix_len;         // read by the append; read and advanced by the compaction
  const int32_t* capacity;
  const __nv_bfloat16* draft;  // [B*T, 576]
  const int32_t* accept_len;
  const int32_t* accept_nodes;
  int32_t* out_cache_loc;
  uint32_t* status;
  int B, T;
};

// Row of draft node i of request b, or -1 when the request's reserved range
// cannot hold its prefix and draft, or the row falls outside the pool.
__device__ __forceinline__ int64_t draft_row(const PlaceParams& p, int b, int i) {
  const int64_t P = p.prefix_len[b];
  if (P < 0 || P + p.T > int64_t(p.capacity[b])) return -1;
  const int64_t row = p.kv_start[b] + P + i;
  return (row >= 0 && row < p.num_slots && row <= 0x7fffffff) ? row : -1;
}

// One warp per draft row: row b*T + i of the draft latents into the first
// 576 columns of the request's row kv_start[b] + prefix_len[b] + i.
__global__ void __launch_bounds__(kPlaceWarps * 32) append_contiguous_kernel(PlaceParams p) {
  griddep_wait();                // the stream's previous kernel has completed
  griddep_launch_dependents();   // the next kernel may start its set-up
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kPlaceWarps + (threadIdx.x >> 5);
  if (r >= p.B * p.T) return;
  const int b = r / p.T, i = r - b * p.T;
  const int64_t row = draft_row(p, b, i);
  if (lane == 0) {
    if (p.out_cache_loc) p.out_cache_loc[r] = row >= 0 ? int32_t(row) : -1;
    if (row < 0 && p.status) atomicOr(p.status, VA_STATUS_BAD_DST);
  }
  if (row < 0) return;
  const uint4* src = reinterpret_cast<const uint4*>(p.draft + size_t(r) * kDqk);
  uint4* dst = reinterpret_cast<uint4*>(p.pool + row * p.stride);
  for (int c = lane; c < kRowChunks; c += 32) dst[c] = src[c];
}

// One CTA per request: the k-th accepted node's row (kv_start + P + node)
// moves to kv_start + P + k, every row read into shared memory before any is
// written (a path may list its nodes in any order), then prefix_len += n.  A
// request whose accept count, nodes or rows are out of range is left as it is
// and flagged.  Thread k checks node k, all at once.
__global__ void __launch_bounds__(kPlaceWarps * 32) compact_accepted_kernel(PlaceParams p) {
  extern __shared__ __align__(16) uint4 stage[];   // [T][72]
  __shared__ int s_node[VA_T_MAX];
  griddep_wait();                // the stream's previous kernel has completed
  griddep_launch_dependents();   // the next kernel may start its set-up
  const int b = blockIdx.x, tid = threadIdx.x;
  const int T = p.T;
  const int n = p.accept_len[b];
  const int64_t P = p.prefix_len[b];
  const int64_t base = p.kv_start[b] + P;
  const bool req_ok = n >= 0 && n <= T && P >= 0 && P + T <= int64_t(p.capacity[b]) &&
                      base >= 0 && base + T <= p.num_slots;
  bool ok = true;
  if (req_ok && tid < n) {
    const int node = p.accept_nodes[size_t(b) * T + tid];
    ok = node >= 0 && node < T;
    s_node[tid] = node;
  }
  if (!__syncthreads_and(req_ok && ok)) {
    if (tid == 0 && p.status) atomicOr(p.status, VA_STATUS_BAD_DST);
    return;
  }
  for (int e = tid; e < n * kRowChunks; e += blockDim.x) {
    const int k = e / kRowChunks, c = e - k * kRowChunks;
    stage[e] = reinterpret_cast<const uint4*>(p.pool + (base + s_node[k]) * p.stride)[c];
  }
  __syncthreads();
  for (int e = tid; e < n * kRowChunks; e += blockDim.x) {
    const int k = e / kRowChunks, c = e - k * kRowChunks;
    reinterpret_cast<uint4*>(p.pool + (base + k) * p.stride)[c] = stage[e];
  }
  if (tid == 0) p.prefix_len[b] = int32_t(P + n);
}

bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

// A programmatic dependent of the stream's previous kernel: the CTAs may
// become resident while it finishes; each waits for it (griddepcontrol.wait)
// before reading anything.
int launch_dependent(void (*kernel)(PlaceParams), dim3 grid, int smem, va_stream_t stream,
                     const PlaceParams& p) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kPlaceWarps * 32, 1u, 1u);
  cfg.dynamicSmemBytes = size_t(smem);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p) == cudaSuccess ? VA_OK : VA_ERR_LAUNCH;
}

int check_common(const void* pool, int64_t num_slots, int64_t stride, const int64_t* kv_start,
                 const int32_t* prefix_len, const int32_t* capacity, int B, int T,
                 const uint32_t* status) {
  if (!pool || !kv_start || !prefix_len || !capacity) return VA_ERR_NULL;
  if (B < 1 || B > 65535 || T < 1 || T > VA_T_MAX || num_slots < 1 || stride < VA_D_QK)
    return VA_ERR_SHAPE;
  if (stride % 8 != 0) return VA_ERR_ALIGN;
  if (!aligned(pool, 16) || !aligned(kv_start, 8) || !aligned(prefix_len, 4) ||
      !aligned(capacity, 4) || (status && !aligned(status, 4)))
    return VA_ERR_ALIGN;
  return VA_OK;
}

}  // namespace
}  // namespace va

VA_API int va_kv_append_contiguous(void* kv_pool, int64_t num_slots, int64_t kv_row_stride,
                                   const int64_t* kv_start, const int32_t* prefix_len,
                                   const int32_t* kv_capacity, const void* draft_kv, int B,
                                   int T, int32_t* out_cache_loc, uint32_t* status,
                                   va_stream_t stream) {
  using namespace va;
  int rc = check_common(kv_pool, num_slots, kv_row_stride, kv_start, prefix_len, kv_capacity, B,
                        T, status);
  if (rc != VA_OK) return rc;
  if (!draft_kv) return VA_ERR_NULL;
  if (!aligned(draft_kv, 16) || (out_cache_loc && !aligned(out_cache_loc, 4))) return VA_ERR_ALIGN;
  PlaceParams p;
  memset(&p, 0, sizeof p);
  p.pool = static_cast<__nv_bfloat16*>(kv_pool);
  p.num_slots = num_slots;
  p.stride = kv_row_stride;
  p.kv_start = kv_start;
  p.prefix_len = const_cast<int32_t*>(prefix_len);
  p.capacity = kv_capacity;
  p.draft = static_cast<const __nv_bfloat16*>(draft_kv);
  p.out_cache_loc = out_cache_loc;
  p.status = status;
  p.B = B;
  p.T = T;
  const int rows = B * T;
  return launch_dependent(append_contiguous_kernel, dim3(unsigned((rows + kPlaceWarps - 1) / kPlaceWarps)),
                          0, stream, p);
}

VA_API int va_kv_compact_accepted(void* kv_pool, int64_t num_slots, int64_t kv_row_stride,
                                  const int64_t* kv_start, int32_t* prefix_len,
                                  const int32_t* kv_capacity, const int32_t* accept_len,
                                  const int32_t* accept_nodes, int B, int T, uint32_t* status,
                                  va_stream_t stream) {
  using namespace va;
  int rc = check_common(kv_pool, num_slots, kv_row_stride, kv_start, prefix_len, kv_capacity, B,
                        T, status);
  if (rc != VA_OK) return rc;
  if (!accept_len || !accept_nodes) return VA_ERR_NULL;
  if (!aligned(accept_len, 4) || !aligned(accept_nodes, 4)) return VA_ERR_ALIGN;
  const int smem = T * kRowChunks * 16;   // <= 64 rows x 1152 bytes
  if (cudaFuncSetAttribute(compact_accepted_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return VA_ERR_CUDA;
  PlaceParams p;
  memset(&p, 0, sizeof p);
  p.pool = static_cast<__nv_bfloat16*>(kv_pool);
  p.num_slots = num_slots;
  p.stride = kv_row_stride;
  p.kv_start = kv_start;
  p.prefix_len = prefix_len;
  p.capacity = kv_capacity;
  p.accept_len = accept_len;
  p.accept_nodes = accept_nodes;
  p.status = status;
  p.B = B;
  p.T = T;
  return launch_dependent(compact_accepted_kernel, dim3(unsigned(B)), smem, stream, p);
}
