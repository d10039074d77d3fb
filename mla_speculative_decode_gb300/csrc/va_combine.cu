// va_combine.cu -- LSE-merge of split partials (K2) and KV defragmentation.
//
// Merge (The Milestone Commit, "The Deeper Significance": the reduction
// kernel; The Commit That Locked In 6x Decode, "Input Knowledge Required":
// NSPLIT partial-reduce).  Split s of a row holds a normalised partial output
// o_s and lse_s over its keys; the row's result is
//     lse = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) o_s
// with a max shift, splits at -inf skipped and a row with no key at all
// producing out = 0, lse = -inf.  The split order is fixed, so the result is
// deterministic.
//
// Defragmentation (The Checkpoint Report, "Input Knowledge Required": keep
// each request's KV contiguous).  A warp copies whole rows with 16-byte
// loads and stores; every source and destination row is range-checked.
#include <math.h>
#include <string.h>

#include "va_common.cuh"

namespace va {
namespace {

constexpr int kCombineThreads = 256;   // 8 warps
constexpr int kCombineCols = 128;      // value columns per CTA (a float4 per lane)
constexpr int kMaxSplits = VA_NSPLIT_MAX;

__device__ __forceinline__ float block_reduce(float v, float* red, bool is_max) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, w) : v + w;
  }
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int i = 1; i < kCombineThreads / 32; ++i) r = is_max ? fmaxf(r, red[i]) : r + red[i];
  __syncthreads();
  return r;
}

// Grid (row, 128-column chunk).  Each warp first issues the loads of its
// share of the splits' partial outputs for the chunk (a float4 per lane, up to
// kBuf splits per warp in flight) -- they do not depend on the weights, so
// their round trip to memory overlaps the one of the lse values.  The split
// weights exp(lse_s - lse) are formed once per CTA in shared memory; each warp
// then sums its splits and the eight partial sums are added.  Only the
// request's effective splits are loaded: slots past them were not written by
// this call (they may hold an earlier call's data) and are never read.
constexpr int kBuf = 10;   // splits per warp per round (80 per CTA)

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

// The call's status word on the tensor-core path: the OR of the status words
// of every split-K CTA of the grid (a CTA past its request's splits stores
// 0), loaded by a whole block, four independent loads in flight per thread.
__device__ __forceinline__ uint32_t cta_flags_or(const Params& p, int tid, int nthreads) {
  const size_t n = size_t(p.B) * p.flag_blocks * p.nsplit * 2;
  const size_t step = size_t(nthreads);
  uint32_t v = 0u;
  size_t i = size_t(tid);
  for (; i + 3 * step < n; i += 4 * step)
    v |= p.cta_flags[i] | p.cta_flags[i + step] | p.cta_flags[i + 2 * step] |
         p.cta_flags[i + 3 * step];
  for (; i < n; i += step) v |= p.cta_flags[i];
  return v;
}

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(Params p) {
  __shared__ float wsplit[kMaxSplits];
  __shared__ float red[kCombineThreads / 32];
  __shared__ float4 part[kCombineThreads / 32][kCombineCols / 4];
  const int rows_total = p.B * p.rows_per_req;
  const int row = blockIdx.x, chunk = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = row / p.rows_per_req;
  constexpr int kWarps = kCombineThreads / 32;
  // The request's split count comes from its bounds, which are inputs of the
  // call rather than results of the split-K kernel (this kernel is scheduled
  // only once every split-K CTA has passed its own wait for the stream's
  // earlier work), so they are read before the wait; only the splits that ran
  // are loaded below.
  const ReqInfo ri = req_info(p, b, false);
  const int ne = split_range(ri.N, p.nsplit, 0).nsplit_eff;
  griddep_wait();   // the split-K kernel's partials are complete and visible
  // the stream's next kernel, when launched as a programmatic dependent (the
  // next call's split-K kernel), may start its set-up now; it waits for
  // this kernel's completion before reading anything
  griddep_launch_dependents();
  const __nv_bfloat16* po = p.part_o + size_t(row) * kDv + chunk * kCombineCols + lane * 4;
  const size_t sstride = size_t(rows_total) * kDv;

  // first round of partial-output loads (splits warp, warp + 8, ...)
  uint2 buf[kBuf];   // four bf16 partial values per lane
#pragma unroll
  for (int i = 0; i < kBuf; ++i) {
    const int s = warp + kWarps * i;
    buf[i] = s < ne ? *reinterpret_cast<const uint2*>(po + size_t(s) * sstride)
                    : make_uint2(0u, 0u);
  }

  const float* pl = p.part_lse + row;
  float m = -INFINITY;
  for (int s = tid; s < ne; s += kCombineThreads) {
    const float ls = pl[size_t(s) * rows_total];
    wsplit[s] = ls;
    m = fmaxf(m, ls);
  }
  m = block_reduce(m, red, true);
  float z = 0.f;
  if (m != -INFINITY)
    for (int s = tid; s < ne; s += kCombineThreads)
      if (wsplit[s] != -INFINITY) z += expf(wsplit[s] - m);
  z = block_reduce(z, red, false);
  const float L = m == -INFINITY ? -INFINITY : m + logf(z);
  for (int s = tid; s < ne; s += kCombineThreads)
    wsplit[s] = (L == -INFINITY || wsplit[s] == -INFINITY) ? 0.f : expf(wsplit[s] - L);
  __syncthreads();

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int base = 0; base < ne; base += kWarps * kBuf) {
    if (base > 0) {
#pragma unroll
      for (int i = 0; i < kBuf; ++i) {
        const int s = base + warp + kWarps * i;
        buf[i] = s < ne ? *reinterpret_cast<const uint2*>(po + size_t(s) * sstride)
                        : make_uint2(0u, 0u);
      }
    }
#pragma unroll
    for (int i = 0; i < kBuf; ++i) {
      const int s = base + warp + kWarps * i;
      if (s < ne) {
        const float w = wsplit[s];
        const float2 lo = bf16x2_to_float2(buf[i].x), hi = bf16x2_to_float2(buf[i].y);
        acc.x = fmaf(w, lo.x, acc.x);
        acc.y = fmaf(w, lo.y, acc.y);
        acc.z = fmaf(w, hi.x, acc.z);
        acc.w = fmaf(w, hi.y, acc.w);
      }
    }
  }
  part[warp][lane] = acc;
  __syncthreads();
  if (warp == 0) {
    float4 t = part[0][lane];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) {
      const float4 u = part[w][lane];
      t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
    }
    uint2 packed;
    packed.x = uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(t.x))) |
               (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(t.y))) << 16);
    packed.y = uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(t.z))) |
               (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(t.w))) << 16);
    *reinterpret_cast<uint2*>(p.out + size_t(row) * kDv + chunk * kCombineCols + lane * 4) = packed;
    if (chunk == 0 && lane == 0) p.lse[row] = L;
  }
  if (p.cta_flags && row == 0 && chunk == 0) {
    __shared__ uint32_t acc;
    if (tid == 0) acc = 0u;
    __syncthreads();
    const uint32_t v = cta_flags_or(p, tid, kCombineThreads);
    if (v) atomicOr(&acc, v);
    __syncthreads();
    if (tid == 0) *p.status = acc;
  }
}

// Merge for few splits and many rows (nsplit <= kRowSplits, e.g. a batch of
// requests at full H): one warp per (row, 32*kVec-column chunk), no shared
// memory and no block-wide reductions.  Lane j < nsplit_eff holds split j's
// lse; the warp forms the maximum, the sum and the weights with shuffles;
// every lane loads its kVec columns of every split up front (while the
// weights are formed) and sums them.  The launch sizes the split buffer to
// the split count: up to 8 splits, 16-byte lanes (kVec = 8); 9 to 16, 8-byte
// lanes (kVec = 4), so that the buffer stays small enough for the warps that
// keep the loads in flight.  Same arithmetic as combine_kernel (the split
// order is fixed, so the result is deterministic).
constexpr int kRowSplits = 16;
constexpr int kRowWarps = 8;    // warps per CTA

template <int kVec>
struct RowVec;
template <>
struct RowVec<8> {
  using T = uint4;
  __device__ static uint32_t word(const uint4& v, int k) {
    return k == 0 ? v.x : k == 1 ? v.y : k == 2 ? v.z : v.w;
  }
  __device__ static uint4 zero() { return make_uint4(0u, 0u, 0u, 0u); }
  __device__ static uint4 make(const uint32_t* w) { return make_uint4(w[0], w[1], w[2], w[3]); }
};
template <>
struct RowVec<4> {
  using T = uint2;
  __device__ static uint32_t word(const uint2& v, int k) { return k == 0 ? v.x : v.y; }
  __device__ static uint2 zero() { return make_uint2(0u, 0u); }
  __device__ static uint2 make(const uint32_t* w) { return make_uint2(w[0], w[1]); }
};

template <int kMax, int kVec>
__global__ void __launch_bounds__(kRowWarps * 32) combine_rows_kernel(Params p) {
  using V = RowVec<kVec>;
  constexpr int kChunks = kDv / (32 * kVec);   // warps per row
  const int rows_total = p.B * p.rows_per_req;
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  const int row = item / kChunks, chunk = item % kChunks;
  const bool live = row < rows_total;
  const int b = live ? row / p.rows_per_req : 0;
  // the request's split count from its bounds (inputs of the call, not
  // results of the split-K kernel), before the wait
  const int ne = live ? split_range(req_info(p, b, false).N, p.nsplit, 0).nsplit_eff : 0;
  griddep_wait();   // the split-K kernel's partials are complete and visible
  // the stream's next kernel, when launched as a programmatic dependent (the
  // next call's split-K kernel), may start its set-up now; it waits for
  // this kernel's completion before reading anything
  griddep_launch_dependents();
  if (live) {
    const size_t col = size_t(chunk) * (32 * kVec) + size_t(lane) * kVec;
    const __nv_bfloat16* po = p.part_o + size_t(row) * kDv + col;
    const size_t sstride = size_t(rows_total) * kDv;
    typename V::T buf[kMax];
#pragma unroll
    for (int s = 0; s < kMax; ++s)
      buf[s] = s < ne ? *reinterpret_cast<const typename V::T*>(po + size_t(s) * sstride) : V::zero();
    const float ls = lane < ne ? p.part_lse[size_t(lane) * rows_total + row] : -INFINITY;
    float m = ls;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = (m == -INFINITY || ls == -INFINITY) ? 0.f : expf(ls - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const float L = m == -INFINITY ? -INFINITY : m + logf(z);
    const float w = (L == -INFINITY || ls == -INFINITY) ? 0.f : expf(ls - L);
    float acc[kVec];
#pragma unroll
    for (int k = 0; k < kVec; ++k) acc[k] = 0.f;
#pragma unroll
    for (int s = 0; s < kMax; ++s) {
      const float ws = __shfl_sync(0xffffffffu, w, s);
      if (s < ne) {
#pragma unroll
        for (int k = 0; k < kVec / 2; ++k) {
          const float2 f = bf16x2_to_float2(V::word(buf[s], k));
          acc[2 * k] = fmaf(ws, f.x, acc[2 * k]);
          acc[2 * k + 1] = fmaf(ws, f.y, acc[2 * k + 1]);
        }
      }
    }
    uint32_t pk[kVec / 2];
#pragma unroll
    for (int k = 0; k < kVec / 2; ++k)
      pk[k] = uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * k]))) |
              (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * k + 1]))) << 16);
    *reinterpret_cast<typename V::T*>(p.out + size_t(row) * kDv + col) = V::make(pk);
    if (chunk == 0 && lane == 0) p.lse[row] = L;
  }
  if (p.cta_flags && blockIdx.x == 0) {
    __shared__ uint32_t acc_flags;
    if (threadIdx.x == 0) acc_flags = 0u;
    __syncthreads();
    uint32_t v = cta_flags_or(p, threadIdx.x, kRowWarps * 32);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0 && v) atomicOr(&acc_flags, v);
    __syncthreads();
    if (threadIdx.x == 0) *p.status = acc_flags;
  }
}

constexpr int kDefragThreads = 256;

// A warp moves four rows per round: the four source slots arrive with one
// load, then every chunk of the four rows is loaded before any is stored, so
// a round pays the memory latency about twice rather than twice per row.
constexpr int kDefragRows = 4;

__global__ void __launch_bounds__(kDefragThreads)
    defrag_kernel(uint4* pool, int64_t num_slots, int64_t vec_per_row, const int32_t* src,
                  const int32_t* indptr, const int64_t* dst_base, int32_t* slots_out,
                  uint32_t* status) {
  const int b = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int64_t warp = int64_t(blockIdx.x) * (kDefragThreads / 32) + (threadIdx.x >> 5);
  const int64_t nwarps = int64_t(gridDim.x) * (kDefragThreads / 32);
  const int64_t i0 = indptr[b], n = int64_t(indptr[b + 1]) - i0;
  const int64_t dbase = dst_base[b];
  for (int64_t r0 = warp * kDefragRows; r0 < n; r0 += nwarps * kDefragRows) {
    const int64_t s_lane = (lane < kDefragRows && r0 + lane < n) ? int64_t(src[i0 + r0 + lane]) : 0;
    bool ok[kDefragRows];
    int64_t sr[kDefragRows];
#pragma unroll
    for (int k = 0; k < kDefragRows; ++k) {
      const int64_t i = r0 + k;
      const int64_t s = __shfl_sync(0xffffffffu, s_lane, k);
      const int64_t d = dbase + i;
      const bool s_ok = s >= 0 && s < num_slots;
      const bool d_ok = d >= 0 && d < num_slots;
      sr[k] = s;
      ok[k] = i < n && s_ok && d_ok;
      if (i < n && !(s_ok && d_ok) && lane == 0 && status)
        atomicOr(status, (s_ok ? 0u : VA_STATUS_BAD_SLOT) | (d_ok ? 0u : VA_STATUS_BAD_DST));
    }
    if (vec_per_row <= 96) {
      uint4 v[kDefragRows][3];
#pragma unroll
      for (int k = 0; k < kDefragRows; ++k)
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          const int64_t c = lane + 32 * j;
          if (ok[k] && c < vec_per_row) v[k][j] = pool[sr[k] * vec_per_row + c];
        }
#pragma unroll
      for (int k = 0; k < kDefragRows; ++k)
#pragma unroll
        for (int j = 0; j < 3; ++j) {
          const int64_t c = lane + 32 * j;
          if (ok[k] && c < vec_per_row) pool[(dbase + r0 + k) * vec_per_row + c] = v[k][j];
        }
    } else {
      for (int k = 0; k < kDefragRows; ++k) {
        if (!ok[k]) continue;
        const uint4* from = pool + sr[k] * vec_per_row;
        uint4* to = pool + (dbase + r0 + k) * vec_per_row;
        for (int64_t c = lane; c < vec_per_row; c += 32) to[c] = from[c];
      }
    }
    if (lane < kDefragRows && r0 + lane < n && slots_out) {
      bool okl = false;
#pragma unroll
      for (int k = 0; k < kDefragRows; ++k)
        if (k == lane) okl = ok[k];
      if (okl) slots_out[i0 + r0 + lane] = int32_t(dbase + r0 + lane);
    }
  }
}

}  // namespace

cudaError_t launch_combine(const Params& p, cudaStream_t st) {
  const int rows_total = p.B * p.rows_per_req;
  const bool by_rows = p.nsplit <= kRowSplits;
  const int row_vec = p.nsplit <= 8 ? 8 : 4;   // columns per lane of the warp-per-row merge
  dim3 grid = by_rows ? dim3(unsigned((rows_total * (kDv / (32 * row_vec)) + kRowWarps - 1) / kRowWarps),
                             1u, 1u)
                      : dim3(unsigned(rows_total), unsigned(kDv / kCombineCols), 1u);
  // launched with programmatic stream serialization: its blocks may be
  // scheduled as the split-K kernel's clusters retire and wait in-kernel
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = grid;
  cfg.blockDim = dim3(by_rows ? kRowWarps * 32 : kCombineThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!by_rows) return cudaLaunchKernelEx(&cfg, combine_kernel, p);
  if (p.nsplit <= 4) return cudaLaunchKernelEx(&cfg, combine_rows_kernel<4, 8>, p);
  if (p.nsplit <= 8) return cudaLaunchKernelEx(&cfg, combine_rows_kernel<8, 8>, p);
  return cudaLaunchKernelEx(&cfg, combine_rows_kernel<kRowSplits, 4>, p);
}

cudaError_t launch_defrag(void* pool, int64_t num_slots, int64_t stride, const int32_t* src,
                          const int32_t* indptr, const int64_t* dst_base, int32_t* slots_out,
                          int B, int64_t max_rows, uint32_t* status, cudaStream_t st) {
  const int64_t per_req = (max_rows + B - 1) / B;
  int64_t blocks = (per_req + kDefragRows * (kDefragThreads / 32) - 1) /
                   (kDefragRows * (kDefragThreads / 32));
  if (blocks < 1) blocks = 1;
  if (blocks > 65535) blocks = 65535;
  dim3 grid{unsigned(blocks), unsigned(B), 1u};
  defrag_kernel<<<grid, kDefragThreads, 0, st>>>(reinterpret_cast<uint4*>(pool), num_slots,
                                                 stride / 8, src, indptr, dst_base, slots_out,
                                                 status);
  return cudaGetLastError();
}

}  // namespace va
