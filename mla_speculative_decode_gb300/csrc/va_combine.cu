// va_combine.cu -- LSE-merge of split partials (K2) and KV defragmentation.
//
// Merge (The Milestone Commit, "The Deeper Significance": the reduction
// kernel; The Commit That Locked In 6x Decode, "Input Knowledge Required":
// NSPLIT partial-reduce).  Split s of a row holds a normalised partial output
// o_s and lse_s over its keys; the row's result is
//     lse = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) o_s
// with a max shift, splits at -inf skipped and a row with no key at all
// producing out = 0, lse = -inf.  The split order is fixed, so the result is
// deterministic.  A CTA of 128 threads merges one row, 4 columns per thread.
//
// Defragmentation (The Checkpoint Report, "Input Knowledge Required": keep
// each request's KV contiguous).  A warp copies whole rows with 16-byte
// loads and stores; every source and destination row is range-checked.
#include <math.h>

#include "va_common.cuh"

namespace va {
namespace {

constexpr int kCombineThreads = kDv / 4;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(Params p) {
  const int rows_total = p.B * p.rows_per_req;
  const int tid = threadIdx.x;
  for (int row = blockIdx.x; row < rows_total; row += gridDim.x) {
    const int b = row / p.rows_per_req;
    const ReqInfo ri = req_info(p, b, false);
    const int ne = split_range(ri.N, p.nsplit, 0).nsplit_eff;
    const float* pl = p.part_lse + row;
    float m = -INFINITY;
    for (int s = 0; s < ne; ++s) m = fmaxf(m, pl[size_t(s) * rows_total]);
    float L = -INFINITY;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (m != -INFINITY) {
      float z = 0.f;
      for (int s = 0; s < ne; ++s) {
        const float ls = pl[size_t(s) * rows_total];
        if (ls != -INFINITY) z += expf(ls - m);
      }
      L = m + logf(z);
      for (int s = 0; s < ne; ++s) {
        const float ls = pl[size_t(s) * rows_total];
        if (ls == -INFINITY) continue;
        const float w = expf(ls - L);
        const float4 o = *reinterpret_cast<const float4*>(
            p.part_o + ((size_t)s * rows_total + row) * kDv + tid * 4);
        acc.x = fmaf(w, o.x, acc.x);
        acc.y = fmaf(w, o.y, acc.y);
        acc.z = fmaf(w, o.z, acc.z);
        acc.w = fmaf(w, o.w, acc.w);
      }
    }
    uint2 packed;
    packed.x = uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(acc.x))) |
               (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(acc.y))) << 16);
    packed.y = uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(acc.z))) |
               (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(acc.w))) << 16);
    *reinterpret_cast<uint2*>(p.out + size_t(row) * kDv + tid * 4) = packed;
    if (tid == 0) p.lse[row] = L;
  }
}

constexpr int kDefragThreads = 256;

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
  for (int64_t i = warp; i < n; i += nwarps) {
    int64_t s = 0;
    if (lane == 0) s = src[i0 + i];
    s = __shfl_sync(0xffffffffu, s, 0);
    const int64_t d = dbase + i;
    const bool s_ok = s >= 0 && s < num_slots;
    const bool d_ok = d >= 0 && d < num_slots;
    if (!s_ok || !d_ok) {
      if (lane == 0 && status)
        atomicOr(status, (s_ok ? 0u : VA_STATUS_BAD_SLOT) | (d_ok ? 0u : VA_STATUS_BAD_DST));
      continue;
    }
    const uint4* from = pool + s * vec_per_row;
    uint4* to = pool + d * vec_per_row;
    for (int64_t c = lane; c < vec_per_row; c += 32) to[c] = from[c];
    if (lane == 0 && slots_out) slots_out[i0 + i] = int32_t(d);
  }
}

}  // namespace

cudaError_t launch_combine(const Params& p, cudaStream_t st) {
  const int rows_total = p.B * p.rows_per_req;
  const int grid = rows_total < 65535 ? rows_total : 65535;
  combine_kernel<<<grid, kCombineThreads, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_defrag(void* pool, int64_t num_slots, int64_t stride, const int32_t* src,
                          const int32_t* indptr, const int64_t* dst_base, int32_t* slots_out,
                          int B, int64_t max_rows, uint32_t* status, cudaStream_t st) {
  const int64_t per_req = (max_rows + B - 1) / B;
  int64_t blocks = (per_req + 4 * (kDefragThreads / 32) - 1) / (4 * (kDefragThreads / 32));
  if (blocks < 1) blocks = 1;
  if (blocks > 65535) blocks = 65535;
  dim3 grid{unsigned(blocks), unsigned(B), 1u};
  defrag_kernel<<<grid, kDefragThreads, 0, st>>>(reinterpret_cast<uint4*>(pool), num_slots,
                                                 stride / 8, src, indptr, dst_base, slots_out,
                                                 status);
  return cudaGetLastError();
}

}  // namespace va
