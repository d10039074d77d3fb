// va_fma.cu -- split-K partial kernel on CUDA cores (K1, FMA path).
//
// Design after the pages' own kernel (The Milestone Commit, "The Thinking
// Process Revealed": split-K over the KV range, warp-per-key scoring, online
// softmax; The Commit That Locked In 6x Decode, "3. Vectorized bf16 Loads":
// 128-bit gathers of 8 bf16 per thread), kept for row blocks too small for a
// tensor-core tile and as a second, independent device implementation.
//
// Grid (split, row block of 16 rows, request).  Per CTA, 256 threads:
//   - the 16 query rows are staged once as fp32 in shared memory;
//   - 32-key tiles are gathered with 16-byte cp.async (zero-filled for keys
//     without a valid slot), double buffered;
//   - scores: each warp takes 4 keys; a lane owns 16-24 of the 576 columns,
//     forms partial dot products for 16 rows x 4 keys and the warp sums the 64
//     partials with a halving butterfly (62 shuffles, not 5 x 64);
//   - online softmax in the log2 domain: a warp per row, a lane per key;
//   - PV: a thread owns two value columns for all 16 rows (32 fp32
//     accumulators), probabilities read as broadcast float4s;
//   - the split's normalised partial output and its lse go to the workspace.
#include <math.h>

#include "va_common.cuh"

namespace va {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRB = kFmaRows;          // rows per CTA
constexpr int kKT = 32;                // keys per tile
constexpr int kChunks = kDqk / 8;      // 16-byte chunks per key row (72)
constexpr int kHalf = kDqk / 2;        // 288
static_assert(kKT == kWarps * 4, "4 keys per warp");
static_assert(kRB * 4 == 64, "butterfly sized for 64 partials");
static_assert(kThreads * 2 == kDv, "two value columns per thread");

struct __align__(16) FmaSmem {
  // q[r][h*288 + c*4 + e]: the 8 values of 16-byte chunk c are split in two
  // float4 halves so that a warp's float4 loads are conflict free.
  float q[kRB * kDqk];
  __nv_bfloat16 k[2][kKT * kDqk];
  float pt[kKT][kRB];                  // raw dots, then probabilities (key-major)
  float alpha[kRB];
  float m[kRB];
  float l[kRB];
  int valid[2][kKT];
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
  f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
  f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
  f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

__global__ void __launch_bounds__(kThreads) partial_fma_kernel(Params p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  FmaSmem& S = *reinterpret_cast<FmaSmem*>(smem_raw);
  const int split = blockIdx.x, rb = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const ReqInfo ri = req_info(p, b, split == 0 && rb == 0);
  const SplitRange sr = split_range(ri.N, p.nsplit, split);
  if (split >= sr.nsplit_eff) return;
  const int R = p.rows_per_req;
  const int row0 = rb * kRB;
  if (row0 >= R) return;
  const size_t rows_total = size_t(p.B) * R;
  const size_t grow0 = size_t(b) * R + row0;

  // ---- gather one tile of keys [tk0, tk0 + 32) into buffer `buf`
  auto load_tile = [&](int tk0, int buf) {
    for (int idx = tid; idx < kKT * kChunks; idx += kThreads) {
      const int key = idx / kChunks, c = idx - key * kChunks;
      const int j = tk0 + key;
      const int64_t row = j < sr.k1 ? key_row(p, ri, j) : -1;
      const __nv_bfloat16* src = row >= 0 ? p.kv + row * p.kv_stride + c * 8 : p.kv;
      const uint32_t dst = smem_u32(&S.k[buf][key * kDqk + c * 8]);
      const int nbytes = row >= 0 ? 16 : 0;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                   "r"(nbytes)
                   : "memory");
      if (c == 0) {
        S.valid[buf][key] = row >= 0;
        if (row < 0 && j < sr.k1) atomicOr(p.status, VA_STATUS_BAD_SLOT);
      }
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  };

  const int ntiles = ceil_div(sr.k1 - sr.k0, kKT);
  load_tile(sr.k0, 0);

  // ---- stage the 16 query rows as fp32 (rows past the request are zero)
  for (int idx = tid; idx < kRB * kChunks; idx += kThreads) {
    const int r = idx / kChunks, c = idx - r * kChunks;
    float f[8];
    if (row0 + r < R) {
      const uint4 v = *reinterpret_cast<const uint4*>(p.q + (grow0 + r) * kDqk + c * 8);
      unpack8(v, f);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = 0.f;
    }
    *reinterpret_cast<float4*>(&S.q[r * kDqk + c * 4]) = make_float4(f[0], f[1], f[2], f[3]);
    *reinterpret_cast<float4*>(&S.q[r * kDqk + kHalf + c * 4]) =
        make_float4(f[4], f[5], f[6], f[7]);
  }
  if (tid < kRB) {
    S.m[tid] = -INFINITY;
    S.l[tid] = 0.f;
  }

  float acc[kRB][2];
#pragma unroll
  for (int r = 0; r < kRB; ++r) acc[r][0] = acc[r][1] = 0.f;

  for (int t = 0; t < ntiles; ++t) {
    const int buf = t & 1;
    const int tk0 = sr.k0 + t * kKT;
    if (t + 1 < ntiles) {
      load_tile(tk0 + kKT, buf ^ 1);
      asm volatile("cp.async.wait_group 1;\n" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    }
    __syncthreads();

    // ---- scores: warp -> 4 keys, lane -> its columns, 16 rows
    {
      float a[kRB * 4];
#pragma unroll
      for (int e = 0; e < kRB * 4; ++e) a[e] = 0.f;
      const int kb = warp * 4;
#pragma unroll
      for (int ci = 0; ci < 3; ++ci) {
        const int c = lane + ci * 32;
        if (c < kChunks) {
          float kf[4][8];
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint4 v = *reinterpret_cast<const uint4*>(&S.k[buf][(kb + kk) * kDqk + c * 8]);
            unpack8(v, kf[kk]);
          }
#pragma unroll
          for (int r = 0; r < kRB; ++r) {
            const float4 q0 = *reinterpret_cast<const float4*>(&S.q[r * kDqk + c * 4]);
            const float4 q1 = *reinterpret_cast<const float4*>(&S.q[r * kDqk + kHalf + c * 4]);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              float s = a[r * 4 + kk];
              s = fmaf(q0.x, kf[kk][0], s);
              s = fmaf(q0.y, kf[kk][1], s);
              s = fmaf(q0.z, kf[kk][2], s);
              s = fmaf(q0.w, kf[kk][3], s);
              s = fmaf(q1.x, kf[kk][4], s);
              s = fmaf(q1.y, kf[kk][5], s);
              s = fmaf(q1.z, kf[kk][6], s);
              s = fmaf(q1.w, kf[kk][7], s);
              a[r * 4 + kk] = s;
            }
          }
        }
      }
      // halving butterfly: after level o each lane keeps the half of its
      // values selected by lane bit o and adds the partner's copy.
#pragma unroll
      for (int lvl = 0; lvl < 5; ++lvl) {
        const int o = 16 >> lvl;
        const int half = 32 >> lvl;
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
          const float send = upper ? a[i] : a[i + half];
          const float keep = upper ? a[i + half] : a[i];
          a[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      const int idx0 = 2 * lane;   // lane bit 4 picked the upper 32, bit 3 the upper 16, ...
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int idx = idx0 + e;
        S.pt[kb + (idx & 3)][idx >> 2] = a[e];
      }
    }
    __syncthreads();

    // ---- online softmax: warp -> 2 rows, lane -> key
#pragma unroll
    for (int rr = 0; rr < kRB / kWarps; ++rr) {
      const int r = warp * (kRB / kWarps) + rr;
      const int lrow = row0 + r;
      const int j = tk0 + lane;
      const float m_old = S.m[r];
      const float l_old = S.l[r];
      float s = -INFINITY;
      if (lrow < R && j < sr.k1 && S.valid[buf][lane]) {
        if (key_visible(p, ri, b, lrow / p.H, j)) s = S.pt[lane][r] * p.scale_log2;
      }
      const float m_new = fmaxf(m_old, warp_max(s));
      float pr = 0.f, alpha = 1.f;
      if (m_new != -INFINITY) {
        alpha = exp2f(m_old - m_new);
        pr = s == -INFINITY ? 0.f : exp2f(s - m_new);
      }
      const float sum = warp_sum(pr);
      S.pt[lane][r] = pr;
      __syncwarp();
      if (lane == 0) {
        S.alpha[r] = alpha;
        S.m[r] = m_new;
        S.l[r] = l_old * alpha + sum;
      }
    }
    __syncthreads();

    // ---- PV: thread -> value columns 2*tid, 2*tid+1
    {
      const int d = tid * 2;
#pragma unroll
      for (int r = 0; r < kRB; ++r) {
        const float al = S.alpha[r];
        acc[r][0] *= al;
        acc[r][1] *= al;
      }
#pragma unroll 4
      for (int key = 0; key < kKT; ++key) {
        const uint32_t vw = *reinterpret_cast<const uint32_t*>(&S.k[buf][key * kDqk + d]);
        const float v0 = bf16lo(vw), v1 = bf16hi(vw);
        const float4* p4 = reinterpret_cast<const float4*>(S.pt[key]);
#pragma unroll
        for (int g = 0; g < kRB / 4; ++g) {
          const float4 pp = p4[g];
          acc[g * 4 + 0][0] = fmaf(pp.x, v0, acc[g * 4 + 0][0]);
          acc[g * 4 + 0][1] = fmaf(pp.x, v1, acc[g * 4 + 0][1]);
          acc[g * 4 + 1][0] = fmaf(pp.y, v0, acc[g * 4 + 1][0]);
          acc[g * 4 + 1][1] = fmaf(pp.y, v1, acc[g * 4 + 1][1]);
          acc[g * 4 + 2][0] = fmaf(pp.z, v0, acc[g * 4 + 2][0]);
          acc[g * 4 + 2][1] = fmaf(pp.z, v1, acc[g * 4 + 2][1]);
          acc[g * 4 + 3][0] = fmaf(pp.w, v0, acc[g * 4 + 3][0]);
          acc[g * 4 + 3][1] = fmaf(pp.w, v1, acc[g * 4 + 3][1]);
        }
      }
    }
    __syncthreads();
  }

  // ---- the split's normalised partial output and lse
  const int d = tid * 2;
#pragma unroll
  for (int r = 0; r < kRB; ++r) {
    if (row0 + r < R) {
      const float l = S.l[r];
      const float inv = l > 0.f ? 1.f / l : 0.f;
      *reinterpret_cast<__nv_bfloat162*>(p.part_o + ((size_t)split * rows_total + grow0 + r) * kDv +
                                         d) = __floats2bfloat162_rn(acc[r][0] * inv, acc[r][1] * inv);
    }
  }
  if (tid < kRB && row0 + tid < R) {
    const float l = S.l[tid];
    p.part_lse[(size_t)split * rows_total + grow0 + tid] =
        l > 0.f ? (S.m[tid] + log2f(l)) * kLn2 : -INFINITY;
  }
}

}  // namespace

cudaError_t init_partial_fma() {
  return cudaFuncSetAttribute(partial_fma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(sizeof(FmaSmem)));
}

cudaError_t launch_partial_fma(const Params& p, int /*num_sms*/, cudaStream_t st) {
  dim3 grid(p.nsplit, ceil_div(p.rows_per_req, kRB), p.B);
  partial_fma_kernel<<<grid, kThreads, sizeof(FmaSmem), st>>>(p);
  return cudaGetLastError();
}

}  // namespace va
