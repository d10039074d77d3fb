// va_host.cu -- the C ABI: argument checks, workspace layout and launches.
//
// Every entry point checks its arguments on the host and returns a VA_ERR_*
// code before touching the device; it then enqueues its kernels on the
// caller's stream and returns without synchronising or allocating, so that a
// call can be captured into a CUDA graph and replayed (The Commit That Locked
// In 6x Decode, "1. Capture-Safe Design").
#include <math.h>
#include <string.h>

#include "va_common.cuh"

#define VA_API extern "C" __attribute__((visibility("default")))

namespace va {
cudaError_t init_partial_fma();
cudaError_t init_partial_tc(int* max_pairs, int* max_quads);
bool tc_supported(int B, int T, int H);
bool tc_use_pair(int T, int H, int flags);
int tc_auto_nsplit(int B, int T, int H, int clusters, bool pair);
int tc_flag_blocks(int T, int H, bool pair);
cudaError_t launch_partial_tc(const Params& p, int num_sms, cudaStream_t st);
}  // namespace va

namespace {

constexpr int kMaxDevices = 64;
struct DeviceState {
  int ready;
  int num_sms;
  int tc_pairs;   // two-CTA clusters of the tensor-core kernel resident at once
  int tc_quads;   // four-CTA clusters (two-SM products) resident at once
};
DeviceState g_dev[kMaxDevices];   // written by va_init only
cudaEvent_t g_ev_before = nullptr; // benchmark timing hook (va_set_partial_events)
cudaEvent_t g_ev_after = nullptr;

// Event record that also works under stream capture (as an external event node).
cudaError_t record_event(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return cudaErrorUnknown;
  return cs == cudaStreamCaptureStatusActive
             ? cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal)
             : cudaEventRecord(ev, st);
}

bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

int current_state(DeviceState* out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return VA_ERR_CUDA;
  if (!g_dev[dev].ready) return VA_ERR_UNSUPPORTED;
  *out = g_dev[dev];
  return VA_OK;
}

int auto_nsplit_fma(int B, int T, int H, int num_sms) {
  const long rowblocks = (long(T) * H + va::kFmaRows - 1) / va::kFmaRows;
  const long items = rowblocks * B;
  long ns = (2L * num_sms + items - 1) / items;
  if (ns < 1) ns = 1;
  if (ns > 256) ns = 256;
  return int(ns);
}

int pick_path(int flags, int B, int T, int H) {
  if (flags == VA_PATH_FMA) return VA_PATH_FMA;
  if (flags == VA_PATH_TC || flags == VA_PATH_TC_1SM)
    return va::tc_supported(B, T, H) ? VA_PATH_TC : -1;
  return va::tc_supported(B, T, H) ? VA_PATH_TC : VA_PATH_FMA;
}

int auto_nsplit(const DeviceState& ds, int path, int flags, int B, int T, int H) {
  if (path != VA_PATH_TC) return auto_nsplit_fma(B, T, H, ds.num_sms);
  const bool pair = va::tc_use_pair(T, H, flags);
  return va::tc_auto_nsplit(B, T, H, pair ? ds.tc_quads : ds.tc_pairs, pair);
}

// Shared by the entry points.  Key addressing: kv_start (contiguous rows),
// else slot_idx + indptr (paged), with draft_slots the draft nodes' own list
// (segmented; prefix lengths then come from indptr and prefix_len is NULL).
// Tree: dense_mask, else bits, else parent.
int verify_common(const void* q, const void* kv, int64_t num_slots, int64_t stride,
                  const int32_t* slot_idx, const int32_t* indptr, const int64_t* kv_start,
                  const int32_t* draft_slots, const void* draft_kv, const int32_t* prefix_len,
                  const uint8_t* dense_mask,
                  int64_t dense_mask_len, const int32_t* parent, const uint64_t* bits, int B,
                  int T, int H, float sm_scale, int nsplit, int flags, void* ws, size_t ws_bytes,
                  void* out, float* lse, cudaStream_t st) {
  const bool paged = kv_start == nullptr;
  const bool segmented = draft_slots != nullptr;
  if (!q || !kv || !ws || !out || !lse) return VA_ERR_NULL;
  if (!segmented && !prefix_len) return VA_ERR_NULL;
  if (paged && (!slot_idx || !indptr)) return VA_ERR_NULL;
  if (!parent && !bits && !dense_mask) return VA_ERR_NULL;
  if (dense_mask && dense_mask_len < 0) return VA_ERR_SHAPE;
  if (B < 1 || B > 65535 || T < 1 || T > VA_T_MAX || H < 1) return VA_ERR_SHAPE;
  if (int64_t(B) * T * H > (int64_t(1) << 24)) return VA_ERR_SHAPE;
  if (num_slots < 1 || stride < VA_D_QK) return VA_ERR_SHAPE;
  if (nsplit < 0 || nsplit > VA_NSPLIT_MAX) return VA_ERR_SHAPE;
  if (flags < VA_PATH_AUTO || flags > VA_PATH_TC_1SM) return VA_ERR_SHAPE;
  if (!isfinite(sm_scale)) return VA_ERR_SHAPE;
  if (stride % 8 != 0) return VA_ERR_ALIGN;
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(out, 16) || !aligned(ws, 256) ||
      !aligned(lse, 4) || (prefix_len && !aligned(prefix_len, 4)) ||
      (draft_slots && !aligned(draft_slots, 4)) || (draft_kv && !aligned(draft_kv, 16)))
    return VA_ERR_ALIGN;
  if (draft_kv && !draft_slots) return VA_ERR_SHAPE;
  if ((slot_idx && !aligned(slot_idx, 4)) || (indptr && !aligned(indptr, 4)) ||
      (parent && !aligned(parent, 4)) || (bits && !aligned(bits, 8)) ||
      (kv_start && !aligned(kv_start, 8)))
    return VA_ERR_ALIGN;

  // an explicit split count lets the workspace be checked before any CUDA call
  if (nsplit > 0 && ws_bytes < va::ws_layout(B, T, H, nsplit).total) return VA_ERR_WORKSPACE;

  DeviceState ds;
  int rc = current_state(&ds);
  if (rc != VA_OK) return rc;
  const int path = pick_path(flags, B, T, H);
  if (path < 0) return VA_ERR_UNSUPPORTED;
  int ns = nsplit;
  if (ns == 0)
    ns = auto_nsplit(ds, path, flags, B, T, H);
  const va::WsLayout L = va::ws_layout(B, T, H, ns);
  if (ws_bytes < L.total) return VA_ERR_WORKSPACE;

  uint8_t* w = static_cast<uint8_t*>(ws);
  va::Params p;
  memset(&p, 0, sizeof p);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.kv = static_cast<const __nv_bfloat16*>(kv);
  p.num_slots = num_slots;
  p.kv_stride = stride;
  p.slot_idx = paged ? slot_idx : nullptr;
  p.kv_indptr = paged ? indptr : nullptr;
  p.kv_start = kv_start;
  p.draft_slots = draft_slots;
  p.draft_kv = static_cast<const __nv_bfloat16*>(draft_kv);
  p.prefix_len = segmented ? nullptr : prefix_len;
  p.dense_mask = dense_mask;
  p.dense_mask_len = dense_mask ? dense_mask_len : 0;
  p.tree_parent = (bits || dense_mask) ? nullptr : parent;
  p.bits = (bits && !dense_mask) ? bits : reinterpret_cast<const uint64_t*>(w + L.bits);
  p.B = B;
  p.T = T;
  p.H = H;
  p.rows_per_req = T * H;
  p.nsplit = ns;
  p.sm_scale = sm_scale;
  p.scale_log2 = sm_scale * va::kLog2e;
  p.part_lse = reinterpret_cast<float*>(w + L.plse);
  p.part_o = reinterpret_cast<__nv_bfloat16*>(w + L.po);
  p.status = reinterpret_cast<uint32_t*>(w);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;

  // The tensor-core path computes the masks in its split-K kernel and keeps
  // per-CTA status words that the merge combines, so the mask kernel runs
  // there only to append draft rows.  The FMA path reads the masks the mask
  // kernel writes, and the mask kernel clears the status word for it.
  if (path == VA_PATH_TC) {
    p.cta_flags = reinterpret_cast<uint32_t*>(w + L.flags);
    p.tc_pair = va::tc_use_pair(T, H, flags) ? 1 : 0;
    p.flag_blocks = va::tc_flag_blocks(T, H, p.tc_pair != 0);
  }
  if (path != VA_PATH_TC || p.draft_kv) {
    if (va::launch_tree_bits(p, reinterpret_cast<uint64_t*>(w + L.bits), st) != cudaSuccess)
      return VA_ERR_LAUNCH;
  }
  const bool timed = g_ev_before && g_ev_after;
  if (timed && record_event(g_ev_before, st) != cudaSuccess) return VA_ERR_CUDA;
  cudaError_t e = path == VA_PATH_TC ? va::launch_partial_tc(p, ds.num_sms, st)
                                     : va::launch_partial_fma(p, ds.num_sms, st);
  if (e != cudaSuccess) return VA_ERR_LAUNCH;
  if (timed && record_event(g_ev_after, st) != cudaSuccess) return VA_ERR_CUDA;
  if (va::launch_combine(p, st) != cudaSuccess) return VA_ERR_LAUNCH;
  return VA_OK;
}

// Scratch of verify_attn_paged_noalloc: one fixed device array per GPU that
// loads this library, held until the process exits.  Host code must not pass
// the symbol itself to a kernel (on the host it names a host-side stand-in);
// it passes the device address from cudaGetSymbolAddress instead.
static __device__ __align__(256) uint8_t g_noalloc_scratch[VA_NOALLOC_SCRATCH_BYTES];
void* g_noalloc_ptr[kMaxDevices];   // device address per device (va_init, else first use)

// Resolves the scratch array's device address on the current device.  This
// translation unit is a module of its own (no relocatable device code), and
// under lazy module loading the driver loads a module -- and places its
// device arrays in memory -- on first use, so this call is where the array's
// memory is claimed.  va_init makes it, so that the array is in place before
// a caller reserves the rest of device memory or begins a stream capture.
cudaError_t resolve_noalloc(int dev) {
  if (g_noalloc_ptr[dev]) return cudaSuccess;
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess || !ptr) return e != cudaSuccess ? e : cudaErrorUnknown;
  g_noalloc_ptr[dev] = ptr;
  return cudaSuccess;
}

}  // namespace

VA_API int va_version(void) { return 100; }

VA_API int va_init(int device) {
  if (device < 0 || device >= kMaxDevices) return VA_ERR_SHAPE;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return VA_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return VA_ERR_UNSUPPORTED;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return VA_ERR_CUDA;
  if (cudaSetDevice(device) != cudaSuccess) return VA_ERR_CUDA;
  cudaError_t e1 = va::init_partial_fma();
  int pairs = 0, quads = 0;
  cudaError_t e2 = va::init_partial_tc(&pairs, &quads);
  // the no-allocation scratch array: placed now, with the device current; a
  // failure here (no memory left for it) is not an error of va_init -- the
  // first verify_attn_paged_noalloc call on the device retries and reports it
  if (resolve_noalloc(device) != cudaSuccess) (void)cudaGetLastError();
  cudaSetDevice(prev);
  if (e1 != cudaSuccess || e2 != cudaSuccess) return VA_ERR_CUDA;
  g_dev[device].num_sms = prop.multiProcessorCount;
  g_dev[device].tc_pairs = pairs > 0 ? pairs : prop.multiProcessorCount / 2;
  g_dev[device].tc_quads = quads > 0 ? quads : prop.multiProcessorCount / 4;
  g_dev[device].ready = 1;
  return VA_OK;
}

VA_API int va_auto_nsplit(int B, int T, int H, int flags) {
  if (B < 1 || T < 1 || T > VA_T_MAX || H < 1) return VA_ERR_SHAPE;
  if (flags < VA_PATH_AUTO || flags > VA_PATH_TC_1SM) return VA_ERR_SHAPE;
  DeviceState ds;
  int rc = current_state(&ds);
  if (rc != VA_OK) return rc;
  const int path = pick_path(flags, B, T, H);
  if (path < 0) return VA_ERR_UNSUPPORTED;
  return auto_nsplit(ds, path, flags, B, T, H);
}

VA_API size_t va_workspace_bytes(int B, int T, int H, int nsplit) {
  if (B < 1 || T < 1 || T > VA_T_MAX || H < 1 || nsplit < 1 || nsplit > VA_NSPLIT_MAX) return 0;
  return va::ws_layout(B, T, H, nsplit).total;
}

VA_API int verify_attn_paged(const void* q, const void* kv_pool, int64_t num_slots,
                             int64_t kv_row_stride, const int32_t* slot_idx,
                             const int32_t* kv_indptr, const int32_t* prefix_len,
                             const int32_t* tree_parent, const uint64_t* tree_bits, int B, int T,
                             int H, float sm_scale, int nsplit, int flags, void* workspace,
                             size_t workspace_bytes, void* out, float* lse, va_stream_t stream) {
  if (!slot_idx || !kv_indptr) return VA_ERR_NULL;
  return verify_common(q, kv_pool, num_slots, kv_row_stride, slot_idx, kv_indptr, nullptr, nullptr,
                       nullptr, prefix_len, nullptr, 0, tree_parent, tree_bits, B, T, H, sm_scale,
                       nsplit, flags, workspace, workspace_bytes, out, lse,
                       reinterpret_cast<cudaStream_t>(stream));
}

VA_API int verify_attn_contiguous(const void* q, const void* kv_pool, int64_t num_slots,
                                  int64_t kv_row_stride, const int64_t* kv_start,
                                  const int32_t* prefix_len, const int32_t* tree_parent,
                                  const uint64_t* tree_bits, int B, int T, int H, float sm_scale,
                                  int nsplit, int flags, void* workspace, size_t workspace_bytes,
                                  void* out, float* lse, va_stream_t stream) {
  if (!kv_start) return VA_ERR_NULL;
  return verify_common(q, kv_pool, num_slots, kv_row_stride, nullptr, nullptr, kv_start, nullptr,
                       nullptr, prefix_len, nullptr, 0, tree_parent, tree_bits, B, T, H, sm_scale,
                       nsplit, flags, workspace, workspace_bytes, out, lse,
                       reinterpret_cast<cudaStream_t>(stream));
}

VA_API int verify_attn_segmented(const void* q, const void* kv_pool, int64_t num_slots,
                                 int64_t kv_row_stride, const int32_t* kv_indices,
                                 const int32_t* kv_indptr, const int32_t* out_cache_loc,
                                 const void* draft_kv, const uint8_t* custom_mask,
                                 int64_t custom_mask_len,
                                 const int32_t* tree_parent, const uint64_t* tree_bits, int B,
                                 int T, int H, float sm_scale, int nsplit, int flags,
                                 void* workspace, size_t workspace_bytes, void* out, float* lse,
                                 va_stream_t stream) {
  if (!kv_indices || !kv_indptr || !out_cache_loc) return VA_ERR_NULL;
  return verify_common(q, kv_pool, num_slots, kv_row_stride, kv_indices, kv_indptr, nullptr,
                       out_cache_loc, draft_kv, nullptr, custom_mask, custom_mask_len, tree_parent,
                       tree_bits, B, T, H, sm_scale, nsplit, flags, workspace, workspace_bytes,
                       out, lse, reinterpret_cast<cudaStream_t>(stream));
}

VA_API int verify_attn_defrag(void* kv_pool, int64_t num_slots, int64_t kv_row_stride,
                              const int32_t* src_slots, const int32_t* src_indptr,
                              const int64_t* dst_base, int32_t* slot_idx_out, int B,
                              int64_t max_rows, uint32_t* status, va_stream_t stream) {
  if (!kv_pool || !src_slots || !src_indptr || !dst_base) return VA_ERR_NULL;
  if (B < 1 || B > 65535 || num_slots < 1 || kv_row_stride < VA_D_QK || max_rows < 1)
    return VA_ERR_SHAPE;
  if (kv_row_stride % 8 != 0) return VA_ERR_ALIGN;
  if (!aligned(kv_pool, 16) || !aligned(src_slots, 4) || !aligned(src_indptr, 4) ||
      !aligned(dst_base, 8) || (slot_idx_out && !aligned(slot_idx_out, 4)) ||
      (status && !aligned(status, 4)))
    return VA_ERR_ALIGN;
  DeviceState ds;
  int rc = current_state(&ds);
  if (rc != VA_OK) return rc;
  if (va::launch_defrag(kv_pool, num_slots, kv_row_stride, src_slots, src_indptr, dst_base,
                        slot_idx_out, B, max_rows, status,
                        reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return VA_ERR_LAUNCH;
  return VA_OK;
}

VA_API int verify_attn_paged_noalloc(const void* q, const void* kv_pool, int64_t num_slots,
                                     int64_t kv_row_stride, const int32_t* slot_idx,
                                     const int32_t* kv_indptr, const int32_t* prefix_len,
                                     const int32_t* tree_parent, const uint64_t* tree_bits, int B,
                                     int T, int H, float sm_scale, int nsplit, int flags,
                                     void* out, float* lse, va_stream_t stream) {
  if (B < 1 || T < 1 || T > VA_T_MAX || H < 1 || nsplit < 0 || nsplit > VA_NSPLIT_MAX)
    return VA_ERR_SHAPE;
  if (flags < VA_PATH_AUTO || flags > VA_PATH_TC_1SM) return VA_ERR_SHAPE;
  const size_t cap = VA_NOALLOC_SCRATCH_BYTES;
  // an explicit split count that does not fit is rejected before any CUDA call
  if (nsplit > 0 && va::ws_layout(B, T, H, nsplit).total > cap) return VA_ERR_WORKSPACE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return VA_ERR_CUDA;
  DeviceState ds;
  int rc = current_state(&ds);
  if (rc != VA_OK) return rc;
  // normally resolved by va_init; otherwise (va_init could not place the
  // array) this first call on the device tries again
  if (!g_noalloc_ptr[dev] && resolve_noalloc(dev) != cudaSuccess) return VA_ERR_CUDA;
  int ns = nsplit;
  if (ns == 0) {
    const int path = pick_path(flags, B, T, H);
    if (path < 0) return VA_ERR_UNSUPPORTED;
    ns = auto_nsplit(ds, path, flags, B, T, H);
    while (ns > 1 && va::ws_layout(B, T, H, ns).total > cap) --ns;
  }
  if (va::ws_layout(B, T, H, ns).total > cap) return VA_ERR_WORKSPACE;
  return verify_common(q, kv_pool, num_slots, kv_row_stride, slot_idx, kv_indptr, nullptr, nullptr,
                       nullptr, prefix_len, nullptr, 0, tree_parent, tree_bits, B, T, H, sm_scale, ns,
                       flags, g_noalloc_ptr[dev], cap, out, lse,
                       reinterpret_cast<cudaStream_t>(stream));
}

VA_API int va_set_partial_events(void* before, void* after) {
  g_ev_before = static_cast<cudaEvent_t>(before);
  g_ev_after = static_cast<cudaEvent_t>(after);
  return VA_OK;
}

VA_API int va_read_status(const void* workspace, uint32_t* status_host, va_stream_t stream) {
  if (!workspace || !status_host) return VA_ERR_NULL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return VA_ERR_CUDA;
  if (cudaMemcpy(status_host, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
    return VA_ERR_CUDA;
  return VA_OK;
}
