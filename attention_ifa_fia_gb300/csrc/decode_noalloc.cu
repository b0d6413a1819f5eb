// decode_noalloc.cu -- fia_decode for callers that cannot allocate device memory.
//
// fia_decode needs a caller-provided workspace (the split plan and the per-chunk
// partial results).  Some callers have no way to provide one: plugins whose host
// application owns every byte of device memory through its own allocator, modules
// that are not allowed to touch the CUDA allocator at all, and latency-critical
// loops in which cudaMalloc (which may synchronise the device) is forbidden.  For
// them this file keeps the workspace in a fixed, file-scope device array instead.
//
// Costs and limits, stated for the user:
//   * Every GPU that loads the library holds kScratchBytes (16 MiB) of device
//     memory for this array until the process exits, whether or not the entry
//     point is ever called.
//   * Problems whose workspace (fia_decode_workspace_size) exceeds kScratchBytes
//     are rejected with FIA_ERR_PARAM_INVALID and a message naming the limit.
//   * All calls on a device share the one array.  It keeps whatever the previous
//     call left in it; nothing in it needs to start at zero (the split plan kernel
//     rewrites the work counter and item list at the start of every call).  Calls
//     whose work overlaps on the GPU -- different streams, or different host
//     threads without ordering between them -- race on the array and give wrong
//     results.  Issue them on one stream, or order them.
//   * The first call on each device looks up the array's device address with
//     cudaGetSymbolAddress while that device is current.  Make that first call
//     before any stream capture begins.  The address is kept per device together
//     with the device's context; a call that finds another context current (after
//     a device reset, which reloads the module) looks it up again, so the first
//     call after a reset must also come before any stream capture.
//   * Arguments are checked exactly as fia_decode checks them (same codes, same
//     order) before the workspace size is compared with the scratch.
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <cstdio>
#include <mutex>

#include "fia.h"
#include "fia_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB per device

// The scratch itself.  In host code this name is only a host-side stand-in for the
// symbol, never a device address: its address must come from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchAddr {
  void* ctx = nullptr;  // the context the address belongs to
  void* ptr = nullptr;
};
ScratchAddr g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of this device's scratch array, looked up with the device current
// the first time and again whenever the device's current context has changed.
// Returns 0, or a non-zero fia status.
int scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fia::report_error(FIA_ERR_RUNTIME, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fia::report_error(FIA_ERR_RUNTIME, "device ordinal %d out of range", dev);
  void* ctx = nullptr;
  if (int rc = fia::current_context(&ctx)) return rc;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  ScratchAddr& a = g_scratch[dev];
  if (!a.ptr || a.ctx != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || !p)
      return fia::report_error(FIA_ERR_RUNTIME, "cudaGetSymbolAddress of the decode scratch: %s",
                               cudaGetErrorString(e));
    if (int rc = fia::current_context(&a.ctx)) return rc;  // current now, if it was not before
    a.ptr = p;
  }
  *out = a.ptr;
  return FIA_SUCCESS;
}

}  // namespace

extern "C" int fia_decode_noalloc(const void* q, fia_dtype q_dtype, const void* k_cache, const void* v_cache,
                                  fia_dtype kv_dtype, const int32_t* block_table, int64_t bt_stride,
                                  const int64_t* actual_seq_lengths, int max_kv_len, int B, int Nq, int Nkv, int D,
                                  int block_size, int64_t num_blocks, double scale, const float* antiquant_scale,
                                  const float* antiquant_offset, const float* sink, void* out, float* softmax_max,
                                  float* softmax_sum, int num_splits, fia_stream_t stream) {
  int rc = fia::decode_check(q, q_dtype, k_cache, v_cache, kv_dtype, block_table, bt_stride, actual_seq_lengths,
                             max_kv_len, B, Nq, Nkv, D, block_size, num_blocks, scale, antiquant_scale,
                             antiquant_offset, sink, out, softmax_max, softmax_sum, num_splits);
  if (rc != FIA_SUCCESS) return rc;  // the code and message fia_decode would give
  size_t need = 0;
  rc = fia_decode_workspace_size(B, Nq, Nkv, D, max_kv_len, block_size, num_splits, &need);
  if (rc != FIA_SUCCESS) return rc;  // fia_last_error() describes the bad argument
  if (need > kScratchBytes)
    return fia::report_error(FIA_ERR_PARAM_INVALID,
                             "fia_decode_noalloc: this problem needs %zu bytes of workspace, more than the fixed "
                             "%zu-byte scratch; call fia_decode with a caller-provided workspace instead",
                             need, kScratchBytes);
  void* scratch = nullptr;
  rc = scratch_for_current_device(&scratch);
  if (rc != FIA_SUCCESS) return rc;
  return fia_decode(q, q_dtype, k_cache, v_cache, kv_dtype, block_table, bt_stride, actual_seq_lengths, max_kv_len,
                    B, Nq, Nkv, D, block_size, num_blocks, scale, antiquant_scale, antiquant_offset, sink, out,
                    softmax_max, softmax_sum, num_splits, scratch, kScratchBytes, stream);
}
