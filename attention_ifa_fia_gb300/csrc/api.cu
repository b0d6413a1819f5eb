// api.cu -- the extern "C" entry points declared in include/fia.h.
//
// Host side only: argument validation (before any launch), the split planner,
// TMA tensor-map encoding, the device status word, and dispatch to the kernels.
#include <cudaTypedefs.h>

#include <algorithm>
#include <map>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <utility>
#include <vector>

#include "fia.h"
#include "fia_internal.h"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_err[0] = '\0';
  return FIA_SUCCESS;
}

// One status word per device.  Kernels OR bits into it (see fia_device_status).
__device__ unsigned int g_status_word;

constexpr int kMaxDevices = 64;
struct DeviceInfo {
  bool init = false;
  void* ctx = nullptr;  // the context the cached addresses belong to
  int num_sms = 0;
  unsigned int* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Per-device set-up with that device current: SM count and the status word's address,
// looked up again whenever the device's current context changes (a device reset destroys
// the context and the module; the next context loads the module at new addresses).
int device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FIA_ERR_RUNTIME, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(FIA_ERR_RUNTIME, "device ordinal %d out of range", dev);
  void* ctx = nullptr;
  if (int rc = fia::current_context(&ctx)) return rc;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.init || d.ctx != ctx) {
    d.init = false;
    e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(FIA_ERR_RUNTIME, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status_word);
    if (e != cudaSuccess) return fail(FIA_ERR_RUNTIME, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    if (int rc = fia::current_context(&d.ctx)) return rc;  // current now, if it was not before
    d.init = true;
  }
  *out = &d;
  return FIA_SUCCESS;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D tensor map over a row-major matrix of `rows` rows of `cols` elements;
// box = box_cols x box_rows; swizzle span = box_cols * element bytes (128 or 64).
int make_tmap(CUtensorMap* m, const void* base, int dtype, uint64_t cols, uint64_t rows, uint32_t box_cols,
              uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(FIA_ERR_RUNTIME, "cuTensorMapEncodeTiled is not available from the driver");
  const uint32_t elem = dtype == fia::kI8 ? 1 : 2;
  CUtensorMapDataType t = dtype == fia::kI8    ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                          : dtype == fia::kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                               : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint32_t span = box_cols * elem;
  CUtensorMapSwizzle sw = span == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                          : span == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                       : CU_TENSOR_MAP_SWIZZLE_32B;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * elem};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, t, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FIA_ERR_RUNTIME, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return FIA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 3-D tensor map over queries (rows, Nq, D) -> dims (D, Nq, rows), boxes of 64 channels x G
// heads x qs rows, 128-byte swizzle: one kv head's G query heads at qs consecutive positions,
// landing as qs * G rows of 128 bytes (row i * G + g).
int make_tmap_q3(CUtensorMap* m, const void* base, int dtype, uint64_t D, uint64_t Nq, uint64_t rows, uint32_t G,
                 uint32_t qs) {
  auto fn = encode_fn();
  if (!fn) return fail(FIA_ERR_RUNTIME, "cuTensorMapEncodeTiled is not available from the driver");
  const CUtensorMapDataType t = dtype == fia::kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[3] = {D, Nq, rows};
  cuuint64_t strides[2] = {D * 2, Nq * D * 2};
  cuuint32_t box[3] = {64, G, qs};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, t, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FIA_ERR_RUNTIME, "cuTensorMapEncodeTiled (queries) failed (%d)", (int)r);
  return FIA_SUCCESS;
}

int gcd(int a, int b) { return b ? gcd(b, a % b) : a; }

// ---------------------------------------------------------------- decode planner
struct DecodePlan {
  int chunk_tokens = 0;
  int max_items = 0;
};

// Work items are (b, kv head, chunk) triples of `chunk_tokens` tokens.  With
// num_splits = n > 0 each sequence splits into at most n chunks; with 0 the
// chunk is sized so that the upper bound of the work (every sequence at
// max_kv_len) gives about `items_per_sm` items per SM, between one tile and 8192
// tokens.  Fewer items per SM mean fewer, larger chunks (a smaller workspace).
constexpr int kItemsPerSm = 12;      // 16-bit caches
constexpr int kItemsPerSmInt8 = 6;   // int8 caches: an item boundary costs the int8 kernel more
int plan_decode(int B, int Nkv, int max_kv_len, int num_splits, int num_sms, DecodePlan* plan,
                int items_per_sm = kItemsPerSm) {
  const int64_t T = fia::kDecodeTileTC;  // items are whole tiles of either attention kernel
  int64_t c;
  if (num_splits > 0) {
    c = ((int64_t)max_kv_len + num_splits - 1) / num_splits;
  } else {
    const int64_t upper = (int64_t)B * Nkv * max_kv_len;
    c = upper / ((int64_t)items_per_sm * std::max(num_sms, 1));
    c = std::min<int64_t>(std::max<int64_t>(c, T), 8192);
  }
  c = (c + T - 1) / T * T;
  if (c < T) c = T;
  const int64_t chunks = max_kv_len > 0 ? ((int64_t)max_kv_len + c - 1) / c : 1;
  const int64_t items = (int64_t)B * Nkv * chunks;
  if (items > (1LL << 30) || c > (1LL << 30))
    return fail(FIA_ERR_INNER_TILING, "split plan too large (%lld items)", (long long)items);
  const int64_t max_chunks_merge = 48 * 1024 / 4 / 8;  // merge weights held in shared memory
  if (chunks > max_chunks_merge)
    return fail(FIA_ERR_INNER_TILING, "%lld chunks per sequence exceed the merge limit %lld", (long long)chunks,
                (long long)max_chunks_merge);
  plan->chunk_tokens = (int)c;
  plan->max_items = (int)std::max<int64_t>(items, 1);
  return FIA_SUCCESS;
}

int check_decode_shape(int B, int Nq, int* Nkv, int D, int max_kv_len, int block_size, int num_splits) {
  if (B < 0 || B > 65536) return fail(FIA_ERR_PARAM_INVALID, "B = %d outside [0, 65536]", B);
  if (Nq < 1 || Nq > 256) return fail(FIA_ERR_PARAM_INVALID, "Nq = %d outside [1, 256]", Nq);
  if (*Nkv == 0) *Nkv = Nq;
  if (*Nkv < 0 || Nq % *Nkv != 0)
    return fail(FIA_ERR_PARAM_INVALID, "Nq = %d is not a multiple of Nkv = %d", Nq, *Nkv);
  if (Nq / *Nkv > 16)
    return fail(FIA_ERR_PARAM_INVALID, "GQA group %d > 16 is not supported in this build", Nq / *Nkv);
  if (D != 64 && D != 128) return fail(FIA_ERR_PARAM_INVALID, "D = %d not supported (64 or 128)", D);
  if (block_size <= 0 || block_size > 512 || block_size % 16 != 0)
    return fail(FIA_ERR_PARAM_INVALID, "block_size = %d must be a multiple of 16 in (0, 512]", block_size);
  if (max_kv_len < 0) return fail(FIA_ERR_PARAM_INVALID, "max_kv_len = %d < 0", max_kv_len);
  if (num_splits < 0) return fail(FIA_ERR_PARAM_INVALID, "num_splits = %d < 0", num_splits);
  return FIA_SUCCESS;
}

// ---------------------------------------------------------------- launch tracer
struct TraceState {
  bool on = false;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> marks[fia::kKernelCount];
  cudaEvent_t pending[fia::kKernelCount] = {};
  std::vector<cudaEvent_t> pool;
};
thread_local TraceState g_trace;

cudaEvent_t trace_event() {
  if (!g_trace.pool.empty()) {
    cudaEvent_t e = g_trace.pool.back();
    g_trace.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

namespace fia {
int current_context(void** ctx) {
  using GetCurrent = CUresult (*)(CUcontext*);
  static GetCurrent fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<GetCurrent>(p);
  });
  if (!fn) return report_error(FIA_ERR_RUNTIME, "cuCtxGetCurrent is not available from the driver");
  // NULL until the runtime has made the device's primary context current (it does so on the
  // first runtime call that needs a context, e.g. cudaGetSymbolAddress)
  CUcontext c = nullptr;
  if (fn(&c) != CUDA_SUCCESS) return report_error(FIA_ERR_RUNTIME, "cuCtxGetCurrent failed");
  *ctx = c;
  return FIA_SUCCESS;
}

cudaError_t ensure_smem(const void* func, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<void*, const void*>, size_t> done;  // (context, function) -> limit set
  void* ctx = nullptr;
  if (current_context(&ctx) != FIA_SUCCESS) ctx = nullptr;  // unknown context: always set
  std::lock_guard<std::mutex> lk(mu);
  auto key = std::make_pair(ctx, func);
  auto it = done.find(key);
  if (ctx && it != done.end() && it->second >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && ctx) done[key] = bytes;
  return e;
}

int report_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return code;
}

void trace_mark(int kernel, int phase, cudaStream_t stream) {
  if (!g_trace.on || kernel < 0 || kernel >= kKernelCount) return;
  cudaEvent_t e = trace_event();
  if (!e) return;
  cudaEventRecord(e, stream);
  if (phase == 0) {
    g_trace.pending[kernel] = e;
  } else if (g_trace.pending[kernel]) {
    g_trace.marks[kernel].emplace_back(g_trace.pending[kernel], e);
    g_trace.pending[kernel] = nullptr;
  }
}
}  // namespace fia

extern "C" {

const char* fia_last_error(void) { return g_err; }

int fia_trace_enable(int on) {
  g_trace.on = on != 0;
  return ok();
}

int fia_trace_collect(int kernel, double* total_ms, int* launches) {
  if (!total_ms || !launches) return fail(FIA_ERR_PARAM_NULLPTR, "total_ms and launches are required");
  if (kernel < 0 || kernel >= fia::kKernelCount) return fail(FIA_ERR_PARAM_INVALID, "unknown kernel id %d", kernel);
  double tot = 0.0;
  int n = 0;
  for (auto& pr : g_trace.marks[kernel]) {
    cudaError_t e = cudaEventSynchronize(pr.second);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, pr.first, pr.second);
    if (e != cudaSuccess) return fail(FIA_ERR_RUNTIME, "trace events: %s", cudaGetErrorString(e));
    tot += ms;
    ++n;
    g_trace.pool.push_back(pr.first);
    g_trace.pool.push_back(pr.second);
  }
  g_trace.marks[kernel].clear();
  *total_ms = tot;
  *launches = n;
  return ok();
}

int fia_device_status(fia_stream_t stream, unsigned int* flags) {
  if (!flags) return fail(FIA_ERR_PARAM_NULLPTR, "flags is NULL");
  DeviceInfo* d;
  if (int rc = device_info(&d)) return rc;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return fail(FIA_ERR_RUNTIME, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  unsigned int v = 0;
  e = cudaMemcpy(&v, d->status, sizeof v, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(d->status, 0, sizeof v);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(FIA_ERR_RUNTIME, "reading the status word: %s", cudaGetErrorString(e));
  *flags = v;
  return ok();
}

int fia_decode_workspace_size(int B, int Nq, int Nkv, int D, int max_kv_len, int block_size, int num_splits,
                              size_t* bytes) {
  if (!bytes) return fail(FIA_ERR_PARAM_NULLPTR, "bytes is NULL");
  if (int rc = check_decode_shape(B, Nq, &Nkv, D, max_kv_len, block_size, num_splits)) return rc;
  DeviceInfo* d;
  if (int rc = device_info(&d)) return rc;
  DecodePlan plan;
  if (int rc = plan_decode(B, Nkv, max_kv_len, num_splits, d->num_sms, &plan)) return rc;
  *bytes = fia::decode_workspace_bytes(B, Nkv, Nq / Nkv, D, plan.max_items);
  return ok();
}

static int decode_impl(const void* q, fia_dtype q_dtype, const void* k_cache, const void* v_cache,
                       fia_dtype kv_dtype, const int32_t* block_table, int64_t bt_stride,
                       const int64_t* actual_seq_lengths, int max_kv_len, int B, int Nq, int Nkv, int D,
                       int block_size, int64_t num_blocks, double scale, const float* antiquant_scale,
                       const float* antiquant_offset, const float* sink, void* out, float* softmax_max,
                       float* softmax_sum, int num_splits, void* workspace, size_t workspace_bytes,
                       fia_stream_t stream, const fia_decode_options* opt, bool check_only = false) {
  const int kv_layout = opt ? opt->kv_layout : FIA_KV_BNNBSD;
  const int aq_mode = opt ? opt->antiquant_mode : FIA_AQ_PER_CHANNEL;
  float* lse = opt ? opt->softmax_lse : nullptr;
  const uint8_t* mask = opt ? opt->atten_mask : nullptr;
  const int64_t mask_stride = opt ? opt->atten_mask_stride : 0;
  const float* qs2 = opt ? opt->quant_scale2 : nullptr;
  const float* qo2 = opt ? opt->quant_offset2 : nullptr;
  const int q2_per_channel = opt ? opt->quant2_per_channel : 0;
  const bool windowed = opt && opt->band;
  const int qs = (opt && opt->q_len > 1) ? opt->q_len : 1;  // query positions per batch
  // -- 161001: required pointers
  if (!q || !k_cache || !v_cache || !block_table || !actual_seq_lengths || !out)
    return fail(FIA_ERR_PARAM_NULLPTR, "q, k_cache, v_cache, block_table, actual_seq_lengths and out are required");
  if (kv_dtype == FIA_I8 && !antiquant_scale)
    return fail(FIA_ERR_PARAM_NULLPTR, "int8 KV needs antiquant_scale");
  if (!workspace && !check_only) return fail(FIA_ERR_PARAM_NULLPTR, "workspace is NULL");
  // -- 161002: dtypes, shapes, attributes
  if (q_dtype != FIA_F16 && q_dtype != FIA_BF16)
    return fail(FIA_ERR_PARAM_INVALID, "query dtype must be fp16 or bf16");
  if (kv_dtype != q_dtype && kv_dtype != FIA_I8)
    return fail(FIA_ERR_PARAM_INVALID, "key/value dtype must equal the query dtype or be int8");
  if (int rc = check_decode_shape(B, Nq, &Nkv, D, max_kv_len, block_size, num_splits)) return rc;
  if (kv_dtype == FIA_I8 && block_size % 32 != 0)
    return fail(FIA_ERR_PARAM_INVALID, "int8 KV needs block_size %% 32 == 0 (got %d)", block_size);
  if (kv_dtype == FIA_I8 && Nq / Nkv > 8)
    return fail(FIA_ERR_PARAM_INVALID, "int8 KV supports GQA groups up to 8 in this build (got %d)", Nq / Nkv);
  if (kv_dtype == FIA_I8 && sink)
    return fail(FIA_ERR_PARAM_INVALID, "the learnable sink is supported only without KV quantisation");
  if (kv_layout != FIA_KV_BNNBSD && kv_layout != FIA_KV_BNBSH)
    return fail(FIA_ERR_PARAM_INVALID, "unknown KV layout %d", kv_layout);
  if (aq_mode != FIA_AQ_PER_CHANNEL && aq_mode != FIA_AQ_PER_TENSOR)
    return fail(FIA_ERR_PARAM_INVALID, "unknown antiquant mode %d", aq_mode);
  if (aq_mode == FIA_AQ_PER_TENSOR && kv_dtype != FIA_I8)
    return fail(FIA_ERR_PARAM_INVALID, "per-tensor antiquant needs int8 KV");
  if (mask && mask_stride < (int64_t)max_kv_len)
    return fail(FIA_ERR_PARAM_INVALID, "atten_mask rows of %lld bytes are shorter than max_kv_len %d",
                (long long)mask_stride, max_kv_len);
  if (qo2 && !qs2) return fail(FIA_ERR_PARAM_INVALID, "quant_offset2 without quant_scale2");
  if (q2_per_channel != 0 && q2_per_channel != 1)
    return fail(FIA_ERR_PARAM_INVALID, "quant2_per_channel must be 0 or 1 (got %d)", q2_per_channel);
  if (opt && (opt->q_len < 0 || opt->q_len > 16))
    return fail(FIA_ERR_PARAM_INVALID, "q_len = %d outside [0, 16]", opt->q_len);
  if (qs > 1 && (Nq / Nkv) * qs > (kv_dtype == FIA_I8 ? 8 : 16))
    return fail(FIA_ERR_PARAM_INVALID, "GQA group %d x q_len %d exceeds %d in this build", Nq / Nkv, qs,
                kv_dtype == FIA_I8 ? 8 : 16);
  if (qs > 1 && Nq * qs > 256)
    return fail(FIA_ERR_PARAM_INVALID, "Nq x q_len = %d exceeds 256", Nq * qs);
  if (qs > 1 && (mask || windowed))
    return fail(FIA_ERR_PARAM_INVALID, "q_len > 1 takes the causal cut only (no attenMask or band) in this build");
  // the band in keys around the query (position L - 1), clamped to +-2^30 (no length is that large)
  constexpr int64_t kBandCap = 1LL << 30;
  int64_t win_pre = kBandCap, win_next = kBandCap;
  if (windowed) {
    win_pre = std::min(std::max(opt->pre_tokens, -kBandCap), kBandCap);
    win_next = std::min(std::max(opt->next_tokens, -kBandCap), kBandCap);
    if (win_pre + win_next < 0)
      return fail(FIA_ERR_PARAM_INVALID, "band with pre_tokens %lld and next_tokens %lld holds no key",
                  (long long)opt->pre_tokens, (long long)opt->next_tokens);
  }
  if (bt_stride < 1 || (int64_t)max_kv_len > bt_stride * block_size)
    return fail(FIA_ERR_PARAM_INVALID, "block table too narrow: max_kv_len %d > bt_stride %lld * block_size %d",
                max_kv_len, (long long)bt_stride, block_size);
  if (num_blocks < 1) return fail(FIA_ERR_PARAM_INVALID, "num_blocks = %lld < 1", (long long)num_blocks);
  if (num_blocks * Nkv * (int64_t)block_size >= (1LL << 31))
    return fail(FIA_ERR_PARAM_INVALID, "KV pool has 2^31 or more rows");
  if (!std::isfinite(scale)) return fail(FIA_ERR_PARAM_INVALID, "scale is not finite");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return fail(FIA_ERR_PARAM_INVALID, "q, k_cache, v_cache and out must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(FIA_ERR_PARAM_INVALID, "workspace must be 256-byte aligned");
  DeviceInfo* d;
  if (int rc = device_info(&d)) return rc;
  DecodePlan plan;
  if (int rc = plan_decode(B, Nkv, max_kv_len, num_splits, d->num_sms, &plan,
                           kv_dtype == FIA_I8 ? kItemsPerSmInt8 : kItemsPerSm))
    return rc;
  const int G = Nq / Nkv;
  const size_t need = fia::decode_workspace_bytes(B, Nkv, G * qs, D, plan.max_items);
  if (check_only) return ok();
  if (workspace_bytes < need)
    return fail(FIA_ERR_PARAM_INVALID, "workspace of %zu bytes is smaller than the %zu required", workspace_bytes,
                need);
  if (B == 0) return ok();  // empty query: nothing to do

  fia::DecodeParams p{};
  p.q = q;
  p.out = out;
  p.softmax_max = softmax_max;
  p.softmax_sum = softmax_sum;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.seq_lens = actual_seq_lengths;
  p.aq_scale = antiquant_scale;
  p.aq_offset = antiquant_offset;
  p.sink = sink;
  p.B = B;
  p.Nq = Nq;
  p.Nkv = Nkv;
  p.G = G;
  p.qs = qs;
  p.GV = G * qs;
  p.D = D;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.max_kv_len = max_kv_len;
  p.chunk_tokens = plan.chunk_tokens;
  p.max_items = plan.max_items;
  p.scale_log2 = (float)(scale * 1.4426950408889634);
  p.q_dtype = q_dtype;
  p.kv_dtype = kv_dtype;
  p.kv_layout = kv_layout;
  p.kv_row_blk = kv_layout == FIA_KV_BNBSH ? block_size : Nkv * block_size;
  p.kv_row_h = kv_layout == FIA_KV_BNBSH ? 0 : block_size;
  p.kv_x_h = kv_layout == FIA_KV_BNBSH ? D : 0;
  p.atten_mask = mask;
  p.mask_stride = mask ? mask_stride : 0;
  p.pq_scale = qs2;
  p.pq_offset = qo2;
  p.pq_stride = q2_per_channel;
  p.partials_only = qs2 != nullptr;
  p.windowed = windowed ? 1 : 0;
  // 16-bit KV runs on the tensor-core kernel, which schedules its own work when the batch
  // fits its shared-memory schedule (otherwise a plan launch precedes it)
  p.fused_plan = (kv_dtype != FIA_I8 && B <= fia::kFusedPlanMaxB) ? 1 : 0;
  p.win_pre = (int)win_pre;
  p.win_next = (int)win_next;
  p.ws = fia::decode_workspace_carve(workspace, B, Nkv, G * qs, D, plan.max_items);
  p.status = d->status;
  if (aq_mode == FIA_AQ_PER_TENSOR) {  // the kernels read the per-channel form
    float* sc = p.ws.aux;
    float* of = antiquant_offset ? p.ws.aux + 2 * Nkv * D : nullptr;
    cudaError_t e0 = fia::launch_aq_expand(antiquant_scale, antiquant_offset, Nkv, D, sc, of, stream);
    if (e0 != cudaSuccess) return fail(FIA_ERR_RUNTIME, "antiquant expansion: %s", cudaGetErrorString(e0));
    p.aq_scale = sc;
    p.aq_offset = of;
  }
  if (lse) {  // max and sum are needed for the log-sum-exp; scratch if not requested
    if (!p.softmax_max) p.softmax_max = p.ws.aux + 4 * Nkv * D;
    if (!p.softmax_sum) p.softmax_sum = p.ws.aux + 4 * Nkv * D + (size_t)B * qs * Nq;
  }

  // 16-bit KV runs on the tensor-core kernel (128-token tiles), int8 KV with D = 128 on the
  // int8 tensor-core kernel (128-token tiles), other int8 shapes on the CUDA-core one.
  const bool tc = kv_dtype != FIA_I8;
  const bool tile128 = tc || fia::decode_uses_i8tc(kv_dtype, D);
  const int elem = kv_dtype == FIA_I8 ? 1 : 2;
  const uint32_t box_cols = (uint32_t)std::min(D * elem, 128) / elem;
  const int box_rows = gcd(block_size, tile128 ? fia::kDecodeTileTC : fia::kDecodeTile);
  // layout 0: a row of D channels per (block, kv head, token); layout 1: a row of Nkv * D
  // channels per (block, token), the kernels adding the head's column offset
  const uint64_t cols = kv_layout == FIA_KV_BNBSH ? (uint64_t)Nkv * D : (uint64_t)D;
  const uint64_t rows = kv_layout == FIA_KV_BNBSH ? (uint64_t)num_blocks * block_size
                                                  : (uint64_t)num_blocks * Nkv * block_size;
  CUtensorMap tmK, tmV, tmQ, tail[2];
  if (int rc = make_tmap(&tmK, k_cache, kv_dtype, cols, rows, box_cols, box_rows)) return rc;
  if (int rc = make_tmap(&tmV, v_cache, kv_dtype, cols, rows, box_cols, box_rows)) return rc;
  // boxes of 16 rows (32 for int8: its block size is a multiple of 32) for tiles with fewer
  // than 128 keys, so that rows past a sequence's keys are not read
  const int tail_rows = kv_dtype == FIA_I8 ? 32 : 16;
  if (tile128 && box_rows > tail_rows) {
    if (int rc = make_tmap(&tail[0], k_cache, kv_dtype, cols, rows, box_cols, tail_rows)) return rc;
    if (int rc = make_tmap(&tail[1], v_cache, kv_dtype, cols, rows, box_cols, tail_rows)) return rc;
  } else {
    tail[0] = tmK;
    tail[1] = tmV;
  }
  if (tc) {
    if (qs == 1) {
      if (int rc = make_tmap(&tmQ, q, q_dtype, D, (uint64_t)B * Nq, 64, 16)) return rc;
    } else {  // (D, Nq, B * q_len) with (64, G, q_len) boxes: a kv head's G x q_len query rows
      if (int rc = make_tmap_q3(&tmQ, q, q_dtype, D, Nq, (uint64_t)B * qs, G, qs)) return rc;
    }
  }
  cudaError_t e = fia::launch_decode(p, tmK, tmV, tc ? &tmQ : nullptr, tail, box_rows, d->num_sms, stream);
  if (e != cudaSuccess) return fail(FIA_ERR_RUNTIME, "decode launch: %s", cudaGetErrorString(e));
  if (lse) {
    e = fia::launch_lse(p.softmax_max, p.softmax_sum, lse, (int64_t)B * qs * Nq, stream);
    if (e != cudaSuccess) return fail(FIA_ERR_RUNTIME, "log-sum-exp launch: %s", cudaGetErrorString(e));
  }
  return ok();
}

}  // extern "C"

namespace fia {
int decode_check(const void* q, int q_dtype, const void* k_cache, const void* v_cache, int kv_dtype,
                 const int32_t* block_table, int64_t bt_stride, const int64_t* actual_seq_lengths, int max_kv_len,
                 int B, int Nq, int Nkv, int D, int block_size, int64_t num_blocks, double scale,
                 const float* antiquant_scale, const float* antiquant_offset, const float* sink, void* out,
                 float* softmax_max, float* softmax_sum, int num_splits) {
  return decode_impl(q, static_cast<fia_dtype>(q_dtype), k_cache, v_cache, static_cast<fia_dtype>(kv_dtype), block_table, bt_stride, actual_seq_lengths, max_kv_len,
                     B, Nq, Nkv, D, block_size, num_blocks, scale, antiquant_scale, antiquant_offset, sink, out,
                     softmax_max, softmax_sum, num_splits, nullptr, 0, nullptr, nullptr, true);
}
}  // namespace fia

extern "C" {

int fia_decode(const void* q, fia_dtype q_dtype, const void* k_cache, const void* v_cache, fia_dtype kv_dtype,
               const int32_t* block_table, int64_t bt_stride, const int64_t* actual_seq_lengths, int max_kv_len,
               int B, int Nq, int Nkv, int D, int block_size, int64_t num_blocks, double scale,
               const float* antiquant_scale, const float* antiquant_offset, const float* sink, void* out,
               float* softmax_max, float* softmax_sum, int num_splits, void* workspace, size_t workspace_bytes,
               fia_stream_t stream) {
  return decode_impl(q, q_dtype, k_cache, v_cache, kv_dtype, block_table, bt_stride, actual_seq_lengths, max_kv_len,
                     B, Nq, Nkv, D, block_size, num_blocks, scale, antiquant_scale, antiquant_offset, sink, out,
                     softmax_max, softmax_sum, num_splits, workspace, workspace_bytes, stream, nullptr);
}

int fia_decode_ex(const void* q, fia_dtype q_dtype, const void* k_cache, const void* v_cache, fia_dtype kv_dtype,
                  const int32_t* block_table, int64_t bt_stride, const int64_t* actual_seq_lengths, int max_kv_len,
                  int B, int Nq, int Nkv, int D, int block_size, int64_t num_blocks, double scale,
                  const float* antiquant_scale, const float* antiquant_offset, const float* sink, void* out,
                  float* softmax_max, float* softmax_sum, int num_splits, void* workspace, size_t workspace_bytes,
                  fia_stream_t stream, const fia_decode_options* options) {
  return decode_impl(q, q_dtype, k_cache, v_cache, kv_dtype, block_table, bt_stride, actual_seq_lengths, max_kv_len,
                     B, Nq, Nkv, D, block_size, num_blocks, scale, antiquant_scale, antiquant_offset, sink, out,
                     softmax_max, softmax_sum, num_splits, workspace, workspace_bytes, stream, options);
}

int ring_attention_update(const void* prev_out, const float* prev_max, const float* prev_sum, const void* cur_out,
                          const float* cur_max, const float* cur_sum, fia_dtype out_dtype, int64_t rows, int N,
                          int D, void* out, float* max_out, float* sum_out, fia_stream_t stream) {
  if (!prev_out || !prev_max || !prev_sum || !cur_out || !cur_max || !cur_sum || !out || !max_out || !sum_out)
    return fail(FIA_ERR_PARAM_NULLPTR, "every input and output of ring_attention_update is required");
  if (out_dtype != FIA_F32 && out_dtype != FIA_F16 && out_dtype != FIA_BF16)
    return fail(FIA_ERR_PARAM_INVALID, "out dtype must be fp32, fp16 or bf16");
  if (rows < 0) return fail(FIA_ERR_PARAM_INVALID, "rows = %lld < 0", (long long)rows);
  if (N < 1 || N > 256) return fail(FIA_ERR_PARAM_INVALID, "N = %d outside [1, 256]", N);
  if (D < 8 || D > 768 || D % 8 != 0) return fail(FIA_ERR_PARAM_INVALID, "D = %d must be a multiple of 8 <= 768", D);
  if (!aligned16(prev_out) || !aligned16(cur_out) || !aligned16(out))
    return fail(FIA_ERR_PARAM_INVALID, "attention outputs must be 16-byte aligned");
  cudaError_t e = fia::launch_rau(prev_out, prev_max, prev_sum, cur_out, cur_max, cur_sum, out_dtype, rows, N, D,
                                  out, max_out, sum_out, stream);
  if (e != cudaSuccess) return fail(FIA_ERR_RUNTIME, "ring_attention_update launch: %s", cudaGetErrorString(e));
  return ok();
}

int fia_debug_dequant(const int8_t* codes, const float* scale, const float* offset, int64_t n, float* out,
                      fia_stream_t stream) {
  if (!codes || !scale || !offset || !out) return fail(FIA_ERR_PARAM_NULLPTR, "all pointers are required");
  if (n < 0) return fail(FIA_ERR_PARAM_INVALID, "n < 0");
  cudaError_t e = fia::launch_debug_dequant(codes, scale, offset, n, out, stream);
  if (e != cudaSuccess) return fail(FIA_ERR_RUNTIME, "dequant probe launch: %s", cudaGetErrorString(e));
  return ok();
}

int fia_debug_gather(const void* k_cache, fia_dtype kv_dtype, const int32_t* block_table, int64_t bt_stride,
                     const int64_t* actual_seq_lengths, int max_kv_len, int B, int Nkv, int D, int block_size,
                     int64_t num_blocks, int b, int hkv, void* dst, fia_stream_t stream) {
  if (!k_cache || !block_table || !actual_seq_lengths || !dst)
    return fail(FIA_ERR_PARAM_NULLPTR, "k_cache, block_table, actual_seq_lengths and dst are required");
  if (kv_dtype != FIA_F16 && kv_dtype != FIA_BF16 && kv_dtype != FIA_I8)
    return fail(FIA_ERR_PARAM_INVALID, "kv dtype must be fp16, bf16 or int8");
  int nkv = Nkv;
  if (int rc = check_decode_shape(B, std::max(Nkv, 1), &nkv, D, max_kv_len, block_size, 0)) return rc;
  if (b < 0 || b >= B || hkv < 0 || hkv >= nkv) return fail(FIA_ERR_PARAM_INVALID, "(b, hkv) out of range");
  if (bt_stride < 1 || (int64_t)max_kv_len > bt_stride * block_size || num_blocks < 1)
    return fail(FIA_ERR_PARAM_INVALID, "block table / pool shape");
  if (!aligned16(k_cache)) return fail(FIA_ERR_PARAM_INVALID, "k_cache must be 16-byte aligned");
  DeviceInfo* d;
  if (int rc = device_info(&d)) return rc;
  fia::DecodeParams p{};
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.seq_lens = actual_seq_lengths;
  p.B = B;
  p.Nkv = nkv;
  p.D = D;
  p.block_size = block_size;
  p.kv_row_blk = nkv * block_size;  // (num_blocks, Nkv, block_size, D)
  p.kv_row_h = block_size;
  p.num_blocks = num_blocks;
  p.max_kv_len = max_kv_len;
  p.kv_dtype = kv_dtype;
  p.status = d->status;
  const int elem = kv_dtype == FIA_I8 ? 1 : 2;
  const uint32_t box_cols = (uint32_t)std::min(D * elem, 128) / elem;
  const int box_rows = gcd(block_size, fia::kDecodeTile);
  CUtensorMap tmK;
  if (int rc = make_tmap(&tmK, k_cache, kv_dtype, D, (uint64_t)num_blocks * nkv * block_size, box_cols, box_rows))
    return rc;
  cudaError_t e = fia::launch_debug_gather(p, tmK, box_rows, b, hkv, dst, stream);
  if (e != cudaSuccess) return fail(FIA_ERR_RUNTIME, "gather probe launch: %s", cudaGetErrorString(e));
  return ok();
}

int fia_debug_i8_codes(const int8_t* codes, int64_t n, uint16_t* out, fia_stream_t stream) {
  if (!codes || !out) return fail(FIA_ERR_PARAM_NULLPTR, "codes and out are required");
  if (n < 0 || n % 4 != 0) return fail(FIA_ERR_PARAM_INVALID, "n = %lld must be a non-negative multiple of 4",
                                       (long long)n);
  if ((reinterpret_cast<uintptr_t>(codes) & 3u) || (reinterpret_cast<uintptr_t>(out) & 7u))
    return fail(FIA_ERR_PARAM_INVALID, "codes must be 4-byte and out 8-byte aligned");
  cudaError_t e = fia::launch_debug_i8_codes(codes, n, out, stream);
  if (e != cudaSuccess) return fail(FIA_ERR_RUNTIME, "code conversion probe launch: %s", cudaGetErrorString(e));
  return ok();
}

int fia_debug_i8_qprep(const void* q, fia_dtype q_dtype, const float* antiquant_scale, const float* antiquant_offset,
                       int B, int Nq, int Nkv, double scale, void* blocks, size_t blocks_bytes, uint16_t* q_hi,
                       uint16_t* q_lo, float* kq_nq, fia_stream_t stream) {
  if (!q || !antiquant_scale || !blocks || !q_hi || !q_lo || !kq_nq)
    return fail(FIA_ERR_PARAM_NULLPTR, "q, antiquant_scale, blocks, q_hi, q_lo and kq_nq are required");
  if (q_dtype != FIA_F16 && q_dtype != FIA_BF16) return fail(FIA_ERR_PARAM_INVALID, "query dtype must be fp16 or bf16");
  int nkv = Nkv;
  if (int rc = check_decode_shape(B, Nq, &nkv, 128, 0, 128, 0)) return rc;
  if (!std::isfinite(scale)) return fail(FIA_ERR_PARAM_INVALID, "scale is not finite");
  if (!aligned16(q) || (reinterpret_cast<uintptr_t>(blocks) & 255u))
    return fail(FIA_ERR_PARAM_INVALID, "q must be 16-byte and blocks 256-byte aligned");
  const size_t need = fia::debug_i8_qprep_block_bytes() * (size_t)B * nkv;
  if (blocks_bytes < need)
    return fail(FIA_ERR_PARAM_INVALID, "blocks of %zu bytes are smaller than the %zu required", blocks_bytes, need);
  fia::DecodeParams p{};
  p.q = q;
  p.q_dtype = q_dtype;
  p.aq_scale = antiquant_scale;
  p.aq_offset = antiquant_offset;
  p.B = B;
  p.Nq = Nq;
  p.Nkv = nkv;
  p.G = Nq / nkv;
  p.qs = 1;
  p.GV = p.G;
  p.D = 128;
  p.scale_log2 = (float)(scale * 1.4426950408889634);
  p.ws.qprep = static_cast<uint8_t*>(blocks);
  cudaError_t e = fia::launch_debug_i8_qprep(p, q_hi, q_lo, kq_nq, stream);
  if (e != cudaSuccess) return fail(FIA_ERR_RUNTIME, "query preparation probe launch: %s", cudaGetErrorString(e));
  return ok();
}

}  // extern "C"

namespace {

// 3-D tensor map over a (rows, heads, D) row-major tensor, box = 64 x 1 x 128 rows,
// 128-byte swizzle: one head's 128 consecutive rows, 64 channels per box.
int make_tmap_thd(CUtensorMap* m, const void* base, int dtype, uint64_t D, uint64_t heads, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return fail(FIA_ERR_RUNTIME, "cuTensorMapEncodeTiled is not available from the driver");
  const CUtensorMapDataType t = dtype == fia::kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[3] = {D, heads, rows};
  cuuint64_t strides[2] = {D * 2, heads * D * 2};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, t, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FIA_ERR_RUNTIME, "cuTensorMapEncodeTiled (3-D) failed (%d)", (int)r);
  return FIA_SUCCESS;
}

// A paged K or V pool as a 3-D tensor (cols channels, block_size rows, zs blocks [x kv
// heads]) read in boxes of 64 channels x box_rows rows x 1 block: 128 / box_rows boxes side
// by side land in shared memory as the (64, 1, 128) box of the TND map does, 128 rows of 128
// bytes (box_rows is a multiple of 16, so every box starts on a whole swizzle pattern).
int make_tmap_paged(CUtensorMap* m, const void* base, int dtype, uint64_t cols, int block_size, uint64_t zs,
                    int box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(FIA_ERR_RUNTIME, "cuTensorMapEncodeTiled is not available from the driver");
  const CUtensorMapDataType t = dtype == fia::kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[3] = {cols, (cuuint64_t)block_size, zs};
  cuuint64_t strides[2] = {cols * 2, (cuuint64_t)block_size * cols * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, t, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FIA_ERR_RUNTIME, "cuTensorMapEncodeTiled (paged 3-D) failed (%d)", (int)r);
  return FIA_SUCCESS;
}

int check_prefill_shape(int B, int Nq, int* Nkv, int D, int max_seqlen_q) {
  if (B < 0 || B > 65536) return fail(FIA_ERR_PARAM_INVALID, "B = %d outside [0, 65536]", B);
  if (Nq < 1 || Nq > 256) return fail(FIA_ERR_PARAM_INVALID, "Nq = %d outside [1, 256]", Nq);
  if (*Nkv == 0) *Nkv = Nq;
  if (*Nkv < 0 || Nq % *Nkv != 0)
    return fail(FIA_ERR_PARAM_INVALID, "Nq = %d is not a multiple of Nkv = %d", Nq, *Nkv);
  if (D != 64 && D != 128) return fail(FIA_ERR_PARAM_INVALID, "prefill supports D = 64 or 128 in this build (got %d)", D);
  if (max_seqlen_q < 0) return fail(FIA_ERR_PARAM_INVALID, "max_seqlen_q = %d < 0", max_seqlen_q);
  if ((int64_t)B * ((max_seqlen_q + 127) / 128) >= (1LL << 31) / 256)
    return fail(FIA_ERR_PARAM_INVALID, "too many query tiles");
  return FIA_SUCCESS;
}

}  // namespace

extern "C" {

int fia_prefill_workspace_size(int B, int Nq, int Nkv, int D, int max_seqlen_q, size_t* bytes) {
  if (!bytes) return fail(FIA_ERR_PARAM_NULLPTR, "bytes is NULL");
  if (int rc = check_prefill_shape(B, Nq, &Nkv, D, max_seqlen_q)) return rc;
  *bytes = fia::prefill_workspace_bytes(B, Nq, max_seqlen_q);
  return ok();
}

static int prefill_impl(const void* q, const void* k, const void* v, fia_dtype dtype, const int64_t* cu_seqlens_q,
                        const int64_t* cu_seqlens_kv, int B, int64_t T, int64_t Tkv, int max_seqlen_q,
                        int max_seqlen_kv, int Nq, int Nkv, int D, double scale, int mask, const float* sink,
                        void* out, float* softmax_max, float* softmax_sum, void* workspace, size_t workspace_bytes,
                        fia_stream_t stream, const fia_prefill_options* opt) {
  const bool paged = opt && opt->block_table;
  if (!q || !k || !v || !cu_seqlens_q || !out || (!paged && !cu_seqlens_kv))
    return fail(FIA_ERR_PARAM_NULLPTR, "q, k, v, cu_seqlens_q, cu_seqlens_kv (unless paged) and out are required");
  if (paged && !opt->seq_lens_kv) return fail(FIA_ERR_PARAM_NULLPTR, "paged keys need seq_lens_kv");
  if (!workspace) return fail(FIA_ERR_PARAM_NULLPTR, "workspace is NULL");
  if (dtype != FIA_F16 && dtype != FIA_BF16) return fail(FIA_ERR_PARAM_INVALID, "dtype must be fp16 or bf16");
  if (int rc = check_prefill_shape(B, Nq, &Nkv, D, max_seqlen_q)) return rc;
  if (T < 0 || Tkv < 0 || T >= (1LL << 31) || Tkv >= (1LL << 31))
    return fail(FIA_ERR_PARAM_INVALID, "T = %lld, Tkv = %lld outside [0, 2^31)", (long long)T, (long long)Tkv);
  if (max_seqlen_kv < 0 || max_seqlen_kv > (1 << 20))
    return fail(FIA_ERR_PARAM_INVALID, "max_seqlen_kv = %d outside [0, 2^20] (this build)", max_seqlen_kv);
  if (mask != 0 && mask != 3 && mask != 4)
    return fail(FIA_ERR_PARAM_INVALID, "mask = %d: 0 (none), 3 (rightDownCausal) and 4 (band) are supported", mask);
  // the band in keys around the rightDownCausal diagonal, clamped to +-2^30 (no sequence is
  // longer than 2^21 here, so clamping changes no visible set)
  constexpr int64_t kBandCap = 1LL << 30;
  int64_t pre = kBandCap, next = mask == 3 ? 0 : kBandCap;
  if (mask == 4) {
    if (!opt) return fail(FIA_ERR_PARAM_NULLPTR, "mask 4 (band) needs options with pre_tokens and next_tokens");
    pre = std::min(std::max(opt->pre_tokens, -kBandCap), kBandCap);
    next = std::min(std::max(opt->next_tokens, -kBandCap), kBandCap);
    if (pre + next < 0)
      return fail(FIA_ERR_PARAM_INVALID, "band with pre_tokens %lld and next_tokens %lld holds no key",
                  (long long)opt->pre_tokens, (long long)opt->next_tokens);
  }
  if (paged) {
    const int bs = opt->block_size;
    if (bs < 16 || bs > 512 || bs % 16 != 0)
      return fail(FIA_ERR_PARAM_INVALID, "paged prefill needs block_size a multiple of 16 up to 512 (got %d)", bs);
    if (opt->kv_layout != FIA_KV_BNNBSD && opt->kv_layout != FIA_KV_BNBSH)
      return fail(FIA_ERR_PARAM_INVALID, "unknown KV layout %d", opt->kv_layout);
    if (opt->num_blocks < 1 || opt->num_blocks * Nkv >= (1LL << 31))
      return fail(FIA_ERR_PARAM_INVALID, "num_blocks = %lld outside [1, 2^31 / Nkv)", (long long)opt->num_blocks);
    if (opt->bt_stride < 1 || (int64_t)max_seqlen_kv > opt->bt_stride * bs)
      return fail(FIA_ERR_PARAM_INVALID, "block table too narrow: max_seqlen_kv %d > bt_stride %lld * block_size %d",
                  max_seqlen_kv, (long long)opt->bt_stride, bs);
  }
  const float* qs2 = opt ? opt->quant_scale2 : nullptr;
  const float* qo2 = opt ? opt->quant_offset2 : nullptr;
  const int q2_per_channel = opt ? opt->quant2_per_channel : 0;
  if (qo2 && !qs2) return fail(FIA_ERR_PARAM_INVALID, "quant_offset2 without quant_scale2");
  if (q2_per_channel != 0 && q2_per_channel != 1)
    return fail(FIA_ERR_PARAM_INVALID, "quant2_per_channel must be 0 or 1 (got %d)", q2_per_channel);
  if (!std::isfinite(scale)) return fail(FIA_ERR_PARAM_INVALID, "scale is not finite");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(FIA_ERR_PARAM_INVALID, "q, k, v and out must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(FIA_ERR_PARAM_INVALID, "workspace must be 256-byte aligned");
  const size_t need = fia::prefill_workspace_bytes(B, Nq, max_seqlen_q);
  if (workspace_bytes < need)
    return fail(FIA_ERR_PARAM_INVALID, "workspace of %zu bytes is smaller than the %zu required", workspace_bytes,
                need);
  DeviceInfo* d;
  if (int rc = device_info(&d)) return rc;
  if (B == 0 || T == 0) return ok();

  fia::PrefillParams p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.softmax_max = softmax_max;
  p.softmax_sum = softmax_sum;
  p.cu_q = cu_seqlens_q;
  p.cu_kv = cu_seqlens_kv;
  p.sink = sink;
  p.B = B;
  p.Nq = Nq;
  p.Nkv = Nkv;
  p.G = Nq / Nkv;
  p.D = D;
  p.T = T;
  p.Tkv = Tkv;
  p.max_seqlen_q = max_seqlen_q;
  p.max_seqlen_kv = max_seqlen_kv;
  p.pre = (int)pre;
  p.next = (int)next;
  if (paged) {
    const bool bsh = opt->kv_layout == FIA_KV_BNBSH;
    p.block_table = opt->block_table;
    p.bt_stride = opt->bt_stride;
    p.seq_lens_kv = opt->seq_lens_kv;
    p.block_size = opt->block_size;
    p.box_rows = gcd(opt->block_size, 128);
    p.num_blocks = opt->num_blocks;
    p.kv_x_h = bsh ? D : 0;
    p.kv_z_blk = bsh ? 1 : Nkv;
    p.kv_z_h = bsh ? 0 : 1;
  }
  p.dtype = dtype;
  p.scale_log2 = (float)(scale * 1.4426950408889634);
  p.pq_scale = qs2;
  p.pq_offset = qo2;
  p.pq_stride = q2_per_channel;
  p.tile_counter = static_cast<int*>(workspace);
  p.tile_list = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + 256);
  p.max_tiles = (int)((need - 256) / sizeof(int));
  p.status = d->status;
  CUtensorMap tmQ, tmK, tmV;
  if (int rc = make_tmap_thd(&tmQ, q, dtype, D, Nq, T)) return rc;
  if (paged) {  // (channels, rows of a block, block [x kv head]) with (64, 128, 1) boxes
    const bool bsh = opt->kv_layout == FIA_KV_BNBSH;
    const uint64_t cols = bsh ? (uint64_t)Nkv * D : (uint64_t)D;
    const uint64_t zs = bsh ? (uint64_t)opt->num_blocks : (uint64_t)opt->num_blocks * Nkv;
    if (int rc = make_tmap_paged(&tmK, k, dtype, cols, opt->block_size, zs, p.box_rows)) return rc;
    if (int rc = make_tmap_paged(&tmV, v, dtype, cols, opt->block_size, zs, p.box_rows)) return rc;
  } else {
    if (int rc = make_tmap_thd(&tmK, k, dtype, D, Nkv, Tkv > 0 ? Tkv : 1)) return rc;
    if (int rc = make_tmap_thd(&tmV, v, dtype, D, Nkv, Tkv > 0 ? Tkv : 1)) return rc;
  }
  cudaError_t e = fia::launch_prefill(p, tmQ, tmK, tmV, d->num_sms, stream);
  if (e != cudaSuccess) return fail(FIA_ERR_RUNTIME, "prefill launch: %s", cudaGetErrorString(e));
  return ok();
}

int fia_prefill(const void* q, const void* k, const void* v, fia_dtype dtype, const int64_t* cu_seqlens_q,
                const int64_t* cu_seqlens_kv, int B, int64_t T, int64_t Tkv, int max_seqlen_q, int max_seqlen_kv,
                int Nq, int Nkv, int D, double scale, int mask, const float* sink, void* out, float* softmax_max,
                float* softmax_sum, void* workspace, size_t workspace_bytes, fia_stream_t stream) {
  return prefill_impl(q, k, v, dtype, cu_seqlens_q, cu_seqlens_kv, B, T, Tkv, max_seqlen_q, max_seqlen_kv, Nq, Nkv,
                      D, scale, mask, sink, out, softmax_max, softmax_sum, workspace, workspace_bytes, stream,
                      nullptr);
}

int fia_prefill_ex(const void* q, const void* k, const void* v, fia_dtype dtype, const int64_t* cu_seqlens_q,
                   const int64_t* cu_seqlens_kv, int B, int64_t T, int64_t Tkv, int max_seqlen_q, int max_seqlen_kv,
                   int Nq, int Nkv, int D, double scale, int mask, const float* sink, void* out, float* softmax_max,
                   float* softmax_sum, void* workspace, size_t workspace_bytes, fia_stream_t stream,
                   const fia_prefill_options* options) {
  return prefill_impl(q, k, v, dtype, cu_seqlens_q, cu_seqlens_kv, B, T, Tkv, max_seqlen_q, max_seqlen_kv, Nq, Nkv,
                      D, scale, mask, sink, out, softmax_max, softmax_sum, workspace, workspace_bytes, stream,
                      options);
}

}  // extern "C"
