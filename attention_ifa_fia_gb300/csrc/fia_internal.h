// fia_internal.h -- declarations shared between the C-ABI layer (api.cu) and
// the kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fia {

// storage types (same numbering as fia_dtype in include/fia.h)
enum : int { kF32 = 0, kF16 = 1, kBF16 = 2, kI8 = 3 };

// bits of the device status word
enum : unsigned int {
  kStatusWaitTimeout = 1u << 0,    // a bounded mbarrier wait gave up
  kStatusBadBlockIndex = 1u << 1,  // a block-table entry outside [0, num_blocks)
  kStatusLengthClamped = 1u << 2,  // a device length outside [0, max_kv_len] was clamped
  kStatusBadSeqlens = 1u << 3,     // cumulative sequence lengths not monotone / out of range
};

// kernels known to the launch tracer (fia_trace_enable / fia_trace_collect)
enum : int { kKernelDecodePlan = 0, kKernelDecodeAttention = 1, kKernelDecodeMerge = 2, kKernelPrefill = 3,
             kKernelRau = 4, kKernelCount = 5 };

// Sets the text fia_last_error() returns on this thread and returns `code`.
int report_error(int code, const char* fmt, ...);

// Raises the dynamic shared-memory limit of kernel `func` to at least `bytes`, calling
// cudaFuncSetAttribute only the first time a (context, function) pair needs a larger value,
// so that repeated launches (and stream capture) do not repeat it.
cudaError_t ensure_smem(const void* func, size_t bytes);
template <typename K>
inline cudaError_t ensure_smem(K* kern, size_t bytes) {
  return ensure_smem(reinterpret_cast<const void*>(kern), bytes);
}

// The calling thread's current CUDA context (a CUcontext; NULL if none is current yet).
// Returns 0 or a non-zero fia status.
int current_context(void** ctx);

// Every check fia_decode makes on these arguments, in the same order and with the same
// codes and messages, except those on the workspace; launches nothing.
int decode_check(const void* q, int q_dtype, const void* k_cache, const void* v_cache, int kv_dtype,
                 const int32_t* block_table, int64_t bt_stride, const int64_t* actual_seq_lengths, int max_kv_len,
                 int B, int Nq, int Nkv, int D, int block_size, int64_t num_blocks, double scale,
                 const float* antiquant_scale, const float* antiquant_offset, const float* sink, void* out,
                 float* softmax_max, float* softmax_sum, int num_splits);

// Records a CUDA event on `stream` before (phase 0) or after (phase 1) a launch
// of `kernel` when tracing is enabled on the calling thread; otherwise nothing.
void trace_mark(int kernel, int phase, cudaStream_t stream);

constexpr float kLog2e = 1.4426950408889634f;  // log2(e)
constexpr float kLn2 = 0.6931471805599453f;    // ln(2)

// ---------------------------------------------------------------------------
// Decode
// ---------------------------------------------------------------------------
constexpr int kDecodeTile = 64;        // tokens per pipeline stage
constexpr int kDecodeStages = 4;       // stages in the TMA ring
constexpr int kDecodeConsumers = 256;  // math threads (8 warps)

struct DecodeWorkspace {
  int* counter;     // dynamic work counter (reset by the plan kernel)
  int* n_items;     // number of work items written by the plan kernel
  int* seg_base;    // (B + 1) first item of batch b; [B] = the number of items
  int4* items;      // (max_items) {b, hkv | nch << 16, first token, last token + 1}
  int* order;       // (max_items) execution order: order[k] is the k-th item to be claimed
  float* part_o;    // (max_items, G, D) normalised partial outputs
  float2* part_ml;  // (max_items, G) {max (log2 units), sum}
  uint8_t* qprep;   // (B * Nkv) q' blocks of the int8 tensor-core path (D = 128), else null
  float* aux;       // (4 Nkv D + 2 B Nq): per-tensor antiquant expanded to (2, Nkv, D) scale and
                    // offset, then max and sum scratch for the log-sum-exp output
};

struct DecodeParams {
  const void* q;
  void* out;
  float* softmax_max;
  float* softmax_sum;
  const int32_t* block_table;
  int64_t bt_stride;
  const int64_t* seq_lens;
  const float* aq_scale;   // (2, Nkv, D) or null
  const float* aq_offset;  // (2, Nkv, D) or null
  const float* sink;       // (Nq) or null
  int B, Nq, Nkv, G, D, block_size;
  int64_t num_blocks;
  int max_kv_len;     // device lengths are clamped to [0, max_kv_len]
  int chunk_tokens;   // tokens per work item (a multiple of kDecodeTile)
  int max_items;
  float scale_log2;   // scale * log2(e)
  int q_dtype, kv_dtype;
  int kv_layout;      // 0: (num_blocks, Nkv, block_size, D); 1: (num_blocks, block_size, Nkv * D)
  // tensor-map coordinates of a pool token: row = blk * kv_row_blk + hkv * kv_row_h + t % block_size,
  // column of the head's first channel = hkv * kv_x_h (set from kv_layout by the host)
  int kv_row_blk, kv_row_h, kv_x_h;
  const uint8_t* atten_mask;  // (B, mask_stride) bytes, nonzero = key masked out; or null
  int64_t mask_stride;
  // int8 output: code = sat8(rint(out * pq_scale[c * pq_stride] + pq_offset[c * pq_stride])) for
  // channel c = h * D + d; pq_scale null for a 16-bit output.  With it every segment, of one
  // item or none, is finished by the merge kernel (partials_only).
  const float* pq_scale;
  const float* pq_offset;  // or null
  int pq_stride;           // 0: one value for the tensor; 1: one per channel
  int partials_only;
  // band of the one query (windowed != 0): batch b of length L sees keys
  // L - 1 - win_pre .. L - 1 + win_next (both within [-2^30, 2^30], win_pre + win_next >= 0)
  int windowed, win_pre, win_next;
  // nonzero: the tensor-core attention kernel schedules its own work items (no plan launch;
  // B <= kFusedPlanMaxB)
  int fused_plan;
  // query positions per batch (FusedInferAttentionScore, Q_S > 1 over the paged cache): q and
  // out are (B, qs, Nq, D), position i of batch b (at key L_b - qs + i) sees keys
  // t <= L_b - qs + i.  The kernels treat the qs positions of a kv head's G query heads as
  // GV = G * qs virtual heads v = i * G + g; qs = 1 is plain decode
  int qs, GV;
  DecodeWorkspace ws;
  unsigned int* status;  // device status word
};

size_t decode_workspace_bytes(int B, int Nkv, int G, int D, int max_items);
// (2) per-tensor antiquant scale and offset (offset may be null) -> (2, Nkv, D) in dst_scale,
// dst_offset; log-sum-exp of n rows from their max and sum.
cudaError_t launch_aq_expand(const float* scale2, const float* offset2, int Nkv, int D, float* dst_scale,
                             float* dst_offset, cudaStream_t stream);
cudaError_t launch_lse(const float* mx, const float* sm, float* lse, int64_t n, cudaStream_t stream);
DecodeWorkspace decode_workspace_carve(void* base, int B, int Nkv, int G, int D, int max_items);

// Launches plan + attention + merge on `stream`.  tmK / tmV describe the K and V
// pools as 2-D tensors (D, num_blocks * Nkv * block_size) with boxes of box_rows
// rows.  With tmQ (the query as a 2-D tensor (D, B * Nq), 16-row boxes) the
// tensor-core attention kernel runs (16-bit KV, G <= 16, 128-token tiles);
// without it the CUDA-core kernel (any KV type, G <= 8, 64-token tiles).
// tail[0], tail[1]: the K and V pools again with 16-row boxes, used for tiles with fewer
// than 128 keys (the same maps as tmK / tmV when box_rows is 16).
cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          const CUtensorMap* tmQ, const CUtensorMap* tail, int box_rows, int num_sms,
                          cudaStream_t stream);
cudaError_t launch_decode_tc_attention(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                       const CUtensorMap& tmQ, const CUtensorMap* tail, int box_rows, int grid,
                                       cudaStream_t stream);
cudaError_t launch_merge(const DecodeParams& p, cudaStream_t stream);
constexpr int kDecodeTileTC = 128;  // tokens per tensor-core tile; work items are multiples of it
constexpr int kFusedPlanMaxB = 256;  // batches the in-kernel schedule of the 16-bit kernel holds

// int8 KV with D = 128 runs on the tensor-core kernel of decode_i8tc.cu (128-token
// tiles, G <= 8); other int8 shapes on the CUDA-core kernel.
inline bool decode_uses_i8tc(int kv_dtype, int D) { return kv_dtype == kI8 && D == 128; }
cudaError_t launch_decode_i8tc_attention(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                         const CUtensorMap* tail, int box_rows, int grid, cudaStream_t stream);

// ---------------------------------------------------------------------------
// RingAttentionUpdate
// ---------------------------------------------------------------------------
cudaError_t launch_rau(const void* prev_out, const float* prev_max, const float* prev_sum, const void* cur_out,
                       const float* cur_max, const float* cur_sum, int out_dtype, int64_t rows, int N, int D,
                       void* out, float* max_out, float* sum_out, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Prefill
// ---------------------------------------------------------------------------
struct PrefillParams {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* softmax_max;
  float* softmax_sum;
  const int64_t* cu_q;
  const int64_t* cu_kv;
  const float* sink;
  int B, Nq, Nkv, G, D;
  int64_t T, Tkv;
  int max_seqlen_q, max_seqlen_kv;
  // band on the rightDownCausal diagonal: key j is visible to query i of a sequence iff
  // i + d - pre <= j <= i + d + next, d = Lkv - Lq (pre + next >= 0, both within
  // [-2^30, 2^30]); rightDownCausal is (2^30, 0), no mask (2^30, 2^30)
  int pre, next;
  // paged K/V (block_table non-null): k and v are pools of blocks of block_size tokens (a
  // multiple of 16); key t of sequence b is row t % block_size of block
  // block_table[b][t / block_size], at tensor-map coordinates (x = hkv * kv_x_h + channel,
  // y = row in block, z = blk * kv_z_blk + hkv * kv_z_h); a key tile of 128 keys arrives as
  // 128 / box_rows boxes of box_rows rows, each inside one block; sequence b has
  // seq_lens_kv[b] keys (clamped to [0, max_seqlen_kv]); cu_kv is unused
  const int32_t* block_table;
  int64_t bt_stride;
  const int64_t* seq_lens_kv;
  int block_size;
  int box_rows;  // rows of one tensor-map box: gcd(block_size, 128), so a box lies in one block
  int64_t num_blocks;
  int kv_x_h, kv_z_blk, kv_z_h;
  int dtype;          // kBF16 or kF16
  float scale_log2;
  // int8 output (pq_scale non-null): code = saturate(rne(o * pq_scale[c] + pq_offset[c])),
  // c = (h * D + d) * pq_stride (pq_stride 0: one value for every channel)
  const float* pq_scale;
  const float* pq_offset;
  int pq_stride;
  int* tile_list;     // workspace: (sequence << 16 | query tile) pairs, longest first
  int* tile_counter;  // workspace: [0] unit counter, [1] number of units
  int max_tiles;
  unsigned int* status;
};

size_t prefill_workspace_bytes(int B, int Nq, int max_seqlen_q);
cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                           const CUtensorMap& tmV, int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Probes used by the bit-exactness tests
// ---------------------------------------------------------------------------
cudaError_t launch_debug_dequant(const int8_t* codes, const float* scale, const float* offset, int64_t n,
                                 float* out, cudaStream_t stream);
cudaError_t launch_debug_gather(const DecodeParams& p, const CUtensorMap& tmK, int box_rows, int b, int hkv,
                                void* dst, cudaStream_t stream);
// The int8 tensor-core kernel's exact steps: n codes (n % 4 == 0) -> fp16 bit patterns; the
// q' blocks of p (written to p.ws.qprep, B * Nkv blocks of debug_i8_qprep_block_bytes()) and
// their hi / lo parts (B * Nkv * 16 rows x 128) and {kq, nq} pairs (B * Nkv * 16) read back.
size_t debug_i8_qprep_block_bytes();
cudaError_t launch_debug_i8_codes(const int8_t* codes, int64_t n, uint16_t* out, cudaStream_t stream);
cudaError_t launch_debug_i8_qprep(const DecodeParams& p, uint16_t* hi, uint16_t* lo, float* kn,
                                  cudaStream_t stream);

}  // namespace fia
