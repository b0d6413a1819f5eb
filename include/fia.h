/*
 * fia.h -- C interface of libfia_gb300: fused inference attention on one GB300
 * (sm_103a).
 *
 * Operators (semantics from the operator documentation pages cited per call):
 *   fia_decode             paged GQA decode attention, query S = 1, optional int8
 *                          KV antiquant and learnable sink, split-KV partials merged
 *                          by the RingAttentionUpdate rule
 *   fia_decode_ex          the same with the operator's variants: the (blocknum,
 *                          blocksize, H) cache layout, per-tensor antiquant, attenMask,
 *                          softmaxLse, an int8 output (quantScale2 / quantOffset2) and
 *                          a band window (preTokens / nextTokens)
 *   fia_decode_noalloc     fia_decode without a workspace argument
 *   fia_prefill            causal variable-length attention, TND layout
 *   fia_prefill_ex         the same with the band mask (preTokens / nextTokens) and
 *                          keys and values in a paged cache (chunked prefill)
 *   ring_attention_update  merge of two attention partials by softmax max/sum
 *
 * Conventions shared by every call:
 *   - Pointers marked "device" are CUDA device addresses; the caller allocates and
 *     owns all of them, including the workspace.  The library allocates nothing on
 *     the device and keeps no state between calls except the device status word
 *     (see fia_device_status).
 *   - All work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  Results are valid once the stream has synchronised.
 *   - Arguments are checked on the host before anything is launched.  On any
 *     non-zero return nothing was launched and no output was touched, except for
 *     FIA_ERR_RUNTIME, which reports a failed launch.
 *   - Results are bitwise reproducible for fixed inputs and arguments (no float
 *     atomics; partials are merged in a fixed order).
 *   - Return codes follow the aclnn codes of the pages (aclnnIncreFlashAttentionV3,
 *     "Return Value"): 0 success; 161001 a required pointer is NULL; 161002 an
 *     invalid dtype, shape, attribute or alignment, a size this build does not
 *     support, or a workspace that is too small; 361001 a CUDA runtime error;
 *     561002 the split planner could not partition the work.
 *     fia_last_error() returns a text description of the last failure on the
 *     calling thread.
 */
#ifndef FIA_H_
#define FIA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fia_stream_t; /* identical to cudaStream_t */

typedef enum { FIA_F32 = 0, FIA_F16 = 1, FIA_BF16 = 2, FIA_I8 = 3 } fia_dtype;

enum {
  FIA_SUCCESS = 0,
  FIA_ERR_PARAM_NULLPTR = 161001,
  FIA_ERR_PARAM_INVALID = 161002,
  FIA_ERR_RUNTIME = 361001,
  FIA_ERR_INNER_TILING = 561002
};

/* Bits of the device status word (fia_device_status). */
enum {
  FIA_STATUS_WAIT_TIMEOUT = 1,    /* a bounded on-chip wait gave up; results of that launch are invalid */
  FIA_STATUS_BAD_BLOCK_INDEX = 2, /* a block-table entry in use was outside [0, num_blocks); its tile was skipped */
  FIA_STATUS_LENGTH_CLAMPED = 4,  /* a device length was outside [0, max_kv_len] and was clamped */
  FIA_STATUS_BAD_SEQLENS = 8      /* cumulative sequence lengths were not monotone or exceeded T */
};

/* Text of the last error returned on the calling thread ("" if none). */
const char* fia_last_error(void);

/* Synchronises `stream`, returns in *flags the device status bits raised by any
 * launch of this library on the current device since the previous call, and
 * clears them.  Returns 0, or 361001 if the synchronisation itself failed. */
int fia_device_status(fia_stream_t stream, unsigned int* flags);

/* Launch tracing.  While enabled on the calling thread, every launch of one of the
 * library's kernels is bracketed by two CUDA events recorded on the launching stream.
 * fia_trace_collect synchronises on the recorded events, returns the summed device time
 * (ms) and the number of launches of one kernel since the previous collect, and forgets
 * them.  Kernel ids: */
enum {
  FIA_KERNEL_DECODE_PLAN = 0,      /* per-call split plan (one CTA) */
  FIA_KERNEL_DECODE_ATTENTION = 1, /* split-KV attention over the paged cache */
  FIA_KERNEL_DECODE_MERGE = 2,     /* merge of split partials, sink, outputs */
  FIA_KERNEL_PREFILL = 3,          /* TND prefill */
  FIA_KERNEL_RAU = 4               /* ring_attention_update */
};
int fia_trace_enable(int on);
int fia_trace_collect(int kernel, double* total_ms, int* launches);

/* ------------------------------------------------------------------------- decode
 * aclnnIncreFlashAttentionV3 ("Function", parameter table, "Constraints / page
 * attention"); FusedInferAttentionScore (learnableSink, softmax max/sum for ring
 * merging); aclnnFlashAttentionScoreV4 (sink formula).
 *
 *   out[b][h] = softmax(scale * q[b][h] . K^T) V over the first L_b = actual_seq_lengths[b]
 *   tokens of batch b, with query head h reading kv head h / (Nq / Nkv).  Token t of batch
 *   b lives in pool block block_table[b * bt_stride + t / block_size], row t % block_size.
 *   With a sink s_h:  m = max(s_h, max_t z_t),  out = sum_t e^{z_t - m} v_t / (sum_t e^{z_t - m} + e^{s_h - m}).
 *   softmax_max[b][h] = m and softmax_sum[b][h] = sum_t e^{z_t - m} (+ e^{s_h - m}), where z_t is
 *   the scaled logit (natural-exp domain).  A row with no visible key and no sink gives
 *   out = 0, max = -inf, sum = 0; with a sink, out = 0, max = s_h, sum = 1.
 *
 * q, out             device, (B, Nq, D) row-major in q_dtype (FIA_F16 or FIA_BF16); with query
 *                    length 1 this is the memory of the BNSD, BSND and BSH layouts alike.
 *                    16-byte aligned.
 * k_cache, v_cache   device, (num_blocks, Nkv, block_size, D) row-major (the pages'
 *                    (blocknum, KV_N, blocksize, D) layout), in kv_dtype: q_dtype, or FIA_I8.
 *                    16-byte aligned.  Only rows of visible tokens are read.
 * block_table        device int32, B rows of bt_stride entries; entries past
 *                    ceil(L_b / block_size) are never read.
 * actual_seq_lengths device int64 (B).  Values are clamped to [0, max_kv_len]
 *                    (FIA_STATUS_LENGTH_CLAMPED is raised if any is outside).
 * max_kv_len         host upper bound of the lengths; <= bt_stride * block_size.
 * Nkv                0 means Nkv = Nq.  Nq % Nkv == 0; Nq / Nkv <= 16 (<= 8 with int8 KV) in
 *                    this build.
 * D                  64 or 128 in this build.
 * block_size         > 0, <= 512, a multiple of 16 (16-bit KV) or 32 (int8 KV).
 * scale              the scaleValue of the pages, usually 1/sqrt(D).
 * antiquant_scale    device fp32 (2, Nkv, D): [0] for K, [1] for V; required iff kv_dtype is
 *                    FIA_I8.  Dequantisation is (x - offset) * scale in fp32.
 * antiquant_offset   device fp32 (2, Nkv, D) or NULL (zero).
 * sink               device fp32 (Nq) or NULL; not allowed with int8 KV.
 * softmax_max/sum    device fp32 (B, Nq) or NULL (not written).
 * num_splits         0 picks the split automatically; n > 0 splits each sequence into at most
 *                    n chunks of ceil(max_kv_len / n) tokens (rounded up to 128).
 * workspace          device, at least fia_decode_workspace_size() bytes, 256-byte aligned.
 *                    Holds the split plan and partials; contents need no initialisation.
 */
int fia_decode_workspace_size(int B, int Nq, int Nkv, int D, int max_kv_len, int block_size, int num_splits,
                              size_t* bytes);

int fia_decode(const void* q, fia_dtype q_dtype, const void* k_cache, const void* v_cache, fia_dtype kv_dtype,
               const int32_t* block_table, int64_t bt_stride, const int64_t* actual_seq_lengths, int max_kv_len,
               int B, int Nq, int Nkv, int D, int block_size, int64_t num_blocks, double scale,
               const float* antiquant_scale, const float* antiquant_offset, const float* sink, void* out,
               float* softmax_max, float* softmax_sum, int num_splits, void* workspace, size_t workspace_bytes,
               fia_stream_t stream);

/* fia_decode with decode variants of the same kernels (aclnnIncreFlashAttentionV3,
 * "Constraints / page attention": the (blocknum, blocksize, H) KV layout beside
 * (blocknum, KV_N, blocksize, D); the per-tensor antiquant of shape (2); the parameter
 * table's attenMask and quantScale2 / quantOffset2; FusedInferAttentionScore's
 * softmaxLse output).  Arguments as for fia_decode, plus:
 *
 * options->kv_layout        FIA_KV_BNNBSD: k_cache/v_cache are (num_blocks, Nkv, block_size, D)
 *                           as for fia_decode.  FIA_KV_BNBSH: (num_blocks, block_size, Nkv * D)
 *                           row-major (H = Nkv * D): token t of a block is one row holding
 *                           every kv head's channels, head h at columns [h * D, (h + 1) * D).
 * options->antiquant_mode   FIA_AQ_PER_CHANNEL: antiquant_scale/offset are (2, Nkv, D) as for
 *                           fia_decode.  FIA_AQ_PER_TENSOR: they are (2): one scale (offset)
 *                           for all keys, one for all values.  Int8 KV only.
 * options->softmax_lse      device fp32 (B, Nq) or NULL: ln(sum_t e^{z_t}) (+ e^{s_h} with a
 *                           sink) = softmax_max + ln(softmax_sum); -inf for a row with
 *                           neither a visible key nor a sink.
 * options->atten_mask       device bytes (B, 1, 1, S) -- bool, int8 or uint8 holding 0 or 1 --
 *                           or NULL: byte b * atten_mask_stride + t nonzero removes key t of
 *                           batch b from the softmax (1 = masked out).  A batch whose keys are
 *                           all masked gives the rows of an empty sequence (out 0, max -inf,
 *                           sum 0, or the sink's values).  Masked keys contribute nothing,
 *                           whatever the cache holds for them (NaN included).
 * options->atten_mask_stride  S, bytes per mask row; >= max_kv_len.
 * options->quant_scale2     device fp32 or NULL.  Non-NULL makes out an int8 (B, Nq, D) tensor:
 *                           out = saturate(round-half-even(o * quant_scale2[c] +
 *                           quant_offset2[c])) to [-128, 127], o the fp32 attention output and
 *                           c = h * D + d with quant2_per_channel = 1 (Nq * D values), c = 0
 *                           with quant2_per_channel = 0 (one value).
 * options->quant_offset2    device fp32, as many values as quant_scale2, or NULL (zero).
 * options->band             nonzero: FusedInferAttentionScore's band (sparseMode 4) for the one
 *                           query, at position L - 1 of a batch of length L: keys
 *                           L - 1 - pre_tokens .. L - 1 + next_tokens are visible (a sliding
 *                           window of W keys is pre_tokens = W - 1, next_tokens = 0).  Only
 *                           the window's tiles are read.  Values beyond +-2^30 are clamped;
 *                           pre_tokens + next_tokens < 0 is FIA_ERR_PARAM_INVALID.  A batch
 *                           with no key in the window gets the empty-row outputs.
 * options->q_len            s > 1: s query positions per batch (FusedInferAttentionScore runs
 *                           Q_S > 1 against a paged cache with blockTable / actualSeqLengths,
 *                           e.g. draft tokens of speculative decoding).  q and out are
 *                           (B, s, Nq, D) row-major (BSND), softmax max / sum / lse (B, s, Nq);
 *                           position i of batch b sits at key L_b - s + i and sees keys
 *                           t <= L_b - s + i (rightDownCausal; a position before the first key
 *                           gets the empty-row outputs).  The cache is read once for all s
 *                           positions.  In this build (Nq / Nkv) * s <= 16 (<= 8 with int8
 *                           KV), Nq * s <= 256, and neither atten_mask nor band with s > 1.
 *                           The workspace is fia_decode_workspace_size() with Nq * s in place
 *                           of Nq.
 * options == NULL behaves as fia_decode.  The workspace is fia_decode_workspace_size()
 * bytes, as for fia_decode.  Errors: an unknown layout or mode, the per-tensor mode
 * without int8 KV, a mask row shorter than max_kv_len, quant_offset2 without
 * quant_scale2, quant2_per_channel outside {0, 1}, or an empty band is FIA_ERR_PARAM_INVALID. */
typedef enum { FIA_KV_BNNBSD = 0, FIA_KV_BNBSH = 1 } fia_kv_layout;
typedef enum { FIA_AQ_PER_CHANNEL = 0, FIA_AQ_PER_TENSOR = 1 } fia_antiquant_mode;
typedef struct {
  int kv_layout;       /* fia_kv_layout */
  int antiquant_mode;  /* fia_antiquant_mode */
  float* softmax_lse;  /* device fp32 (B, Nq) or NULL */
  const uint8_t* atten_mask;   /* device (B, atten_mask_stride) bytes or NULL */
  int64_t atten_mask_stride;   /* bytes per mask row, >= max_kv_len */
  const float* quant_scale2;   /* device fp32, 1 or Nq * D values, or NULL (16-bit out) */
  const float* quant_offset2;  /* device fp32, as quant_scale2, or NULL */
  int quant2_per_channel;      /* 0: one value; 1: Nq * D values */
  int band;                    /* nonzero: keys L-1-pre_tokens .. L-1+next_tokens only */
  int64_t pre_tokens;
  int64_t next_tokens;
  int q_len;                   /* 0 or 1: one query per batch; s > 1: q and out (B, s, Nq, D) */
} fia_decode_options;

int fia_decode_ex(const void* q, fia_dtype q_dtype, const void* k_cache, const void* v_cache, fia_dtype kv_dtype,
                  const int32_t* block_table, int64_t bt_stride, const int64_t* actual_seq_lengths, int max_kv_len,
                  int B, int Nq, int Nkv, int D, int block_size, int64_t num_blocks, double scale,
                  const float* antiquant_scale, const float* antiquant_offset, const float* sink, void* out,
                  float* softmax_max, float* softmax_sum, int num_splits, void* workspace, size_t workspace_bytes,
                  fia_stream_t stream, const fia_decode_options* options);

/* Allocation-free variant of fia_decode.  The operator pages have no counterpart:
 * it exists for callers that cannot allocate device memory for the workspace --
 * plugins whose host application owns all device memory through its own allocator,
 * modules that may not call the CUDA allocator, and loops in which cudaMalloc's
 * possible device synchronisation is not allowed.  Arguments and results are those
 * of fia_decode without the workspace: the workspace is a fixed 16 MiB array in the
 * library's device memory (every GPU that loads the library holds it until exit).
 *   - Problems whose fia_decode_workspace_size exceeds 16 MiB return
 *     FIA_ERR_PARAM_INVALID (fia_last_error names the limit).
 *   - All calls on a device share the array, which keeps the last call's contents;
 *     nothing in it needs to start at zero.  Calls that overlap on the GPU (other
 *     streams, or unordered host threads) race on it: order them.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make it before any stream
 *     capture begins.
 *   - Nothing is allocated or freed by this call. */
int fia_decode_noalloc(const void* q, fia_dtype q_dtype, const void* k_cache, const void* v_cache,
                       fia_dtype kv_dtype, const int32_t* block_table, int64_t bt_stride,
                       const int64_t* actual_seq_lengths, int max_kv_len, int B, int Nq, int Nkv, int D,
                       int block_size, int64_t num_blocks, double scale, const float* antiquant_scale,
                       const float* antiquant_offset, const float* sink, void* out, float* softmax_max,
                       float* softmax_sum, int num_splits, fia_stream_t stream);

/* ------------------------------------------------------------------------ prefill
 * FusedInferAttentionScore (prefill mode Q_S > 1, sparseMode 3 rightDownCausal, TND);
 * aclnnFlashAttentionScoreV4 (TND, cumulative actual_seq_qlen, zero-length sequences).
 *
 *   For sequence b with Lq = cu_seqlens_q[b+1] - cu_seqlens_q[b] queries and
 *   Lkv = cu_seqlens_kv[b+1] - cu_seqlens_kv[b] keys, query i sees key j iff mask == 0, or
 *   mask == 3 and j <= i + Lkv - Lq (rightDownCausal; lower-triangular when Lq == Lkv).
 *   Outputs as for decode, per (token, head).
 *
 * q, out           device (T, Nq, D) row-major, dtype FIA_BF16 or FIA_F16, 16-byte aligned.
 * k, v             device (Tkv, Nkv, D) row-major, same dtype, 16-byte aligned.
 * cu_seqlens_q/kv  device int64 (B + 1), cu[0] = 0, non-decreasing, cu[B] = T (resp. Tkv).
 * max_seqlen_q/kv  host upper bounds of the per-sequence lengths (max_seqlen_kv <= 2^20 here).
 * D                64 or 128 in this build; Nq % Nkv == 0; max_seqlen_q must bound every Lq.
 * mask             0 (none) or 3 (rightDownCausal); 4 (band) through fia_prefill_ex.
 * sink             device fp32 (Nq) or NULL.
 * softmax_max/sum  device fp32 (T, Nq) or NULL.
 * workspace        device, at least fia_prefill_workspace_size() bytes, 256-byte aligned.
 */
int fia_prefill_workspace_size(int B, int Nq, int Nkv, int D, int max_seqlen_q, size_t* bytes);

int fia_prefill(const void* q, const void* k, const void* v, fia_dtype dtype, const int64_t* cu_seqlens_q,
                const int64_t* cu_seqlens_kv, int B, int64_t T, int64_t Tkv, int max_seqlen_q, int max_seqlen_kv,
                int Nq, int Nkv, int D, double scale, int mask, const float* sink, void* out, float* softmax_max,
                float* softmax_sum, void* workspace, size_t workspace_bytes, fia_stream_t stream);

/* fia_prefill with the band mask (FusedInferAttentionScore sparseMode 4 with preTokens /
 * nextTokens) and keys in a paged cache (FusedInferAttentionScore PagedAttention: blockTable,
 * blockSize, actualSeqLengthsKv; a chunk of queries against a long cached context).
 * Arguments as for fia_prefill; mask may also be 4 (band), which needs options:
 *
 *   query i of a sequence sees key j iff
 *     i + (Lkv - Lq) - pre_tokens <= j <= i + (Lkv - Lq) + next_tokens,
 *   the band around the rightDownCausal diagonal (pre_tokens = large, next_tokens = 0 is
 *   mask 3; pre_tokens = W - 1, next_tokens = 0 a causal sliding window of W keys).  Values
 *   beyond +-2^30 are clamped; pre_tokens + next_tokens < 0 (a band that holds no key, which
 *   the pages forbid) is FIA_ERR_PARAM_INVALID.  Rows with no key in the band get the
 *   empty-row outputs.  Only key tiles that meet a query tile's band are read.
 *
 * options->block_table non-NULL: k and v are paged pools instead of TND tensors --
 *   (num_blocks, Nkv, block_size, D) with kv_layout FIA_KV_BNNBSD, or (num_blocks,
 *   block_size, Nkv * D) with FIA_KV_BNBSH -- key j of sequence b is row j % block_size of
 *   block block_table[b * bt_stride + j / block_size]; sequence b has seq_lens_kv[b] keys
 *   (device int64 (B), clamped to [0, max_seqlen_kv] with FIA_STATUS_LENGTH_CLAMPED);
 *   cu_seqlens_kv and Tkv are not used.  block_size is a multiple of 16 up to 512
 *   (aclnnIncreFlashAttentionV3, "Constraints / page attention"); a key tile of 128 keys is
 *   read in gcd(block_size, 128)-row pieces, one block each.  max_seqlen_kv <= bt_stride *
 *   block_size.  A block
 *   index outside [0, num_blocks) raises FIA_STATUS_BAD_BLOCK_INDEX.  Queries stay TND: a
 *   sequence's Lq queries are its last Lq positions (the rightDownCausal diagonal).  Rows
 *   of a sequence's last block past its length, and blocks past it, may hold anything
 *   (NaN included): they are masked in the scores and zeroed in the values.
 *
 * options->quant_scale2 non-NULL: out is an int8 (T, Nq, D) tensor, the output quantised
 *   as fia_decode_ex quantises it (aclnnIncreFlashAttentionV3 quantScale2 / quantOffset2;
 *   FusedInferAttentionScore takes the same pair in both of its modes):
 *   out = saturate(round-half-even(o * quant_scale2[c] + quant_offset2[c])) to [-128, 127],
 *   o the fp32 attention output, c = h * D + d with quant2_per_channel = 1 (Nq * D values),
 *   c = 0 with quant2_per_channel = 0 (one value); quant_offset2 NULL is zero.
 *   quant_offset2 without quant_scale2, or quant2_per_channel outside {0, 1}, is
 *   FIA_ERR_PARAM_INVALID.
 *
 * options may be NULL for masks 0 and 3 without paging or quantised output (NULL with
 * mask 4 is FIA_ERR_PARAM_NULLPTR). */
typedef struct {
  int64_t pre_tokens;           /* mask 4 only */
  int64_t next_tokens;          /* mask 4 only */
  const int32_t* block_table;   /* NULL: k, v are TND (Tkv, Nkv, D) */
  int64_t bt_stride;
  const int64_t* seq_lens_kv;   /* device int64 (B) */
  int block_size;
  int64_t num_blocks;
  int kv_layout;                /* fia_kv_layout */
  const float* quant_scale2;    /* device fp32, 1 or Nq * D values, or NULL (16-bit out) */
  const float* quant_offset2;   /* device fp32, as quant_scale2, or NULL */
  int quant2_per_channel;       /* 1: Nq * D values, 0: one value */
} fia_prefill_options;

int fia_prefill_ex(const void* q, const void* k, const void* v, fia_dtype dtype, const int64_t* cu_seqlens_q,
                   const int64_t* cu_seqlens_kv, int B, int64_t T, int64_t Tkv, int max_seqlen_q, int max_seqlen_kv,
                   int Nq, int Nkv, int D, double scale, int mask, const float* sink, void* out, float* softmax_max,
                   float* softmax_sum, void* workspace, size_t workspace_bytes, fia_stream_t stream,
                   const fia_prefill_options* options);

/* ---------------------------------------------------------- ring_attention_update
 * aclnnRingAttentionUpdate ("功能说明 / 计算公式").  Per row r and head n:
 *   m = max(pm, cm);  wp = ps e^{pm - m};  wc = cs e^{cm - m};  sum = wp + wc;
 *   out = (prev_out wp + cur_out wc) / sum.
 * The page prints the formula without the ps / cs factors on the outputs and without cs in
 * the sum; that form is exact only when both sums are 1.  This library applies the sums,
 * the form under which merging the partials of any split gives the unsplit result.  A side
 * with max = -inf weighs 0; if both do, out = 0, max = -inf, sum = 0.
 *
 * rows             T for TND, or S * B for SBH (the two layouts are the same elementwise).
 * prev_out, cur_out, out   device (rows, N, D) in out_dtype (FIA_F32, FIA_F16, FIA_BF16),
 *                  16-byte aligned.  D % 8 == 0 and D <= 768; N <= 256.
 * prev/cur_max, prev/cur_sum, max_out, sum_out   device fp32 (rows, N); one value per (row,
 *                  head) (the pages' trailing axis of 8 equal copies is not stored).
 * Outputs may alias the prev_* (or cur_*) inputs, so an n-way fold can run in place.
 */
int ring_attention_update(const void* prev_out, const float* prev_max, const float* prev_sum, const void* cur_out,
                          const float* cur_max, const float* cur_sum, fia_dtype out_dtype, int64_t rows, int N,
                          int D, void* out, float* max_out, float* sum_out, fia_stream_t stream);

/* ------------------------------------------------------------------------- probes
 * Test hooks for the bit-exact parts of the decode path.  The pages have no
 * counterpart; they exist so that tests can compare the exact integer and
 * floating-point steps with the oracle.
 *
 * fia_debug_dequant: out[i] = (codes[i] - offset[i]) * scale[i] in fp32 with two roundings,
 *   through the element-wise antiquant function of the CUDA-core decode kernel, the one that
 *   serves int8 KV with D = 64.  The int8 tensor-core kernel (D = 128) never forms a
 *   dequantised element: it applies the affine map to the query and to the output, and its
 *   exact steps have the two probes below.  All pointers device.
 * fia_debug_gather: copies the K rows of the first L_b tokens of (b, hkv) into dst (device,
 *   L_b * D elements of kv_dtype, row-major) through the attention kernel's block-table walk,
 *   tensor-map tile loads and swizzled addressing.  Other arguments as for fia_decode.
 */
int fia_debug_dequant(const int8_t* codes, const float* scale, const float* offset, int64_t n, float* out,
                      fia_stream_t stream);

int fia_debug_gather(const void* k_cache, fia_dtype kv_dtype, const int32_t* block_table, int64_t bt_stride,
                     const int64_t* actual_seq_lengths, int max_kv_len, int B, int Nkv, int D, int block_size,
                     int64_t num_blocks, int b, int hkv, void* dst, fia_stream_t stream);

/* The int8 tensor-core decode kernel (int8 KV, D = 128) computes a score as
 *   sum_d q_d (x_td - o_d) s_d = sum_d (q_d s_d) x_td - sum_d q_d s_d o_d
 * with the codes x_td entering the tensor-core product as fp16 and q'_d = q_d s_d as an fp16
 * pair hi + lo (aclnnIncreFlashAttentionV3, "antiquantScale / antiquantOffset").  These probes
 * run those steps through the kernel's own device functions.
 *
 * fia_debug_i8_codes: out[i] = the binary16 bit pattern the kernel's converter warps produce
 *   for codes[i]; n % 4 == 0, codes 4-byte and out 8-byte aligned.  The conversion is exact.
 * fia_debug_i8_qprep: the query operand of every (b, kv head) as the plan kernel prepares it,
 *   read back through the kernel's shared-memory layout.  q (B, Nq, 128) as for fia_decode;
 *   antiquant_scale / offset (2, Nkv, 128) (the key half [0] is used; offset may be NULL).
 *   blocks: device scratch of at least B * Nkv * 8320 bytes, 256-byte aligned (the blocks in
 *   the kernel's layout).  q_hi, q_lo: device (B, Nkv, 16, 128) binary16 bit patterns of the
 *   two parts of q'_d 2^e for query head hkv * G + g in row g (rows g >= G are zero), e the
 *   power of two, chosen per row, that puts the row's largest |q'_d| in [2^14, 2^15).  kq_nq: device
 *   (B, Nkv, 16, 2) fp32: kq = scale log2(e) 2^-e and nq = -scale log2(e) sum_d q'_d o_d, so
 *   that the score in log2 units is (sum_d (hi_d + lo_d) x_td) kq + nq.
 */
int fia_debug_i8_codes(const int8_t* codes, int64_t n, uint16_t* out, fia_stream_t stream);

int fia_debug_i8_qprep(const void* q, fia_dtype q_dtype, const float* antiquant_scale, const float* antiquant_offset,
                       int B, int Nq, int Nkv, double scale, void* blocks, size_t blocks_bytes, uint16_t* q_hi,
                       uint16_t* q_lo, float* kq_nq, fia_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FIA_H_ */
