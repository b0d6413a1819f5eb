// decode_common.cuh -- pieces shared by the two decode attention kernels: the work-item
// format written by the plan kernel, the direct output of a (batch, kv-head) segment
// made of one work item, and the launch with programmatic dependent launch.
#pragma once

#include "fia_device.cuh"

namespace fia {

// Tensor-map coordinates of the tile row of token t of kv head hkv in pool block blk: the
// row, and the column of the head's first channel.  Layout 0, (num_blocks, Nkv,
// block_size, D): a row of D channels per (block, head, token).  Layout 1, (num_blocks,
// block_size, Nkv * D): a row of Nkv * D channels per (block, token), the head selecting a
// column range (aclnnIncreFlashAttentionV3, "Constraints / page attention").
struct KvCoord {
  int32_t x0, row;
};
__device__ __forceinline__ KvCoord kv_coord(const DecodeParams& p, int32_t blk, int t, int hkv) {
  KvCoord c;  // (rows < 2^31 is checked by the host)
  c.x0 = hkv * p.kv_x_h;
  c.row = blk * p.kv_row_blk + hkv * p.kv_row_h + t % p.block_size;
  return c;
}

// Work item {b, kv head | (chunk count of the segment) << 16, first token, last token + 1}.
// A segment's chunks start at its span's base, a multiple of 128 tokens, so the tiles of
// every chunk are aligned; the first chunk starts at the span's first key (which the
// producer rounds down to its tile, masking the keys below it).
struct DecodeItem {
  int b, hkv, nch, t_begin, t_end;
};

__device__ __forceinline__ DecodeItem decode_item(int4 d) {
  DecodeItem it;
  it.b = d.x;
  it.hkv = d.y & 0xffff;
  it.nch = (unsigned)d.y >> 16;
  it.t_begin = d.z;
  it.t_end = d.w;
  return it;
}

// The keys [lo, end) the query of a batch of length L sees, and base = lo rounded down to a
// 128-token tile, where the batch's chunks start: [0, L) without a window; with the band
// (FusedInferAttentionScore preTokens / nextTokens, one query at position L - 1) keys
// L - 1 - win_pre .. L - 1 + win_next.  An empty window is [0, 0).
struct DecodeSpan {
  int lo, end, base;
};
__device__ __forceinline__ DecodeSpan decode_span(const DecodeParams& p, int L) {
  DecodeSpan s{0, L, 0};
  if (p.windowed) {
    s.lo = max(L - 1 - p.win_pre, 0);
    s.end = min(L, L + p.win_next);
    if (s.end <= s.lo) s.lo = s.end = 0;
    s.base = s.lo & ~(kDecodeTileTC - 1);
  }
  return s;
}
// chunks of a span
__device__ __forceinline__ int span_chunks(const DecodeSpan& s, int C) { return (s.end - s.base + C - 1) / C; }
// item j of a span: first and last + 1 token
__device__ __forceinline__ int4 span_item(const DecodeSpan& s, int C, int b, int hkv, int nch, int j) {
  return make_int4(b, hkv | (nch << 16), j == 0 ? s.lo : s.base + j * C, min(s.end, s.base + (j + 1) * C));
}

// Work items for the producer warp of a persistent CTA.  Slots are claimed from the
// global counter one item ahead and resolved through the execution order (longest
// first), so that the latency of the claim and of the two dependent loads overlaps
// the current item's tiles.  All lanes call every member; lane 0 holds the state.
struct ItemQueue {
  int n_items, claimed, next;
  int4 next_desc;

  __device__ __forceinline__ void start(const DecodeParams& p, int lane) {
    n_items = *p.ws.n_items;
    if (lane == 0) resolve(p, atomicAdd(p.ws.counter, 1));
  }
  __device__ __forceinline__ void resolve(const DecodeParams& p, int slot) {
    next = slot < n_items ? p.ws.order[slot] : -1;
    next_desc = next >= 0 ? p.ws.items[next] : make_int4(0, 0, 0, 0);
  }
  // The next item (-1 when the work is exhausted) and its descriptor; claims the
  // slot after it.
  __device__ __forceinline__ int pop(const DecodeParams& p, int lane, int4* desc) {
    const int item = __shfl_sync(0xffffffffu, next, 0);
    desc->x = __shfl_sync(0xffffffffu, next_desc.x, 0);
    desc->y = __shfl_sync(0xffffffffu, next_desc.y, 0);
    desc->z = __shfl_sync(0xffffffffu, next_desc.z, 0);
    desc->w = __shfl_sync(0xffffffffu, next_desc.w, 0);
    if (item >= 0 && lane == 0) claimed = atomicAdd(p.ws.counter, 1);
    return item;
  }
  // Resolves the claimed slot; call once per popped item, after its first tile is issued.
  __device__ __forceinline__ void prefetch(const DecodeParams& p, int lane) {
    if (lane == 0) resolve(p, claimed);
  }
};

// Output of a segment made of one item, straight from the item's running state:
// acc = sum_t 2^{s_t - m} v_t (not normalised), l = sum_t 2^{s_t - m}, m in log2 units.
// Returns the value to store for one output channel; *M_out / *W_out receive the
// softmax max (log2 units) and sum for the head.
// attenMask: a nonzero byte at (b, t) removes key t of batch b from the softmax.
__device__ __forceinline__ bool key_masked(const DecodeParams& p, int b, int t) {
  return p.atten_mask != nullptr && __ldg(p.atten_mask + (int64_t)b * p.mask_stride + t) != 0;
}

__device__ __forceinline__ float single_item_output(float acc, float m, float l, const float* sink, int h,
                                                    float* M_out, float* W_out) {
  const float sink2 = sink ? sink[h] * kLog2e : -INFINITY;
  const float M = fmaxf(m, sink2);
  float W = 0.f, scale = 0.f;
  if (M != -INFINITY) {
    scale = (m == -INFINITY) ? 0.f : exp2f(m - M);
    W = l * scale;
    if (sink) W += exp2f(sink2 - M);
  }
  *M_out = M;
  *W_out = W;
  return W > 0.f ? acc * scale / W : 0.f;
}

// Launches `kern` with programmatic stream serialisation, so that it may start while the
// preceding kernel on the stream still runs; the kernel calls griddep_wait() before it
// reads anything that kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), int grid, int threads, size_t smem, cudaStream_t stream,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

}  // namespace fia
