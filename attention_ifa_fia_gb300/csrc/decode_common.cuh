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

// Row of virtual head v (position v / G, query head hkv * G + v % G) of batch b in the
// (B, qs, Nq) rows of q, out, softmax max and sum; and its query head.
__device__ __forceinline__ int64_t q_row(const DecodeParams& p, int b, int hkv, int v) {
  if (p.qs == 1) return (int64_t)b * p.Nq + hkv * p.G + v;
  const int i = v / p.G;
  return ((int64_t)b * p.qs + i) * p.Nq + hkv * p.G + (v - i * p.G);
}
__device__ __forceinline__ int q_head(const DecodeParams& p, int hkv, int v) {
  return hkv * p.G + (p.qs == 1 ? v : v % p.G);
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

constexpr int kPlanMaxTiles = 64;  // size classes of the execution order (tiles per item, capped)

// A batch's key count from the device array, clamped to [0, max_kv_len] (flag: raise the
// status bit if it was outside).
__device__ __forceinline__ int clamp_len(const DecodeParams& p, int b, bool flag) {
  const int64_t raw = p.seq_lens[b];
  if (flag && (raw < 0 || raw > p.max_kv_len)) raise_status(p.status, kStatusLengthClamped);
  return (int)(raw < 0 ? 0 : (raw > p.max_kv_len ? p.max_kv_len : raw));
}

// Rows of a batch with no visible key: out 0, max -inf and sum 0, or with a sink
// max = sink and sum 1 (no work item covers them).
__device__ inline void write_empty_batch(const DecodeParams& p, int b) {
  for (int h = 0; h < p.Nq; ++h) {
    if (p.softmax_max) p.softmax_max[(int64_t)b * p.Nq + h] = p.sink ? p.sink[h] : -INFINITY;
    if (p.softmax_sum) p.softmax_sum[(int64_t)b * p.Nq + h] = p.sink ? 1.f : 0.f;
  }
  uint4* o = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + (int64_t)b * p.Nq * p.D * 2);
  for (int i = 0; i < p.Nq * p.D * 2 / 16; ++i) o[i] = make_uint4(0u, 0u, 0u, 0u);
}

// ----------------------------------------------------------------------------
// In-kernel schedule.  With p.fused_plan the attention kernel plans for itself, with no
// plan launch and no claim counter: every CTA derives from the lengths, in shared memory,
// the same longest-first order of the work items -- first every full chunk (batch, kv
// head, chunk in order), then each batch's last chunk, batches sorted by that chunk's
// tiles, most first -- and takes the slots c, 2G - 1 - c, 2G + c, 4G - 1 - c, ... of it
// (a snake over the G CTAs).  For items ordered longest first this balances the CTAs as
// well as claiming items from a counter (the per-CTA tile counts come out the same), and
// saves the plan launch, its completion and the first claim's round trips.
struct FusedPlan {
  int lo[kFusedPlanMaxB], end[kFusedPlanMaxB];  // span of keys [lo, end) of each batch
  int nch[kFusedPlanMaxB];                       // chunks (items per kv head) of each batch
  int lastk[kFusedPlanMaxB];                     // tiles of each batch's last chunk (0: no key)
  int nat[kFusedPlanMaxB + 1];                   // first item of batch b in (b, h, j) order
  int full[kFusedPlanMaxB + 1];                  // first full-chunk slot of batch b
  int last_ord[kFusedPlanMaxB];                  // batches with keys, longest last chunk first
  int cls[kPlanMaxTiles + 2];                    // batches per last-chunk size, then class starts
  int n_full, n_items;
};

// Builds the schedule; called by every thread of the CTA (nthreads of them), with
// __syncthreads inside.  CTA 0 also writes the rows of batches without keys (unless every
// segment goes through the merge kernel), raises the clamped-length flag, and writes each
// batch's first item index for the merge kernel.
__device__ inline void fused_plan_build(const DecodeParams& p, FusedPlan& fp, int tid, int nthreads) {
  const int C = p.chunk_tokens, lane = tid & 31, warp = tid >> 5;
  const bool cta0 = blockIdx.x == 0;
  for (int i = tid; i < kPlanMaxTiles + 2; i += nthreads) fp.cls[i] = 0;
  __syncthreads();
  for (int b = tid; b < p.B; b += nthreads) {
    const DecodeSpan sp = decode_span(p, clamp_len(p, b, cta0));
    const int nch = span_chunks(sp, C);
    fp.lo[b] = sp.lo;
    fp.end[b] = sp.end;
    fp.nch[b] = nch;
    const int lk = nch ? min((sp.end - sp.base - (nch - 1) * C + kDecodeTileTC - 1) / kDecodeTileTC, kPlanMaxTiles) : 0;
    fp.lastk[b] = lk;
    if (nch) atomicAdd(&fp.cls[lk], 1);
    if (!nch && cta0 && !p.partials_only) write_empty_batch(p, b);
  }
  __syncthreads();
  if (warp == 0) {
    // prefix sums over the batches, 8 consecutive batches per lane (B <= 256)
    int nat_run = 0, full_run = 0, nat_l[8], full_l[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int b = lane * 8 + i;
      const int nch = b < p.B ? fp.nch[b] : 0;
      nat_l[i] = nat_run;
      full_l[i] = full_run;
      nat_run += nch * p.Nkv;
      full_run += (nch ? nch - 1 : 0) * p.Nkv;
    }
    // and the class starts, largest class first: lane l holds classes 64 - 2l and 63 - 2l
    const int k0 = kPlanMaxTiles - 2 * lane, k1 = k0 - 1;
    const int c0 = fp.cls[k0], c1 = k1 >= 1 ? fp.cls[k1] : 0;
    int nat_x = nat_run, full_x = full_run, cls_x = c0 + c1;  // inclusive warp scans
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, nat_x, o), f = __shfl_up_sync(0xffffffffu, full_x, o);
      const int c = __shfl_up_sync(0xffffffffu, cls_x, o);
      if (lane >= o) { nat_x += a; full_x += f; cls_x += c; }
    }
    __syncwarp();
    fp.cls[k0] = cls_x - c0 - c1;
    if (k1 >= 1) fp.cls[k1] = cls_x - c1;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int b = lane * 8 + i;
      if (b <= p.B) {
        fp.nat[b] = nat_x - nat_run + nat_l[i];
        fp.full[b] = full_x - full_run + full_l[i];
      }
    }
    if (lane == 31) {
      fp.nat[p.B] = nat_x;
      fp.full[p.B] = full_x;
      fp.n_full = full_x;
      fp.n_items = nat_x;  // every item: the full chunks and one last chunk per batch and kv head
    }
    __syncwarp();
    // batches with keys in order of their last chunk's tiles (descending), by index within a
    // class: each group of equal sizes among 32 batches takes consecutive places
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int b = b0 + lane;
      const int k = (b < p.B) ? fp.lastk[b] : 0;
      const unsigned peers = __match_any_sync(0xffffffffu, k);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      if (k > 0) fp.last_ord[fp.cls[k] + rank] = b;
      __syncwarp();
      if (k > 0 && rank == 0) fp.cls[k] += __popc(peers);
      __syncwarp();
    }
    if (cta0)
      for (int b = lane; b <= p.B; b += 32) p.ws.seg_base[b] = fp.nat[b];
  }
  __syncthreads();
}

// The work item at slot `slot` of the schedule: its descriptor and its index in (b, h, j)
// order (where its partial goes).
__device__ inline int fused_plan_item(const DecodeParams& p, const FusedPlan& fp, int slot, int4* desc) {
  const int C = p.chunk_tokens;
  int b, h, j, nch;
  if (slot < fp.n_full) {  // a full chunk: the last batch whose first full slot is <= slot
    int lo = 0, hi = p.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (fp.full[mid] <= slot) lo = mid;
      else hi = mid;
    }
    b = lo;
    nch = fp.nch[b];
    const int r = slot - fp.full[b];
    h = r / (nch - 1);
    j = r - h * (nch - 1);
  } else {  // a last chunk
    const int i = slot - fp.n_full;
    b = fp.last_ord[i / p.Nkv];
    h = i % p.Nkv;
    nch = fp.nch[b];
    j = nch - 1;
  }
  const DecodeSpan sp{fp.lo[b], fp.end[b], fp.lo[b] & ~(kDecodeTileTC - 1)};
  *desc = span_item(sp, C, b, h, nch, j);
  return fp.nat[b] + h * nch + j;
}

// Slot of round r for this CTA in the snake over G CTAs.
__device__ __forceinline__ int fused_plan_slot(int r, int G) {
  return r * G + ((r & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x);
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
