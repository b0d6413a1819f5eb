// decode.cu -- paged GQA decode attention (query S = 1) on CUDA cores.
//
// What it computes (aclnnIncreFlashAttentionV3, "Function" and "Constraints /
// page attention"; aclnnFlashAttentionScoreV4, sink formula): for each batch b
// and query head h, out = softmax(scale * q K^T) V over the first L_b tokens of
// the paged cache, token t read from block block_table[b][t / bs], row t % bs of
// the (blocknum, KV_N, blocksize, D) pool, with kv head h / (Nq / Nkv).
//
// Structure (three launches on the caller's stream, each a programmatic dependent
// launch of the one before, so that launches and prologues overlap):
//   1. plan      -- one CTA splits every (b, kv-head) sequence into work items of
//                   `chunk_tokens` tokens, writes their execution order (longest
//                   first) and resets the work counter; rows of empty sequences are
//                   written here.  For int8 KV with D = 128, further CTAs prepare the
//                   query operand of the tensor-core kernel (decode_i8.cuh).
//   2. attention -- persistent CTAs (one per SM) claim items from the counter
//                   (ItemQueue, decode_common.cuh).  Three variants: tcgen05 for
//                   16-bit KV (decode_tc.cu), tcgen05 for int8 KV with D = 128
//                   (decode_i8tc.cu), and the CUDA-core kernel of this file for the
//                   remaining int8 shapes.  Here warp 8 is the producer: it reads the
//                   block table and issues TMA tile loads (2-D tensor maps over the
//                   pool, 128- or 64-byte swizzle) of K and V into a 4-stage mbarrier
//                   ring, plus the item's G query rows by a 1-D bulk copy.  Warps 0-7
//                   compute, for the whole GQA group at once: scores from
//                   register-resident q, a warp-shuffle online softmax (max and sum),
//                   and P.V.  A segment of one item writes the final output directly;
//                   otherwise each item leaves a normalised partial (o, max, sum).
//   3. merge     -- one CTA per (b, kv head) with two or more items folds the
//                   partials in order by the RingAttentionUpdate rule, adds the sink
//                   once and writes out, softmax max and sum.
// Scores are kept in log2 units (scale * log2 e folded into the dot product) and
// converted back to the natural-exp domain for the max output.
#include "decode_common.cuh"
#include "decode_i8.cuh"

namespace fia {
namespace {

constexpr int kTT = kDecodeTile;
constexpr int kConsumerWarps = kDecodeConsumers / 32;
constexpr int kThreads = kDecodeConsumers + 32;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kBarConsumers = 1;  // named barrier id for the 256 math threads
constexpr int kAqHeads = 8;       // kv heads whose antiquant parameters stay in shared memory

template <int KVT, int D, int GP>
struct Cfg {
  static constexpr int kElem = (KVT == kI8) ? 1 : 2;
  static constexpr int kRowBytes = D * kElem;
  static constexpr int kBoxBytes = kRowBytes < 128 ? kRowBytes : 128;  // swizzle span of one box
  static constexpr int kNumBoxes = kRowBytes / kBoxBytes;
  static constexpr uint32_t kSwzMask = kBoxBytes == 128 ? 7u : 3u;
  static constexpr int kTileBytes = kTT * kRowBytes;  // K (or V) of one stage
  // score mapping: each thread owns E channels of one token; P threads per token
  static constexpr int E = (64 / GP) < D ? (64 / GP) : D;
  static constexpr int P = D / E;
  static constexpr int PB = (E * kElem) < 16 ? (E * kElem) : 16;  // bytes per shared load
  static constexpr int NPC = E * kElem / PB;                      // loads per token
  static constexpr int PE = PB / kElem;                           // elements per load
  static constexpr int TPP = kDecodeConsumers / P;                // tokens per pass
  static constexpr int PASSES = (kTT + TPP - 1) / TPP;
  static constexpr bool kPartsMinor = P >= 8;
  static constexpr int TW = 32 / P;  // tokens per warp per pass
  static constexpr int LOGP = (P >= 32) ? 5 : (P >= 16) ? 4 : (P >= 8) ? 3 : (P >= 4) ? 2 : (P >= 2) ? 1 : 0;
  static constexpr int LOGG = (GP >= 8) ? 3 : (GP >= 4) ? 2 : (GP >= 2) ? 1 : 0;
  static constexpr int MS = kPartsMinor ? 1 : TW;  // lane stride between parts of a token
  // P.V mapping: each thread owns 8 channels (one chunk) for a group of tokens
  static constexpr int EV = 8;
  static constexpr int CH = D / EV;
  static constexpr int NTG = kDecodeConsumers / CH;
  static constexpr int TPG = kTT / NTG;
  static_assert(LOGG <= LOGP || P == 1, "score reduction needs at least G lanes per token");
  static_assert(kTT % NTG == 0, "token groups must tile the stage");
};

struct __align__(16) StageMeta {
  int b, hkv, tok0, n;  // tile start token and valid tokens
  int item, first, last, nch;  // nch: items of this (b, kv head) segment
  int nlo, qlim, pad1, pad2;   // tokens below tok0 + nlo lie before the window (masked); query
                               // position i sees tokens up to qlim + i
};

template <int KVT, int D, int GP>
struct Smem {
  using C = Cfg<KVT, D, GP>;
  alignas(1024) uint8_t kv[kDecodeStages][2][C::kTileBytes];  // [stage][K|V]
  alignas(16) uint16_t q[kDecodeStages][GP * D];              // query rows of the item (storage bits)
  float red[kConsumerWarps][GP * D];                          // end-of-item reduction
  float s[GP][kTT];                                           // scores (log2 units)
  float p[kTT][GP];                                           // probabilities
  float alpha[GP], m_run[GP], l_run[GP];
  // int8: [k_scale, k_offset, v_scale, v_offset][hkv * D + d] for up to kAqHeads kv heads
  float aq[KVT == kI8 ? 4 : 1][KVT == kI8 ? D * kAqHeads : 1];
  StageMeta meta[kDecodeStages];
  uint64_t full[kDecodeStages], empty[kDecodeStages];
};

// Pool row of token t of (b, hkv): block_table entry, then the row inside the block.
// Load one 16- or 8-byte piece of a swizzled tile row.
template <int PB>
__device__ __forceinline__ void load_piece(uint32_t addr, uint32_t (&w)[4]) {
  if constexpr (PB == 16) {
    uint4 v = lds128(addr);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else {
    uint2 v = lds64(addr);
    w[0] = v.x; w[1] = v.y; w[2] = 0; w[3] = 0;
  }
}

// Widen element e of a loaded piece to fp32 (int8: exact code, not yet dequantised).
template <int KVT>
__device__ __forceinline__ float piece_elem(const uint32_t (&w)[4], int e) {
  if constexpr (KVT == kBF16) return (e & 1) ? bf16hi(w[e >> 1]) : bf16lo(w[e >> 1]);
  else if constexpr (KVT == kF16) return (e & 1) ? f16hi(w[e >> 1]) : f16lo(w[e >> 1]);
  else return i8_to_f32(w[e >> 2], e & 3);
}

__device__ __forceinline__ float q_elem(const uint16_t* q, int idx, int q_dtype) {
  const uint32_t u = q[idx];
  return q_dtype == kBF16 ? __uint_as_float(u << 16) : __half2float(__ushort_as_half((unsigned short)u));
}

// ------------------------------------------------------------------- plan
constexpr int kPlanSmemB = 4096;  // batches whose item offsets and order slots fit in shared memory

__global__ void __launch_bounds__(1024) decode_plan_kernel(DecodeParams p) {
  // Launched as a dependent of whatever precedes it on the stream (often the previous
  // call's merge), so that its launch overlaps that kernel's end: nothing is read or
  // written before the preceding work is complete.
  griddep_wait();
  griddep_launch_dependents();  // the attention kernel may begin its prologue
  if (blockIdx.x > 0) {  // int8 tensor-core path: q' blocks, one warp per (b, kv head, padded row)
    const int64_t R = (int64_t)(blockIdx.x - 1) * 32 + (threadIdx.x >> 5);
    if (R < (int64_t)p.B * p.Nkv * kI8Heads) i8_qprep_row(p, R, threadIdx.x & 31);
    return;
  }
  // When B <= kPlanSmemB: sbase[B + 1] item offsets, then fpos[B] and tpos[B], the
  // first execution-order slots of each batch's full chunks and of its last chunks, then
  // send[B] and slo[B], the end and first key of each batch's span (its clamped length,
  // windowed by a band; read from global memory once, not in every pass).
  extern __shared__ int sbase[];
  __shared__ int warp_tot[32];
  __shared__ int carry;
  __shared__ int bucket[kPlanMaxTiles + 1];  // items per size (tiles), then the next free slot
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool in_smem = p.B <= kPlanSmemB;
  int* send = sbase + 3 * p.B + 1;
  int* slo = send + p.B;
  if (tid == 0) carry = 0;
  __syncthreads();
  const int C = p.chunk_tokens;
  for (int b0 = 0; b0 < p.B; b0 += 1024) {
    const int b = b0 + tid;
    int nch = 0;
    DecodeSpan sp{0, 0, 0};
    if (b < p.B) {
      sp = decode_span(p, clamp_len(p, b, true));
      if (in_smem) {
        send[b] = sp.end;
        slo[b] = sp.lo;
      }
      nch = span_chunks(sp, C);
      if (nch == 0 && !p.partials_only) write_empty_batch(p, b);
    }
    const int cnt = nch * p.Nkv;
    int x = cnt;  // inclusive warp scan, then across warps
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int t = warp_tot[lane];
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, t, o);
        if (lane >= o) t += y;
      }
      warp_tot[lane] = t;
    }
    __syncthreads();
    const int base = carry + (warp ? warp_tot[warp - 1] : 0) + x - cnt;
    if (b < p.B) {
      p.ws.seg_base[b] = base;
      if (in_smem) sbase[b] = base;
      if (!in_smem)  // large batch counts: each thread lists its own batch's items
        for (int h = 0; h < p.Nkv; ++h)
          for (int j = 0; j < nch; ++j)
            p.ws.items[base + h * nch + j] = span_item(sp, C, b, h, nch, j);
    }
    __syncthreads();
    if (tid == 1023) carry = base + cnt;
    __syncthreads();
  }
  const int total = carry;
  if (in_smem) {
    // Execution order, longest first (a persistent CTA that takes a long item last
    // would finish late): a counting sort of the items by their number of tiles.
    // Full chunks all have kt = C / 128 tiles; the last chunk of a batch has
    // ceil((end - base - (nch - 1) C) / 128) for its span [base, end).  Slots inside a size class are claimed in any
    // order, which changes only the order in which CTAs pick up the items.
    int* fpos = sbase + p.B + 1;
    int* tpos = fpos + p.B;
    const int kt = min(C / kDecodeTileTC, kPlanMaxTiles);  // larger items share the top class
    for (int k = tid; k <= kPlanMaxTiles; k += blockDim.x) bucket[k] = 0;
    if (tid == 0) sbase[p.B] = total;
    __syncthreads();
    for (int b = tid; b < p.B; b += blockDim.x) {
      const int nch = (sbase[b + 1] - sbase[b]) / p.Nkv;
      if (nch == 0) continue;
      const int last = send[b] - (slo[b] & ~(kDecodeTileTC - 1)) - (nch - 1) * C;  // tokens of the last chunk
      atomicAdd(&bucket[kt], (nch - 1) * p.Nkv);
      atomicAdd(&bucket[min((last + kDecodeTileTC - 1) / kDecodeTileTC, kPlanMaxTiles)], p.Nkv);
    }
    __syncthreads();
    if (tid == 0) {  // first slot of each size class, largest class first
      int run = 0;
      for (int k = kPlanMaxTiles; k >= 1; --k) {
        const int c = bucket[k];
        bucket[k] = run;
        run += c;
      }
    }
    __syncthreads();
    for (int b = tid; b < p.B; b += blockDim.x) {
      const int nch = (sbase[b + 1] - sbase[b]) / p.Nkv;
      if (nch == 0) continue;
      const int last = send[b] - (slo[b] & ~(kDecodeTileTC - 1)) - (nch - 1) * C;
      fpos[b] = atomicAdd(&bucket[kt], (nch - 1) * p.Nkv);
      tpos[b] = atomicAdd(&bucket[min((last + kDecodeTileTC - 1) / kDecodeTileTC, kPlanMaxTiles)], p.Nkv);
    }
    __syncthreads();
    for (int i = tid; i < total; i += blockDim.x) {  // all items in parallel
      int lo = 0, hi = p.B;                          // last b with sbase[b] <= i
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (sbase[mid] <= i) lo = mid;
        else hi = mid;
      }
      const int b = lo, r = i - sbase[b];
      const int nch = (sbase[b + 1] - sbase[b]) / p.Nkv;
      const int h = r / nch, j = r - h * nch;
      const DecodeSpan sp{slo[b], send[b], slo[b] & ~(kDecodeTileTC - 1)};
      p.ws.items[i] = span_item(sp, C, b, h, nch, j);
      p.ws.order[j < nch - 1 ? fpos[b] + h * (nch - 1) + j : tpos[b] + h] = i;
    }
  } else {
    for (int i = tid; i < total; i += blockDim.x) p.ws.order[i] = i;  // item order
  }
  if (tid == 0) {
    *p.ws.n_items = total;
    *p.ws.counter = 0;
    p.ws.seg_base[p.B] = total;
  }
}

// ------------------------------------------------------------------- attention
template <int KVT, int D, int GP>
__global__ void __launch_bounds__(kThreads, 1)
    decode_splitkv_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                          const DecodeParams p, const int box_rows) {
  using C = Cfg<KVT, D, GP>;
  extern __shared__ uint8_t smem_raw[];
  Smem<KVT, D, GP>& sm =
      *reinterpret_cast<Smem<KVT, D, GP>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.GV;  // virtual heads (query heads x query positions) of a kv head

  if (tid == 0) {
    for (int s = 0; s < kDecodeStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kConsumerWarps);
    }
    fence_mbar_init();
  }
  if (KVT == kI8 && p.Nkv <= kAqHeads) {  // per-channel antiquant parameters stay resident
    for (int i = tid; i < p.Nkv * D; i += kThreads) {
      sm.aq[0][i] = p.aq_scale[i];
      sm.aq[1][i] = p.aq_offset ? p.aq_offset[i] : 0.f;
      sm.aq[2][i] = p.aq_scale[p.Nkv * D + i];
      sm.aq[3][i] = p.aq_offset ? p.aq_offset[p.Nkv * D + i] : 0.f;
    }
  }
  __syncthreads();
  griddep_wait();  // the plan kernel's item list, counters and reset are complete and visible
  griddep_launch_dependents();  // the merge kernel may be scheduled; it waits for this grid to finish

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    ItemQueue queue;
    queue.start(p, lane);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    const int bs = p.block_size;
    const uint32_t piece_bytes = (uint32_t)box_rows * C::kBoxBytes * C::kNumBoxes;  // one of K/V
    while (ok) {
      int4 desc;
      const int item = queue.pop(p, lane, &desc);
      if (item < 0) break;
      const DecodeItem it = decode_item(desc);
      const int b = it.b, hkv = it.hkv, t_begin = it.t_begin, t_end = it.t_end;
      const int t0 = t_begin & ~(kTT - 1);  // the first tile (t_begin is aligned but for a window)
      const int qlim = p.qs > 1 ? clamp_len(p, b, false) - p.qs : (1 << 30);  // position 0's last key
      const int32_t* bt_row = p.block_table + (int64_t)b * p.bt_stride;
      for (int tok0 = t0; tok0 < t_end; tok0 += kTT) {
        const int n = min(kTT, t_end - tok0);
        const int npieces = (n + box_rows - 1) / box_rows;
        int32_t blk = 0;
        bool valid = false;
        if (lane < npieces) {
          blk = bt_row[(tok0 + lane * box_rows) / bs];
          valid = blk >= 0 && (int64_t)blk < p.num_blocks;
          if (!valid) raise_status(p.status, kStatusBadBlockIndex);
        }
        const unsigned vmask = __ballot_sync(0xffffffffu, valid);
        const bool first = tok0 == t0;
        uint32_t bytes = 2u * piece_bytes * __popc(vmask);
        if (first) bytes += (uint32_t)(G * D * 2);
        if (!mbar_wait(&sm.empty[stage], phase ^ 1u, p.status)) { ok = false; break; }
        if (lane == 0) {
          StageMeta& m = sm.meta[stage];
          m.b = b; m.hkv = hkv; m.tok0 = tok0; m.n = n;
          m.item = item; m.first = first; m.last = (tok0 + kTT >= t_end); m.nch = it.nch;
          m.nlo = max(t_begin - tok0, 0);
          m.qlim = qlim;
          mbar_arrive_expect_tx(&sm.full[stage], bytes);
        }
        __syncwarp();
        if (valid) {
          const KvCoord kc = kv_coord(p, blk, tok0 + lane * box_rows, hkv);
          for (int bx = 0; bx < C::kNumBoxes; ++bx) {
            const uint32_t off = bx * (kTT * C::kBoxBytes) + lane * box_rows * C::kBoxBytes;
            const int32_t x = kc.x0 + bx * (C::kBoxBytes / C::kElem);
            tma_load_2d(sm.kv[stage][0] + off, &tmK, x, kc.row, &sm.full[stage]);
            tma_load_2d(sm.kv[stage][1] + off, &tmV, x, kc.row, &sm.full[stage]);
          }
        }
        if (first && lane == 0) {  // the G query rows of each query position
          for (int i = 0; i < p.qs; ++i) {
            const uint16_t* qsrc = static_cast<const uint16_t*>(p.q) + q_row(p, b, hkv, i * p.G) * D;
            bulk_load(sm.q[stage] + i * p.G * D, qsrc, (uint32_t)(p.G * D * 2), &sm.full[stage]);
          }
        }
        if (first) queue.prefetch(p, lane);
        if (++stage == kDecodeStages) { stage = 0; phase ^= 1u; }
      }
    }
    // sentinel: tells the math warps that no item follows
    if (ok && mbar_wait(&sm.empty[stage], phase ^ 1u, p.status)) {
      if (lane == 0) {
        sm.meta[stage].item = -1;
        mbar_arrive(&sm.full[stage]);
      }
    } else {
      // give every copy already issued a bounded chance to land before exiting
      for (int s = 0; s < kDecodeStages; ++s) mbar_wait(&sm.full[s], phase, p.status);
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  // score mapping
  const int part = C::kPartsMinor ? (lane % C::P) : (lane / C::TW);
  const int tok_w = C::kPartsMinor ? (lane / C::P) : (lane % C::TW);
  // head held after the reduce-scatter, and whether this lane writes it
  int gh = 0;
  bool writer = true;
  {
    int cnt = GP;
#pragma unroll
    for (int l = 0; l < C::LOGP; ++l) {
      const int mask = C::MS << l;
      if (cnt > 1) {
        cnt >>= 1;
        if (lane & mask) gh += cnt;
      } else if (lane & mask) {
        writer = false;
      }
    }
  }
  // P.V mapping
  const int pv_c = tid % C::CH, pv_tg = tid / C::CH;

  float qr[GP][C::E];
  float kdq[2][C::E];  // int8: k scale / offset of this thread's channels
  float vdq[2][C::EV]; // int8: v scale / offset of this thread's P.V channels
  float acc[GP][C::EV];
#pragma unroll
  for (int g = 0; g < GP; ++g)
#pragma unroll
    for (int e = 0; e < C::EV; ++e) acc[g][e] = 0.f;

  int stage = 0;
  uint32_t phase = 0;
  while (true) {
    if (!mbar_wait(&sm.full[stage], phase, p.status)) break;
    const StageMeta meta = sm.meta[stage];
    if (meta.item < 0) break;
    const uint8_t* kt = sm.kv[stage][0];
    const uint8_t* vt = sm.kv[stage][1];
    const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);

    if (meta.first) {
      const uint16_t* qs = sm.q[stage];
#pragma unroll
      for (int g = 0; g < GP; ++g)
#pragma unroll
        for (int j = 0; j < C::NPC; ++j)
#pragma unroll
          for (int e = 0; e < C::PE; ++e) {
            const int d = (part + C::P * j) * C::PE + e;
            qr[g][j * C::PE + e] = (g < G) ? q_elem(qs, g * D + d, p.q_dtype) : 0.f;
          }
      if (KVT == kI8) {
        const bool resident = p.Nkv <= kAqHeads;
        const int64_t vofs = (int64_t)p.Nkv * D;
#pragma unroll
        for (int j = 0; j < C::NPC; ++j)
#pragma unroll
          for (int e = 0; e < C::PE; ++e) {
            const int d = meta.hkv * D + (part + C::P * j) * C::PE + e;
            kdq[0][j * C::PE + e] = resident ? sm.aq[0][d] : p.aq_scale[d];
            kdq[1][j * C::PE + e] = resident ? sm.aq[1][d] : (p.aq_offset ? p.aq_offset[d] : 0.f);
          }
#pragma unroll
        for (int e = 0; e < C::EV; ++e) {
          const int d = meta.hkv * D + pv_c * C::EV + e;
          vdq[0][e] = resident ? sm.aq[2][d] : p.aq_scale[vofs + d];
          vdq[1][e] = resident ? sm.aq[3][d] : (p.aq_offset ? p.aq_offset[vofs + d] : 0.f);
        }
      }
    }

    // ---- scores: s[g][t] = scale * log2(e) * q_g . k_t
#pragma unroll
    for (int pass = 0; pass < C::PASSES; ++pass) {
      const int t = pass * C::TPP + warp * C::TW + tok_w;
      float v[GP];
#pragma unroll
      for (int g = 0; g < GP; ++g) v[g] = 0.f;
      if (t < kTT) {
#pragma unroll
        for (int j = 0; j < C::NPC; ++j) {
          const uint32_t ob = (part + C::P * j) * C::PB;  // byte offset in the row
          const uint32_t addr = kbase + (ob / C::kBoxBytes) * (kTT * C::kBoxBytes) +
                                swz(t * C::kBoxBytes + (ob % C::kBoxBytes), C::kSwzMask);
          uint32_t w[4];
          load_piece<C::PB>(addr, w);
#pragma unroll
          for (int e = 0; e < C::PE; ++e) {
            float kf = piece_elem<KVT>(w, e);
            if (KVT == kI8) kf = dequant_i8(kf, kdq[1][j * C::PE + e], kdq[0][j * C::PE + e]);
#pragma unroll
            for (int g = 0; g < GP; ++g) v[g] = fmaf(qr[g][j * C::PE + e], kf, v[g]);
          }
        }
      }
      // reduce-scatter across the P lanes of this token: halve the head set per level
      int cnt = GP;
#pragma unroll
      for (int l = 0; l < C::LOGP; ++l) {
        const int mask = C::MS << l;
        const bool upper = lane & mask;
        if (cnt > 1) {
          const int half = cnt >> 1;
#pragma unroll
          for (int i = 0; i < GP / 2; ++i) {
            if (i < half) {
              const float send = upper ? v[i] : v[i + half];
              const float keep = upper ? v[i + half] : v[i];
              v[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
            }
          }
          cnt = half;
        } else {
          v[0] += __shfl_xor_sync(0xffffffffu, v[0], mask);
        }
      }
      if (t < kTT && writer) {
#pragma unroll
        for (int i = 0; i < GP; ++i)
          if (i < cnt)
            sm.s[gh + i][t] = (t < meta.n && t >= meta.nlo && !key_masked(p, meta.b, meta.tok0 + t) &&
                               meta.tok0 + t <= meta.qlim + (gh + i) / p.G)
                                  ? v[i] * p.scale_log2 : -INFINITY;
      }
    }
    named_bar_sync(kBarConsumers, kDecodeConsumers);

    // ---- online softmax, one warp per head
    for (int g = warp; g < GP; g += kConsumerWarps) {
      const float s0 = sm.s[g][lane], s1 = sm.s[g][lane + 32];
      float mx = fmaxf(s0, s1);
#pragma unroll
      for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_old = meta.first ? -INFINITY : sm.m_run[g];
      const float m_new = fmaxf(m_old, mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = (m_old == -INFINITY) ? 0.f : exp2f(m_old - m_use);
      const float p0 = exp2f(s0 - m_use), p1 = exp2f(s1 - m_use);
      sm.p[lane][g] = p0;
      sm.p[lane + 32][g] = p1;
      float sum = p0 + p1;
#pragma unroll
      for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (lane == 0) {
        const float l_old = meta.first ? 0.f : sm.l_run[g];
        sm.l_run[g] = l_old * alpha + sum;
        sm.m_run[g] = m_new;
        sm.alpha[g] = alpha;
      }
    }
    named_bar_sync(kBarConsumers, kDecodeConsumers);

    // ---- acc = acc * alpha + P . V for this thread's 8 channels
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      const float a = sm.alpha[g];
#pragma unroll
      for (int e = 0; e < C::EV; ++e) acc[g][e] = meta.first ? 0.f : acc[g][e] * a;
    }
#pragma unroll
    for (int i = 0; i < C::TPG; ++i) {
      const int t = pv_tg + C::NTG * i;
      if (t < meta.n) {
        const uint32_t ob = pv_c * C::EV * C::kElem;
        const uint32_t addr = vbase + (ob / C::kBoxBytes) * (kTT * C::kBoxBytes) +
                              swz(t * C::kBoxBytes + (ob % C::kBoxBytes), C::kSwzMask);
        uint32_t w[4];
        load_piece<C::EV * C::kElem>(addr, w);
        float vf[C::EV];
#pragma unroll
        for (int e = 0; e < C::EV; ++e) {
          vf[e] = piece_elem<KVT>(w, e);
          if (KVT == kI8) vf[e] = dequant_i8(vf[e], vdq[1][e], vdq[0][e]);
        }
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          const float pg = sm.p[t][g];
#pragma unroll
          for (int e = 0; e < C::EV; ++e) acc[g][e] = fmaf(pg, vf[e], acc[g][e]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[stage]);

    // ---- end of item: reduce over token groups and write the normalised partial
    if (meta.last) {
#pragma unroll
      for (int mask = C::CH; mask < 32; mask <<= 1)
#pragma unroll
        for (int g = 0; g < GP; ++g)
#pragma unroll
          for (int e = 0; e < C::EV; ++e) acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], mask);
      if (lane < C::CH) {
#pragma unroll
        for (int g = 0; g < GP; ++g)
#pragma unroll
          for (int e = 0; e < C::EV; ++e) sm.red[warp][g * D + pv_c * C::EV + e] = acc[g][e];
      }
      named_bar_sync(kBarConsumers, kDecodeConsumers);
      if (meta.nch == 1 && !p.partials_only) {
        // the segment is this one item: write the final output directly
        for (int o = tid; o < G * D; o += kDecodeConsumers) {
          float s = 0.f;
#pragma unroll
          for (int w2 = 0; w2 < kConsumerWarps; ++w2) s += sm.red[w2][o];
          const int g = o / D;
          const int64_t row = q_row(p, meta.b, meta.hkv, g);
          float M, W;
          const float v = single_item_output(s, sm.m_run[g], sm.l_run[g], p.sink, q_head(p, meta.hkv, g), &M, &W);
          const int64_t oi = row * D + (o - g * D);
          if (p.q_dtype == kBF16) store_out<kBF16>(p.out, oi, v);
          else store_out<kF16>(p.out, oi, v);
          if (o % D == 0) {
            if (p.softmax_max) p.softmax_max[row] = (M == -INFINITY) ? -INFINITY : M * kLn2;
            if (p.softmax_sum) p.softmax_sum[row] = W;
          }
        }
      } else {
        float* po = p.ws.part_o + (int64_t)meta.item * G * D;
        for (int o = tid; o < G * D; o += kDecodeConsumers) {
          float s = 0.f;
#pragma unroll
          for (int w2 = 0; w2 < kConsumerWarps; ++w2) s += sm.red[w2][o];
          const float l = sm.l_run[o / D];
          po[o] = l > 0.f ? s / l : 0.f;
        }
        if (tid < G) p.ws.part_ml[(int64_t)meta.item * G + tid] = make_float2(sm.m_run[tid], sm.l_run[tid]);
      }
      named_bar_sync(kBarConsumers, kDecodeConsumers);
    }
    if (++stage == kDecodeStages) { stage = 0; phase ^= 1u; }
  }
}

// ------------------------------------------------------------------- merge
// One CTA per (b, kv head) segment of two or more work items (segments of one item are
// written by the attention kernel, empty batches by the plan; with partials_only, for the
// int8 output, every segment is finished here, an empty one as zero partials).
// Partials are folded in
// order by the RingAttentionUpdate rule, each weighted by its own sum, with the sink
// added once (aclnnRingAttentionUpdate; aclnnFlashAttentionScoreV4 sink formula):
//   M = max(sink, max_j m_j),  W = sum_j l_j 2^{m_j - M} + 2^{sink - M},
//   out = sum_j o_j l_j 2^{m_j - M} / W,  softmax_max = M ln 2,  softmax_sum = W.
// The int8 output (aclnnIncreFlashAttentionV3 quantScale2 / quantOffset2) is taken from the
// fp32 out: code = saturate(round-to-nearest-even(out * scale2 + offset2)) to [-128, 127].
// Launched dependent on the attention kernel: its launch overlaps that kernel's tail.
constexpr int kMergeThreads = 256;

template <int QT>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(const DecodeParams p) {
  griddep_wait();  // every partial of the attention kernel is written and visible
  griddep_launch_dependents();  // a following plan kernel may launch; it waits for this grid
  extern __shared__ float2 ml[];  // [G][nch]: (max, sum), then (weight, -) per partial
  const int b = blockIdx.x / p.Nkv, hkv = blockIdx.x % p.Nkv;
  const int seg0 = p.ws.seg_base[b], seg1 = p.ws.seg_base[b + 1];  // batch b's items, all kv heads
  const int nch = (seg1 - seg0) / p.Nkv;
  if (nch <= 1 && !p.partials_only) return;
  // G: virtual heads (query heads x query positions) of the kv head
  const int G = p.GV, D = p.D, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int first = seg0 + hkv * nch;
  const float4* po = reinterpret_cast<const float4*>(p.ws.part_o + (int64_t)first * G * D);
  const int q4n = G * D / 4;  // float4 outputs per partial
  // this thread's outputs of the first kPre partials, loaded now so that their latency overlaps
  // that of the maxima and sums
  constexpr int kPre = 8;
  float4 pre[kPre];
#pragma unroll
  for (int j = 0; j < kPre; ++j)
    pre[j] = (tid < q4n && j < nch) ? po[(int64_t)j * q4n + tid] : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = tid; i < G * nch; i += kMergeThreads) {  // coalesced: partial-major in memory
    const int j = i / G, g = i - j * G;
    ml[g * nch + j] = p.ws.part_ml[(int64_t)first * G + i];
  }
  __syncthreads();
  for (int g = warp; g < G; g += kMergeThreads / 32) {
    const int h = q_head(p, hkv, g);
    const int64_t orow = q_row(p, b, hkv, g);
    float2* row = ml + g * nch;
    float M = -INFINITY;
    for (int j = lane; j < nch; j += 32) M = fmaxf(M, row[j].x);
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float sink2 = p.sink ? p.sink[h] * kLog2e : -INFINITY;
    M = fmaxf(M, sink2);
    float W = 0.f;
    for (int j = lane; j < nch; j += 32) {
      const float w = (M == -INFINITY || row[j].x == -INFINITY) ? 0.f : row[j].y * exp2f(row[j].x - M);
      row[j].x = w;
      W += w;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
    if (p.sink && M != -INFINITY) W += exp2f(sink2 - M);
    const float inv = W > 0.f ? 1.f / W : 0.f;
    __syncwarp();
    for (int j = lane; j < nch; j += 32) row[j].x *= inv;
    if (lane == 0) {
      if (p.softmax_max) p.softmax_max[orow] = (M == -INFINITY) ? -INFINITY : M * kLn2;
      if (p.softmax_sum) p.softmax_sum[orow] = W;
    }
  }
  __syncthreads();
  for (int q4 = tid; q4 < q4n; q4 += kMergeThreads) {
    const float2* row = ml + ((q4 * 4) / D) * nch;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int j = 0;
    if (q4 == tid) {  // the prefetched partials
#pragma unroll
      for (int k = 0; k < kPre; ++k)
        if (k < nch) {
          const float w = row[k].x;
          acc.x = fmaf(w, pre[k].x, acc.x);
          acc.y = fmaf(w, pre[k].y, acc.y);
          acc.z = fmaf(w, pre[k].z, acc.z);
          acc.w = fmaf(w, pre[k].w, acc.w);
        }
      j = min(nch, kPre);
    }
    for (; j + 4 <= nch; j += 4) {  // four independent loads in flight
      const float4 v0 = po[(int64_t)(j + 0) * q4n + q4], v1 = po[(int64_t)(j + 1) * q4n + q4];
      const float4 v2 = po[(int64_t)(j + 2) * q4n + q4], v3 = po[(int64_t)(j + 3) * q4n + q4];
      const float w0 = row[j].x, w1 = row[j + 1].x, w2 = row[j + 2].x, w3 = row[j + 3].x;
      acc.x = fmaf(w3, v3.x, fmaf(w2, v2.x, fmaf(w1, v1.x, fmaf(w0, v0.x, acc.x))));
      acc.y = fmaf(w3, v3.y, fmaf(w2, v2.y, fmaf(w1, v1.y, fmaf(w0, v0.y, acc.y))));
      acc.z = fmaf(w3, v3.z, fmaf(w2, v2.z, fmaf(w1, v1.z, fmaf(w0, v0.z, acc.z))));
      acc.w = fmaf(w3, v3.w, fmaf(w2, v2.w, fmaf(w1, v1.w, fmaf(w0, v0.w, acc.w))));
    }
    for (; j < nch; ++j) {
      const float4 v = po[(int64_t)j * q4n + q4];
      const float w = row[j].x;
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    const int v = (q4 * 4) / D, d = q4 * 4 - v * D;
    const int64_t o = q_row(p, b, hkv, v) * D + d;
    if (p.pq_scale) {
      const int c = q_head(p, hkv, v) * D + d;  // channel of acc.x within the (Nq, D) row
      const float a[4] = {acc.x, acc.y, acc.z, acc.w};
      uint32_t w = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int pc = (c + i) * p.pq_stride;
        const float y = fmaf(a[i], p.pq_scale[pc], p.pq_offset ? p.pq_offset[pc] : 0.f);
        const int v = min(max(__float2int_rn(y), -128), 127);
        w |= (uint32_t)(v & 0xff) << (8 * i);
      }
      *reinterpret_cast<uint32_t*>(static_cast<int8_t*>(p.out) + o) = w;  // o % 4 == 0 (D % 4 == 0)
    } else {
      store_out<QT>(p.out, o, acc.x);
      store_out<QT>(p.out, o + 1, acc.y);
      store_out<QT>(p.out, o + 2, acc.z);
      store_out<QT>(p.out, o + 3, acc.w);
    }
  }
}

// ------------------------------------------------------------------- probes
__global__ void debug_dequant_kernel(const int8_t* codes, const float* scale, const float* offset, int64_t n,
                                     float* out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const uint32_t w = (uint32_t)(uint8_t)codes[i];
    out[i] = dequant_i8(i8_to_f32(w, 0), offset[i], scale[i]);
  }
}

// Copies the visible K rows of one (b, hkv) sequence into dst (L x D, storage
// bytes) through the same block-table walk, tensor map, box shape and swizzled
// read addressing as the attention kernel.
template <int KVT, int D>
__global__ void __launch_bounds__(128) debug_gather_kernel(const __grid_constant__ CUtensorMap tmK,
                                                           const DecodeParams p, const int box_rows, const int b,
                                                           const int hkv, uint8_t* dst) {
  using C = Cfg<KVT, D, 1>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tile = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar;
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  int64_t raw = p.seq_lens[b];
  const int L = (int)(raw < 0 ? 0 : (raw > p.max_kv_len ? p.max_kv_len : raw));
  const int32_t* bt_row = p.block_table + (int64_t)b * p.bt_stride;
  uint32_t phase = 0;
  for (int tok0 = 0; tok0 < L; tok0 += kTT) {
    const int n = min(kTT, L - tok0);
    const int npieces = (n + box_rows - 1) / box_rows;
    if (tid == 0) {
      uint32_t bytes = 0;
      for (int r = 0; r < npieces; ++r) {
        const int32_t blk = bt_row[(tok0 + r * box_rows) / p.block_size];
        if (blk >= 0 && blk < p.num_blocks) bytes += box_rows * C::kBoxBytes * C::kNumBoxes;
      }
      mbar_arrive_expect_tx(&bar, bytes);
      for (int r = 0; r < npieces; ++r) {
        const int32_t blk = bt_row[(tok0 + r * box_rows) / p.block_size];
        if (!(blk >= 0 && blk < p.num_blocks)) continue;
        const KvCoord kc = kv_coord(p, blk, tok0 + r * box_rows, hkv);
        for (int bx = 0; bx < C::kNumBoxes; ++bx)
          tma_load_2d(tile + bx * (kTT * C::kBoxBytes) + r * box_rows * C::kBoxBytes, &tmK,
                      kc.x0 + bx * (C::kBoxBytes / C::kElem), kc.row, &bar);
      }
    }
    __syncthreads();
    if (!mbar_wait(&bar, phase, p.status)) return;
    phase ^= 1u;
    for (int i = tid; i < n * C::kRowBytes; i += blockDim.x) {
      const int t = i / C::kRowBytes, ob = i % C::kRowBytes;
      const uint32_t off = (ob / C::kBoxBytes) * (kTT * C::kBoxBytes) +
                           swz(t * C::kBoxBytes + (ob % C::kBoxBytes), C::kSwzMask);
      dst[(int64_t)(tok0 + t) * C::kRowBytes + ob] = tile[off];
    }
    __syncthreads();
  }
}

template <int KVT, int D, int GP>
cudaError_t launch_attention(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV, int box_rows,
                             int grid, cudaStream_t stream) {
  const size_t smem = sizeof(Smem<KVT, D, GP>) + 1024;
  auto kern = decode_splitkv_kernel<KVT, D, GP>;
  cudaError_t e = ensure_smem(kern, (int)smem);
  if (e != cudaSuccess) return e;
  trace_mark(kKernelDecodeAttention, 0, stream);
  e = launch_dependent(kern, grid, kThreads, smem, stream, tmK, tmV, p, box_rows);
  trace_mark(kKernelDecodeAttention, 1, stream);
  return e;
}

template <int KVT, int D>
cudaError_t launch_attention_g(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV, int box_rows,
                               int grid, cudaStream_t stream) {
  if (p.GV <= 1) return launch_attention<KVT, D, 1>(p, tmK, tmV, box_rows, grid, stream);
  if (p.GV <= 2) return launch_attention<KVT, D, 2>(p, tmK, tmV, box_rows, grid, stream);
  if (p.GV <= 4) return launch_attention<KVT, D, 4>(p, tmK, tmV, box_rows, grid, stream);
  return launch_attention<KVT, D, 8>(p, tmK, tmV, box_rows, grid, stream);
}

}  // namespace

size_t decode_workspace_bytes(int B, int Nkv, int G, int D, int max_items) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  size_t s = 256;                                      // counter, n_items
  s += up(sizeof(int) * (size_t)(B + 1));              // seg_base
  s += up(sizeof(int4) * (size_t)max_items);           // items
  s += up(sizeof(int) * (size_t)max_items);            // order
  s += up(sizeof(float) * (size_t)max_items * G * D);  // part_o
  s += up(sizeof(float2) * (size_t)max_items * G);     // part_ml
  if (D == 128) s += up((size_t)kI8QBlockBytes * B * Nkv);  // qprep
  s += up(sizeof(float) * ((size_t)4 * Nkv * D + (size_t)2 * (B > 0 ? B : 1) * Nkv * G));  // aux
  return s;
}

DecodeWorkspace decode_workspace_carve(void* base, int B, int Nkv, int G, int D, int max_items) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  uint8_t* c = static_cast<uint8_t*>(base);
  DecodeWorkspace w;
  w.counter = reinterpret_cast<int*>(c);
  w.n_items = reinterpret_cast<int*>(c + 4);
  c += 256;
  w.seg_base = reinterpret_cast<int*>(c);
  c += up(sizeof(int) * (size_t)(B + 1));
  w.items = reinterpret_cast<int4*>(c);
  c += up(sizeof(int4) * (size_t)max_items);
  w.order = reinterpret_cast<int*>(c);
  c += up(sizeof(int) * (size_t)max_items);
  w.part_o = reinterpret_cast<float*>(c);
  c += up(sizeof(float) * (size_t)max_items * G * D);
  w.part_ml = reinterpret_cast<float2*>(c);
  c += up(sizeof(float2) * (size_t)max_items * G);
  w.qprep = (D == 128) ? c : nullptr;
  if (D == 128) c += up((size_t)kI8QBlockBytes * B * Nkv);
  w.aux = reinterpret_cast<float*>(c);
  return w;
}

// Per-tensor antiquant (scale and offset of shape (2): keys, values) written out as the
// per-channel (2, Nkv, D) arrays the kernels read: the same dequantisation, (x - o) s.
__global__ void aq_expand_kernel(const float* scale2, const float* offset2, int n_per, float* dst_scale,
                                 float* dst_offset) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= 2 * n_per) return;
  const int sel = i / n_per;  // 0 keys, 1 values
  dst_scale[i] = scale2[sel];
  if (dst_offset) dst_offset[i] = offset2 ? offset2[sel] : 0.f;
}

// softmaxLse = ln(sum_t e^{z_t}) = max + ln(sum), the max and sum of the same row
// (natural-exp units); -inf for a row with an empty sum.
__global__ void lse_kernel(const float* mx, const float* sm, float* lse, int64_t n) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float m = mx[i], s = sm[i];
  lse[i] = (s > 0.f && m != -INFINITY) ? m + logf(s) : -INFINITY;
}

cudaError_t launch_aq_expand(const float* scale2, const float* offset2, int Nkv, int D, float* dst_scale,
                             float* dst_offset, cudaStream_t stream) {
  const int n = 2 * Nkv * D;
  aq_expand_kernel<<<(n + 255) / 256, 256, 0, stream>>>(scale2, offset2, Nkv * D, dst_scale, dst_offset);
  return cudaGetLastError();
}

cudaError_t launch_lse(const float* mx, const float* sm, float* lse, int64_t n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  lse_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(mx, sm, lse, n);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          const CUtensorMap* tmQ, const CUtensorMap* tail, int box_rows, int num_sms,
                          cudaStream_t stream) {
  if (tmQ && p.fused_plan) {  // the tensor-core kernel plans for itself: attention, then merge
    cudaError_t e = launch_decode_tc_attention(p, tmK, tmV, *tmQ, tail, box_rows, num_sms, stream);
    if (e != cudaSuccess) return e;
    return launch_merge(p, stream);
  }
  trace_mark(kKernelDecodePlan, 0, stream);
  const size_t plan_smem = p.B <= kPlanSmemB ? sizeof(int) * (size_t)(5 * p.B + 1) : 0;
  if (plan_smem > 48 * 1024) {
    cudaError_t e0 = ensure_smem(decode_plan_kernel, (int)(sizeof(int) * (5 * kPlanSmemB + 1)));
    if (e0 != cudaSuccess) return e0;
  }
  const bool i8tc = !tmQ && decode_uses_i8tc(p.kv_dtype, p.D);
  const int64_t prep_blocks = i8tc ? ((int64_t)p.B * p.Nkv * kI8Heads + 31) / 32 : 0;
  cudaError_t e = launch_dependent(decode_plan_kernel, (int)(1 + prep_blocks), 1024, plan_smem, stream, p);
  trace_mark(kKernelDecodePlan, 1, stream);
  if (e != cudaSuccess) return e;
  const int grid = num_sms;
  if (tmQ) {
    e = launch_decode_tc_attention(p, tmK, tmV, *tmQ, tail, box_rows, grid, stream);
  } else if (i8tc) {
    e = launch_decode_i8tc_attention(p, tmK, tmV, tail, box_rows, grid, stream);
  } else if (p.kv_dtype == kBF16) {
    e = (p.D == 64) ? launch_attention_g<kBF16, 64>(p, tmK, tmV, box_rows, grid, stream)
                    : launch_attention_g<kBF16, 128>(p, tmK, tmV, box_rows, grid, stream);
  } else if (p.kv_dtype == kF16) {
    e = (p.D == 64) ? launch_attention_g<kF16, 64>(p, tmK, tmV, box_rows, grid, stream)
                    : launch_attention_g<kF16, 128>(p, tmK, tmV, box_rows, grid, stream);
  } else {
    e = (p.D == 64) ? launch_attention_g<kI8, 64>(p, tmK, tmV, box_rows, grid, stream)
                    : launch_attention_g<kI8, 128>(p, tmK, tmV, box_rows, grid, stream);
  }
  if (e != cudaSuccess) return e;
  return launch_merge(p, stream);
}

// merge of segments with two or more items (of every segment with partials_only);
// dependent launch on the attention kernel
cudaError_t launch_merge(const DecodeParams& p, cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
  const int max_chunks = (p.max_kv_len + p.chunk_tokens - 1) / p.chunk_tokens;
  if (max_chunks <= 1 && !p.partials_only) return cudaSuccess;
  const size_t msmem = sizeof(float2) * (size_t)p.GV * (max_chunks > 1 ? max_chunks : 1);
  auto merge = (p.q_dtype == kBF16) ? decode_merge_kernel<kBF16> : decode_merge_kernel<kF16>;
  if (msmem > 48 * 1024) {
    e = ensure_smem(merge, (int)msmem);
    if (e != cudaSuccess) return e;
  }
  trace_mark(kKernelDecodeMerge, 0, stream);
  e = launch_dependent(merge, p.B * p.Nkv, kMergeThreads, msmem, stream, p);
  trace_mark(kKernelDecodeMerge, 1, stream);
  return e;
}

cudaError_t launch_debug_dequant(const int8_t* codes, const float* scale, const float* offset, int64_t n,
                                 float* out, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int grid = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  debug_dequant_kernel<<<grid, 256, 0, stream>>>(codes, scale, offset, n, out);
  return cudaGetLastError();
}

cudaError_t launch_debug_gather(const DecodeParams& p, const CUtensorMap& tmK, int box_rows, int b, int hkv,
                                void* dst, cudaStream_t stream) {
  auto run = [&](auto kern, int tile_bytes) {
    const int smem = tile_bytes + 1024;
    cudaError_t e = ensure_smem(kern, smem);
    if (e != cudaSuccess) return e;
    kern<<<1, 128, smem, stream>>>(tmK, p, box_rows, b, hkv, static_cast<uint8_t*>(dst));
    return cudaGetLastError();
  };
  if (p.kv_dtype == kI8)
    return p.D == 64 ? run(debug_gather_kernel<kI8, 64>, Cfg<kI8, 64, 1>::kTileBytes)
                     : run(debug_gather_kernel<kI8, 128>, Cfg<kI8, 128, 1>::kTileBytes);
  if (p.kv_dtype == kF16)
    return p.D == 64 ? run(debug_gather_kernel<kF16, 64>, Cfg<kF16, 64, 1>::kTileBytes)
                     : run(debug_gather_kernel<kF16, 128>, Cfg<kF16, 128, 1>::kTileBytes);
  return p.D == 64 ? run(debug_gather_kernel<kBF16, 64>, Cfg<kBF16, 64, 1>::kTileBytes)
                   : run(debug_gather_kernel<kBF16, 128>, Cfg<kBF16, 128, 1>::kTileBytes);
}

}  // namespace fia
