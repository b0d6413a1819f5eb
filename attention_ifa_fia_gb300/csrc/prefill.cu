// prefill.cu -- causal / band variable-length prefill attention (TND) on tcgen05 tensor cores.
//
// What it computes (FusedInferAttentionScore: prefill mode with query length > 1 and
// sparseMode 3 = rightDownCausal; aclnnFlashAttentionScoreV4: TND layout, cumulative
// sequence lengths, sink formula): for sequence b with Lq queries and Lkv keys, query i
// of head h attends to keys j <= i + (Lkv - Lq) of kv head h / (Nq / Nkv).
//
// Work unit: (sequence, 128-query tile, query head).  A one-CTA plan kernel lists the
// (sequence, tile) pairs longest-first (by number of visible key tiles); persistent
// CTAs take units from a counter.  Per key tile of 128 keys:
//
//   S [128 q x 128 k] = Q . K^T     A = Q tile, B = K tile, both K-major (TMA, 128B swizzle)
//   O [128 q x D]    += P . V       A = P in tensor memory (16-bit pairs per column)
//                                   B = V tile read MN-major
//
// S (double buffered), P (double buffered) and O all live in tensor memory, so the PV
// product reads only V from shared memory.  Warp roles (320 threads): warp 0 issues TMA
// (Q per unit, double buffered; K and V tiles in separate 2-stage rings, each V one tile
// behind its K); warp 1 owns TMEM and issues MMAs (QK of tile j+1 overlaps the softmax of
// tile j); warps 2-9 are two warpgroups that split every query row between them (key
// columns / output channels 0-63 and 64-127): mask, row max and sum in registers with
// only the per-row maximum exchanged through shared memory, P, the rescale of O, and the
// epilogue.  O is rescaled only when the running row max
// grows by more than 8 (log2 units); otherwise the stale max keeps every exponent
// <= 2^8, and the softmax max/sum outputs are converted to the true max at the end.
//
// Head dim D = 64 or 128 (template parameter kD): tiles are 128 rows of D channels in
// boxes of 64 channels; the QK product takes D / 16 K-steps and the PV product N = D.
// Keys from a paged cache (FusedInferAttentionScore PagedAttention) arrive in boxes of
// gcd(blockSize, 128) rows, each from its own block; rows of a key tile past the
// sequence's keys are masked in S, and in V they are zeroed before the PV product (a
// cache may hold anything there, NaN included, and P = 0 would not cancel a NaN).
// The output is 16-bit, or int8 with quantScale2 / quantOffset2 (aclnnIncreFlashAttentionV3
// parameter table): each normalised fp32 output is scaled, offset, rounded to the nearest
// integer and saturated in the epilogue (template parameter kQuant).
#include "decode_common.cuh"

namespace fia {
namespace {

constexpr int kQT = 128;           // queries per tile (MMA M)
constexpr int kKT = 128;           // keys per tile (MMA N of QK, K of PV)
constexpr int kPThreads = 320;   // warp 0 TMA, warp 1 MMA, warps 2-9 softmax (two column halves)
constexpr int kSoftmaxThreads = 256;
constexpr int kBarSoftmax = 3;   // named barrier of the softmax warps
constexpr int kPStages = 2;
constexpr uint32_t kRescaleThreshold = 8;  // log2 units

// a Q, K or V tile: 128 rows of kD channels (kD / 64 boxes of 128 rows x 128 bytes)
template <int kD>
constexpr int tile_bytes() { return kQT * kD * 2; }

struct __align__(16) PTileMeta {
  int b, h, q0, kvt;      // sequence, query head, first query (within the sequence), key tile
  int tq, tk, Lq, Lkv;    // first token of the sequence in q / kv, sequence lengths
  int first, last, qbuf, unit;
  int vrows, pad0, pad1, pad2;  // rows of the V tile to keep; rows from vrows on are zeroed
};

constexpr int kMetaRing = 4;

template <int kD>
struct PSmem {
  static constexpr int kTileB = tile_bytes<kD>();
  alignas(1024) uint8_t q[2][kTileB];
  alignas(1024) uint8_t k[kPStages][kTileB];
  alignas(1024) uint8_t v[kPStages][kTileB];
  PTileMeta meta[kMetaRing];
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[kPStages], k_empty[kPStages];
  uint64_t v_full[kPStages], v_empty[kPStages];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[2], p_free[2];
  // PV(j) completes phase j >> 1 of pv_done[j & 1]: a waiter for PV(j) is then never two
  // phases behind (PV(j - 2) has completed once S(j) is ready) nor ahead (PV(j + 2) needs
  // this tile's successor's P), which a parity wait on one barrier could not ensure
  uint64_t pv_done[2], o_free;
  float rmax[2][2][kQT];  // [tile parity][column half][row]: partial row maxima
  float lsum[2][kQT];     // [column half][row]: partial row sums at the epilogue
  uint32_t tmem_base;
};
// The dynamic shared memory must fit the 227 KB a CTA may use.
static_assert(sizeof(PSmem<128>) <= 232448, "prefill shared memory exceeds the per-CTA limit");

// per (sequence, query tile): the key tiles holding at least one visible key, {first,
// count}.  A row's visible keys form one interval of the band; the rows' intervals shift
// by one key per row and hold pre + next + 1 >= 1 keys, so their union is one interval.
__device__ __forceinline__ int2 key_tile_range(const PrefillParams& p, int q0, int Lq, int Lkv) {
  const int q_last = min(q0 + kQT - 1, Lq - 1);
  const int d = Lkv - Lq;
  const int k_min = max(q0 + d - p.pre, 0);
  const int k_max = min(q_last + d + p.next, Lkv - 1);
  if (k_max < k_min) return make_int2(0, 0);
  return make_int2(k_min / kKT, k_max / kKT - k_min / kKT + 1);
}

__device__ __forceinline__ void seq_bounds(const PrefillParams& p, int b, int& tq, int& Lq, int& tk, int& Lkv) {
  int64_t q0 = p.cu_q[b], q1 = p.cu_q[b + 1], k0 = 0, k1;
  if (p.block_table) {  // paged keys: a length per sequence
    k1 = p.seq_lens_kv[b];
    if (k1 < 0 || k1 > p.max_seqlen_kv) {
      raise_status(p.status, kStatusLengthClamped);
      k1 = k1 < 0 ? 0 : p.max_seqlen_kv;
    }
  } else {
    k0 = p.cu_kv[b];
    k1 = p.cu_kv[b + 1];
  }
  if (q0 < 0 || q1 < q0 || q1 > p.T || k0 < 0 || k1 < k0 || (!p.block_table && k1 > p.Tkv)) {
    raise_status(p.status, kStatusBadSeqlens);
    q0 = q1 = k0 = k1 = 0;
  }
  tq = (int)q0;
  Lq = (int)(q1 - q0);
  tk = (int)k0;
  Lkv = (int)(k1 - k0);
}

// Issues the TMA loads of key tile kt of kv head hkv of sequence b (keys from tk in the TND
// layout, or Lkv keys in the paged pool) into dst, completing on bar: kD / 64 boxes of 64
// channels, and in the paged pool 128 / box_rows boxes of box_rows rows along the tile, each
// from its own block.  A paged box past the keys (rows the tile masks) reads block 0; a block
// index outside the pool raises the status flag and reads block 0 instead.  The bytes that
// land are always tile_bytes<kD>().
template <int kD>
__device__ __forceinline__ void load_key_tile(uint8_t* dst, const CUtensorMap* m, const PrefillParams& p, int b,
                                              int tk, int Lkv, int kt, int hkv, uint64_t* bar) {
  constexpr int kBoxes = kD / 64;
  if (!p.block_table) {
#pragma unroll
    for (int bx = 0; bx < kBoxes; ++bx) tma_load_3d(dst + bx * (kKT * 128), m, bx * 64, hkv, tk + kt * kKT, bar);
    return;
  }
  const int rows = p.box_rows, n = kKT / rows;
  int32_t blk[8];  // block of each box (at most 8: box_rows >= 16); the table loads are independent
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int tok = kt * kKT + i * rows;
    blk[i] = (i < n && tok < Lkv) ? p.block_table[(int64_t)b * p.bt_stride + tok / p.block_size] : 0;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (i >= n) break;
    if (blk[i] < 0 || (int64_t)blk[i] >= p.num_blocks) {
      raise_status(p.status, kStatusBadBlockIndex);
      blk[i] = 0;
    }
    const int tok = kt * kKT + i * rows;
    const int z = blk[i] * p.kv_z_blk + hkv * p.kv_z_h;
#pragma unroll
    for (int bx = 0; bx < kBoxes; ++bx)
      tma_load_3d(dst + bx * (kKT * 128) + i * rows * 128, m, hkv * p.kv_x_h + bx * 64, tok % p.block_size, z, bar);
  }
}

// Rows of key tile kt that hold keys of a paged sequence of Lkv keys (the rest are zeroed in
// V); a TND tile keeps every row (rows past the sequence are the next sequence's keys, or
// zeros that TMA fills past the tensor's end).
__device__ __forceinline__ int v_rows_kept(const PrefillParams& p, int Lkv, int kt) {
  return p.block_table ? min(max(Lkv - kt * kKT, 0), kKT) : kKT;
}

// Zeroes rows [vrows, 128) of a V tile in shared memory (every box), by the 32 lanes of a
// warp, and makes the stores visible to the tensor cores (async proxy).
template <int kD>
__device__ __forceinline__ void zero_v_rows(uint8_t* vt, int vrows, int lane) {
  const int n16 = (kKT - vrows) * 8;  // 16-byte chunks per box (a row is 128 bytes of a box)
#pragma unroll
  for (int bx = 0; bx < kD / 64; ++bx)
    for (int i = lane; i < n16; i += 32)
      *reinterpret_cast<uint4*>(vt + bx * (kKT * 128) + vrows * 128 + i * 16) = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  __syncwarp();
}

// ------------------------------------------------------------------ plan
// Lists (sequence, query tile) pairs ordered by decreasing number of key tiles
// (counting sort), resets the unit counter.  Units are list entry x query head, or
// list entry x pair of query heads for the head-pair kernel.  The bounds of a chunk of
// sequences are read once into shared memory (the two passes would otherwise wait on
// dependent global loads sequence after sequence); warp w handles sequences w, w + 32, ...
// of the chunk, its lanes the query tiles.  Launched as a dependent of the preceding
// kernel: it waits for that kernel before touching memory and lets the attention kernel
// start its prologue at once.
constexpr int kPlanChunk = 256;  // sequences whose bounds are staged at a time

size_t prefill_plan_smem(int max_key_tiles) {
  return sizeof(int) * (size_t)((max_key_tiles + 2 + 3) & ~3) + sizeof(int4) * kPlanChunk;
}

__global__ void __launch_bounds__(1024) prefill_plan_kernel(PrefillParams p, int max_key_tiles, int unit_heads) {
  extern __shared__ int sh[];
  int* hist = sh;                                                          // [max_key_tiles + 2]
  int4* bounds = reinterpret_cast<int4*>(sh + ((max_key_tiles + 2 + 3) & ~3));  // {tq, Lq, tk, Lkv}
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  griddep_wait();
  griddep_launch_dependents();
  for (int i = tid; i < max_key_tiles + 2; i += blockDim.x) hist[i] = 0;
  for (int pass = 0; pass < 2; ++pass) {  // pass 0: histogram of key-tile counts; pass 1: scatter
    for (int b0 = 0; b0 < p.B; b0 += kPlanChunk) {
      const int nb = min(kPlanChunk, p.B - b0);
      __syncthreads();  // the previous chunk's bounds are no longer read (pass 1: the offsets are set)
      if (pass == 0 || p.B > kPlanChunk) {  // one chunk: pass 1 reads the bounds pass 0 staged
        for (int i = tid; i < nb; i += blockDim.x) {
          int tq, Lq, tk, Lkv;
          seq_bounds(p, b0 + i, tq, Lq, tk, Lkv);
          bounds[i] = make_int4(tq, Lq, tk, Lkv);
        }
        __syncthreads();
      }
      for (int i = warp; i < nb; i += nwarps) {
        const int4 bd = bounds[i];
        for (int qt = lane; qt * kQT < bd.y; qt += 32) {
          const int n = min(max(key_tile_range(p, qt * kQT, bd.y, bd.w).y, 1), max_key_tiles);
          if (pass == 0) {
            atomicAdd(&hist[n], 1);
          } else {
            const int pos = atomicAdd(&hist[n], 1);
            if (pos < p.max_tiles) p.tile_list[pos] = ((b0 + i) << 16) | qt;
          }
        }
      }
    }
    __syncthreads();
    if (pass == 0 && tid == 0) {  // exclusive offsets, largest count first
      int run = 0;
      for (int n = max_key_tiles; n >= 1; --n) {
        const int c = hist[n];
        hist[n] = run;
        run += c;
      }
      hist[0] = run;  // total pairs
    }
  }
  if (tid == 0) {
    p.tile_counter[0] = 0;
    p.tile_counter[1] = min(hist[0], p.max_tiles) * (p.Nq / unit_heads);  // number of units
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_f16(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// int8 output (quantScale2 / quantOffset2): the codes of channels c0 .. c0 + 3 of a row, each
// the fp32 output v * inv scaled and offset by its channel's values, rounded to the nearest
// integer (ties to even) and saturated to [-128, 127]; packed low byte first
__device__ __forceinline__ uint32_t quant4(const float* v, float inv, const PrefillParams& p, int c0) {
  uint32_t w = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int pc = (c0 + i) * p.pq_stride;
    const float y = fmaf(v[i] * inv, p.pq_scale[pc], p.pq_offset ? p.pq_offset[pc] : 0.f);
    const int q = min(max(__float2int_rn(y), -128), 127);
    w |= (uint32_t)(q & 0xff) << (8 * i);
  }
  return w;
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]),
      "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]),
      "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]),
      "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, issued by one thread (A: rows on lanes, 16-bit pairs per column).
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// As umma_f16_ta, executed by a whole converged warp (one elected lane issues).
__device__ __forceinline__ void umma_f16_ta_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// ------------------------------------------------------------------ attention
// kBand: a band's lower edge may fall inside a key tile (pre_tokens below the longest key
// sequence); without it the lower edge is never inside a tile and the softmax masks the
// upper edge only.  kQuant: int8 output.
template <int kD, int DT, bool kBand, bool kQuant>
__global__ void __launch_bounds__(kPThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using Sm = PSmem<kD>;
  constexpr int kTileB = Sm::kTileB;
  constexpr int kOH = kD / 2;  // output channels per softmax half
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Sm& sm = *reinterpret_cast<Sm*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (smem_u32(smem_raw) & 1023u) {  // the swizzled operand layouts need 1 KB alignment
    if (tid == 0) raise_status(p.status, kStatusWaitTimeout);
    return;
  }

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.q_full[i], 1);
      mbar_init(&sm.q_empty[i], 1);
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.s_free[i], 8);
      mbar_init(&sm.p_full[i], 8);
      mbar_init(&sm.p_free[i], 1);
    }
    for (int st = 0; st < kPStages; ++st) {
      mbar_init(&sm.k_full[st], 1);
      mbar_init(&sm.k_empty[st], 1);
      mbar_init(&sm.v_full[st], 1);
      mbar_init(&sm.v_empty[st], 1);
    }
    mbar_init(&sm.pv_done[0], 1);
    mbar_init(&sm.pv_done[1], 1);
    mbar_init(&sm.o_free, 8);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&sm.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;  // S: 2 x 128, O: kD, P: 2 x 64

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int n_units = p.tile_counter[1];
      const int G = p.G;
      int j = 0, u_local = 0;
      int v_next = 0;  // next tile whose V is to be loaded
      bool ok = true;
      // V of tile jv, one tile behind its K
      auto load_v = [&](int jv) -> bool {
        const int st = jv % kPStages;
        if (!mbar_wait(&sm.v_empty[st], ((uint32_t)(jv / kPStages) & 1u) ^ 1u, p.status)) return false;
        const PTileMeta& m = sm.meta[jv % kMetaRing];
        mbar_arrive_expect_tx(&sm.v_full[st], kTileB);
        load_key_tile<kD>(sm.v[st], &tmV, p, m.b, m.tk, m.Lkv, m.kvt, m.h / G, &sm.v_full[st]);
        return true;
      };
      while (ok) {
        const int u = atomicAdd(&p.tile_counter[0], 1);
        if (u >= n_units) break;
        const int pair = p.tile_list[u / p.Nq];
        const int h = u % p.Nq, b = pair >> 16, qt = pair & 0xffff;
        int tq, Lq, tk, Lkv;
        seq_bounds(p, b, tq, Lq, tk, Lkv);
        const int q0 = qt * kQT;
        const int2 kr = key_tile_range(p, q0, Lq, Lkv);  // a query tile with no key still runs one
        const int nkv = max(kr.y, 1);                     // (all-masked) tile
        const int qb = u_local & 1;
        if (!mbar_wait(&sm.q_empty[qb], ((uint32_t)(u_local >> 1) & 1u) ^ 1u, p.status)) { ok = false; break; }
        mbar_arrive_expect_tx(&sm.q_full[qb], kTileB);
        for (int bx = 0; bx < kD / 64; ++bx)
          tma_load_3d(sm.q[qb] + bx * (kQT * 128), &tmQ, bx * 64, h, tq + q0, &sm.q_full[qb]);
        const int hkv = h / G;
        for (int i = 0; i < nkv; ++i, ++j) {
          const int kt = kr.x + i;
          const int st = j % kPStages;
          if (!mbar_wait(&sm.k_empty[st], ((uint32_t)(j / kPStages) & 1u) ^ 1u, p.status)) { ok = false; break; }
          PTileMeta& m = sm.meta[j % kMetaRing];
          m.b = b; m.h = h; m.q0 = q0; m.kvt = kt;
          m.tq = tq; m.tk = tk; m.Lq = Lq; m.Lkv = Lkv;
          m.first = i == 0; m.last = i == nkv - 1; m.qbuf = qb; m.unit = u;
          m.vrows = v_rows_kept(p, Lkv, kt);
          mbar_arrive_expect_tx(&sm.k_full[st], kTileB);
          load_key_tile<kD>(sm.k[st], &tmK, p, b, tk, Lkv, kt, hkv, &sm.k_full[st]);
          if (v_next < j) {
            if (!load_v(v_next)) { ok = false; break; }
            ++v_next;
          }
        }
        ++u_local;
      }
      while (ok && v_next < j) {  // V of the last tiles
        if (!load_v(v_next)) { ok = false; break; }
        ++v_next;
      }
      if (ok) {  // sentinel tile
        const int st = j % kPStages;
        if (mbar_wait(&sm.k_empty[st], ((uint32_t)(j / kPStages) & 1u) ^ 1u, p.status)) {
          sm.meta[j % kMetaRing].unit = -1;
          mbar_arrive(&sm.k_full[st]);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (whole warp)
    // All lanes wait; one elected lane issues and commits (a converged warp issues sooner than
    // one thread in a divergent branch), and the lanes together zero V rows when needed.
    {
      constexpr uint32_t idesc_qk = umma_idesc_f16(DT == kBF16, 0, 0, kQT, kKT);
      constexpr uint32_t idesc_pv = umma_idesc_f16(DT == kBF16, 0, 1, kQT, kD);
      int o_uses = 0;  // units whose first PV (which overwrites O) has been issued
      // O += P(jj) . V(jj), P from TMEM; the first PV of a unit overwrites O, after the
      // previous unit's epilogue has read it (o_free phase o_uses - 1)
      auto issue_pv = [&](int jj, bool first_of_unit) -> bool {
        const int pb = jj & 1, vs = jj % kPStages;
        const int vrows = sm.meta[jj % kMetaRing].vrows;  // (slot not yet reused: see the producer)
        if (!mbar_wait_warp(&sm.p_full[pb], (uint32_t)(jj >> 1) & 1u, p.status)) return false;
        if (!mbar_wait_warp(&sm.v_full[vs], (uint32_t)(jj / kPStages) & 1u, p.status)) return false;
        if (first_of_unit && o_uses > 0 && !mbar_wait_warp(&sm.o_free, (uint32_t)(o_uses - 1) & 1u, p.status))
          return false;
        if (vrows < kKT) zero_v_rows<kD>(sm.v[vs], vrows, lane);
        tc_fence_after();
        const uint32_t vbase = smem_u32(sm.v[vs]);
#pragma unroll
        for (int s = 0; s < kKT / 16; ++s) {
          const uint64_t bd = umma_desc(vbase + s * 16 * 128, kKT * 128, 1024);
          umma_f16_ta_w(tmem + kColO, tmem + kColP + pb * 64 + s * 8, bd, idesc_pv,
                        (first_of_unit && s == 0) ? 0u : 1u);
        }
        umma_commit_w(&sm.pv_done[pb]);
        umma_commit_w(&sm.p_free[pb]);
        umma_commit_w(&sm.v_empty[vs]);
        if (first_of_unit) ++o_uses;
        return true;
      };
      int j = 0, u_local = 0;
      bool prev_first = false;
      while (true) {
        const int st = j % kPStages;
        if (!mbar_wait_warp(&sm.k_full[st], (uint32_t)(j / kPStages) & 1u, p.status)) break;
        const PTileMeta& meta = sm.meta[j % kMetaRing];
        const int unit = meta.unit, first = meta.first, last = meta.last, qb = meta.qbuf;
        if (unit < 0) {
          if (j > 0) issue_pv(j - 1, prev_first);
          if (lane == 0) mbar_arrive(&sm.s_full[j & 1]);  // lets the softmax warps see the sentinel
          break;
        }
        if (first && !mbar_wait_warp(&sm.q_full[qb], (uint32_t)(u_local >> 1) & 1u, p.status)) break;
        const int sb = j & 1;
        if (!mbar_wait_warp(&sm.s_free[sb], ((uint32_t)(j >> 1) & 1u) ^ 1u, p.status)) break;
        tc_fence_after();
        const uint32_t qbase = smem_u32(sm.q[qb]), kbase = smem_u32(sm.k[st]);
#pragma unroll
        for (int s = 0; s < kD / 16; ++s) {
          const uint64_t a = umma_desc(qbase + (s >> 2) * (kQT * 128) + (s & 3) * 32, 16, 1024);
          const uint64_t bd = umma_desc(kbase + (s >> 2) * (kKT * 128) + (s & 3) * 32, 16, 1024);
          umma_f16_w(tmem + kColS + sb * kKT, a, bd, idesc_qk, s > 0);
        }
        umma_commit_w(&sm.s_full[sb]);
        umma_commit_w(&sm.k_empty[st]);
        if (last) {
          umma_commit_w(&sm.q_empty[qb]);
          ++u_local;
        }
        if (j > 0 && !issue_pv(j - 1, prev_first)) break;
        prev_first = first;
        ++j;
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax, rescale, epilogue
    // Two warpgroups split each query row: half 0 owns key columns 0-63 of S (and output
    // channels [0, kD/2) of O), half 1 columns 64-127 (and channels [kD/2, kD)).  Only the
    // per-row tile maximum (and, at the end, the row sum) is exchanged through shared memory.
    const int half = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // query row of the tile = TMEM lane
    const uint32_t tq_lane = tmem + ((uint32_t)(quad * 32) << 16);
    const int c_base = half * 64;   // key columns of this half
    const int o_base = half * kOH;  // output channels of this half
    float m_run = -INFINITY;   // max used for the exponents (may lag the true max by < 2^8)
    float m_true = -INFINITY;  // true running max
    float l_run = 0.f;         // this half's sum of exponents relative to m_run
    int j = 0;
    while (true) {
      const int sb = j & 1;
      if (!mbar_wait(&sm.s_full[sb], (uint32_t)(j >> 1) & 1u, p.status)) break;
      const PTileMeta meta = sm.meta[j % kMetaRing];
      if (meta.unit < 0) break;
      tc_fence_after();
      if (meta.first) {
        m_run = -INFINITY;
        m_true = -INFINITY;
        l_run = 0.f;
      }
      const int qi = meta.q0 + r;            // query index within the sequence
      const bool row_ok = qi < meta.Lq;
      const int k0 = meta.kvt * kKT + c_base;
      // visible keys of this row among this half's columns: [k0 + nlo, k0 + nvis)
      const int dq = qi + (meta.Lkv - meta.Lq);
      const int k_hi = min(meta.Lkv, dq + p.next + 1);
      const int nvis = row_ok ? max(0, min(k_hi - k0, 64)) : 0;
      const int nlo = kBand ? min(max(dq - p.pre - k0, 0), 64) : 0;
      float s[64];
#pragma unroll
      for (int c = 0; c < 64; c += 32) {
        float v[32];
        tmem_ld32(tq_lane + kColS + sb * kKT + c_base + c, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c + i] = v[i];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.s_free[sb]);
      float mt = -INFINITY;
      if (kBand && __any_sync(0xffffffffu, nlo > 0)) {  // a band's lower edge crosses the tile
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          s[c] = (c >= nlo && c < nvis) ? s[c] * p.scale_log2 : -INFINITY;
          mt = fmaxf(mt, s[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          s[c] = (c < nvis) ? s[c] * p.scale_log2 : -INFINITY;
          mt = fmaxf(mt, s[c]);
        }
      }
      sm.rmax[sb][half][r] = mt;
      named_bar_sync(kBarSoftmax, kSoftmaxThreads);
      mt = fmaxf(mt, sm.rmax[sb][half ^ 1][r]);
      const float m_old = m_run;
      m_true = fmaxf(m_true, mt);
      bool rescale = false;
      float alpha = 1.f;
      if (mt > m_run + (float)kRescaleThreshold || (m_run == -INFINITY && mt != -INFINITY)) {
        m_run = mt;
        if (m_old != -INFINITY) {
          rescale = true;
          alpha = fast_exp2(m_old - m_run);
        }
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      float lsum = 0.f;
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const float e0 = fast_exp2(s[c] - m_use), e1 = fast_exp2(s[c + 1] - m_use);
        lsum += e0 + e1;
        pk[c >> 1] = (DT == kBF16) ? pack_bf16(e0, e1) : pack_f16(e0, e1);
      }
      l_run = fmaf(l_run, alpha, lsum);
      // O rescale (rare): the previous tile's PV must be complete and this tile's not begun.
      // tcgen05.ld/st are warp-collective (.sync.aligned), so the whole warp takes part,
      // rows that do not need it with a factor of 1.
      if (__any_sync(0xffffffffu, rescale && !meta.first)) {
        if (!mbar_wait(&sm.pv_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u, p.status)) break;
        const float f = (rescale && !meta.first) ? alpha : 1.f;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kOH; c += 32) {
          float o[32];
          tmem_ld32(tq_lane + kColO + o_base + c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= f;
          tmem_st32(tq_lane + kColO + o_base + c, o);
        }
      }
      // this half of P row r (64 keys = 32 packed columns) into the P buffer of this tile
      if (!mbar_wait(&sm.p_free[sb], ((uint32_t)(j >> 1) & 1u) ^ 1u, p.status)) break;
      tmem_st32u(tq_lane + kColP + sb * 64 + half * 32, pk);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_full[sb]);
      if (meta.last) {
        // epilogue: wait for this tile's PV, normalise O and write out, max and sum
        if (!mbar_wait(&sm.pv_done[j & 1], (uint32_t)(j >> 1) & 1u, p.status)) break;
        tc_fence_after();
        sm.lsum[half][r] = l_run;
        named_bar_sync(kBarSoftmax, kSoftmaxThreads);
        const float l_row = l_run + sm.lsum[half ^ 1][r];  // relative to m_run
        const float sink2 = p.sink ? p.sink[meta.h] * kLog2e : -INFINITY;
        const float m_fin = fmaxf(m_true, sink2);
        float denom = l_row;
        if (p.sink && m_run != -INFINITY) denom += fast_exp2(sink2 - m_run);
        const float inv = denom > 0.f ? 1.f / denom : 0.f;
        const int64_t tok = (int64_t)meta.tq + qi;
        // every lane takes part in the (warp-collective) TMEM loads; only valid rows store
        uint8_t* orow = static_cast<uint8_t*>(p.out) + ((tok * p.Nq + meta.h) * (int64_t)kD + o_base) * 2;
        uint8_t* qrow = static_cast<uint8_t*>(p.out) + (tok * p.Nq + meta.h) * (int64_t)kD + o_base;  // int8
#pragma unroll
        for (int c = 0; c < kOH; c += 32) {
          float o[32];
          tmem_ld32(tq_lane + kColO + o_base + c, o);
          if constexpr (kQuant) {
            if (row_ok) {
#pragma unroll
              for (int i = 0; i < 32; i += 16) {
                const int ch = meta.h * kD + o_base + c + i;
                const uint4 w = make_uint4(quant4(o + i, inv, p, ch), quant4(o + i + 4, inv, p, ch + 4),
                                           quant4(o + i + 8, inv, p, ch + 8), quant4(o + i + 12, inv, p, ch + 12));
                *reinterpret_cast<uint4*>(qrow + c + i) = w;
              }
            }
          } else if (row_ok) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              uint4 w;
              if (DT == kBF16)
                w = make_uint4(pack_bf16(o[i] * inv, o[i + 1] * inv), pack_bf16(o[i + 2] * inv, o[i + 3] * inv),
                               pack_bf16(o[i + 4] * inv, o[i + 5] * inv), pack_bf16(o[i + 6] * inv, o[i + 7] * inv));
              else
                w = make_uint4(pack_f16(o[i] * inv, o[i + 1] * inv), pack_f16(o[i + 2] * inv, o[i + 3] * inv),
                               pack_f16(o[i + 4] * inv, o[i + 5] * inv), pack_f16(o[i + 6] * inv, o[i + 7] * inv));
              *reinterpret_cast<uint4*>(orow + (c + i) * 2) = w;
            }
          }
        }
        if (row_ok && half == 0) {
          float sum_true = 0.f;
          if (m_fin != -INFINITY) {
            sum_true = (m_run == -INFINITY) ? 0.f : l_row * fast_exp2(m_run - m_fin);
            if (p.sink) sum_true += fast_exp2(sink2 - m_fin);
          }
          if (p.softmax_max) p.softmax_max[tok * p.Nq + meta.h] = (m_fin == -INFINITY) ? -INFINITY : m_fin * kLn2;
          if (p.softmax_sum) p.softmax_sum[tok * p.Nq + meta.h] = sum_true;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.o_free);
      }
      ++j;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ head-pair kernel
// For an even GQA group: a work unit is (sequence, 128-query tile, pair of query heads
// 2hp and 2hp + 1), and both heads share the kv head, so each K and V tile is loaded
// once for two heads.  Tensor memory holds S and O of both heads (4 x 128 columns);
// P of a head is written over the first 64 columns of its own S once they have been
// read.  The products are issued in the strict order
//
//   QK_A(0) QK_B(0) | PV_A(0) QK_A(1) PV_B(0) QK_B(1) | PV_A(1) QK_A(2) ...
//
// so that the softmax of one head overlaps the products of the other (the strict order
// keeps the two heads half a period apart; issued independently they fall into step and
// their softmaxes contend for the same units).  The MMAs of one thread execute in issue
// order, so QK_X(j+1) may overwrite P_X(j) as soon as PV_X(j) is issued.  Each head has its
// own issuing warp, and the two pass a baton: a head's block (PV_X(j), QK_X(j+1)) is issued
// back to back, the baton passed, and only then committed (a commit holds the issuing
// thread until the products before it are under way; with one issuer, the other head's P
// would wait behind it).  PV_X(j) takes keys 0-63 as soon as the softmax has released that
// half of P.  Warp roles (352 threads): warp 0 TMA, warps 1 and 10 MMA of heads A and B,
// warps 2-5 head A and warps 6-9 head B: one query row per thread with the whole S row in
// registers, the softmax of every tile and, after a unit's last tile, its epilogue
// (normalise O, write out, max and sum), during which the other head keeps the tensor
// cores busy.
constexpr int kP2Threads = 352;
constexpr int kP2TmaWarp = 0, kP2MmaWarpA = 1, kP2MmaWarpB = 10;

// d = a * b + c for two lanes at once (one packed fp32 instruction, each lane rounded as fmaf).
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b, float c) {
  uint64_t d;
  asm("{\n\t.reg .b64 a, b, c;\n\tmov.b64 a, {%1, %2};\n\tmov.b64 b, {%3, %3};\n\tmov.b64 c, {%4, %4};\n\t"
      "fma.rn.f32x2 %0, a, b, c;\n\t}"
      : "=l"(d)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
  d0 = __uint_as_float((uint32_t)d);
  d1 = __uint_as_float((uint32_t)(d >> 32));
}

// 64 consecutive 32-bit TMEM columns of this thread's lane, load and wait in one statement.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,"
      "%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]),
        "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]),
        "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]),
        "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]),
        "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// 128 consecutive 32-bit TMEM columns of this thread's lane: two loads, one wait.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float (&v)[128]) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {"
      "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,"
      "%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,"
      "%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63"
      "}, [%128];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {"
      "%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,"
      "%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,"
      "%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127"
      "}, [%129];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]),
        "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]),
        "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]),
        "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]),
        "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]),
        "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]),
        "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]),
        "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]),
        "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]),
        "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]),
        "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]),
        "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]),
        "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]),
        "=r"(r[126]), "=r"(r[127])
      : "r"(taddr), "r"(taddr + 64u)
      : "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}

// P = 2^(s mul - m) of keys [64 h, 64 h + 64) of one S row in 16-bit pairs, stored at
// columns [32 h, 32 h + 32) from taddr; returns their sum of P.
template <int DT, int h>
__device__ __forceinline__ float p_pass(const float (&s)[kKT], float mul, float m, uint32_t taddr) {
  float a[4] = {0.f, 0.f, 0.f, 0.f};  // four independent partial sums
  const float neg_m = -m;
#pragma unroll
  for (int c = 64 * h; c < 64 * h + 64; c += 32) {
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      float t0, t1;
      ffma2(t0, t1, s[c + i], s[c + i + 1], mul, neg_m);
      const float p0 = fast_exp2(t0), p1 = fast_exp2(t1);
      const int k = (i >> 1) & 1;  // (a packed add here would pin register pairs and spill)
      a[2 * k] += p0;
      a[2 * k + 1] += p1;
      pk[i >> 1] = (DT == kBF16) ? pack_bf16(p0, p1) : pack_f16(p0, p1);
    }
    tmem_st16u(taddr + (c >> 1), pk);
  }
  return (a[0] + a[1]) + (a[2] + a[3]);
}

template <int kD>
struct P2Smem {
  static constexpr int kTileB = tile_bytes<kD>();
  alignas(1024) uint8_t q[2][kTileB];  // head A, head B of the current unit
  alignas(1024) uint8_t k[kPStages][kTileB];
  alignas(1024) uint8_t v[kPStages][kTileB];
  alignas(128) uint8_t ostage[8][32 * 128];  // per softmax warp: 32 rows x 64 channels of out
  PTileMeta meta[kMetaRing];
  uint64_t q_full, q_empty;
  uint64_t k_full[kPStages], k_empty[kPStages];
  uint64_t v_full[kPStages], v_empty[kPStages];
  uint64_t s_full[2], p_lo[2], p_full[2], pv_done[2];  // per head, one phase per key tile
  uint64_t o_ready[2], o_free[2];             // per head, one phase per unit
  uint64_t turn[2];                           // the issue baton: head x's MMA warp may issue its next block
  int stop[2];                                // set by head x's MMA warp after the last tile
  uint32_t tmem_base;
};
static_assert(sizeof(P2Smem<128>) <= 232448, "prefill shared memory exceeds the per-CTA limit");

template <int kD, int DT, bool kBand, bool kQuant>
__global__ void __launch_bounds__(kP2Threads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using Sm = P2Smem<kD>;
  constexpr int kTileB = Sm::kTileB;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Sm& sm = *reinterpret_cast<Sm*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (smem_u32(smem_raw) & 1023u) {  // the swizzled operand layouts need 1 KB alignment
    if (tid == 0) raise_status(p.status, kStatusWaitTimeout);
    return;
  }
  if (tid == 0) {
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 2);  // q_empty, k_empty, v_empty: one commit per head's MMA warp
    for (int st = 0; st < kPStages; ++st) {
      mbar_init(&sm.k_full[st], 1);
      mbar_init(&sm.k_empty[st], 2);
      mbar_init(&sm.v_full[st], 1);
      mbar_init(&sm.v_empty[st], 2);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sm.s_full[x], 1);
      mbar_init(&sm.p_lo[x], 4);
      mbar_init(&sm.p_full[x], 4);
      mbar_init(&sm.pv_done[x], 1);
      mbar_init(&sm.o_ready[x], 1);
      mbar_init(&sm.o_free[x], 4);
      mbar_init(&sm.turn[x], 1);
      sm.stop[x] = 0;
    }
    fence_mbar_init();
  }
  if (warp == kP2MmaWarpA) tmem_alloc(&sm.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_wait();  // the plan's unit list (this kernel is a dependent launch)
  const uint32_t tmem = sm.tmem_base;
  constexpr uint32_t kColS[2] = {0, 128}, kColO[2] = {256, 384};

  if (warp == kP2TmaWarp) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int n_units = p.tile_counter[1];
      const int npairs = p.Nq / 2;
      int j = 0, u_local = 0, v_next = 0;
      bool ok = true;
      auto load_v = [&](int jv) -> bool {  // V of tile jv, one tile behind its K
        const int st = jv % kPStages;
        if (!mbar_wait(&sm.v_empty[st], ((uint32_t)(jv / kPStages) & 1u) ^ 1u, p.status)) return false;
        const PTileMeta& m = sm.meta[jv % kMetaRing];
        mbar_arrive_expect_tx(&sm.v_full[st], kTileB);
        load_key_tile<kD>(sm.v[st], &tmV, p, m.b, m.tk, m.Lkv, m.kvt, m.h / p.G, &sm.v_full[st]);
        return true;
      };
      while (ok) {
        const int u = atomicAdd(&p.tile_counter[0], 1);
        if (u >= n_units) break;
        const int pair = p.tile_list[u / npairs];
        const int hp = u % npairs, b = pair >> 16, qt = pair & 0xffff;
        const int h0 = 2 * hp;
        int tq, Lq, tk, Lkv;
        seq_bounds(p, b, tq, Lq, tk, Lkv);
        const int q0 = qt * kQT;
        const int2 kr = key_tile_range(p, q0, Lq, Lkv);  // a query tile with no key still runs one
        const int nkv = max(kr.y, 1);                     // (all-masked) tile
        // both Q tiles; the previous unit's last QK_B has completed
        if (!mbar_wait(&sm.q_empty, ((uint32_t)u_local & 1u) ^ 1u, p.status)) { ok = false; break; }
        mbar_arrive_expect_tx(&sm.q_full, 2 * kTileB);
        for (int x = 0; x < 2; ++x)
          for (int bx = 0; bx < kD / 64; ++bx)
            tma_load_3d(sm.q[x] + bx * (kQT * 128), &tmQ, bx * 64, h0 + x, tq + q0, &sm.q_full);
        const int hkv = h0 / p.G;
        for (int i = 0; i < nkv; ++i, ++j) {
          const int kt = kr.x + i;
          const int st = j % kPStages;
          if (!mbar_wait(&sm.k_empty[st], ((uint32_t)(j / kPStages) & 1u) ^ 1u, p.status)) { ok = false; break; }
          PTileMeta& m = sm.meta[j % kMetaRing];
          m.b = b; m.h = h0; m.q0 = q0; m.kvt = kt;
          m.tq = tq; m.tk = tk; m.Lq = Lq; m.Lkv = Lkv;
          m.first = i == 0; m.last = i == nkv - 1; m.qbuf = 0; m.unit = u;
          m.vrows = v_rows_kept(p, Lkv, kt);
          mbar_arrive_expect_tx(&sm.k_full[st], kTileB);
          load_key_tile<kD>(sm.k[st], &tmK, p, b, tk, Lkv, kt, hkv, &sm.k_full[st]);
          if (v_next < j) {
            if (!load_v(v_next)) { ok = false; break; }
            ++v_next;
          }
        }
        // the unit's remaining V tiles before the next unit's Q, whose buffer frees only
        // after the unit's last QK
        while (ok && v_next < j) {
          if (!load_v(v_next)) { ok = false; break; }
          ++v_next;
        }
        ++u_local;
      }
      while (ok && v_next < j) {
        if (!load_v(v_next)) { ok = false; break; }
        ++v_next;
      }
      if (ok) {  // sentinel tile
        const int st = j % kPStages;
        if (mbar_wait(&sm.k_empty[st], ((uint32_t)(j / kPStages) & 1u) ^ 1u, p.status)) {
          sm.meta[j % kMetaRing].unit = -1;
          mbar_arrive(&sm.k_full[st]);
        }
      }
    }
  } else if (warp == kP2MmaWarpA || warp == kP2MmaWarpB) {
    // ------------------------------------------------------------------ MMA issuer of head x (whole warp)
    const int x = warp == kP2MmaWarpA ? 0 : 1;
    constexpr uint32_t idesc_qk = umma_idesc_f16(DT == kBF16, 0, 0, kQT, kKT);
    constexpr uint32_t idesc_pv = umma_idesc_f16(DT == kBF16, 0, 1, kQT, kD);
    const uint64_t qdesc = umma_desc(smem_u32(sm.q[x]), 16, 1024);
    const uint32_t col_s = tmem + kColS[x], col_o = tmem + kColO[x];
    int o_units = 0;  // units whose first PV into O_x has been issued
    int u_local = 0;
    // S_x = Q_x K(jj)^T (8 MMAs, no commit)
    auto qk = [&](int jj) {
      const uint64_t b0 = umma_desc(smem_u32(sm.k[jj % kPStages]), 16, 1024);
#pragma unroll
      for (int s = 0; s < kD / 16; ++s) {
        const uint32_t off = (uint32_t)(((s >> 2) * (kQT * 128) + (s & 3) * 32) >> 4);
        umma_f16_w(col_s, qdesc + off, b0 + off, idesc_qk, s > 0);
      }
    };
    // O_x (+)= P_x(jj) V(jj) (8 MMAs, no commit): keys 0-63 once the softmax has released
    // that half of P, keys 64-127 once it has released all of it.  flags of a tile: bit 0
    // first, bit 1 last; vrows: rows of its V tile to keep (head A zeroes the rest, once,
    // before its product; head B issues after head A's block)
    auto pv = [&](int jj, int flags, int vrows) -> bool {
      if ((flags & 1) && o_units > 0 && !mbar_wait_warp(&sm.o_free[x], (uint32_t)(o_units - 1) & 1u, p.status))
        return false;
      if (x == 0 && vrows < kKT) zero_v_rows<kD>(sm.v[jj % kPStages], vrows, lane);
      const uint64_t b0 = umma_desc(smem_u32(sm.v[jj % kPStages]), kKT * 128, 1024);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        if (!mbar_wait_warp(hf ? &sm.p_full[x] : &sm.p_lo[x], (uint32_t)jj & 1u, p.status)) return false;
        tc_fence_after();
#pragma unroll
        for (int s = 4 * hf; s < 4 * hf + 4; ++s)
          umma_f16_ta_w(col_o, col_s + s * 8, b0 + (uint64_t)((s * 16 * 128) >> 4), idesc_pv,
                        ((flags & 1) && s == 0) ? 0u : 1u);
      }
      if (flags & 1) ++o_units;
      return true;
    };
    // waits for K of tile jj; returns its flags, -1 at the sentinel, -2 on error; *vrows
    // receives the rows of its V tile to keep
    auto load_tile = [&](int jj, int* vrows) -> int {
      if (!mbar_wait_warp(&sm.k_full[jj % kPStages], (uint32_t)(jj / kPStages) & 1u, p.status)) return -2;
      const PTileMeta& m = sm.meta[jj % kMetaRing];
      if (m.unit < 0) return -1;
      *vrows = m.vrows;
      return (m.first ? 1 : 0) | (m.last ? 2 : 0);
    };
    // the unit's Q before the QK products of its first tile
    auto wait_q = [&](int flags) -> bool {
      if ((flags & 1) && !mbar_wait_warp(&sm.q_full, (uint32_t)u_local & 1u, p.status)) return false;
      tc_fence_after();
      return true;
    };
    // the baton: head A's block b follows head B's block b - 1, head B's block b follows
    // head A's block b
    int block = 0;
    auto take_turn = [&]() -> bool {
      if (x == 0 && block == 0) return true;
      return mbar_wait_warp(&sm.turn[x], (uint32_t)(x == 0 ? block - 1 : block) & 1u, p.status);
    };
    auto pass_turn = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.turn[x ^ 1]);
      ++block;
    };
    int vr_cur = kKT, vr_nxt = kKT;
    int cur = load_tile(0, &vr_cur);
    if (cur >= 0 && !wait_q(cur)) cur = -2;
    if (cur >= 0 && take_turn()) {  // block 0: QK_x(0)
      qk(0);
      pass_turn();
      umma_commit_w(&sm.s_full[x]);
      umma_commit_w(&sm.k_empty[0]);
      if (cur & 2) {
        umma_commit_w(&sm.q_empty);
        ++u_local;
      }
    } else {
      cur = -2;
    }
    // Block j + 1: PV_x(j), then QK_x(j + 1), then (after the baton) the commits: S_x(j + 1)
    // is complete when s_full fires; pv_done fires once PV_x(j) (and QK_x(j + 1)) are, which
    // the rescale of O in the softmax of tile j + 1 needs and has by then.
    for (int j = 0; cur >= 0; ++j) {
      const int vs = j % kPStages;
      if (!mbar_wait_warp(&sm.v_full[vs], (uint32_t)(j / kPStages) & 1u, p.status)) break;
      // within a unit, the next K tile (loaded long before) is checked before PV_x(j), so that
      // QK_x(j + 1) follows PV_x(j) without a gap; the next unit's first K tile is requested
      // only as this unit's last QK completes and is waited for after PV_x(j)
      int nxt = -3;
      if (!(cur & 2)) {
        nxt = load_tile(j + 1, &vr_nxt);
        if (nxt == -2) break;
      }
      if (!take_turn()) break;
      if (!pv(j, cur, vr_cur)) break;
      if (cur & 2) umma_commit_w(&sm.o_ready[x]);  // the epilogue need not wait for QK_x(j + 1)
      if (nxt == -3) {
        nxt = load_tile(j + 1, &vr_nxt);
        if (nxt == -2) break;
      }
      if (nxt >= 0 && !wait_q(nxt)) break;
      if (nxt >= 0) qk(j + 1);
      pass_turn();
      if (nxt >= 0) umma_commit_w(&sm.s_full[x]);
      umma_commit_w(&sm.pv_done[x]);
      umma_commit_w(&sm.v_empty[vs]);
      if (nxt >= 0) {
        umma_commit_w(&sm.k_empty[(j + 1) % kPStages]);
        if (nxt & 2) {
          umma_commit_w(&sm.q_empty);
          ++u_local;
        }
      }
      cur = nxt;
      vr_cur = vr_nxt;
    }
    // No more tiles.  The softmax warps of head x have consumed every S phase (PV of the last
    // tile waited for their P), so a plain arrival completes the next one and they see the flag.
    if (lane == 0) {
      sm.stop[x] = 1;
      mbar_arrive(&sm.s_full[x]);
    }
  } else {
    // ------------------------------------------------------------------ softmax and epilogue of head x
    const int x = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // query row of the tile = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
    float m_run = -INFINITY, m_true = -INFINITY, l_run = 0.f;
    int units = 0;  // units finished by this warp group
    for (int j = 0;; ++j) {
      if (!mbar_wait(&sm.s_full[x], (uint32_t)j & 1u, p.status)) break;
      if (sm.stop[x]) break;
      // this tile's descriptor: its slot is rewritten only after QK(j + 2), which waits for
      // this warp group's P(j + 1), so fields are read where they are needed (fewer live
      // registers across the softmax)
      const PTileMeta& meta = sm.meta[j % kMetaRing];
      tc_fence_after();
      const bool first = meta.first;
      if (first) {
        m_run = -INFINITY;
        m_true = -INFINITY;
        l_run = 0.f;
      }
      int nvis, nlo;  // visible keys of the row in this tile: [k0 + nlo, k0 + nvis)
      bool all_keys;  // the row sees every key of the tile, or is past the sequence's queries
      {
        const int qi = meta.q0 + r, Lq = meta.Lq, Lkv = meta.Lkv;
        const int k0 = meta.kvt * kKT;
        const int dq = qi + (Lkv - Lq);
        const int k_hi = min(Lkv, dq + p.next + 1);
        nvis = qi < Lq ? max(0, min(k_hi - k0, kKT)) : 0;
        nlo = kBand ? min(max(dq - p.pre - k0, 0), kKT) : 0;
        all_keys = qi >= Lq || (nvis == kKT && nlo == 0);
      }
      // the S row in registers (raw scores)
      float s[kKT];
      tmem_ld128(tl + kColS[x], s);
      const float sc = p.scale_log2;
      // every row of the warp sees all 128 keys (rows past the sequence's queries are never
      // written out: any finite values do) and the scale is positive: the row max may be
      // taken on the raw scores and the scale applied once
      const bool full = __all_sync(0xffffffffu, all_keys) && sc > 0.f;
      const uint32_t col_p = tl + kColS[x];  // P (16-bit pairs) over the first 64 columns of S
      float alpha = 1.f;
      bool rescale = false;
      float lsum;
      {
        // the tile max; scores scaled in place unless full, keys outside the visible range at
        // -inf; four independent chains
        float mt = -INFINITY;
        if (full) {
          float e[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
          for (int i = 4; i < kKT; i += 8)
#pragma unroll
            for (int k = 0; k < 4; ++k) e[k] = fmax3(e[k], s[i + 2 * k], s[i + 2 * k + 1]);
          mt = fmax3(fmaxf(e[0], e[1]), e[2], e[3]) * sc;
        } else if (kBand && __any_sync(0xffffffffu, nlo > 0)) {  // a band's lower edge crosses the tile
          float e[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int i = 0; i < kKT; i += 8)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int i0 = i + 2 * k, i1 = i0 + 1;
              s[i0] = (i0 >= nlo && i0 < nvis) ? s[i0] * sc : -INFINITY;
              s[i1] = (i1 >= nlo && i1 < nvis) ? s[i1] * sc : -INFINITY;
              e[k] = fmax3(e[k], s[i0], s[i1]);
            }
          mt = fmax3(fmaxf(e[0], e[1]), e[2], e[3]);
        } else {
          float e[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int i = 0; i < kKT; i += 8)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int i0 = i + 2 * k, i1 = i0 + 1;
              s[i0] = (i0 < nvis) ? s[i0] * sc : -INFINITY;
              s[i1] = (i1 < nvis) ? s[i1] * sc : -INFINITY;
              e[k] = fmax3(e[k], s[i0], s[i1]);
            }
          mt = fmax3(fmaxf(e[0], e[1]), e[2], e[3]);
        }
        const float m_old = m_run;
        m_true = fmaxf(m_true, mt);
        if (mt > m_run + (float)kRescaleThreshold || (m_run == -INFINITY && mt != -INFINITY)) {
          m_run = mt;
          if (m_old != -INFINITY) {
            rescale = true;
            alpha = fast_exp2(m_old - m_run);
          }
        }
      }
      // P = 2^(s - m) in 16-bit pairs (raw scores times the scale when full), released in
      // two halves: the PV product of keys 0-63 starts while keys 64-127 are exponentiated.
      // A tile that rescales O (rare) releases both halves after the rescale, which needs
      // PV(j - 1) complete (pv_done fires with QK(j), before S(j)) and PV(j) not begun.
      const bool rescale_o = __any_sync(0xffffffffu, rescale && !first);
      {
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        const float mul = full ? sc : 1.f;
        lsum = p_pass<DT, 0>(s, mul, m_use, col_p);
        if (!rescale_o) {
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.p_lo[x]);
        }
        lsum += p_pass<DT, 1>(s, mul, m_use, col_p);
      }
      if (rescale_o) {
        if (!mbar_wait(&sm.pv_done[x], (uint32_t)(j - 1) & 1u, p.status)) break;
        const float f = (rescale && !first) ? alpha : 1.f;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kD; c += 32) {
          float o[32];
          tmem_ld32(tl + kColO[x] + c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= f;
          tmem_st32(tl + kColO[x] + c, o);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_lo[x]);
      }
      l_run = fmaf(l_run, alpha, lsum);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_full[x]);
      if (meta.last) {
        // epilogue: PV of this tile complete, normalise O, write out, max and sum, release O
        if (!mbar_wait(&sm.o_ready[x], (uint32_t)units & 1u, p.status)) break;
        tc_fence_after();
        const int h = meta.h + x;
        const float sink2 = p.sink ? p.sink[h] * kLog2e : -INFINITY;
        const float m_fin = fmaxf(m_true, sink2);
        float denom = l_run;
        if (p.sink && m_run != -INFINITY) denom += fast_exp2(sink2 - m_run);
        const float inv = denom > 0.f ? 1.f / denom : 0.f;
        const int qi = meta.q0 + r;
        const bool row_ok = qi < meta.Lq;
        const int64_t tok = (int64_t)meta.tq + qi;
        // out, 64 channels at a time: normalise and pack the warp's 32 rows into its staging
        // slot (16-byte chunk c of row l at position c ^ (l & 7): no bank conflicts either
        // way), then store 4 rows x 128 bytes per instruction
        uint8_t* stg = sm.ostage[warp - 2];
        const int row0 = meta.q0 + quad * 32;  // query row of lane 0
        const int rows_ok = min(max(meta.Lq - row0, 0), 32);
        uint8_t* obase = static_cast<uint8_t*>(p.out) + (((int64_t)meta.tq + row0) * p.Nq + h) * (int64_t)kD * 2;
        const int64_t orow_stride = (int64_t)p.Nq * kD * 2;
#pragma unroll
        for (int half = 0; half < kD / 64; ++half) {
          float o[64];
          tmem_ld64(tl + kColO[x] + half * 64, o);
          if (half == kD / 64 - 1) {  // every read of O_x is done: the next unit may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.o_free[x]);
          }
          if constexpr (kQuant) {  // int8: the half's 64 codes are chunks 4 half .. 4 half + 3 of the row
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const float* v = o + 16 * c;
              const int ch = h * kD + half * 64 + 16 * c;
              const uint4 w = make_uint4(quant4(v, inv, p, ch), quant4(v + 4, inv, p, ch + 4),
                                         quant4(v + 8, inv, p, ch + 8), quant4(v + 12, inv, p, ch + 12));
              *reinterpret_cast<uint4*>(stg + lane * 128 + (((4 * half + c) ^ (lane & 7)) << 4)) = w;
            }
            continue;  // the rows go out once both halves are staged
          }
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float* v = o + 8 * c;
            uint4 w;
            if (DT == kBF16)
              w = make_uint4(pack_bf16(v[0] * inv, v[1] * inv), pack_bf16(v[2] * inv, v[3] * inv),
                             pack_bf16(v[4] * inv, v[5] * inv), pack_bf16(v[6] * inv, v[7] * inv));
            else
              w = make_uint4(pack_f16(v[0] * inv, v[1] * inv), pack_f16(v[2] * inv, v[3] * inv),
                             pack_f16(v[4] * inv, v[5] * inv), pack_f16(v[6] * inv, v[7] * inv));
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) = w;
          }
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int rr = 4 * k + (lane >> 3), c = lane & 7;
            const uint4 w = *reinterpret_cast<const uint4*>(stg + rr * 128 + ((c ^ (rr & 7)) << 4));
            if (rr < rows_ok) *reinterpret_cast<uint4*>(obase + rr * orow_stride + half * 128 + c * 16) = w;
          }
          __syncwarp();
        }
        if constexpr (kQuant) {  // int8 rows of kD bytes: kD / 16 chunks, 32 / (kD / 16) rows per store
          constexpr int kChunks = kD / 16, kRowsPer = 32 / kChunks;
          uint8_t* qbase = static_cast<uint8_t*>(p.out) + (((int64_t)meta.tq + row0) * p.Nq + h) * (int64_t)kD;
          const int64_t qrow_stride = (int64_t)p.Nq * kD;
          __syncwarp();
#pragma unroll
          for (int k = 0; k < kChunks; ++k) {
            const int rr = kRowsPer * k + lane / kChunks, c = lane % kChunks;
            const uint4 w = *reinterpret_cast<const uint4*>(stg + rr * 128 + ((c ^ (rr & 7)) << 4));
            if (rr < rows_ok) *reinterpret_cast<uint4*>(qbase + rr * qrow_stride + c * 16) = w;
          }
          __syncwarp();
        }
        if (row_ok) {
          float sum_true = 0.f;
          if (m_fin != -INFINITY) {
            sum_true = (m_run == -INFINITY) ? 0.f : l_run * fast_exp2(m_run - m_fin);
            if (p.sink) sum_true += fast_exp2(sink2 - m_fin);
          }
          if (p.softmax_max) p.softmax_max[tok * p.Nq + h] = (m_fin == -INFINITY) ? -INFINITY : m_fin * kLn2;
          if (p.softmax_sum) p.softmax_sum[tok * p.Nq + h] = sum_true;
        }
        ++units;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kP2MmaWarpA) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

size_t prefill_workspace_bytes(int B, int Nq, int max_seqlen_q) {
  (void)Nq;
  const int64_t pairs = (int64_t)B * ((max_seqlen_q + kQT - 1) / kQT);
  return 256 + (size_t)(pairs > 0 ? pairs : 1) * sizeof(int);
}

namespace {

template <int kD, int DT>
cudaError_t launch_prefill_attention(const PrefillParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                     const CUtensorMap& tmV, int num_sms, cudaStream_t stream) {
  // a query sees keys d + i - pre.. with d + i <= Lkv - 1: a lower edge inside the keys needs
  // pre < the longest key sequence
  const bool band = p.pre < p.max_seqlen_kv;
  if (p.G % 2 == 0) {  // heads 2hp and 2hp + 1 share a kv head
    const size_t smem = sizeof(P2Smem<kD>);
    auto kern = p.pq_scale ? (band ? prefill_pair_kernel<kD, DT, true, true> : prefill_pair_kernel<kD, DT, false, true>)
                           : (band ? prefill_pair_kernel<kD, DT, true, false> : prefill_pair_kernel<kD, DT, false, false>);
    cudaError_t e = ensure_smem(kern, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_dependent(kern, num_sms, kP2Threads, smem, stream, tmQ, tmK, tmV, p);
  }
  const size_t smem = sizeof(PSmem<kD>);
  auto kern = p.pq_scale ? (band ? prefill_tc_kernel<kD, DT, true, true> : prefill_tc_kernel<kD, DT, false, true>)
                         : (band ? prefill_tc_kernel<kD, DT, true, false> : prefill_tc_kernel<kD, DT, false, false>);
  cudaError_t e = ensure_smem(kern, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<num_sms, kPThreads, smem, stream>>>(tmQ, tmK, tmV, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                           const CUtensorMap& tmV, int num_sms, cudaStream_t stream) {
  const int max_key_tiles = (p.max_seqlen_kv + kKT - 1) / kKT + 1;
  trace_mark(kKernelPrefill, 0, stream);
  const bool pairs = p.G % 2 == 0;
  const size_t plan_smem = prefill_plan_smem(max_key_tiles);
  cudaError_t e = cudaSuccess;
  if (plan_smem > 48 * 1024) {
    e = ensure_smem(prefill_plan_kernel, (int)plan_smem);
    if (e != cudaSuccess) return e;
  }
  // a warp per sequence of a chunk: a short batch needs few warps (fewer to synchronise)
  const int plan_threads = std::min(1024, std::max(128, (std::min(p.B, kPlanChunk) * 32 + 127) / 128 * 128));
  e = launch_dependent(prefill_plan_kernel, 1, plan_threads, plan_smem, stream, p, max_key_tiles, pairs ? 2 : 1);
  if (e != cudaSuccess) return e;
  if (p.D == 64)
    e = p.dtype == kBF16 ? launch_prefill_attention<64, kBF16>(p, tmQ, tmK, tmV, num_sms, stream)
                         : launch_prefill_attention<64, kF16>(p, tmQ, tmK, tmV, num_sms, stream);
  else
    e = p.dtype == kBF16 ? launch_prefill_attention<128, kBF16>(p, tmQ, tmK, tmV, num_sms, stream)
                         : launch_prefill_attention<128, kF16>(p, tmQ, tmK, tmV, num_sms, stream);
  trace_mark(kKernelPrefill, 1, stream);
  return e;
}

}  // namespace fia
