// decode_i8tc.cu -- paged GQA decode attention over an int8 KV cache on tcgen05 tensor
// cores (D = 128).
//
// Same operator, plan, work items, partial format and merge as decode.cu.  The
// per-channel antiquant (aclnnIncreFlashAttentionV3, "antiquantScale /
// antiquantOffset": k^ = (x - offset) * scale, the same for V with its own
// parameters) is affine, so this kernel never forms k^ or v^ element by element:
//
//   scores  S^T [128 tok x 32] = X_K [128 x D] . [Q'hi; Q'lo]^T   (decode_i8.cuh)
//           score (log2 units) = (S_hi + S_lo) kq + nq
//   values  O^T [D x 16]       = X_V^T [D x 128] . P^T
//           out_d              = s_v[d] * (O_d / l - o_v[d])
//
// X_K and X_V are the int8 codes, exact as fp16 integers.  The output side uses
// sum_t p_t (x_td - o_d) s_d = s_d (sum_t p_t x_td - o_d sum_t p_t); the PV MMA
// weighs with P rounded to fp16, the correction with the fp32 sum l, a difference
// of at most |o_d s_d| 2^-11 per output.
//
// Warp roles (608 threads):
//   warp 0      TMA producer: the item's q' block (one bulk copy from the workspace),
//               int8 K and V tiles (128 rows x 128 bytes, 128-byte swizzle) into a
//               6-stage ring; a slot is released by the commit of its tile's PV.
//   warp 1      TMEM allocation; one thread issues the score MMAs.
//   warp 14     one thread issues the PV MMAs (a second issue stream on another SM
//               sub-partition: an MMA blocks its issuing thread for about 50 cycles).
//   warps 2-5   online softmax of tile j (one token per TMEM lane); the PV products
//   and 15-18   of an item accumulate in TMEM (items alternate between two O buffers),
//               rescaled there in the rare tile that raises a head's reference; at the
//               item's end the final output or split partial (one channel per lane);
//               each group takes half of the heads.
//   warps 6-9   K codes -> fp16 pairs in TMEM (one token row per lane): the A
//               operand of the score MMA, double buffered.
//   warps 10-13 V codes -> fp16 in the tile's own ring slot (over the K codes already
//               read and the V codes as they are read), in the MN-major layout of the
//               A operand of the PV MMA.
// Each code takes one integer and one half-precision operation: the byte (plus
// 128) is placed under the exponent of 1024 and 1152 is subtracted.
#include <algorithm>

#include "decode_common.cuh"
#include "decode_i8.cuh"

namespace fia {
namespace {

constexpr int kT = 128;     // tokens per tile: the M of the score MMA
constexpr int kNP = 16;     // query heads per group, padded: the N of both MMAs
constexpr int kD = 128;     // head dim (the M of the PV MMA)
constexpr int kStages = 6;  // int8 ring (a slot also holds its tile's fp16 V until PV)
constexpr int kThreads = 608;
constexpr int kPvWarp = 14;     // issues the PV MMAs (warp 1 the score MMAs)
constexpr int kSm2Warp0 = 15;   // warps 15-18: the second softmax warp group
constexpr float kLazyMax = 8.f;  // log2 units: P stays below 2^8 between exchanges of maxima
// The reference of an item before any exchange: finite, so that a tile whose keys are all
// masked (scores -inf) gives P = 2^(-inf - kNoRef) = 0 on the no-exchange path, and below
// any real score by far more than kLazyMax, so that the first unmasked score exchanges.
constexpr float kNoRef = -1e30f;
constexpr int kBarSoftmax = 2;  // named barriers 2 and 3: the two softmax warp groups (128 threads each)
// TMEM columns.  An MMA of M = 128 costs the tensor pipe about the same for any
// N <= 64, so the hi and lo parts of q' share one MMA of N = 32.
constexpr int kNS = 2 * kNP;     // N of the score MMA
constexpr uint32_t kColS = 0;    // S: 2 buffers x 32 columns (hi scores, then lo scores)
constexpr uint32_t kColO = 64;   // O: 2 buffers x 16 columns
constexpr uint32_t kColK = 128;  // K codes: 2 buffers x 64 columns
constexpr uint32_t kTmemCols = 256;
constexpr int kI8Tile = kT * kD;      // bytes of one int8 K or V tile
constexpr int kPBytes = kNP * kT * 2;

struct __align__(16) I8Meta {
  int b, hkv, n, item;
  int first, last, qbuf, nch;
  int tok0, nlo, qlim, pad2;  // tok0: the tile's first token; tokens below tok0 + nlo are masked;
                              // query position i sees tokens up to qlim + i
};

constexpr int kMetaRing = 4;  // tile descriptors in flight between the K converters, MMA and softmax warps
constexpr int kQBufs = 2;     // q' blocks (the producer may run one item ahead of the one in the softmax)

struct I8Smem {
  // int8 K and V codes of a tile; after the K converters have read the K half, the V
  // converters write the tile's fp16 V over both halves (the PV MMA's A operand)
  alignas(1024) uint8_t kv[kStages][2][kI8Tile];
  alignas(1024) uint8_t q[kQBufs][kI8QBytes];
  alignas(1024) uint8_t p[2][kPBytes];
  alignas(16) float2 kn[kQBufs][kNP];
  alignas(16) float red[2][kNP][4];  // [S buffer][head][warp]: per-warp maxima
  float lsum[4][kNP];
  float lmax[4][kNP];  // [warp][head]: per-warp true maxima at an item's end
  float lref[kNP];     // [head]: the item's final reference (m_run) at its end
  I8Meta meta[kStages];    // per int8 stage (producer)
  I8Meta tmeta[kMetaRing];  // per tile j at j % kMetaRing (K converters)
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t kconv[kStages];  // K converters -> V converters: the slot's K codes have been read
  uint64_t k_full[2], q_full[kQBufs], q_empty[kQBufs];
  uint64_t v_full[kStages];  // per ring slot: the V converters may run ahead of PV by several tiles
  uint64_t s_full[2], p_full[2], pv_done[2];
  int pflag[2];  // per P buffer: bit 0 the tile starts its item, bit 1 the item's O buffer
  int pv_stop;  // index of the sentinel tile, set by the softmax warps when they reach it
  uint32_t tmem_base;
};
static_assert(sizeof(I8Smem) + 1024 <= 232448, "shared memory of the int8 decode kernel");


// Offset of element (row g, token t) of the P^T operand: two 64-token slabs of
// 16 rows x 128 bytes, 128-byte swizzle.
__device__ __forceinline__ uint32_t i8_p_offset(int g, int t) {
  const uint32_t slab = t >> 6, col = (t & 63) * 2;
  return slab * (kNP * 128) + swz((uint32_t)g * 128 + col, 7);
}

__device__ __forceinline__ void tmem_st32w(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// N consecutive 32-bit TMEM columns of this thread's lane (32x32b shape, N = 1, 2 or 4).
template <int N>
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const float (&v)[N]);
template <>
__device__ __forceinline__ void tmem_st_n<1>(uint32_t taddr, const float (&v)[1]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(__float_as_uint(v[0])) : "memory");
}
template <>
__device__ __forceinline__ void tmem_st_n<2>(uint32_t taddr, const float (&v)[2]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(taddr), "r"(__float_as_uint(v[0])),
               "r"(__float_as_uint(v[1]))
               : "memory");
}
template <>
__device__ __forceinline__ void tmem_st_n<4>(uint32_t taddr, const float (&v)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3]))
               : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T (A: rows on lanes, 16-bit pairs per column).
__device__ __forceinline__ void umma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Scores of GH heads h0 .. h0 + GH - 1 from one S buffer (hi partial sums in columns 0-15,
// lo in 16-31): only the columns of the calling warp group's heads are read.
template <int GH>
__device__ __forceinline__ void tmem_ld_scores_part(uint32_t taddr, int h0, float (&v)[GH]) {
  float hi[GH], lo[GH];
  tmem_ld_n<GH>(taddr + h0, hi);
  tmem_ld_n<GH>(taddr + kNP + h0, lo);
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < GH; ++i) v[i] = hi[i] + lo[i];
}


__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// kKeyMask: an attenMask or a band window removes keys inside the tiles (the softmax tests
// each token against them); without it a tile's first n tokens are its keys.
template <int QT, int GP, bool kKeyMask>
__global__ void __launch_bounds__(kThreads, 1)
    decode_i8tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmK16, const __grid_constant__ CUtensorMap tmV16,
                       const DecodeParams p, const int box_rows) {
  extern __shared__ uint8_t smem_raw[];
  I8Smem& sm = *reinterpret_cast<I8Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.GV;  // virtual heads (query heads x query positions) of a kv head

  // Synchronisation.  Buffers indexed by tile j use slot j & 1 (j % kStages for the
  // int8 ring); a slot is reused two tiles later, and most "free" signals follow
  // from program order:
  //   kv_full  TMA -> converters: codes of tile j in ring slot j % kStages
  //   kconv    K converters -> V converters: the slot's K codes have been read
  //   k_full   K converters -> MMA: codes of tile j in TMEM, descriptor in tmeta
  //   s_full   MMA commit of QK(j) -> softmax (scores ready) and K converters of
  //            tile j + 2 (the K buffer may be overwritten)
  //   p_full   softmax -> MMA: P(j) written.  Each softmax warp arrives after reading
  //            S(j) (and, when it rescaled it, O): the MMA warp may then overwrite
  //            the S buffer and accumulate into O
  //   v_full   V converters -> MMA: fp16 V of tile j in its ring slot (one barrier per
  //            slot: nothing else keeps the converters within a phase of the PV warp)
  //   pv_done  MMA commit of PV(j) -> softmax (O ready; P buffer free)
  //   kv_empty MMA commit of PV(j) -> TMA: ring slot j % kStages free
  if (tid == 0) {
    for (int i = 0; i < kQBufs; ++i) {
      mbar_init(&sm.q_full[i], 1);
      mbar_init(&sm.q_empty[i], 9);  // MMA commit after the item's last QK + the 8 softmax warps
                                     // after reading the item's constants at its last tile
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);  // the commit of the tile's PV product
      mbar_init(&sm.kconv[s], 4);     // the four K converter warps
      mbar_init(&sm.v_full[s], 4);    // the four V converter warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.k_full[i], 4);

      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.p_full[i], 8);
      mbar_init(&sm.pv_done[i], 1);
    }
    sm.pv_stop = 0x7fffffff;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&sm.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  griddep_wait();               // item list, counters and q' blocks of the plan launch are visible
  griddep_launch_dependents();  // the merge kernel may be scheduled; it waits for this grid to finish

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmK16);
      tma_prefetch_desc(&tmV16);
    }
    ItemQueue queue;
    queue.start(p, lane);
    const int bs = p.block_size;
    int j = 0, local_item = 0;
    bool ok = true;
    while (ok) {
      int4 desc;
      const int item = queue.pop(p, lane, &desc);
      if (item < 0) break;
      const DecodeItem it = decode_item(desc);
      const int b = it.b, hkv = it.hkv, t_begin = it.t_begin, t_end = it.t_end;
      const int t0 = t_begin & ~(kT - 1);  // the first tile (t_begin is aligned but for a window)
      const int qb = local_item % kQBufs;
      const int qlim = p.qs > 1 ? clamp_len(p, b, false) - p.qs : (1 << 30);  // position 0's last key
      if (!mbar_wait(&sm.q_empty[qb], ((uint32_t)(local_item / kQBufs) & 1u) ^ 1u, p.status)) { ok = false; break; }
      if (lane == 0) {
        const uint8_t* src = p.ws.qprep + ((int64_t)b * p.Nkv + hkv) * kI8QBlockBytes;
        mbar_arrive_expect_tx(&sm.q_full[qb], kI8QBlockBytes);
        bulk_load(sm.q[qb], src, kI8QBytes, &sm.q_full[qb]);
        bulk_load(sm.kn[qb], src + kI8QBytes, kI8QBlockBytes - kI8QBytes, &sm.q_full[qb]);
      }
      const int32_t* bt_row = p.block_table + (int64_t)b * p.bt_stride;
      for (int tok0 = t0; tok0 < t_end; tok0 += kT, ++j) {
        const int st = j % kStages;
        const uint32_t ph = (uint32_t)(j / kStages) & 1u;
        const int n = min(kT, t_end - tok0);
        // (tiles of fewer than 128 keys in 32-row pieces, as the 16-bit kernel does with 16-row
        // ones, measured 1% slower here: the tail map is passed but not used)
        const bool fine = false;
        const int prow = box_rows;
        const int npieces = (n + prow - 1) / prow;
        int32_t blk = 0;
        bool valid = false;
        if (lane < npieces) {
          blk = bt_row[(tok0 + lane * prow) / bs];
          valid = blk >= 0 && (int64_t)blk < p.num_blocks;
          if (!valid) raise_status(p.status, kStatusBadBlockIndex);
        }
        const unsigned vmask = __ballot_sync(0xffffffffu, valid);
        const uint32_t bytes = 2u * (uint32_t)prow * 128u * __popc(vmask);
        if (!mbar_wait(&sm.kv_empty[st], ph ^ 1u, p.status)) { ok = false; break; }
        if (lane == 0) {
          I8Meta& m = sm.meta[st];
          m.b = b; m.hkv = hkv; m.n = n; m.item = item;
          m.first = (tok0 == t0); m.last = (tok0 + kT >= t_end); m.qbuf = qb; m.nch = it.nch; m.tok0 = tok0;
          m.nlo = max(t_begin - tok0, 0);
          m.qlim = qlim;
          if (bytes) mbar_arrive_expect_tx(&sm.kv_full[st], bytes);
          else mbar_arrive(&sm.kv_full[st]);
        }
        __syncwarp();
        if (valid) {
          const KvCoord kc = kv_coord(p, blk, tok0 + lane * prow, hkv);
          const uint32_t off = (uint32_t)lane * prow * 128u;
          tma_load_2d(sm.kv[st][0] + off, fine ? &tmK16 : &tmK, kc.x0, kc.row, &sm.kv_full[st]);
          tma_load_2d(sm.kv[st][1] + off, fine ? &tmV16 : &tmV, kc.x0, kc.row, &sm.kv_full[st]);
        }
        if (tok0 == t0) queue.prefetch(p, lane);
      }
      ++local_item;
    }
    if (ok) {  // sentinel tile: no more work
      const int st = j % kStages;
      if (mbar_wait(&sm.kv_empty[st], ((uint32_t)(j / kStages) & 1u) ^ 1u, p.status) && lane == 0) {
        sm.meta[st].item = -1;
        mbar_arrive(&sm.kv_full[st]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ score MMAs
    if (lane == 0) {
      constexpr uint32_t idesc_qk = umma_idesc_f16(0, 0, 0, kT, kNS);  // fp16, A (TMEM) and B K-major
      int local_item = 0;
      for (int j = 0;; ++j) {
        const int kb = j & 1;
        if (!mbar_wait(&sm.k_full[kb], (uint32_t)(j >> 1) & 1u, p.status)) break;
        // the S buffer of tile j - 2 has been read (its P written)
        if (j >= 2 && !mbar_wait(&sm.p_full[kb], ((uint32_t)(j >> 1) & 1u) ^ 1u, p.status)) break;
        const I8Meta meta = sm.tmeta[j % kMetaRing];
        if (meta.item < 0) {
          mbar_arrive(&sm.s_full[kb]);  // the softmax warps see the sentinel
          break;
        }
        const int qb = meta.qbuf;
        if (meta.first && !mbar_wait(&sm.q_full[qb], (uint32_t)(local_item / kQBufs) & 1u, p.status)) break;
        tc_fence_after();
        const uint32_t tk = tmem + kColK + kb * 64;
        const uint32_t ts = tmem + kColS + kb * kNS;
        const uint64_t b0 = umma_desc(smem_u32(sm.q[qb]), 16, 1024);
#pragma unroll
        for (int s = 0; s < kD / 16; ++s)  // 16 channels per step
          umma_f16_tmem_a(ts, tk + s * 8, b0 + ((((s >> 2) * (kI8QRows * 128)) + (s & 3) * 32) >> 4), idesc_qk, s > 0);
        umma_commit(&sm.s_full[kb]);
        if (meta.last) {
          umma_commit(&sm.q_empty[qb]);
          ++local_item;
        }
      }
    }
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------------ PV MMAs
    // A warp of its own on another SM sub-partition, so that the two product streams
    // are issued in parallel; the tensor pipe runs them interleaved.
    if (lane == 0) {
      constexpr uint32_t idesc_pv = umma_idesc_f16(0, 1, 0, kT, kNP);  // fp16, A = V^T read MN-major
      for (int j = 0;; ++j) {
        const int pb = j & 1;
        const uint32_t ph = (uint32_t)(j >> 1) & 1u;
        if (!mbar_wait(&sm.p_full[pb], ph, p.status)) break;
        if (j >= *static_cast<volatile int*>(&sm.pv_stop)) break;  // tile j is the sentinel
        if (!mbar_wait(&sm.v_full[j % kStages], (uint32_t)(j / kStages) & 1u, p.status)) break;
        tc_fence_after();
        // O of the tile's item accumulates over its tiles; its first tile overwrites it
        const int fl = *static_cast<volatile int*>(&sm.pflag[pb]);
        const uint32_t ocol = tmem + kColO + (uint32_t)(fl >> 1) * kNP;
        const uint64_t a0 = umma_desc(smem_u32(sm.kv[j % kStages][0]), kT * 128, 1024);
        const uint64_t b0 = umma_desc(smem_u32(sm.p[pb]), 16, 1024);
#pragma unroll
        for (int s = 0; s < kT / 16; ++s)  // 16 tokens per step
          umma_f16(ocol, a0 + ((s * 16 * 128) >> 4), b0 + ((((s >> 2) * (kNP * 128)) + (s & 3) * 32) >> 4),
                   idesc_pv, (s > 0 || !(fl & 1)) ? 1u : 0u);
        umma_commit(&sm.pv_done[pb]);
        umma_commit(&sm.kv_empty[j % kStages]);  // the tile's codes and fp16 V are no longer needed
      }
    }
  } else if (warp < 6 || warp >= kSm2Warp0) {
    // ------------------------------------------------------------------ softmax + correction
    // Two warp groups share the work of each tile: group 0 (warps 2-5) takes heads
    // [0, GH), group 1 (warps 15-18) heads [GH, 2 GH), so that each thread's chain of
    // dependent steps per tile is half as long.
    constexpr int GH = GP / 2;
    const bool upper = warp >= kSm2Warp0;
    const int h0 = upper ? GH : 0;
    // The groups exchange maxima and sums only among their own four warps.  (At the
    // sentinel, the PV thread sees pv_stop: thread 64 writes it before its warp arrives.)
    const int bar_group = kBarSoftmax + (upper ? 1 : 0);
    const int quad = warp & 3;       // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;  // TMEM lane: token of S, channel of O
    const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16);
    // Lazy maximum: m_run is a reference for each head, the same in all threads of the group,
    // and P = 2^(score - m_run).  A tile whose scores all stay below m_run + kLazyMax (one
    // barrier-reduction tells) keeps the reference, with no exchange of maxima; otherwise
    // the tile's exact maximum is exchanged and the reference raised.  m_thr is each
    // thread's true maximum, combined at the item's end for the max and sum outputs.
    float m_run[GH], l_part[GH], m_thr[GH];
    int vpos[GH];  // query position of each of this group's virtual heads
#pragma unroll
    for (int g = 0; g < GH; ++g) {
      m_run[g] = kNoRef; l_part[g] = 0.f; m_thr[g] = -INFINITY;
      vpos[g] = kKeyMask ? (h0 + g) / p.G : 0;
    }
    float vs_cur = 0.f, vo_cur = 0.f;  // value antiquant of channel r for the current item
    int prev_item = -1, prev_b = 0, prev_hkv = 0, prev_nch = 1;
    int ob = 1;  // O buffer of the current item (items alternate between the two)
    // The epilogue of a finished item waits until the softmax of the next item's first tile
    // has released its P, so that the products of the new item run meanwhile.  Its row
    // partials (sums and maxima reduced over each warp, and the final reference) were left
    // in shared memory at its last tile; these hold the rest.
    bool pending = false;
    int pend_item = 0, pend_b = 0, pend_hkv = 0, pend_nch = 1;
    float pend_vs = 0.f, pend_vo = 0.f;

    // At an item's last tile: this warp's partial sums and maxima, and the reference.
    auto park = [&]() {
      float lv[GH], mt[GH];
#pragma unroll
      for (int g = 0; g < GH; ++g) {
        lv[g] = l_part[g];
        mt[g] = m_thr[g];
      }
#pragma unroll
      for (int off = 16; off; off >>= 1)
#pragma unroll
        for (int g = 0; g < GH; ++g) {
          lv[g] += __shfl_xor_sync(0xffffffffu, lv[g], off);
          mt[g] = fmaxf(mt[g], __shfl_xor_sync(0xffffffffu, mt[g], off));
        }
      if (lane == 0) {
#pragma unroll
        for (int g = 0; g < GH; ++g) {
          sm.lsum[quad][h0 + g] = lv[g];
          sm.lmax[quad][h0 + g] = mt[g];
          if (quad == 0) sm.lref[h0 + g] = m_run[g];
        }
      }
    };

    // The epilogue of the pending item (last tile jj, O buffer obuf): final output, or split
    // partial.
    auto finish = [&](int jj, int obuf) -> bool {
      named_bar_sync(bar_group, 128);  // every warp of the group has parked its partials
      if (!mbar_wait(&sm.pv_done[jj & 1], (uint32_t)(jj >> 1) & 1u, p.status)) return false;
      tc_fence_after();
      float o[GH];  // this group's heads only
      tmem_ld_n<GH>(tq + kColO + obuf * kNP + h0, o);
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      // (mm, lt): the head's true maximum and the sum relative to it; a relative to it too
      float mm[GH], lt[GH], a[GH];
#pragma unroll
      for (int g = 0; g < GH; ++g) {
        mm[g] = fmax3(fmaxf(sm.lmax[0][h0 + g], sm.lmax[1][h0 + g]), sm.lmax[2][h0 + g], sm.lmax[3][h0 + g]);
        const float sc = (mm[g] == -INFINITY) ? 0.f : exp2f(sm.lref[h0 + g] - mm[g]);
        lt[g] = (sm.lsum[0][h0 + g] + sm.lsum[1][h0 + g] + sm.lsum[2][h0 + g] + sm.lsum[3][h0 + g]) * sc;
        a[g] = pend_vs * fmaf(-pend_vo, lt[g], o[g] * sc);  // sum_t 2^(s_t - mm) v^_t, unnormalised
      }
      if (pend_nch == 1 && !p.partials_only) {
#pragma unroll
        for (int g = 0; g < GH; ++g) {
          const int hg = h0 + g;
          if (hg < G) {
            // several query positions run only on the key-mask instantiation; the plain one keeps
            // the one-position rows (measured: the general mapping here slowed every tile by 4%)
            const int64_t row = kKeyMask ? q_row(p, pend_b, pend_hkv, hg) : (int64_t)pend_b * p.Nq + pend_hkv * G + hg;
            const int h = kKeyMask ? q_head(p, pend_hkv, hg) : pend_hkv * G + hg;
            float M, W;
            const float v = single_item_output(a[g], mm[g], lt[g], p.sink, h, &M, &W);
            store_out<QT>(p.out, row * kD + r, v);
            if (r == hg) {
              if (p.softmax_max) p.softmax_max[row] = (M == -INFINITY) ? -INFINITY : M * kLn2;
              if (p.softmax_sum) p.softmax_sum[row] = W;
            }
          }
        }
      } else {
        float* po = p.ws.part_o + (int64_t)pend_item * G * kD;
#pragma unroll
        for (int g = 0; g < GH; ++g)
          if (h0 + g < G) po[(h0 + g) * kD + r] = lt[g] > 0.f ? a[g] / lt[g] : 0.f;
        if (r >= h0 && r < h0 + GH && r < G) {
          float mv = mm[0], lw = lt[0];
#pragma unroll
          for (int g = 1; g < GH; ++g)
            if (r == h0 + g) { mv = mm[g]; lw = lt[g]; }
          p.ws.part_ml[(int64_t)pend_item * G + r] = make_float2(mv, lw);
        }
      }
      named_bar_sync(bar_group, 128);  // the parked partials may be overwritten
      pending = false;
      return true;
    };

    int j = 0;
    bool ok = true;
    while (true) {
      const int sb = j & 1;
      const uint32_t sph = (uint32_t)(j >> 1) & 1u;
      if (!mbar_wait(&sm.s_full[sb], sph, p.status)) { ok = false; break; }
      const I8Meta meta = sm.tmeta[j % kMetaRing];
      if (meta.item < 0) {  // no more tiles: wake the PV warp, which stops
        if (tid == 64) sm.pv_stop = j;
        named_bar_sync(bar_group, 128);
        if (lane == 0) mbar_arrive(&sm.p_full[sb]);
        break;
      }
      if (meta.first) {  // the previous item's epilogue waits (see finish); start this one
        if (j > 0) {
          pending = true;
          pend_item = prev_item; pend_b = prev_b; pend_hkv = prev_hkv; pend_nch = prev_nch;
          pend_vs = vs_cur; pend_vo = vo_cur;
        }
        const int64_t vi = ((int64_t)p.Nkv + meta.hkv) * kD + r;  // value scale/offset: index 1 of (2, Nkv, D)
        vs_cur = p.aq_scale[vi];
        vo_cur = p.aq_offset ? p.aq_offset[vi] : 0.f;
        ob ^= 1;
#pragma unroll
        for (int g = 0; g < GH; ++g) {
          m_run[g] = kNoRef;
          l_part[g] = 0.f;
          m_thr[g] = -INFINITY;
        }
      }
      tc_fence_after();
      float s[GH];  // scores of this group's heads
      tmem_ld_scores_part<GH>(tq + kColS + sb * kNS, h0, s);
      const bool valid = r < meta.n && (!kKeyMask || (r >= meta.nlo && !key_masked(p, meta.b, meta.tok0 + r)));
      float x[GH];
      const float2* kn = sm.kn[meta.qbuf] + h0;  // {kq, nq} of this group's heads (decode_i8.cuh)
      bool above = false;  // a score of this thread exceeds its head's reference by kLazyMax
#pragma unroll
      for (int g = 0; g < GH; ++g) {
        const float2 c = kn[g];
        // (several query positions: position i sees tokens up to qlim + i)
        bool vis = valid;
        if constexpr (kKeyMask) vis = vis && meta.tok0 + r <= meta.qlim + vpos[g];
        x[g] = vis ? fmaf(s[g], c.x, c.y) : -INFINITY;
        above |= x[g] > m_run[g] + kLazyMax;  // (the unset reference, kNoRef, is exceeded by any score)
        m_thr[g] = fmaxf(m_thr[g], x[g]);
      }
      if (meta.last) {  // the q' buffer may be refilled once the MMA thread is done with it too
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.q_empty[meta.qbuf]);
      }
      float alpha[GH], pr[GH];
      if (named_bar_or(bar_group, 128, above)) {  // exact maximum of the tile, reference raised
        float mx[GH];
#pragma unroll
        for (int g = 0; g < GH; ++g) mx[g] = warp_max(x[g]);
        if (lane == 0) {
#pragma unroll
          for (int g = 0; g < GH; ++g) sm.red[sb][h0 + g][quad] = mx[g];
        }
        named_bar_sync(bar_group, 128);
#pragma unroll
        for (int g = 0; g < GH; ++g) {
          const float4 rq = *reinterpret_cast<const float4*>(sm.red[sb][h0 + g]);  // the four quadrants' maxima
          const float tmax = fmax3(fmaxf(rq.x, rq.y), rq.z, rq.w);
          const float m_new = fmaxf(m_run[g], tmax);
          const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
          alpha[g] = fast_exp2(m_run[g] - m_use);
          pr[g] = fast_exp2(x[g] - m_use);
          l_part[g] = fmaf(l_part[g], alpha[g], pr[g]);
          m_run[g] = m_new;
        }
        if (!meta.first) {  // O holds the item's earlier tiles relative to the old reference
          if (!mbar_wait(&sm.pv_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u, p.status)) { ok = false; break; }
          tc_fence_after();
          float o[GH];
          tmem_ld_n<GH>(tq + kColO + ob * kNP + h0, o);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
          for (int g = 0; g < GH; ++g) o[g] *= alpha[g];
          tmem_st_n<GH>(tq + kColO + ob * kNP + h0, o);
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        }
      } else {  // every score within 2^kLazyMax of the reference: keep it
#pragma unroll
        for (int g = 0; g < GH; ++g) {
          alpha[g] = 1.f;
          pr[g] = fast_exp2(x[g] - m_run[g]);
          l_part[g] += pr[g];
        }
      }
      uint8_t* pbuf = sm.p[sb];
      // the P buffer is free once PV(j - 2) has completed
      if (j >= 2 && !mbar_wait(&sm.pv_done[sb], sph ^ 1u, p.status)) { ok = false; break; }
#pragma unroll
      for (int g = 0; g < GH; ++g)
        if (h0 + g < G)
          *reinterpret_cast<uint16_t*>(pbuf + i8_p_offset(h0 + g, r)) = __half_as_ushort(__float2half_rn(pr[g]));
      if (warp == 2 && lane == 0) sm.pflag[sb] = (meta.first ? 1 : 0) | (ob << 1);
      fence_proxy_async_smem();
      tc_fence_before();  // the tensor-memory accesses of S(j) (and O) precede the arrival
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_full[sb]);
      if (pending && !finish(j - 1, ob ^ 1)) { ok = false; break; }  // (this tile starts an item)
      if (meta.last) park();
      prev_item = meta.item;
      prev_b = meta.b;
      prev_hkv = meta.hkv;
      prev_nch = meta.nch;
      ++j;
    }
    if (ok && j > 0) {  // the last item: its partials were parked at its last tile
      pend_item = prev_item; pend_b = prev_b; pend_hkv = prev_hkv; pend_nch = prev_nch;
      pend_vs = vs_cur; pend_vo = vo_cur;
      finish(j - 1, ob);
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------------ K codes -> TMEM
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16);
    for (int j = 0;; ++j) {
      const int st = j % kStages;
      if (!mbar_wait(&sm.kv_full[st], (uint32_t)(j / kStages) & 1u, p.status)) break;
      const I8Meta meta = sm.meta[st];
      const int kb = j & 1;
      // QK(j - 2) has completed: the K buffer is free, and the softmax warps have read tmeta of tile j - 4
      if (!mbar_wait(&sm.s_full[kb], ((uint32_t)(j >> 1) & 1u) ^ 1u, p.status)) break;
      if (warp == 6 && lane == 0) sm.tmeta[j % kMetaRing] = meta;
      if (meta.item < 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.k_full[kb]);
        break;
      }
      const uint32_t row = smem_u32(sm.kv[st][0]) + r * 128;
      tc_fence_after();
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t v[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int chunk = half * 4 + c;
          const uint4 w = lds128(row + ((chunk ^ (r & 7)) << 4));
          codes_to_f16x2(w.x, v[c * 8 + 0], v[c * 8 + 1]);
          codes_to_f16x2(w.y, v[c * 8 + 2], v[c * 8 + 3]);
          codes_to_f16x2(w.z, v[c * 8 + 4], v[c * 8 + 5]);
          codes_to_f16x2(w.w, v[c * 8 + 6], v[c * 8 + 7]);
        }
        tmem_st32w(tq + kColK + kb * 64 + half * 32, v);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.kconv[st]);
        mbar_arrive(&sm.k_full[kb]);
      }
    }
  } else if (warp < 14) {
    // ------------------------------------------------------------------ V codes -> shared memory
    const int r = (warp - 10) * 32 + lane;
    for (int j = 0;; ++j) {
      const int st = j % kStages;
      if (!mbar_wait(&sm.kv_full[st], (uint32_t)(j / kStages) & 1u, p.status)) break;
      if (sm.meta[st].item < 0) break;
      // fp16 channels 0-63 of row r go over K row r: the K converters must have read it.
      // Channels 64-127 go over this row's own codes, each 16-byte chunk after the codes
      // it overwrites have been read (chunk c of codes feeds fp16 chunks 2c and 2c + 1).
      if (!mbar_wait(&sm.kconv[st], (uint32_t)(j / kStages) & 1u, p.status)) break;
      const uint32_t row = smem_u32(sm.kv[st][1]) + r * 128;
      const uint32_t dst = smem_u32(sm.kv[st][0]) + r * 128;
#pragma unroll
      for (int chunk = 0; chunk < 8; ++chunk) {
        const uint4 w = lds128(row + ((chunk ^ (r & 7)) << 4));
        uint32_t h[8];
        codes_to_f16x2(w.x, h[0], h[1]);
        codes_to_f16x2(w.y, h[2], h[3]);
        codes_to_f16x2(w.z, h[4], h[5]);
        codes_to_f16x2(w.w, h[6], h[7]);
        // channels 16 chunk .. +7 and +8 .. +15: fp16 chunks 2 chunk and 2 chunk + 1
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int cc = 2 * chunk + hf;
          const uint32_t a = dst + (cc >> 3) * (kT * 128) + ((((uint32_t)cc & 7u) ^ ((uint32_t)r & 7u)) << 4);
          sts128(a, h[hf * 4 + 0], h[hf * 4 + 1], h[hf * 4 + 2], h[hf * 4 + 3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.v_full[st]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int QT, int GP>
cudaError_t launch_i8(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap* tail,
                      int box_rows, int grid, cudaStream_t stream) {
  const size_t smem = sizeof(I8Smem) + 1024;
  auto kern = (p.atten_mask || p.windowed || p.qs > 1) ? decode_i8tc_kernel<QT, GP, true>
                                                       : decode_i8tc_kernel<QT, GP, false>;
  cudaError_t e = ensure_smem(kern, (int)smem);
  if (e != cudaSuccess) return e;
  trace_mark(kKernelDecodeAttention, 0, stream);
  e = launch_dependent(kern, grid, kThreads, smem, stream, tmK, tmV, tail[0], tail[1], p, box_rows);
  trace_mark(kKernelDecodeAttention, 1, stream);
  return e;
}

template <int QT>
cudaError_t launch_i8_g(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap* tail,
                        int box_rows, int grid, cudaStream_t stream) {
  if (p.GV <= 2) return launch_i8<QT, 2>(p, tmK, tmV, tail, box_rows, grid, stream);
  if (p.GV <= 4) return launch_i8<QT, 4>(p, tmK, tmV, tail, box_rows, grid, stream);
  if (p.GV <= 8) return launch_i8<QT, 8>(p, tmK, tmV, tail, box_rows, grid, stream);
  return cudaErrorInvalidValue;  // int8 groups above 8 are rejected before launch
}

}  // namespace

cudaError_t launch_decode_i8tc_attention(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                         const CUtensorMap* tail, int box_rows, int grid, cudaStream_t stream) {
  return p.q_dtype == kBF16 ? launch_i8_g<kBF16>(p, tmK, tmV, tail, box_rows, grid, stream)
                            : launch_i8_g<kF16>(p, tmK, tmV, tail, box_rows, grid, stream);
}

// ------------------------------------------------------------------- probes
// The exact steps of this kernel on their own: the code -> fp16 conversion of the K and V
// converter warps, and the query operand (q' = q * s_K as an fp16 hi + lo pair after the
// power-of-two prescale, and the per-head constants) that the plan kernel prepares.
namespace {

__global__ void debug_i8_codes_kernel(const uint32_t* words, int64_t nw, uint2* out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nw; i += (int64_t)gridDim.x * blockDim.x) {
    uint32_t h01, h23;
    codes_to_f16x2(words[i], h01, h23);
    out[i] = make_uint2(h01, h23);
  }
}

// One warp per row of a q' block, as in the plan kernel's extra CTAs.
__global__ void debug_i8_qprep_kernel(const DecodeParams p) {
  const int64_t R = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (R < (int64_t)p.B * p.Nkv * kI8Heads) i8_qprep_row(p, R, threadIdx.x & 31);
}

// The blocks read back through the same layout function: hi and lo parts of row g, channel d,
// and the {kq, nq} pair of head g.
__global__ void debug_i8_qunpack_kernel(const uint8_t* blocks, int64_t nblk, uint16_t* hi, uint16_t* lo,
                                        float2* kn) {
  const int64_t n = nblk * kI8Heads * 128;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t blk = i / (kI8Heads * 128);
    const int g = (int)(i / 128 % kI8Heads), d = (int)(i % 128);
    const uint8_t* base = blocks + blk * kI8QBlockBytes;
    hi[i] = *reinterpret_cast<const uint16_t*>(base + i8q_offset(g, d));
    lo[i] = *reinterpret_cast<const uint16_t*>(base + i8q_offset(kI8Heads + g, d));
    if (d == 0) kn[blk * kI8Heads + g] = reinterpret_cast<const float2*>(base + kI8QBytes)[g];
  }
}

}  // namespace

size_t debug_i8_qprep_block_bytes() { return kI8QBlockBytes; }

cudaError_t launch_debug_i8_codes(const int8_t* codes, int64_t n, uint16_t* out, cudaStream_t stream) {
  const int64_t nw = n / 4;
  if (nw <= 0) return cudaSuccess;
  const int grid = (int)std::min<int64_t>((nw + 255) / 256, 4096);
  debug_i8_codes_kernel<<<grid, 256, 0, stream>>>(reinterpret_cast<const uint32_t*>(codes), nw,
                                                   reinterpret_cast<uint2*>(out));
  return cudaGetLastError();
}

cudaError_t launch_debug_i8_qprep(const DecodeParams& p, uint16_t* hi, uint16_t* lo, float* kn,
                                  cudaStream_t stream) {
  const int64_t rows = (int64_t)p.B * p.Nkv * kI8Heads;
  if (rows <= 0) return cudaSuccess;
  debug_i8_qprep_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t n = rows * 128;
  const int grid = (int)std::min<int64_t>((n + 255) / 256, 4096);
  debug_i8_qunpack_kernel<<<grid, 256, 0, stream>>>(p.ws.qprep, (int64_t)p.B * p.Nkv, hi, lo,
                                                    reinterpret_cast<float2*>(kn));
  return cudaGetLastError();
}

}  // namespace fia
