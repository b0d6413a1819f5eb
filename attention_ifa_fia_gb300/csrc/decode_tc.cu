// decode_tc.cu -- paged GQA decode attention on tcgen05 tensor cores (fp16 / bf16 KV).
//
// Same operator, plan, work items, partial format and merge as decode.cu (see the
// header there); only the attention kernel differs.  Per 128-token tile of one
// (b, kv-head) work item, the whole GQA group is computed by two MMAs with the
// tokens on the M dimension ("swap AB"), so that a group of G <= 16 query heads
// only pads N to 16:
//
//   S^T [128 tok x 16] = K [128 x D] . Q^T          A = K tile (K-major, TMA 128B swizzle)
//                                                    B = Q rows of the group (K-major)
//   O^T [D x 16]       = V^T [D x 128] . P^T         A = V tile read MN-major
//                                                    B = P^T written by the softmax warps
//
// Both accumulators live in tensor memory (double buffered).  For D = 64 the PV
// product uses M = 128 by stacking the two 64-token halves of the V tile as the
// two halves of A (rows 0-63: tokens 0-63, rows 64-127: tokens 64-127) and issuing
// one MMA per half against the matching half of P^T into separate accumulators.
//
// Warp roles (352 threads): warp 0 issues TMA loads (Q of each item, K and V tiles
// into a 3- or 5-stage ring); warp 1 allocates tensor memory and one thread issues
// the score MMAs, one thread of warp 6 the PV MMAs.  Warps 2-5 and warps 7-10 are
// two groups that each own TMEM lanes 0-127 for half of the query heads: online
// softmax of tile j (one token per lane, warp max across lanes) followed by the
// rescale-and-accumulate of the PV result of tile j-1 (one output channel per lane).
#include "decode_common.cuh"

namespace fia {
namespace {

constexpr int kT = 128;          // tokens per tile: the M of the score MMA
constexpr int kNP = 16;          // query heads per group, padded: the N of both MMAs
constexpr int kTmemCols = 128;
constexpr int kThreadsTC = 352;
constexpr int kPvWarpTC = 6;     // issues the PV MMAs (warp 1 the score MMAs)
constexpr int kSm2Warp0 = 7;     // warps 7-10: the second softmax warp group
constexpr int kBarCompute = 2;   // named barriers 2 and 3: the two softmax warp groups (128 threads each)

template <int D>
struct TcCfg {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kNumBoxes = kRowBytes / 128;  // 64-element column boxes per row
  static constexpr int kTileBytes = kT * kRowBytes;   // K or V tile
  static constexpr int kStages = (D == 128) ? 3 : 5;
  static constexpr int kQBytes = kNP * kRowBytes;
  static constexpr int kPBytes = kNP * kT * 2;
  static constexpr int kKSteps = D / 16;
  static constexpr bool kStacked = (D == 64);
  static constexpr uint32_t kColS = 0;                       // S buffers: [0, 32)
  static constexpr uint32_t kColO = 32;                      // O buffers: [32, 64) or [32, 96)
  static constexpr uint32_t kOStride = kStacked ? 32 : 16;   // columns per O buffer
};

struct __align__(16) TileMeta {
  int b, hkv, tok0, n;
  int item, first, last, qbuf;
  int nch, nlo, qlim, pad2;  // nch: items of this (b, kv head) segment; tokens tok0 .. tok0 + nlo - 1
                             // lie before the window and are masked; with several query positions
                             // position i sees tokens up to qlim + i
};

template <int D>
struct TcSmem {
  using C = TcCfg<D>;
  alignas(1024) uint8_t kv[C::kStages][2][C::kTileBytes];
  alignas(1024) uint8_t q[2][C::kQBytes];
  alignas(1024) uint8_t p[2][C::kPBytes];
  alignas(16) float red[2][kNP][4];  // [S buffer][head][warp]: per-warp maxima
  float lsum[4][kNP];
  float accx[C::kStacked ? 64 : 1][kNP];
  TileMeta meta[C::kStages];
  uint64_t kv_full[C::kStages], kv_empty[C::kStages];
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2], p_full[2];
  int pv_stop;  // index of the sentinel tile, set by the softmax warps when they reach it
  uint32_t tmem_base;
  FusedPlan plan;  // the in-kernel schedule (p.fused_plan)
};

// Offset of element (row g, token t) of the P^T operand: two 64-token slabs of
// 16 rows x 128 bytes, 128-byte swizzle (8-row atoms of 1 KB).
__device__ __forceinline__ uint32_t p_offset(int g, int t) {
  const uint32_t slab = t >> 6, col = (t & 63) * 2;
  const uint32_t off = (uint32_t)g * 128 + col;  // within the slab (rows of 128 B)
  return slab * (kNP * 128) + swz(off, 7);
}

// kKeyMask: an attenMask or a band window removes keys inside the tiles (the softmax tests
// each token against them); without it a tile's first n tokens are its keys.
template <int D, int DT, int GP, bool kKeyMask>
__global__ void __launch_bounds__(kThreadsTC, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK16,
                     const __grid_constant__ CUtensorMap tmV16, const DecodeParams p, const int box_rows) {
  using C = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  TcSmem<D>& sm = *reinterpret_cast<TcSmem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.G, GV = p.GV;  // GV: virtual heads (query heads x positions) of a kv head

  // Synchronisation.  kv_full: TMA -> score warp.  s_full: QK(j) committed -> softmax.
  // p_full: the four softmax warps -> PV warp (P(j) written) and score warp; each warp
  // arrives after reading S(j) and, earlier in its program, O(j - 2), so QK(j + 2) and
  // PV(j) may overwrite those S and O buffers.  kv_empty: PV(j) committed -> producer
  // (stage free) and softmax (O(j) ready, P buffer free).  q_empty: the item's last QK
  // committed -> producer.
  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.q_full[i], 1);
      mbar_init(&sm.q_empty[i], 1);
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.p_full[i], 8);
    }
    sm.pv_stop = 0x7fffffff;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&sm.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  griddep_wait();  // the plan kernel's item list, counters and reset are complete and visible
  griddep_launch_dependents();  // the merge kernel may be scheduled; it waits for this grid to finish
  if (p.fused_plan) fused_plan_build(p, sm.plan, tid, kThreadsTC);  // (no plan launch preceded)

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK16);
      tma_prefetch_desc(&tmV16);
    }
    ItemQueue queue;
    if (!p.fused_plan) queue.start(p, lane);
    const int bs = p.block_size;
    int j = 0, local_item = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
      int4 desc;
      int item;
      if (p.fused_plan) {  // this CTA's next slot of the in-kernel schedule
        const int slot = fused_plan_slot(round, gridDim.x);
        item = slot < sm.plan.n_items ? fused_plan_item(p, sm.plan, slot, &desc) : -1;
      } else {
        item = queue.pop(p, lane, &desc);
      }
      if (item < 0) break;
      const DecodeItem it = decode_item(desc);
      const int b = it.b, hkv = it.hkv, t_begin = it.t_begin, t_end = it.t_end;
      const int t0 = t_begin & ~(kT - 1);  // the first tile (t_begin is aligned but for a window)
      const int qb = local_item & 1;
      if (!mbar_wait(&sm.q_empty[qb], ((local_item >> 1) & 1) ^ 1u, p.status)) { ok = false; break; }
      int qlim = 1 << 30;  // the last token position 0 sees (several query positions only)
      if (p.qs > 1) qlim = (p.fused_plan ? sm.plan.end[b] : clamp_len(p, b, false)) - p.qs;
      if (lane == 0) {
        if (p.qs == 1) {  // the group's 16 query rows (rows past G belong to other heads: unused)
          mbar_arrive_expect_tx(&sm.q_full[qb], C::kQBytes);
          const int32_t row = b * p.Nq + hkv * G;
          for (int bx = 0; bx < C::kNumBoxes; ++bx)
            tma_load_2d(sm.q[qb] + bx * (kNP * 128), &tmQ, bx * 64, row, &sm.q_full[qb]);
        } else {  // (64 channels, G heads, qs positions) boxes: rows v = i * G + g
          mbar_arrive_expect_tx(&sm.q_full[qb], (uint32_t)(C::kNumBoxes * GV * 128));
          for (int bx = 0; bx < C::kNumBoxes; ++bx)
            tma_load_3d(sm.q[qb] + bx * (kNP * 128), &tmQ, bx * 64, hkv * G, b * p.qs, &sm.q_full[qb]);
        }
      }
      const int32_t* bt_row = p.block_table + (int64_t)b * p.bt_stride;
      for (int tok0 = t0; tok0 < t_end; tok0 += kT, ++j) {
        const int st = j % C::kStages;
        const uint32_t ph = (uint32_t)(j / C::kStages) & 1u;
        const int n = min(kT, t_end - tok0);
        // a tile holding fewer than 128 keys (an item's last) is read in 16-row pieces, so that
        // rows past its keys are not fetched from memory
        const bool fine = n < kT && box_rows > 16;
        const int prow = fine ? 16 : box_rows;
        const int npieces = (n + prow - 1) / prow;
        int32_t blk = 0;
        bool valid = false;
        if (lane < npieces) {
          blk = bt_row[(tok0 + lane * prow) / bs];
          valid = blk >= 0 && (int64_t)blk < p.num_blocks;
          if (!valid) raise_status(p.status, kStatusBadBlockIndex);
        }
        const unsigned vmask = __ballot_sync(0xffffffffu, valid);
        const uint32_t bytes = 2u * (uint32_t)prow * C::kRowBytes * __popc(vmask);
        if (!mbar_wait(&sm.kv_empty[st], ph ^ 1u, p.status)) { ok = false; break; }
        if (lane == 0) {
          TileMeta& m = sm.meta[st];
          m.b = b; m.hkv = hkv; m.tok0 = tok0; m.n = n;
          m.item = item; m.first = (tok0 == t0); m.last = (tok0 + kT >= t_end); m.qbuf = qb;
          m.nch = it.nch; m.nlo = max(t_begin - tok0, 0); m.qlim = qlim;
          if (bytes) mbar_arrive_expect_tx(&sm.kv_full[st], bytes);
          else mbar_arrive(&sm.kv_full[st]);
        }
        __syncwarp();
        if (valid) {
          const KvCoord kc = kv_coord(p, blk, tok0 + lane * prow, hkv);
          const CUtensorMap* mk = fine ? &tmK16 : &tmK;
          const CUtensorMap* mv = fine ? &tmV16 : &tmV;
          for (int bx = 0; bx < C::kNumBoxes; ++bx) {
            const uint32_t off = bx * (kT * 128) + lane * prow * 128;
            tma_load_2d(sm.kv[st][0] + off, mk, kc.x0 + bx * 64, kc.row, &sm.kv_full[st]);
            tma_load_2d(sm.kv[st][1] + off, mv, kc.x0 + bx * 64, kc.row, &sm.kv_full[st]);
          }
        }
        if (tok0 == t0 && !p.fused_plan) queue.prefetch(p, lane);
      }
      ++local_item;
    }
    if (ok) {  // sentinel tile: no more work
      const int st = j % C::kStages;
      if (mbar_wait(&sm.kv_empty[st], ((uint32_t)(j / C::kStages) & 1u) ^ 1u, p.status) && lane == 0) {
        sm.meta[st].item = -1;
        mbar_arrive(&sm.kv_full[st]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ score MMAs
    if (lane == 0) {
      constexpr uint32_t idesc_qk = umma_idesc_f16(DT == kBF16, 0, 0, kT, kNP);
      int local_item = 0;
      for (int j = 0;; ++j) {
        const int st = j % C::kStages;
        const int sb = j & 1;
        if (!mbar_wait(&sm.kv_full[st], (uint32_t)(j / C::kStages) & 1u, p.status)) break;
        // the S buffer of tile j - 2 has been read (its P written)
        if (j >= 2 && !mbar_wait(&sm.p_full[sb], ((uint32_t)(j >> 1) & 1u) ^ 1u, p.status)) break;
        const TileMeta meta = sm.meta[st];
        if (meta.item < 0) {
          mbar_arrive(&sm.s_full[sb]);  // lets the compute warps see the sentinel
          break;
        }
        const int qb = meta.qbuf;
        if (meta.first && !mbar_wait(&sm.q_full[qb], (uint32_t)(local_item >> 1) & 1u, p.status)) break;
        tc_fence_after();
        const uint32_t kbase = smem_u32(sm.kv[st][0]);
        const uint32_t qbase = smem_u32(sm.q[qb]);
#pragma unroll
        for (int s = 0; s < C::kKSteps; ++s) {
          const uint64_t a = umma_desc(kbase + (s >> 2) * (kT * 128) + (s & 3) * 32, 16, 1024);
          const uint64_t bd = umma_desc(qbase + (s >> 2) * (kNP * 128) + (s & 3) * 32, 16, 1024);
          umma_f16(tmem + C::kColS + sb * 16, a, bd, idesc_qk, s > 0);
        }
        umma_commit(&sm.s_full[sb]);
        if (meta.last) {
          umma_commit(&sm.q_empty[qb]);
          ++local_item;
        }
      }
    }
  } else if (warp == kPvWarpTC) {
    // ------------------------------------------------------------------ PV MMAs
    // A second issue stream on another SM sub-partition (an MMA blocks its issuing
    // thread for about 50 cycles); the tensor pipe runs the two streams interleaved.
    if (lane == 0) {
      constexpr uint32_t idesc_pv = umma_idesc_f16(DT == kBF16, 1, 0, kT, kNP);
      for (int j = 0;; ++j) {
        const int pb = j & 1;
        if (!mbar_wait(&sm.p_full[pb], (uint32_t)(j >> 1) & 1u, p.status)) break;
        if (j >= *static_cast<volatile int*>(&sm.pv_stop)) break;  // tile j is the sentinel
        tc_fence_after();
        const int st = j % C::kStages;
        const uint32_t vbase = smem_u32(sm.kv[st][1]);
        const uint32_t pbase = smem_u32(sm.p[pb]);
        const uint32_t ocol = tmem + C::kColO + pb * C::kOStride;
        if constexpr (!C::kStacked) {
#pragma unroll
          for (int s = 0; s < kT / 16; ++s) {
            const uint64_t a = umma_desc(vbase + s * 16 * 128, kT * 128, 1024);
            const uint64_t bd = umma_desc(pbase + (s >> 2) * (kNP * 128) + (s & 3) * 32, 16, 1024);
            umma_f16(ocol, a, bd, idesc_pv, s > 0);
          }
        } else {
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const uint64_t a = umma_desc(vbase + s * 16 * 128, 64 * 128, 1024);
            const uint64_t b0 = umma_desc(pbase + s * 32, 16, 1024);
            const uint64_t b1 = umma_desc(pbase + kNP * 128 + s * 32, 16, 1024);
            umma_f16(ocol, a, b0, idesc_pv, s > 0);
            umma_f16(ocol + 16, a, b1, idesc_pv, s > 0);
          }
        }
        umma_commit(&sm.kv_empty[st]);
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax + correction
    // Two warp groups share the work of each tile: group 0 (warps 2-5) takes heads
    // [0, GH), group 1 (warps 7-10) heads [GH, 2 GH), so that each thread's chain of
    // dependent steps per tile is half as long.  GP (the group size rounded up to a
    // power of two) is a compile-time bound, so the per-head loops unroll into
    // independent chains the scheduler can interleave.
    constexpr int GH = GP / 2;
    const bool upper = warp >= kSm2Warp0;
    const int h0 = upper ? GH : 0;
    // The groups exchange maxima and sums only among their own four warps.  (At the
    // sentinel, the PV thread sees pv_stop: thread 64 writes it before its warp arrives.)
    const int bar_group = kBarCompute + (upper ? 1 : 0);
    const int quad = warp & 3;                 // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;            // TMEM lane: token of S, channel of O
    const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16);
    float m_run[GH], l_part[GH], alpha_prev[GH], acc[GH], m_fin[GH], l_fin[GH];
    int vpos[GH];  // query position of each of this group's virtual heads
#pragma unroll
    for (int g = 0; g < GH; ++g) {
      m_run[g] = -INFINITY; l_part[g] = 0.f; alpha_prev[g] = 0.f; acc[g] = 0.f; m_fin[g] = -INFINITY; l_fin[g] = 0.f;
      vpos[g] = kKeyMask ? (h0 + g) / G : 0;
    }
    int prev_item = -1, prev_b = 0, prev_hkv = 0, prev_nch = 1;
    bool prev_first = false, prev_last = false;

    // rescale-and-accumulate of the PV result of tile jj; finalises its item if it was the last tile
    auto correct = [&](int jj, bool use_fin) -> bool {
      const int ob = jj & 1;
      if (!mbar_wait(&sm.kv_empty[jj % C::kStages], (uint32_t)(jj / C::kStages) & 1u, p.status)) return false;
      tc_fence_after();
      float o[kNP];
      const uint32_t ocol = tq + C::kColO + ob * C::kOStride + ((C::kStacked && r >= 64) ? 16 : 0);
      tmem_ld16(ocol, o);  // read before this warp's next p_full arrival
#pragma unroll
      for (int g = 0; g < GH; ++g) {
        const float og = upper ? o[GH + g] : o[g];  // compile-time indices
        acc[g] = prev_first ? og : fmaf(acc[g], alpha_prev[g], og);
      }
      if (prev_last) {
        float mm[GH], lv[GH];
#pragma unroll
        for (int g = 0; g < GH; ++g) {
          mm[g] = use_fin ? m_fin[g] : m_run[g];
          lv[g] = use_fin ? l_fin[g] : l_part[g];
        }
#pragma unroll
        for (int off = 16; off; off >>= 1)
#pragma unroll
          for (int g = 0; g < GH; ++g) lv[g] += __shfl_xor_sync(0xffffffffu, lv[g], off);
        if (lane == 0) {
#pragma unroll
          for (int g = 0; g < GH; ++g) sm.lsum[quad][h0 + g] = lv[g];
        }
        if (C::kStacked && r >= 64) {
#pragma unroll
          for (int g = 0; g < GH; ++g) sm.accx[r - 64][h0 + g] = acc[g];
        }
        named_bar_sync(bar_group, 128);
        float lt[GH];
#pragma unroll
        for (int g = 0; g < GH; ++g)
          lt[g] = sm.lsum[0][h0 + g] + sm.lsum[1][h0 + g] + sm.lsum[2][h0 + g] + sm.lsum[3][h0 + g];
        if (prev_nch == 1 && !p.partials_only) {
          // the segment is this one item: write the final output directly
          if (!C::kStacked || r < 64) {
#pragma unroll
            for (int g = 0; g < GH; ++g) {
              const int hg = h0 + g;
              if (hg < GV) {
                const float a = C::kStacked ? acc[g] + sm.accx[r][hg] : acc[g];
                // several query positions run only on the key-mask instantiation
                const int64_t row = kKeyMask ? q_row(p, prev_b, prev_hkv, hg) : (int64_t)prev_b * p.Nq + prev_hkv * G + hg;
                const int h = kKeyMask ? q_head(p, prev_hkv, hg) : prev_hkv * G + hg;
                float M, W;
                const float v = single_item_output(a, mm[g], lt[g], p.sink, h, &M, &W);
                store_out<DT>(p.out, row * D + r, v);
                if (r == hg) {
                  if (p.softmax_max) p.softmax_max[row] = (M == -INFINITY) ? -INFINITY : M * kLn2;
                  if (p.softmax_sum) p.softmax_sum[row] = W;
                }
              }
            }
          }
        } else {
          if (!C::kStacked || r < 64) {
            float* po = p.ws.part_o + (int64_t)prev_item * GV * D;
#pragma unroll
            for (int g = 0; g < GH; ++g) {
              const int hg = h0 + g;
              if (hg < GV) {
                const float a = C::kStacked ? acc[g] + sm.accx[r][hg] : acc[g];
                po[hg * D + r] = lt[g] > 0.f ? a / lt[g] : 0.f;
              }
            }
          }
          if (r >= h0 && r < h0 + GH && r < GV) {
            float mv = mm[0], lw = lt[0];
#pragma unroll
            for (int g = 1; g < GH; ++g)
              if (r == h0 + g) { mv = mm[g]; lw = lt[g]; }
            p.ws.part_ml[(int64_t)prev_item * GV + r] = make_float2(mv, lw);
          }
        }
        named_bar_sync(bar_group, 128);
      }
      return true;
    };

    int j = 0;
    bool ok = true;
    while (true) {
      const int sb = j & 1;
      const uint32_t sph = (uint32_t)(j >> 1) & 1u;
      if (!mbar_wait(&sm.s_full[sb], sph, p.status)) { ok = false; break; }
      const int st = j % C::kStages;
      const TileMeta meta = sm.meta[st];
      if (meta.item < 0) {  // no more tiles: wake the PV warp, which stops
        if (tid == 64) sm.pv_stop = j;
        named_bar_sync(bar_group, 128);
        if (lane == 0) mbar_arrive(&sm.p_full[sb]);
        break;
      }
      tc_fence_after();
      float s[kNP];
      tmem_ld16(tq + C::kColS + sb * 16, s);
      if (meta.first) {
#pragma unroll
        for (int g = 0; g < GH; ++g) {
          m_fin[g] = m_run[g];
          l_fin[g] = l_part[g];
          m_run[g] = -INFINITY;
          l_part[g] = 0.f;
        }
      }
      const bool valid = r < meta.n && (!kKeyMask || (r >= meta.nlo && !key_masked(p, meta.b, meta.tok0 + r)));
      // per-head maximum over the tile's tokens: a warp reduction per head, then across
      // the 4 lane quadrants through shared memory
      float x[GH], mx[GH];
#pragma unroll
      for (int g = 0; g < GH; ++g) {
        const float sg = upper ? s[GH + g] : s[g];  // compile-time indices
        // (several query positions: position i sees tokens up to qlim + i)
        const bool vis = valid && (!kKeyMask || meta.tok0 + r <= meta.qlim + vpos[g]);
        x[g] = vis ? sg * p.scale_log2 : -INFINITY;
        mx[g] = warp_max(x[g]);
      }
      if (lane == 0) {
#pragma unroll
        for (int g = 0; g < GH; ++g) sm.red[sb][h0 + g][quad] = mx[g];
      }
      named_bar_sync(bar_group, 128);
      float alpha[GH], pr[GH];
#pragma unroll
      for (int g = 0; g < GH; ++g) {
        const float4 rq = *reinterpret_cast<const float4*>(sm.red[sb][h0 + g]);  // the four quadrants' maxima
        const float tmax = fmax3(fmaxf(rq.x, rq.y), rq.z, rq.w);
        const float m_new = fmaxf(m_run[g], tmax);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        alpha[g] = fast_exp2(m_run[g] - m_use);   // m_run = -inf gives 0
        pr[g] = fast_exp2(x[g] - m_use);          // masked tokens (-inf) give 0
        l_part[g] = fmaf(l_part[g], alpha[g], pr[g]);
        m_run[g] = m_new;
      }
      // P^T (and, from group 0, a zeroed V tail) for the PV MMA; the P buffer is free since
      // PV(j - 2) was waited for in correct(j - 2)
      uint8_t* pbuf = sm.p[sb];
#pragma unroll
      for (int g = 0; g < GH; ++g) {
        if (h0 + g < GV) {
          uint16_t h;
          if (DT == kBF16) h = __bfloat16_as_ushort(__float2bfloat16_rn(pr[g]));
          else h = __half_as_ushort(__float2half_rn(pr[g]));
          *reinterpret_cast<uint16_t*>(pbuf + p_offset(h0 + g, r)) = h;
        }
      }
      // V rows of tokens that are not keys -- past the item's end, and with a key mask also
      // masked keys and keys below a window -- are zeroed: the cache may hold anything there,
      // NaN included, and a weight of 0 would not cancel it in the product
      if ((r >= meta.n || (kKeyMask && !valid)) && !upper) {
        uint8_t* vrow = sm.kv[st][1];
#pragma unroll
        for (int bx = 0; bx < C::kNumBoxes; ++bx) {
          uint4* dst = reinterpret_cast<uint4*>(vrow + bx * (kT * 128) + r * 128);
#pragma unroll
          for (int c = 0; c < 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();  // the tensor-memory reads of S(j) and O(j - 2) precede the arrival
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_full[sb]);
      // rescale-and-accumulate the previous tile's PV result
      if (j > 0 && !correct(j - 1, meta.first)) { ok = false; break; }
#pragma unroll
      for (int g = 0; g < GH; ++g) alpha_prev[g] = alpha[g];
      prev_first = meta.first;
      prev_last = meta.last;
      prev_item = meta.item;
      prev_b = meta.b;
      prev_hkv = meta.hkv;
      prev_nch = meta.nch;
      ++j;
    }
    if (ok && j > 0) correct(j - 1, false);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int DT, int GP>
cudaError_t launch_tc(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmQ,
                      const CUtensorMap* tail, int box_rows, int grid, cudaStream_t stream) {
  const size_t smem = sizeof(TcSmem<D>) + 1024;
  auto kern = (p.atten_mask || p.windowed || p.qs > 1) ? decode_tc_kernel<D, DT, GP, true>
                                                       : decode_tc_kernel<D, DT, GP, false>;
  cudaError_t e = ensure_smem(kern, (int)smem);
  if (e != cudaSuccess) return e;
  trace_mark(kKernelDecodeAttention, 0, stream);
  e = launch_dependent(kern, grid, kThreadsTC, smem, stream, tmK, tmV, tmQ, tail[0], tail[1], p, box_rows);
  trace_mark(kKernelDecodeAttention, 1, stream);
  return e;
}

}  // namespace

template <int D, int DT>
cudaError_t launch_tc_g(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV, const CUtensorMap& tmQ,
                        const CUtensorMap* tail, int box_rows, int grid, cudaStream_t stream) {
  if (p.GV <= 2) return launch_tc<D, DT, 2>(p, tmK, tmV, tmQ, tail, box_rows, grid, stream);
  if (p.GV <= 4) return launch_tc<D, DT, 4>(p, tmK, tmV, tmQ, tail, box_rows, grid, stream);
  if (p.GV <= 8) return launch_tc<D, DT, 8>(p, tmK, tmV, tmQ, tail, box_rows, grid, stream);
  return launch_tc<D, DT, 16>(p, tmK, tmV, tmQ, tail, box_rows, grid, stream);
}

cudaError_t launch_decode_tc_attention(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                       const CUtensorMap& tmQ, const CUtensorMap* tail, int box_rows, int grid,
                                       cudaStream_t stream) {
  if (p.kv_dtype == kBF16)
    return p.D == 64 ? launch_tc_g<64, kBF16>(p, tmK, tmV, tmQ, tail, box_rows, grid, stream)
                     : launch_tc_g<128, kBF16>(p, tmK, tmV, tmQ, tail, box_rows, grid, stream);
  return p.D == 64 ? launch_tc_g<64, kF16>(p, tmK, tmV, tmQ, tail, box_rows, grid, stream)
                   : launch_tc_g<128, kF16>(p, tmK, tmV, tmQ, tail, box_rows, grid, stream);
}

}  // namespace fia
