// prefill.cu -- causal variable-length prefill attention (TND) on tcgen05 tensor cores.
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
//   O [128 q x D]    += P . V       A = P (bf16, K-major, written by the softmax warps)
//                                   B = V tile read MN-major
//
// S (double buffered) and O live in tensor memory.  Warp roles (192 threads): warp 0
// issues TMA (Q per unit, double buffered; K/V tiles in a 2-stage ring), warp 1 owns
// TMEM and issues MMAs (QK of tile j+1 overlaps the softmax of tile j), warps 2-5 own one
// query row each: mask, row max and sum in registers (no cross-thread reduction), P,
// the rescale of O, and the epilogue.  O is rescaled only when the running row max
// grows by more than 8 (log2 units); otherwise the stale max keeps every exponent
// <= 2^8, and the softmax max/sum outputs are converted to the true max at the end.
#include "fia_device.cuh"

namespace fia {
namespace {

constexpr int kQT = 128;           // queries per tile (MMA M)
constexpr int kKT = 128;           // keys per tile (MMA N of QK, K of PV)
constexpr int kPD = 128;           // head dim supported by this kernel
constexpr int kPThreads = 192;
constexpr int kPStages = 2;
constexpr int kTileB = kQT * kPD * 2;  // 32 KB: Q, K, V or P tile
constexpr uint32_t kRescaleThreshold = 8;  // log2 units

struct __align__(16) PTileMeta {
  int b, h, q0, kvt;      // sequence, query head, first query (within the sequence), key tile
  int tq, tk, Lq, Lkv;    // first token of the sequence in q / kv, sequence lengths
  int first, last, qbuf, unit;
};

struct PSmem {
  alignas(1024) uint8_t q[2][kTileB];
  alignas(1024) uint8_t kv[kPStages][2][kTileB];
  alignas(1024) uint8_t p[kTileB];
  PTileMeta meta[kPStages];
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[kPStages], kv_empty[kPStages];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, pv_done, o_free;
  uint32_t tmem_base;
};

// per (sequence, query tile): key tiles that hold at least one visible key
__device__ __forceinline__ int key_tiles(int q0, int Lq, int Lkv, int causal) {
  const int q_last = min(q0 + kQT - 1, Lq - 1);
  int k_max = causal ? q_last + (Lkv - Lq) : Lkv - 1;
  k_max = min(k_max, Lkv - 1);
  return k_max < 0 ? 0 : k_max / kKT + 1;
}

__device__ __forceinline__ void seq_bounds(const PrefillParams& p, int b, int& tq, int& Lq, int& tk, int& Lkv) {
  int64_t q0 = p.cu_q[b], q1 = p.cu_q[b + 1], k0 = p.cu_kv[b], k1 = p.cu_kv[b + 1];
  if (q0 < 0 || q1 < q0 || q1 > p.T || k0 < 0 || k1 < k0 || k1 > p.Tkv) {
    raise_status(p.status, kStatusBadSeqlens);
    q0 = q1 = k0 = k1 = 0;
  }
  tq = (int)q0;
  Lq = (int)(q1 - q0);
  tk = (int)k0;
  Lkv = (int)(k1 - k0);
}

// ------------------------------------------------------------------ plan
// Lists (sequence, query tile) pairs ordered by decreasing number of key tiles
// (counting sort), resets the unit counter.  Units are list entry x query head.
__global__ void __launch_bounds__(1024) prefill_plan_kernel(PrefillParams p, int max_key_tiles) {
  extern __shared__ int hist[];  // [max_key_tiles + 2]
  const int tid = threadIdx.x;
  for (int i = tid; i < max_key_tiles + 2; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (int b = 0; b < p.B; ++b) {  // pass 1: histogram of key-tile counts
    int tq, Lq, tk, Lkv;
    seq_bounds(p, b, tq, Lq, tk, Lkv);
    for (int qt = tid; qt * kQT < Lq; qt += blockDim.x) {
      const int n = min(max(key_tiles(qt * kQT, Lq, Lkv, p.causal), 1), max_key_tiles);
      atomicAdd(&hist[n], 1);
    }
  }
  __syncthreads();
  if (tid == 0) {  // exclusive offsets, largest count first
    int run = 0;
    for (int n = max_key_tiles; n >= 1; --n) {
      const int c = hist[n];
      hist[n] = run;
      run += c;
    }
    hist[0] = run;  // total pairs
  }
  __syncthreads();
  for (int b = 0; b < p.B; ++b) {  // pass 2: scatter
    int tq, Lq, tk, Lkv;
    seq_bounds(p, b, tq, Lq, tk, Lkv);
    for (int qt = tid; qt * kQT < Lq; qt += blockDim.x) {
      const int n = min(max(key_tiles(qt * kQT, Lq, Lkv, p.causal), 1), max_key_tiles);
      const int pos = atomicAdd(&hist[n], 1);
      if (pos < p.max_tiles) p.tile_list[pos] = (b << 16) | qt;
    }
  }
  __syncthreads();
  if (tid == 0) {
    p.tile_counter[0] = 0;
    p.tile_counter[1] = min(hist[0], p.max_tiles) * p.Nq;  // number of units
  }
}

// Offset of (row r, 16-byte chunk c) in a 128-row tile stored as two 64-column
// boxes of 128-byte rows with the 128-byte swizzle.
__device__ __forceinline__ uint32_t tile_chunk_offset(int r, int c) {
  const uint32_t box = c >> 3, cc = c & 7;
  return box * (kQT * 128) + r * 128 + ((cc ^ (r & 7)) << 4);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_f16(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
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

// ------------------------------------------------------------------ attention
template <int DT>
__global__ void __launch_bounds__(kPThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  PSmem& sm = *reinterpret_cast<PSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.q_full[i], 1);
      mbar_init(&sm.q_empty[i], 1);
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.s_free[i], 4);
    }
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    mbar_init(&sm.p_full, 4);
    mbar_init(&sm.pv_done, 1);
    mbar_init(&sm.o_free, 4);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&sm.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  constexpr uint32_t kColS = 0, kColO = 256;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int n_units = p.tile_counter[1];
      const int G = p.G;
      int j = 0, u_local = 0;
      bool ok = true;
      while (ok) {
        const int u = atomicAdd(&p.tile_counter[0], 1);
        if (u >= n_units) break;
        const int pair = p.tile_list[u / p.Nq];
        const int h = u % p.Nq, b = pair >> 16, qt = pair & 0xffff;
        int tq, Lq, tk, Lkv;
        seq_bounds(p, b, tq, Lq, tk, Lkv);
        const int q0 = qt * kQT;
        const int nkv = max(key_tiles(q0, Lq, Lkv, p.causal), 1);
        const int qb = u_local & 1;
        if (!mbar_wait(&sm.q_empty[qb], ((uint32_t)(u_local >> 1) & 1u) ^ 1u, p.status)) { ok = false; break; }
        mbar_arrive_expect_tx(&sm.q_full[qb], kTileB);
        for (int bx = 0; bx < 2; ++bx)
          tma_load_3d(sm.q[qb] + bx * (kQT * 128), &tmQ, bx * 64, h, tq + q0, &sm.q_full[qb]);
        const int hkv = h / G;
        for (int kt = 0; kt < nkv; ++kt, ++j) {
          const int st = j % kPStages;
          if (!mbar_wait(&sm.kv_empty[st], ((uint32_t)(j / kPStages) & 1u) ^ 1u, p.status)) { ok = false; break; }
          PTileMeta& m = sm.meta[st];
          m.b = b; m.h = h; m.q0 = q0; m.kvt = kt;
          m.tq = tq; m.tk = tk; m.Lq = Lq; m.Lkv = Lkv;
          m.first = kt == 0; m.last = kt == nkv - 1; m.qbuf = qb; m.unit = u;
          mbar_arrive_expect_tx(&sm.kv_full[st], 2 * kTileB);
          for (int bx = 0; bx < 2; ++bx) {
            tma_load_3d(sm.kv[st][0] + bx * (kKT * 128), &tmK, bx * 64, hkv, tk + kt * kKT, &sm.kv_full[st]);
            tma_load_3d(sm.kv[st][1] + bx * (kKT * 128), &tmV, bx * 64, hkv, tk + kt * kKT, &sm.kv_full[st]);
          }
        }
        ++u_local;
      }
      if (ok) {  // sentinel
        const int st = j % kPStages;
        if (mbar_wait(&sm.kv_empty[st], ((uint32_t)(j / kPStages) & 1u) ^ 1u, p.status)) {
          sm.meta[st].unit = -1;
          mbar_arrive(&sm.kv_full[st]);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = umma_idesc_f16(DT == kBF16, 0, 0, kQT, kKT);
      constexpr uint32_t idesc_pv = umma_idesc_f16(DT == kBF16, 0, 1, kQT, kPD);
      int o_uses = 0;  // units whose first PV (which overwrites O) has been issued
      // O += P(jj) . V(jj); the first PV of a unit overwrites O, after the previous
      // unit's epilogue has read it (o_free phase o_uses - 1)
      auto issue_pv = [&](int jj, bool first_of_unit) -> bool {
        if (!mbar_wait(&sm.p_full, (uint32_t)jj & 1u, p.status)) return false;
        if (first_of_unit && o_uses > 0 && !mbar_wait(&sm.o_free, (uint32_t)(o_uses - 1) & 1u, p.status))
          return false;
        tc_fence_after();
        const int st = jj % kPStages;
        const uint32_t pbase = smem_u32(sm.p), vbase = smem_u32(sm.kv[st][1]);
#pragma unroll
        for (int s = 0; s < kKT / 16; ++s) {
          const uint64_t a = umma_desc(pbase + (s >> 2) * (kQT * 128) + (s & 3) * 32, 16, 1024);
          const uint64_t bd = umma_desc(vbase + s * 16 * 128, kKT * 128, 1024);
          umma_f16(tmem + kColO, a, bd, idesc_pv, (first_of_unit && s == 0) ? 0u : 1u);
        }
        umma_commit(&sm.pv_done);
        umma_commit(&sm.kv_empty[st]);
        if (first_of_unit) ++o_uses;
        return true;
      };
      int j = 0, u_local = 0;
      bool prev_first = false;
      while (true) {
        const int st = j % kPStages;
        if (!mbar_wait(&sm.kv_full[st], (uint32_t)(j / kPStages) & 1u, p.status)) break;
        const PTileMeta meta = sm.meta[st];
        if (meta.unit < 0) {
          if (j > 0) issue_pv(j - 1, prev_first);
          mbar_arrive(&sm.s_full[j & 1]);  // lets the softmax warps see the sentinel
          break;
        }
        const int qb = meta.qbuf;
        if (meta.first && !mbar_wait(&sm.q_full[qb], (uint32_t)(u_local >> 1) & 1u, p.status)) break;
        const int sb = j & 1;
        if (!mbar_wait(&sm.s_free[sb], ((uint32_t)(j >> 1) & 1u) ^ 1u, p.status)) break;
        tc_fence_after();
        const uint32_t qbase = smem_u32(sm.q[qb]), kbase = smem_u32(sm.kv[st][0]);
#pragma unroll
        for (int s = 0; s < kPD / 16; ++s) {
          const uint64_t a = umma_desc(qbase + (s >> 2) * (kQT * 128) + (s & 3) * 32, 16, 1024);
          const uint64_t bd = umma_desc(kbase + (s >> 2) * (kKT * 128) + (s & 3) * 32, 16, 1024);
          umma_f16(tmem + kColS + sb * kKT, a, bd, idesc_qk, s > 0);
        }
        umma_commit(&sm.s_full[sb]);
        if (meta.last) {
          umma_commit(&sm.q_empty[qb]);
          ++u_local;
        }
        if (j > 0 && !issue_pv(j - 1, prev_first)) break;
        prev_first = meta.first;
        ++j;
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax, rescale, epilogue
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // query row of the tile = TMEM lane
    const uint32_t tq_lane = tmem + ((uint32_t)(quad * 32) << 16);
    float m_run = -INFINITY;   // max used for the exponents (may lag the true max by < 2^8)
    float m_true = -INFINITY;  // true running max
    float l_run = 0.f;         // sum of exponents relative to m_run
    int j = 0;
    bool ok = true;
    while (true) {
      const int sb = j & 1;
      if (!mbar_wait(&sm.s_full[sb], (uint32_t)(j >> 1) & 1u, p.status)) { ok = false; break; }
      const int st = j % kPStages;
      const PTileMeta meta = sm.meta[st];
      if (meta.unit < 0) break;
      tc_fence_after();
      if (meta.first) {
        m_run = -INFINITY;
        m_true = -INFINITY;
        l_run = 0.f;
      }
      const int qi = meta.q0 + r;            // query index within the sequence
      const bool row_ok = qi < meta.Lq;
      const int k0 = meta.kvt * kKT;
      // visible keys of this row in the tile: [k0, k_hi)
      int k_hi = meta.Lkv;
      if (p.causal) k_hi = min(k_hi, qi + (meta.Lkv - meta.Lq) + 1);
      const int nvis = row_ok ? max(0, min(k_hi - k0, kKT)) : 0;
      float s[kKT];
#pragma unroll
      for (int c = 0; c < kKT; c += 32) {
        float v[32];
        tmem_ld32(tq_lane + kColS + sb * kKT + c, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c + i] = v[i];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.s_free[sb]);
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < kKT; ++c) {
        s[c] = (c < nvis) ? s[c] * p.scale_log2 : -INFINITY;
        mt = fmaxf(mt, s[c]);
      }
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
#pragma unroll
      for (int c = 0; c < kKT; ++c) {
        s[c] = fast_exp2(s[c] - m_use);
        lsum += s[c];
      }
      l_run = fmaf(l_run, alpha, lsum);
      // the previous tile's PV must be complete before P is overwritten or O rescaled
      if (j > 0 && !mbar_wait(&sm.pv_done, (uint32_t)(j - 1) & 1u, p.status)) { ok = false; break; }
      // tcgen05.ld/st are warp-collective (.sync.aligned): the whole warp rescales when
      // any of its rows needs it, the other rows with a factor of 1
      if (__any_sync(0xffffffffu, rescale && !meta.first)) {
        const float f = (rescale && !meta.first) ? alpha : 1.f;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kPD; c += 32) {
          float o[32];
          tmem_ld32(tq_lane + kColO + c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= f;
          tmem_st32(tq_lane + kColO + c, o);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
      // P row r: 128 keys as 16 chunks of 8 16-bit values
#pragma unroll
      for (int c = 0; c < kKT / 8; ++c) {
        uint4 w;
        if (DT == kBF16) {
          w = make_uint4(pack_bf16(s[8 * c], s[8 * c + 1]), pack_bf16(s[8 * c + 2], s[8 * c + 3]),
                         pack_bf16(s[8 * c + 4], s[8 * c + 5]), pack_bf16(s[8 * c + 6], s[8 * c + 7]));
        } else {
          w = make_uint4(pack_f16(s[8 * c], s[8 * c + 1]), pack_f16(s[8 * c + 2], s[8 * c + 3]),
                         pack_f16(s[8 * c + 4], s[8 * c + 5]), pack_f16(s[8 * c + 6], s[8 * c + 7]));
        }
        *reinterpret_cast<uint4*>(sm.p + tile_chunk_offset(r, c)) = w;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_full);
      if (meta.last) {
        // epilogue: wait for this tile's PV, normalise O and write out, max and sum
        if (!mbar_wait(&sm.pv_done, (uint32_t)j & 1u, p.status)) { ok = false; break; }
        tc_fence_after();
        const float sink2 = p.sink ? p.sink[meta.h] * kLog2e : -INFINITY;
        const float m_fin = fmaxf(m_true, sink2);
        float denom = l_run;  // relative to m_run
        if (p.sink && m_run != -INFINITY) denom += fast_exp2(sink2 - m_run);
        const float inv = denom > 0.f ? 1.f / denom : 0.f;
        const int64_t tok = (int64_t)meta.tq + qi;
        // every lane takes part in the (warp-collective) TMEM loads; only valid rows store
        uint8_t* orow = static_cast<uint8_t*>(p.out) + (tok * p.Nq + meta.h) * (int64_t)kPD * 2;
#pragma unroll
        for (int c = 0; c < kPD; c += 32) {
          float o[32];
          tmem_ld32(tq_lane + kColO + c, o);
          if (row_ok) {
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
        if (row_ok) {
          float sum_true = 0.f;
          if (m_fin != -INFINITY) {
            sum_true = (m_run == -INFINITY) ? 0.f : l_run * fast_exp2(m_run - m_fin);
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
    (void)ok;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
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

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                           const CUtensorMap& tmV, int num_sms, cudaStream_t stream) {
  const int max_key_tiles = (p.max_seqlen_kv + kKT - 1) / kKT + 1;
  trace_mark(kKernelPrefill, 0, stream);
  prefill_plan_kernel<<<1, 1024, sizeof(int) * (max_key_tiles + 2), stream>>>(p, max_key_tiles);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(PSmem) + 1024;
  if (p.dtype == kBF16) {
    e = cudaFuncSetAttribute(prefill_tc_kernel<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prefill_tc_kernel<kBF16><<<num_sms, kPThreads, smem, stream>>>(tmQ, tmK, tmV, p);
  } else {
    e = cudaFuncSetAttribute(prefill_tc_kernel<kF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prefill_tc_kernel<kF16><<<num_sms, kPThreads, smem, stream>>>(tmQ, tmK, tmV, p);
  }
  trace_mark(kKernelPrefill, 1, stream);
  return cudaGetLastError();
}

}  // namespace fia
