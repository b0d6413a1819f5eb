// decode_i8.cuh -- the query-side preparation of the int8 tensor-core decode path.
//
// Antiquant of a key is affine per channel, k^_td = (x_td - o_d) * s_d
// (aclnnIncreFlashAttentionV3, "antiquantScale / antiquantOffset"), so a score
// separates into a product with the raw codes and a per-head constant:
//
//   sum_d q_d k^_td = sum_d (q_d s_d) x_td - sum_d q_d s_d o_d .
//
// The codes x_td are integers in [-128, 127] and enter the score MMA exactly (as
// fp16).  This file prepares the other operand once per (batch, kv head): the
// scaled query q'_d = q_d s_d, multiplied by a power of two 2^e that puts its
// largest entry in [2^14, 2^15), split into two fp16 parts hi + lo (the pair
// reproduces q' 2^e to about 2^-22 relative), and two per-head constants:
//   kq = scale * log2(e) * 2^-e        nq = -scale * log2(e) * sum_d q'_d o_d
// so that the score in log2 units is S kq + nq, where S = x . (hi + lo) is what
// the two MMAs (one per part) accumulate.
//
// The block of one (b, kv head) is laid out exactly as the B operand of the score
// MMA expects it in shared memory: 32 rows, the hi parts of the 16 (padded) heads
// then their lo parts, K-major with the 128-byte swizzle, so that one MMA of N = 32
// produces both partial scores of every head and the attention kernel moves the
// block with one bulk copy.
#pragma once

#include "decode_common.cuh"

namespace fia {

constexpr int kI8Heads = 16;                              // query heads per block (group, padded)
constexpr int kI8QRows = 2 * kI8Heads;                    // hi rows, then lo rows
constexpr int kI8QBytes = kI8QRows * 128 * 2;             // 32 rows x D = 128 fp16
constexpr int kI8QBlockBytes = kI8QBytes + kI8Heads * 8;  // + {kq, nq} per head

// Byte offset of channel d of row g (0..31) of the block: two 64-channel boxes of
// 32 rows x 128 bytes, the 16-byte chunk index XORed with the row (mod 8).
__device__ __forceinline__ uint32_t i8q_offset(int g, int d) {
  const uint32_t box = (uint32_t)d >> 6, col = ((uint32_t)d & 63u) * 2u;
  return box * (kI8QRows * 128) + (uint32_t)g * 128 + ((((col >> 4) ^ ((uint32_t)g & 7u))) << 4) + (col & 15u);
}

// Four int8 codes (the bytes of w, two's complement) -> two words of fp16 pairs (codes 0,1
// and 2,3; lower code in the low half), exactly: each byte plus 128 is placed under the
// exponent of 1024 (0x6400 | u is the half 1024 + u for u in [0, 255]), and 1152 = 1024 + 128
// is subtracted, which leaves the code itself (an integer of at most 8 bits, exact in fp16).
// The K and V converter warps of the int8 tensor-core kernel and the fia_debug_i8_codes
// probe use this one function.
__device__ __forceinline__ void codes_to_f16x2(uint32_t w, uint32_t& h01, uint32_t& h23) {
  const uint32_t u = w ^ 0x80808080u;  // code + 128 per byte
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
  // each half is now 1024 + code + 128; subtract 1152 (0x6480) from both halves
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(h01) : "r"(a), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(h23) : "r"(b), "r"(0x64806480u));
}

// One warp prepares row g of block (b, hkv); row index R = (b * Nkv + hkv) * 16 + g.  Row g
// is virtual head g: the query of head hkv * G + g % G at position g / G (one position: head
// hkv * G + g).  Lane l handles channels 4l .. 4l + 3.
__device__ __forceinline__ void i8_qprep_row(const DecodeParams& p, int64_t R, int lane) {
  const int64_t blk = R / kI8Heads;
  const int g = (int)(R % kI8Heads);
  const int b = (int)(blk / p.Nkv), hkv = (int)(blk % p.Nkv);
  uint8_t* base = p.ws.qprep + blk * kI8QBlockBytes;
  const int d0 = lane * 4;
  uint2 hi_w = make_uint2(0u, 0u), lo_w = make_uint2(0u, 0u);
  float2 kn = make_float2(0.f, 0.f);
  if (g < p.GV) {
    const uint2 raw = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.q) + q_row(p, b, hkv, g) * 128 + d0);
    float q[4];
    if (p.q_dtype == kBF16) {
      q[0] = bf16lo(raw.x); q[1] = bf16hi(raw.x); q[2] = bf16lo(raw.y); q[3] = bf16hi(raw.y);
    } else {
      q[0] = f16lo(raw.x); q[1] = f16hi(raw.x); q[2] = f16lo(raw.y); q[3] = f16hi(raw.y);
    }
    const float* sc = p.aq_scale + (int64_t)hkv * 128 + d0;  // key scale and offset: index 0 of (2, Nkv, D)
    const float* of = p.aq_offset ? p.aq_offset + (int64_t)hkv * 128 + d0 : nullptr;
    float qs[4], c = 0.f, amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      qs[i] = __fmul_rn(q[i], sc[i]);
      amax = fmaxf(amax, fabsf(qs[i]));
      if (of) c = fmaf(qs[i], of[i], c);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      c += __shfl_xor_sync(0xffffffffu, c, o);
    }
    int e = 0;
    if (amax > 0.f && amax <= 3.0e38f) {
      int ex;
      frexpf(amax, &ex);  // amax in [2^(ex-1), 2^ex)
      e = 15 - ex;
    }
    uint16_t hb[4], lb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float v = ldexpf(qs[i], e);
      const __half hh = __float2half_rn(v);
      const __half ll = __float2half_rn(v - __half2float(hh));  // the difference is exact in fp32
      hb[i] = __half_as_ushort(hh);
      lb[i] = __half_as_ushort(ll);
    }
    hi_w = make_uint2(hb[0] | ((uint32_t)hb[1] << 16), hb[2] | ((uint32_t)hb[3] << 16));
    lo_w = make_uint2(lb[0] | ((uint32_t)lb[1] << 16), lb[2] | ((uint32_t)lb[3] << 16));
    kn = make_float2(ldexpf(p.scale_log2, -e), -c * p.scale_log2);
  }
  *reinterpret_cast<uint2*>(base + i8q_offset(g, d0)) = hi_w;
  *reinterpret_cast<uint2*>(base + i8q_offset(kI8Heads + g, d0)) = lo_w;
  if (lane == 0) reinterpret_cast<float2*>(base + kI8QBytes)[g] = kn;
}

}  // namespace fia
