// rau.cu -- RingAttentionUpdate: merge two attention partials by their softmax
// max and sum (aclnnRingAttentionUpdate, "功能说明 / 计算公式").
//
// Per (row, head):  m = max(m_p, m_c);  w_p = s_p e^{m_p - m};  w_c = s_c e^{m_c - m};
//                   sum = w_p + w_c;    out = (o_p w_p + o_c w_c) / sum.
// Each partial's output is normalised by its own sum, so the sums weight the
// outputs (the formula as printed on the page omits these factors; with them
// the merge of any split equals the unsplit result).  A side whose max is -inf
// (no keys) weighs zero; if both are, out = 0, max = -inf, sum = 0.
//
// One warp handles whole (row, head) groups so that max/sum/out may alias the
// prev_* inputs: every lane reads its inputs before any lane writes.
#include "fia_device.cuh"

namespace fia {
namespace {

template <int DT>
struct Vec;  // 16-byte vector of the output type
template <>
struct Vec<kF32> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void load(const void* p, int64_t i, float (&f)[8]) {
    const float4 v = reinterpret_cast<const float4*>(p)[i];
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
  static __device__ __forceinline__ void store(void* p, int64_t i, const float (&f)[8]) {
    reinterpret_cast<float4*>(p)[i] = make_float4(f[0], f[1], f[2], f[3]);
  }
};
template <int DT>
struct Vec16 {
  static constexpr int N = 8;
  static __device__ __forceinline__ void load(const void* p, int64_t i, float (&f)[8]) {
    const uint4 v = reinterpret_cast<const uint4*>(p)[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (DT == kBF16) {
        f[2 * k] = bf16lo(w[k]);
        f[2 * k + 1] = bf16hi(w[k]);
      } else {
        f[2 * k] = f16lo(w[k]);
        f[2 * k + 1] = f16hi(w[k]);
      }
    }
  }
  static __device__ __forceinline__ void store(void* p, int64_t i, const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (DT == kBF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * k], f[2 * k + 1]);
        w[k] = *reinterpret_cast<uint32_t*>(&h);
      } else {
        __half2 h = __floats2half2_rn(f[2 * k], f[2 * k + 1]);
        w[k] = *reinterpret_cast<uint32_t*>(&h);
      }
    }
    reinterpret_cast<uint4*>(p)[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <>
struct Vec<kF16> : Vec16<kF16> {};
template <>
struct Vec<kBF16> : Vec16<kBF16> {};

template <int DT>
__global__ void __launch_bounds__(256) rau_kernel(const void* prev_out, const float* prev_max,
                                                  const float* prev_sum, const void* cur_out,
                                                  const float* cur_max, const float* cur_sum, int64_t groups, int D,
                                                  void* out, float* max_out, float* sum_out) {
  using V = Vec<DT>;
  const int chunks = D / V::N;                  // 16-byte vectors per group
  const int sg = chunks <= 16 ? 16 : 32;        // lanes per group
  const int lane = threadIdx.x & 31;
  const int sub = lane / sg, sl = lane % sg;
  const int64_t warp_id = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int per_warp = 32 / sg;
  for (int64_t g0 = warp_id * per_warp; g0 < groups; g0 += nwarps * per_warp) {
    const int64_t g = g0 + sub;
    const bool active = g < groups;
    float mp = -INFINITY, mc = -INFINITY, sp = 0.f, sc = 0.f;
    if (active) {
      mp = prev_max[g];
      mc = cur_max[g];
      sp = prev_sum[g];
      sc = cur_sum[g];
    }
    const float m = fmaxf(mp, mc);
    float wp = 0.f, wc = 0.f;
    if (m != -INFINITY) {
      wp = (mp == -INFINITY) ? 0.f : sp * expf(mp - m);
      wc = (mc == -INFINITY) ? 0.f : sc * expf(mc - m);
    }
    const float l = wp + wc;
    const float ap = l > 0.f ? wp / l : 0.f, ac = l > 0.f ? wc / l : 0.f;
    // read every input vector of the group before anything is written
    constexpr int kMaxIter = 6;  // D <= 768: at most 192 fp32 vectors, 6 per lane with 32 lanes
    float po[kMaxIter][8], co[kMaxIter][8];
#pragma unroll
    for (int it = 0; it < kMaxIter; ++it) {
      const int c = sl + it * sg;
      if (active && c < chunks) {
        V::load(prev_out, g * chunks + c, po[it]);
        V::load(cur_out, g * chunks + c, co[it]);
      }
    }
    __syncwarp();
#pragma unroll
    for (int it = 0; it < kMaxIter; ++it) {
      const int c = sl + it * sg;
      if (active && c < chunks) {
        float r[8];
#pragma unroll
        for (int e = 0; e < V::N; ++e) r[e] = po[it][e] * ap + co[it][e] * ac;
        V::store(out, g * chunks + c, r);
      }
    }
    if (active && sl == 0) {
      max_out[g] = m;
      sum_out[g] = l;
    }
    __syncwarp();
  }
}

}  // namespace

cudaError_t launch_rau(const void* prev_out, const float* prev_max, const float* prev_sum, const void* cur_out,
                       const float* cur_max, const float* cur_sum, int out_dtype, int64_t rows, int N, int D,
                       void* out, float* max_out, float* sum_out, cudaStream_t stream) {
  const int64_t groups = rows * N;
  if (groups == 0) return cudaSuccess;
  int64_t blocks = (groups + 15) / 16;  // 8 warps, up to 2 groups per warp
  if (blocks > 152 * 16) blocks = 152 * 16;
  trace_mark(kKernelRau, 0, stream);
  if (out_dtype == kF32)
    rau_kernel<kF32><<<(int)blocks, 256, 0, stream>>>(prev_out, prev_max, prev_sum, cur_out, cur_max, cur_sum,
                                                       groups, D, out, max_out, sum_out);
  else if (out_dtype == kF16)
    rau_kernel<kF16><<<(int)blocks, 256, 0, stream>>>(prev_out, prev_max, prev_sum, cur_out, cur_max, cur_sum,
                                                       groups, D, out, max_out, sum_out);
  else
    rau_kernel<kBF16><<<(int)blocks, 256, 0, stream>>>(prev_out, prev_max, prev_sum, cur_out, cur_max, cur_sum,
                                                        groups, D, out, max_out, sum_out);
  trace_mark(kKernelRau, 1, stream);
  return cudaGetLastError();
}

}  // namespace fia
