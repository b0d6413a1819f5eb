// decode_common.cuh -- pieces shared by the two decode attention kernels: the work-item
// format written by the plan kernel, the direct output of a (batch, kv-head) segment
// made of one work item, and the launch with programmatic dependent launch.
#pragma once

#include "fia_device.cuh"

namespace fia {

// Work item {b, kv head, (chunk count of the segment) << 16 | chunk index, last token + 1};
// the first token is chunk index * chunk_tokens.
struct DecodeItem {
  int b, hkv, j, nch, t_begin, t_end;
};

__device__ __forceinline__ DecodeItem decode_item(int4 d, int chunk_tokens) {
  DecodeItem it;
  it.b = d.x;
  it.hkv = d.y;
  it.j = d.z & 0xffff;
  it.nch = (unsigned)d.z >> 16;
  it.t_begin = it.j * chunk_tokens;
  it.t_end = d.w;
  return it;
}

// Output of a segment made of one item, straight from the item's running state:
// acc = sum_t 2^{s_t - m} v_t (not normalised), l = sum_t 2^{s_t - m}, m in log2 units.
// Returns the value to store for one output channel; *M_out / *W_out receive the
// softmax max (log2 units) and sum for the head.
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
