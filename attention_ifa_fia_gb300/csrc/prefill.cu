// prefill.cu -- causal variable-length prefill (TND) on tcgen05 tensor cores.
#include "fia_device.cuh"

namespace fia {

size_t prefill_workspace_bytes(int B, int Nq, int max_seqlen_q) {
  const int64_t tiles = (int64_t)B * Nq * ((max_seqlen_q + 127) / 128);
  return 256 + (size_t)(tiles > 0 ? tiles : 1) * 16;
}

cudaError_t launch_prefill(const PrefillParams&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, int,
                           cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace fia
