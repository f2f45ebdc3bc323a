// Forward kernel instantiations for bf16 inputs.
#include "fwd_kernel.cuh"

namespace sdpa {

cudaError_t launch_fwd_bf16(int d_qk, int d_v, const CUtensorMap& q, const CUtensorMap& k,
                          const CUtensorMap& v, const FwdParams& p, cudaStream_t st) {
  if (d_qk == 64 && d_v == 64) return launch_fwd_t<64, 64, true>(q, k, v, p, st);
  if (d_qk == 128 && d_v == 128) return launch_fwd_t<128, 128, true>(q, k, v, p, st);
  if (d_qk == 192 && d_v == 128) return launch_fwd_t<192, 128, true>(q, k, v, p, st);
  return cudaErrorInvalidValue;
}

}  // namespace sdpa
