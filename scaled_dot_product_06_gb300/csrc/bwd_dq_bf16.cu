// dQ kernel instantiations for bf16 inputs (a translation unit of their own,
// compiled in parallel with the dK/dV one).
#include "bwd_dq_kernel.cuh"

namespace sdpa {

cudaError_t launch_bwd_dq_bf16(int d_qk, int d_v, const CUtensorMap& q, const CUtensorMap& k,
                             const CUtensorMap& v, const CUtensorMap& dout, const CUtensorMap& bias,
                             const CUtensorMap& dq, const BwdParams& p, cudaStream_t st) {
  if (d_qk == 64 && d_v == 64) return launch_bwd_dq_t<64, 64, true>(q, k, v, dout, bias, dq, p, st);
  if (d_qk == 128 && d_v == 128) return launch_bwd_dq_t<128, 128, true>(q, k, v, dout, bias, dq, p, st);
  if (d_qk == 192 && d_v == 128) return launch_bwd_dq_t<192, 128, true>(q, k, v, dout, bias, dq, p, st);
  return cudaErrorInvalidValue;
}

}  // namespace sdpa
