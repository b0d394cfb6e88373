// rr_inst_hd_bf16.cu -- halving-doubling direct kernels with bfloat16 storage.
#include "rr_hd_direct.cuh"

namespace rr {

cudaError_t launch_hd_direct_bf16(int wire, const RingParams &p, const Launch &l, cudaStream_t s) {
  if (wire == kBF16) return hd::launch_pair<kBF16, kBF16>(p, l, s);
  if (wire == kF32) return hd::launch_pair<kBF16, kF32>(p, l, s);
  return cudaErrorInvalidValue;
}

}  // namespace rr
