// rr_inst_hd_f32.cu -- halving-doubling direct kernels with binary32 storage.
#include "rr_hd_direct.cuh"

namespace rr {

cudaError_t launch_hd_direct_f32(int wire, const RingParams &p, const Launch &l, cudaStream_t s) {
  if (wire == kF32) return hd::launch_pair<kF32, kF32>(p, l, s);
  if (wire == kF16) return hd::launch_pair<kF32, kF16>(p, l, s);
  if (wire == kBF16) return hd::launch_pair<kF32, kBF16>(p, l, s);
  return cudaErrorInvalidValue;
}

}  // namespace rr
