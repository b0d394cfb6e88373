// rr_inst_f32_narrow.cu -- kernels with binary32 storage on a bfloat16 or
// binary16 wire (an ingress rounding, 16-bit hops, an exact egress widening).
#include "rr_kernels.cuh"

namespace rr {

cudaError_t launch_f32_narrow(int op, int wire, const RingParams &p, const Launch &l, cudaStream_t s) {
  switch (op) {
    case kOpAllReduce:
      if (wire == kBF16) return launch_one<kOpAllReduce, kF32, kBF16>(p, l, s);
      if (wire == kF16) return launch_one<kOpAllReduce, kF32, kF16>(p, l, s);
      break;
    case kOpReduceScatter:
      if (wire == kBF16) return launch_one<kOpReduceScatter, kF32, kBF16>(p, l, s);
      if (wire == kF16) return launch_one<kOpReduceScatter, kF32, kF16>(p, l, s);
      break;
  }
  return cudaErrorInvalidValue;
}

}  // namespace rr
