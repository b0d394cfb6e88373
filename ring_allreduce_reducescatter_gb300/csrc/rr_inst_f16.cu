// rr_inst_f16.cu -- kernels with binary16 storage: the binary16 wire, and
// accumulation in binary32.
#include "rr_kernels.cuh"

namespace rr {

cudaError_t launch_f16(int op, int wire, const RingParams &p, const Launch &l, cudaStream_t s) {
  switch (op) {
    case kOpAllReduce:
      if (wire == kF16) return launch_one<kOpAllReduce, kF16, kF16>(p, l, s);
      if (wire == kF32) return launch_one<kOpAllReduce, kF16, kF32>(p, l, s);
      break;
    case kOpReduceScatter:
      if (wire == kF16) return launch_one<kOpReduceScatter, kF16, kF16>(p, l, s);
      if (wire == kF32) return launch_one<kOpReduceScatter, kF16, kF32>(p, l, s);
      break;
    case kOpAllGather:
      if (wire == kF16) return launch_one<kOpAllGather, kF16, kF16>(p, l, s);
      break;
  }
  return cudaErrorInvalidValue;
}

}  // namespace rr
