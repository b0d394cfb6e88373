// rr_inst_bf16.cu -- kernels with bfloat16 storage: the bfloat16 wire, and
// accumulation in binary32.
#include "rr_kernels.cuh"

namespace rr {

cudaError_t launch_bf16(int op, int wire, const RingParams &p, const Launch &l, cudaStream_t s) {
  switch (op) {
    case kOpAllReduce:
      if (wire == kBF16) return launch_one<kOpAllReduce, kBF16, kBF16>(p, l, s);
      if (wire == kF32) return launch_one<kOpAllReduce, kBF16, kF32>(p, l, s);
      break;
    case kOpReduceScatter:
      if (wire == kBF16) return launch_one<kOpReduceScatter, kBF16, kBF16>(p, l, s);
      if (wire == kF32) return launch_one<kOpReduceScatter, kBF16, kF32>(p, l, s);
      break;
    case kOpAllGather:
      if (wire == kBF16) return launch_one<kOpAllGather, kBF16, kBF16>(p, l, s);
      break;
  }
  return cudaErrorInvalidValue;
}

}  // namespace rr
