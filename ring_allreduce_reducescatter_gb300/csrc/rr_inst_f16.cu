// rr_inst_f16.cu -- kernels with binary16 storage and a binary16 wire.
#include "rr_kernels.cuh"

namespace rr {

cudaError_t launch_f16(int op, int wire, const RingParams &p, const Launch &l, cudaStream_t s) {
  if (wire != kF16) return cudaErrorInvalidValue;
  switch (op) {
    case kOpAllReduce:
      return launch_one<kOpAllReduce, kF16, kF16>(p, l, s);
    case kOpReduceScatter:
      return launch_one<kOpReduceScatter, kF16, kF16>(p, l, s);
    case kOpAllGather:
      return launch_one<kOpAllGather, kF16, kF16>(p, l, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace rr
