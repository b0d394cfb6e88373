// rr_inst_bf16.cu -- kernels with bfloat16 storage and a bfloat16 wire.
#include "rr_kernels.cuh"

namespace rr {

cudaError_t launch_bf16(int op, int wire, const RingParams &p, const Launch &l, cudaStream_t s) {
  if (wire != kBF16) return cudaErrorInvalidValue;
  switch (op) {
    case kOpAllReduce:
      return launch_one<kOpAllReduce, kBF16, kBF16>(p, l, s);
    case kOpReduceScatter:
      return launch_one<kOpReduceScatter, kBF16, kBF16>(p, l, s);
    case kOpAllGather:
      return launch_one<kOpAllGather, kBF16, kBF16>(p, l, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace rr
