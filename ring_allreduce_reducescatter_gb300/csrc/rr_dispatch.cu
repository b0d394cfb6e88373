// rr_dispatch.cu -- from (collective, storage format, wire format) to the
// kernels compiled for it (launch_op, one object of rr_inst_one.cu each), and
// the bounded-wait self-test kernel.
#include "rr_device.cuh"

namespace rr {

cudaError_t launch_collective(int op, int dtype, int wire, const RingParams &p, const Launch &l, cudaStream_t s) {
  switch (op) {
    case kOpAllReduce:
    case kOpReduceScatter: {
      const bool ar = op == kOpAllReduce;
      if (dtype == kF32) {
        if (wire == kF32) return ar ? launch_op<kOpAllReduce, kF32, kF32>(p, l, s) : launch_op<kOpReduceScatter, kF32, kF32>(p, l, s);
        if (wire == kBF16) return ar ? launch_op<kOpAllReduce, kF32, kBF16>(p, l, s) : launch_op<kOpReduceScatter, kF32, kBF16>(p, l, s);
        if (wire == kF16) return ar ? launch_op<kOpAllReduce, kF32, kF16>(p, l, s) : launch_op<kOpReduceScatter, kF32, kF16>(p, l, s);
      } else if (dtype == kF16) {
        if (wire == kF16) return ar ? launch_op<kOpAllReduce, kF16, kF16>(p, l, s) : launch_op<kOpReduceScatter, kF16, kF16>(p, l, s);
        if (wire == kF32) return ar ? launch_op<kOpAllReduce, kF16, kF32>(p, l, s) : launch_op<kOpReduceScatter, kF16, kF32>(p, l, s);
      } else if (dtype == kBF16) {
        if (wire == kBF16) return ar ? launch_op<kOpAllReduce, kBF16, kBF16>(p, l, s) : launch_op<kOpReduceScatter, kBF16, kBF16>(p, l, s);
        if (wire == kF32) return ar ? launch_op<kOpAllReduce, kBF16, kF32>(p, l, s) : launch_op<kOpReduceScatter, kBF16, kF32>(p, l, s);
      }
      break;
    }
    case kOpAllGather:
      if (wire != dtype) break;
      if (dtype == kF32) return launch_op<kOpAllGather, kF32, kF32>(p, l, s);
      if (dtype == kF16) return launch_op<kOpAllGather, kF16, kF16>(p, l, s);
      if (dtype == kBF16) return launch_op<kOpAllGather, kBF16, kBF16>(p, l, s);
      break;
  }
  return cudaErrorInvalidValue;
}

__global__ void rr_wait_probe_kernel(unsigned int *status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0, limit_ns)) atomicOr(status, kStatusWaitTimeout);
}

cudaError_t launch_wait_probe(unsigned int *status, unsigned long long limit_ns, cudaStream_t s) {
  rr_wait_probe_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace rr
