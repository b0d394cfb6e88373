// rr_inst_f32.cu -- kernels with binary32 storage (wire: binary32, bfloat16
// or binary16), and the bounded-wait probe kernel.
#include "rr_kernels.cuh"

namespace rr {

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

cudaError_t launch_f32(int op, int wire, const RingParams &p, const Launch &l, cudaStream_t s) {
  switch (op) {
    case kOpAllReduce:
      if (wire == kF32) return launch_one<kOpAllReduce, kF32, kF32>(p, l, s);
      if (wire == kBF16) return launch_one<kOpAllReduce, kF32, kBF16>(p, l, s);
      if (wire == kF16) return launch_one<kOpAllReduce, kF32, kF16>(p, l, s);
      break;
    case kOpReduceScatter:
      if (wire == kF32) return launch_one<kOpReduceScatter, kF32, kF32>(p, l, s);
      if (wire == kBF16) return launch_one<kOpReduceScatter, kF32, kBF16>(p, l, s);
      if (wire == kF16) return launch_one<kOpReduceScatter, kF32, kF16>(p, l, s);
      break;
    case kOpAllGather:
      return launch_one<kOpAllGather, kF32, kF32>(p, l, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace rr
