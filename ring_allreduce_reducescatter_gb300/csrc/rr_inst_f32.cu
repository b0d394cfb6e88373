// rr_inst_f32.cu -- kernels with binary32 storage on a binary32 wire (the
// 16-bit wires are in rr_inst_f32_narrow.cu), and the bounded-wait probe kernel.
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
      return launch_f32_narrow(op, wire, p, l, s);
    case kOpReduceScatter:
      if (wire == kF32) return launch_one<kOpReduceScatter, kF32, kF32>(p, l, s);
      return launch_f32_narrow(op, wire, p, l, s);
    case kOpAllGather:
      return launch_one<kOpAllGather, kF32, kF32>(p, l, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace rr
