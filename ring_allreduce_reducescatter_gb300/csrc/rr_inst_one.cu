// rr_inst_one.cu -- the kernels of one (collective, storage format, wire
// format), chosen when this file is compiled (-DRR_INST_OP, -DRR_INST_DT,
// -DRR_INST_WT, values of the kOp* / kF* constants).  The build script
// compiles it once for every supported combination (INSTANCES in _build.py),
// all at once, so no translation unit carries more than one combination's
// kernels; rr_dispatch.cu calls them through launch_op.
#include "rr_kernels.cuh"

#if !defined(RR_INST_OP) || !defined(RR_INST_DT) || !defined(RR_INST_WT)
#error "rr_inst_one.cu is compiled with -DRR_INST_OP=.. -DRR_INST_DT=.. -DRR_INST_WT=.."
#endif

namespace rr {

template <int OP, int DT, int WT>
cudaError_t launch_op(const RingParams &p, const Launch &l, cudaStream_t s) {
  return launch_one<OP, DT, WT>(p, l, s);
}

template cudaError_t launch_op<RR_INST_OP, RR_INST_DT, RR_INST_WT>(const RingParams &, const Launch &,
                                                                      cudaStream_t);

}  // namespace rr
