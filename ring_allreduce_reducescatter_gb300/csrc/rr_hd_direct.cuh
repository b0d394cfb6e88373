// rr_hd_direct.cuh -- the halving-doubling AllReduce on the direct path: one
// kernel per tree size, so that each is register-allocated for its own tree
// and issues its loads in batches.  Instantiated per storage format by
// rr_inst_hd_<storage>.cu.
//
// The order is the textbook recursive-halving tree the topology switch of the
// page ai6s.net/6a0dd5b5662f9a54cb75ef90.html (TpAllReduceOp::Execute)
// selects for a full mesh: with P the largest power of two <= R and
// E = R - P, leaves L_v = x_{2v} (+) x_{2v+1} for v < E and x_{v+E}
// otherwise, then L_v = L_v (+) L_{v+d} for d = P/2, P/4, ..., 1.
#pragma once

#include "rr_kernels.cuh"

namespace rr {
namespace hd {

// The 2^LOG2N leaves v0 + m * stride (m < 2^LOG2N), loaded together (two
// ranks for a leaf v < E when EXTRA, one otherwise) and combined by the tree
// whose first level pairs m and m + 2^LOG2N / 2.
template <class VT, int E, int LOG2N, bool EXTRA>
__device__ __forceinline__ typename VT::W hd_batch(const RingParams &p, unsigned long long boff, int v0, int stride) {
  using W = typename VT::W;
  constexpr int N = 1 << LOG2N;
  const int Ex = EXTRA ? p.hd_extra : 0;
  uint4 xa[N], xb[N];
#pragma unroll
  for (int m = 0; m < N; ++m) {
    const int v = v0 + m * stride;
    const bool pair = EXTRA && v < Ex;
    xa[m] = load_in<false, E>(p, pair ? 2 * v : v + Ex, boff);
    if constexpr (EXTRA) {
      xb[m] = pair ? load_in<false, E>(p, 2 * v + 1, boff) : make_uint4(0, 0, 0, 0);
    }
  }
  auto leaf = [&](int m) {
    if constexpr (EXTRA) {
      if (v0 + m * stride < Ex) return VT::hop(VT::in(xa[m]), VT::in(xb[m]));
    }
    return VT::in(xa[m]);
  };
  auto add = [](W a, W b) { return VT::hop(a, b); };
  return hd_tree<LOG2N, W>(leaf, add);
}

// The whole tree for P = 2^LOG2P.  Its first three levels (partners P/2, P/4
// and P/8 apart) only combine leaves of one coset {v + m Q : m < 8}, Q = P/8,
// so for P > 8 it is the tree over the Q coset sums (partners Q/2, ..., 1
// apart) of 8-leaf trees: one batch of at most 16 loads per coset.
template <class VT, int E, int LOG2P, bool EXTRA>
__device__ __forceinline__ typename VT::W hd_vec(const RingParams &p, unsigned long long boff) {
  using W = typename VT::W;
  if constexpr (LOG2P <= 3) {
    return hd_batch<VT, E, LOG2P, EXTRA>(p, boff, 0, 1);
  } else {
    constexpr int Q = 1 << (LOG2P - 3);
    auto coset = [&](int v) { return hd_batch<VT, E, 3, EXTRA>(p, boff, v, Q); };
    auto add = [](W a, W b) { return VT::hop(a, b); };
    return hd_tree<LOG2P - 3, W>(coset, add);
  }
}

// Element i by the same tree, with scalar loads (the ragged end).
template <int DT, int WT, int LOG2P, bool EXTRA>
__device__ __forceinline__ typename Fmt<DT>::type hd_scalar(const RingParams &p, unsigned long long i) {
  using S = typename Fmt<DT>::type;
  using SC = Scalar<DT, WT>;
  using W = typename SC::W;
  const int Ex = EXTRA ? p.hd_extra : 0;
  auto x = [&](int r) { return SC::in(load_elem<false, S>(p, r, i)); };
  auto leaf = [&](int v) {
    if constexpr (EXTRA) {
      if (v < Ex) return hop(x(2 * v), x(2 * v + 1));
    }
    return x(v + Ex);
  };
  auto add = [](W a, W b) { return hop(a, b); };
  return SC::out(hd_tree<LOG2P, W>(leaf, add));
}

// OCC: 256-thread CTAs per SM the registers are budgeted for, as for the ring's
// direct kernel.
template <int DT, int WT, int LOG2P, bool EXTRA, int OCC>
__global__ void __launch_bounds__(kDirectThreads, OCC) rr_hd_direct_kernel(const __grid_constant__ RingParams p) {
  grid_dependency_wait();
  grid_dependents_launch();
  using VT = Vec<DT, WT>;
  constexpr int V = VT::V;
  constexpr int E = Fmt<DT>::bytes;
  const unsigned long long nvec = p.n_bulk / V;
  const unsigned long long T = (unsigned long long)gridDim.x * blockDim.x;
  for (unsigned long long v = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += T) {
    const unsigned long long boff = v * V * E;
    const uint4 res = VT::out(hd_vec<VT, E, LOG2P, EXTRA>(p, boff));
    for (int r = 0; r < p.R; ++r) store_out<false, E>(p, r, boff, res);
  }
  // the ragged end (under 16 bytes per rank)
  for (unsigned long long i = p.n_bulk + (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; i < p.count;
       i += T) {
    const typename Fmt<DT>::type y = hd_scalar<DT, WT, LOG2P, EXTRA>(p, i);
    for (int r = 0; r < p.R; ++r) store_elem<false, typename Fmt<DT>::type>(p, r, i, y);
  }
}

template <int DT, int WT, int LOG2P, bool EXTRA>
cudaError_t launch_occ(const RingParams &p, const Launch &l, cudaStream_t s) {
  constexpr bool wide = DT != kF32 && WT == kF32;
  if constexpr (!wide && LOG2P <= 2) {  // the planner asks for three CTAs below seven ranks only
    if (l.direct_occ == 3) return launch_kernel(rr_hd_direct_kernel<DT, WT, LOG2P, EXTRA, 3>, l, 0, s, p);
  }
  return launch_kernel(rr_hd_direct_kernel<DT, WT, LOG2P, EXTRA, 2>, l, 0, s, p);
}

template <int DT, int WT, int LOG2P>
cudaError_t launch_size(const RingParams &p, const Launch &l, cudaStream_t s) {
  if constexpr (LOG2P > 0) {
    if (p.hd_extra > 0) return launch_occ<DT, WT, LOG2P, true>(p, l, s);
  }
  return launch_occ<DT, WT, LOG2P, false>(p, l, s);
}

template <int DT, int WT>
cudaError_t launch_pair(const RingParams &p, const Launch &l, cudaStream_t s) {
  switch (p.hd_log2p) {
    case 0:
      return launch_size<DT, WT, 0>(p, l, s);
    case 1:
      return launch_size<DT, WT, 1>(p, l, s);
    case 2:
      return launch_size<DT, WT, 2>(p, l, s);
    case 3:
      return launch_size<DT, WT, 3>(p, l, s);
    case 4:
      return launch_size<DT, WT, 4>(p, l, s);
    case 5:
      return launch_size<DT, WT, 5>(p, l, s);
    case 6:
      return launch_size<DT, WT, 6>(p, l, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace hd
}  // namespace rr
