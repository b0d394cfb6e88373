// rr_params.h -- the parameter block of every libringred kernel and the
// internal launcher interface between the C ABI (rr_api.cu) and the kernel
// translation units (rr_dispatch.cu, rr_inst_one.cu, rr_inst_hd_*.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ringred.h"

namespace rr {

enum : int { kF32 = 0, kF16 = 1, kBF16 = 2 };
enum : int { kOpAllReduce = 0, kOpReduceScatter = 1, kOpAllGather = 2 };
enum : int { kAlgoRing = 0, kAlgoHalvingDoubling = 1, kAlgoNaive = 2 };

// Device status bits (the word lives in rr_api.cu).  kStatusIndexFault is
// only ever set by a debug build (RR_DEBUG_CHECKS): an access outside its
// buffer was skipped.
enum : unsigned int { kStatusWaitTimeout = 1u, kStatusIndexFault = 2u };

// Limit of one bounded wait inside a kernel.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

// Passed by value as a __grid_constant__ kernel parameter (about 1.1 KB).
struct RingParams {
  const void *in[RR_MAX_RANKS];
  void *out[RR_MAX_RANKS];
  unsigned long long count;       // elements this launch covers (per rank)
  unsigned long long first;       // global index of element 0 of the buffers (AllReduce ranges)
  unsigned long long total;       // N, elements of the whole rank vector (the chunk table's N)
  unsigned long long base;        // floor(N / L): length of every chunk but the last
  unsigned long long n_bulk;      // bulk path: elements [0, n_bulk) go through tiles
  unsigned long long n_tiles;     // bulk path: ceil(n_bulk / tile_elems)
  unsigned int *status;           // device status word
  int R;                          // ranks
  int L;                          // ranks per group (chunk table of (N, L))
  int G;                          // groups, R / L
  int tile_elems;                 // bulk path: elements per rank per tile
  int stages;                     // bulk path: pipeline depth
  int store_lag;                  // bulk path: store groups left in flight before a stage is refilled (1..8)
  int slots;                      // bulk path: tiles of one stage (R, or 1 for AllGather)
  int direct_u;                   // direct path: vectors per thread and iteration (1..4); shifted kernel: rows per warp item
  int algo;                       // AllReduce summation order: kAlgo*
  int hd_log2p;                   // halving-doubling: log2 of P, the largest power of two <= R
  int hd_extra;                   // halving-doubling: R - P ranks folded in pairs first
  int straddle_cta;               // direct AllReduce: 1 if the grid's last CTA folds the vectors over chunk boundaries
  int shifted;                    // direct ReduceScatter / AllGather: chunk boundaries off the 16-byte grid
  int prefetch;                   // direct path: kPrefetch* bits
  unsigned long long debug_margin;  // debug build: bytes taken off every buffer's extent by the checks
  int chunks_on_grid;             // every chunk boundary of this launch falls on the 16-byte vector grid
  int shift_rows;                 // shifted AllGather: rows of 32 output vectors a warp item (else vectors a thread)
};

// L2 prefetch of the direct path's inputs (no data reaches the SM, so no
// registers are held): kPrefetchHead, a thread's first vectors before the
// programmatic-launch wait (their DRAM latency overlaps the previous kernel's
// tail; a prefetch has no effect on the values read after the wait, since L2
// is where the previous kernel's writes land); kPrefetchAhead, the next
// iteration's vectors while the current ones load (twice the requests in
// flight per thread).
enum : int { kPrefetchHead = 1, kPrefetchAhead = 2 };

// Loads a direct-path thread issues together for one group: U vectors of NB
// ranks each.  Eight whatever U is (nine for U = 3, a three-rank group whole).
__host__ __device__ constexpr int direct_batch_ranks(int U) { return U == 3 ? 3 : 8 / U; }

// The direct-path kernels that exist: (collective, wide accumulators, U
// vectors a thread, OCC 256-thread CTAs per SM the registers are budgeted
// for).  Ring / naive AllReduce and ReduceScatter: U = 1, 2 at OCC 2 or 3,
// U = 3, 4 at OCC 2 (at 85 registers a thread they spill); with binary32
// accumulators of 16-bit storage ("wide", eight floats a vector): U = 1, 2 at
// OCC 2; AllGather: U = 1, 2, 4 at OCC 2.  The planner picks only these and
// rejects a forced launch configuration outside them.
__host__ __device__ constexpr bool direct_variant_exists(int op, bool wide, int U, int occ) {
  return op == kOpAllGather ? ((U == 1 || U == 2 || U == 4) && occ == 2)
         : wide             ? ((U == 1 || U == 2) && occ == 2)
                            : (((U == 1 || U == 2) && (occ == 2 || occ == 3)) || ((U == 3 || U == 4) && occ == 2));
}

// The shifted ReduceScatter / AllGather kernels (chunk boundaries off the
// 16-byte grid): US rows of output vectors per warp work item.
// ReduceScatter: US = 1..4 (wide: 1, 2); AllGather: US = 1, 2, 4; AllReduce
// (chunks on the grid): US = 2, 4, not wide.
__host__ __device__ constexpr bool shift_variant_exists(int op, bool wide, int US) {
  return op == kOpAllGather     ? (US == 1 || US == 2 || US == 4)
         : op == kOpAllReduce   ? (!wide && (US == 2 || US == 4))
         : wide                 ? (US == 1 || US == 2)
                                : (US >= 1 && US <= 4);
}

// 256-thread CTAs per SM the shifted kernel of US rows is compiled for.
__host__ __device__ constexpr int shift_occupancy(int US) { return US >= 3 ? 2 : 3; }

// One launch, fully resolved by the planner.
struct Launch {
  int path;         // RR_PATH_BULK, RR_PATH_SIMPLE or RR_PATH_DIRECT
  int grid;
  int threads;
  size_t smem;      // dynamic shared memory bytes
  int ctas_per_sm;
  bool early_launch;   // launch with programmatic stream serialisation
  int direct_occ = 2;  // direct path, one vector per thread: 256-thread CTAs per SM it is compiled for (2 or 3)
};

// The kernel of (OP, storage DT, wire WT) on `stream`; returns the launch
// error.  Explicitly instantiated once per supported combination, each in its
// own object of rr_inst_one.cu.
template <int OP, int DT, int WT>
cudaError_t launch_op(const RingParams &p, const Launch &l, cudaStream_t s);

// Defined in rr_dispatch.cu: the launch_op of (op, storage dtype, wire).
cudaError_t launch_collective(int op, int dtype, int wire, const RingParams &p, const Launch &l, cudaStream_t s);
// Defined in rr_inst_hd_<storage>.cu: the halving-doubling AllReduce on the
// direct path (one kernel per tree size).
cudaError_t launch_hd_direct_f32(int wire, const RingParams &p, const Launch &l, cudaStream_t s);
cudaError_t launch_hd_direct_f16(int wire, const RingParams &p, const Launch &l, cudaStream_t s);
cudaError_t launch_hd_direct_bf16(int wire, const RingParams &p, const Launch &l, cudaStream_t s);
inline cudaError_t launch_hd_direct(int dt, int wire, const RingParams &p, const Launch &l, cudaStream_t s) {
  return dt == kF32 ? launch_hd_direct_f32(wire, p, l, s)
                    : dt == kF16 ? launch_hd_direct_f16(wire, p, l, s) : launch_hd_direct_bf16(wire, p, l, s);
}
// Defined in rr_dispatch.cu: the bounded-wait self test kernel.
cudaError_t launch_wait_probe(unsigned int *status, unsigned long long limit_ns, cudaStream_t s);

}  // namespace rr
