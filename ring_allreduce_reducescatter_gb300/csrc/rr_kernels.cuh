// rr_kernels.cuh -- the kernels of libringred.
//
// Every kernel computes, for each element i of the N-element rank vectors,
//   S_g = x_{gL+c} (+) x_{gL+c+1} (+) ... (+) x_{gL+c+L-1}   (ranks mod L)
//   y   = S_0 (+) S_1 (+) ... (+) S_{G-1}
// with c the chunk of i in the partition of N into L chunks and (+) one hop
// on the wire.  That is the value the ring produces: on the page
// hwcomputing.csdn.net/6a0dc11a10ee7a33f273f7fd.html, section
// "Ring 通信为什么常见", block c starts on card c and picks up cards c+1, c+2,
// ... in turn (the simplified ReduceScatter code on
// ai6s.net/6a102b5410ee7a33f2746c06.html, section "hcomm 与 HCCL 的关系",
// moves the chunk index back by one per step, which is the same order), and
// the AllGather phase copies each finished block to every card.  The two-level
// ring (page hwcomputing.csdn.net/6a0dc11a..., section "通信拓扑与带宽利用率")
// folds the group sums of a chunk once, in group order.
//
// Instead of moving chunks between ranks, a kernel reads every rank's copy of
// an element once, folds it in registers in exactly the ring's order, and
// writes the result once per output: the zero-copy principle of
// ai6s.net/6a102b54..., section "hcomm 的数据传输路径", carried to its end (no
// staging buffers, each byte crosses HBM once).
//
//  rr_simple_kernel: one element per thread, grid-stride, plain loads/stores;
//    any alignment.
//  rr_bulk_kernel: persistent CTAs over tiles of the element range.  Thread 0
//    fills S pipeline stages with bulk asynchronous copies (one tile per rank,
//    completion counted on an mbarrier); all threads fold 16-byte vectors out
//    of shared memory and write the result over slot 0 of the stage; thread 0
//    then writes slot 0 to the outputs with bulk asynchronous stores and
//    refills the stage of the tile D steps back once its stores have read
//    shared memory (D = store_lag): D + 1 tiles of stores and S - D - 1 tiles
//    of loads stay in flight while a tile is folded.  Every wait is bounded.
//  rr_direct_kernel: every thread loads its ranks' 16-byte vectors straight
//    from HBM in batches of eight loads, folds them in registers and stores
//    the result to every output; one extra CTA folds the AllReduce vectors
//    that straddle a chunk boundary.
//  rr_shift_kernel: ReduceScatter / AllGather chunk by chunk, for chunk
//    boundaries off the 16-byte grid (vectors built from two aligned blocks)
//    and, unshifted, for large AllGathers, two-rank ReduceScatters and
//    AllReduces over two to four ranks.
//  The halving-doubling direct kernels are in rr_hd_direct.cuh.
//  Every kernel starts with the programmatic-launch wait, so a launch may
//  overlap the kernel before it on the stream.
#pragma once

#include <mutex>

#include "rr_device.cuh"

namespace rr {

// --------------------------------------------------------------------------
// accesses to the rank buffers.  Every load, store, bulk copy and prefetch of
// a rank buffer goes through these.  A debug build (RR_DEBUG_CHECKS) checks
// each against the buffer's extent in this launch; an access outside it is
// skipped (a load reads zeros, a skipped bulk load's bytes are retired from
// its barrier) and sets kStatusIndexFault in the status word, so an index
// error shows as a status bit, not a fault.  A release build compiles each to
// the plain access.  CH: the buffer holds one chunk (a ReduceScatter output, an
// AllGather input); otherwise the launch's `count` elements.
// --------------------------------------------------------------------------

#ifdef RR_DEBUG_CHECKS
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

__device__ __forceinline__ unsigned long long extent_bytes(const RingParams &p, int r, bool chunk, int E) {
  const unsigned long long n =
      chunk ? (r < p.L - 1 ? p.base : p.total - (unsigned long long)(p.L - 1) * p.base) : p.count;
  return n * (unsigned long long)E;
}

// [off, off + bytes) of buffer r lies inside its extent (always, in a release build).
template <bool CH, int E>
__device__ __forceinline__ bool access_ok(const RingParams &p, int r, unsigned long long off,
                                          unsigned long long bytes) {
  if constexpr (kDebugChecks) {
    if (r < 0 || r >= p.R) {
      atomicOr(p.status, kStatusIndexFault);
      return false;
    }
    const unsigned long long ext = extent_bytes(p, r, CH, E);
    const unsigned long long lim = ext > p.debug_margin ? ext - p.debug_margin : 0;
    if (off > lim || bytes > lim - off) {
      atomicOr(p.status, kStatusIndexFault);
      return false;
    }
  }
  return true;
}

template <bool CH, int E>
__device__ __forceinline__ uint4 load_in(const RingParams &p, int r, unsigned long long off) {
  if (!access_ok<CH, E>(p, r, off, 16)) return make_uint4(0u, 0u, 0u, 0u);
  return ldg_stream(static_cast<const unsigned char *>(p.in[r]) + off);
}

template <bool CH, int E>
__device__ __forceinline__ uint4 load_in_l1(const RingParams &p, int r, unsigned long long off) {
  if (!access_ok<CH, E>(p, r, off, 16)) return make_uint4(0u, 0u, 0u, 0u);
  return ldg_l1(static_cast<const unsigned char *>(p.in[r]) + off);
}

template <bool CH, int E>
__device__ __forceinline__ void store_out(const RingParams &p, int r, unsigned long long off, uint4 v) {
  if (access_ok<CH, E>(p, r, off, 16)) stg_stream(static_cast<unsigned char *>(p.out[r]) + off, v);
}

template <bool CH, int E>
__device__ __forceinline__ void prefetch_in(const RingParams &p, int r, unsigned long long off) {
  if (access_ok<CH, E>(p, r, off, 16)) prefetch_l2(static_cast<const unsigned char *>(p.in[r]) + off);
}

// One element (index i of the buffer).
template <bool CH, class S>
__device__ __forceinline__ S load_elem(const RingParams &p, int r, unsigned long long i) {
  if (!access_ok<CH, (int)sizeof(S)>(p, r, i * sizeof(S), sizeof(S))) return S{};
  return static_cast<const S *>(p.in[r])[i];
}

template <bool CH, class S>
__device__ __forceinline__ void store_elem(const RingParams &p, int r, unsigned long long i, S v) {
  if (access_ok<CH, (int)sizeof(S)>(p, r, i * sizeof(S), sizeof(S))) static_cast<S *>(p.out[r])[i] = v;
}

// Bulk copy of `bytes` from input r at `off` into shared memory (completion on bar).
template <bool CH, int E>
__device__ __forceinline__ void bulk_load_in(const RingParams &p, int r, unsigned long long off, void *smem_dst,
                                             uint32_t bytes, uint64_t *bar, uint64_t pol) {
  if (access_ok<CH, E>(p, r, off, bytes))
    bulk_load(smem_dst, static_cast<const unsigned char *>(p.in[r]) + off, bytes, bar, pol);
  else
    mbar_complete_tx(bar, bytes);
}

template <bool CH, int E>
__device__ __forceinline__ void bulk_store_out(const RingParams &p, int r, unsigned long long off,
                                               const void *smem_src, uint32_t bytes, uint64_t pol) {
  if (access_ok<CH, E>(p, r, off, bytes)) bulk_store(static_cast<unsigned char *>(p.out[r]) + off, smem_src, bytes, pol);
}

// --------------------------------------------------------------------------
// summation orders of the other AllReduce algorithms (page
// ai6s.net/6a0dd5b5662f9a54cb75ef90.html, TpAllReduceOp::Execute)
// --------------------------------------------------------------------------

// The chunk of global element i through a one-entry cache of the chunk last
// looked up: a direct-path thread's vectors advance by a fixed stride, so the
// 64-bit division of chunk_of runs only when one leaves the cached chunk
// (measured at 256 MiB per rank against two divisions a vector: ReduceScatter
// over two / three ranks 165 -> 144 / 179 -> 161 us, AllReduce over two ranks
// 204 -> 179 us; a multiply-and-shift division by the invariant chunk length
// instead was slower than both).  [lo, hi) is the cached chunk's index range
// (the last chunk's reaches the end of the index space, as chunk_of clamps);
// lo == hi is empty.
struct ChunkCache {
  unsigned long long lo = 0, hi = 0;
  int c = 0;
};

__device__ __forceinline__ int cached_chunk(ChunkCache &cc, const RingParams &p, unsigned long long i) {
  if (i - cc.lo < cc.hi - cc.lo) return cc.c;  // lo <= i < hi
  const int c = chunk_of(p, i);
  cc.c = c;
  cc.lo = (unsigned long long)c * p.base;
  cc.hi = c == p.L - 1 ? ~0ull : (unsigned long long)(c + 1) * p.base;
  return c;
}

// Naive (Reduce + Broadcast): the collector adds ranks 0, 1, ..., R-1 in order,
// which is the ring fold started at rank 0 for every element.
__device__ __forceinline__ int start_rank(const RingParams &p, unsigned long long global_index) {
  return p.algo == kAlgoNaive ? 0 : chunk_of(p, global_index);
}

__host__ __device__ constexpr int bit_reverse(int u, int bits) {
  int r = 0;
  for (int i = 0; i < bits; ++i) r |= ((u >> i) & 1) << (bits - 1 - i);
  return r;
}
__host__ __device__ constexpr int trailing_ones(int u) {
  int k = 0;
  while (u & 1) {
    ++k;
    u >>= 1;
  }
  return k;
}

// Halving-doubling: P = 2^LOG2P leaves L_v, combined by recursive halving
// (partners at distance P/2 first): level 1 adds L_v and L_{v+P/2}, level 2
// adds those pair sums at distance P/4, and so on.  Visiting the leaves in
// bit-reversed order turns that tree into adjacent pairs, so a pairwise stack
// of LOG2P + 1 entries, fully unrolled, evaluates it with static indices.
template <int LOG2P, class W, class Leaf, class Add>
__device__ __forceinline__ W hd_tree(const Leaf &leaf, const Add &add) {
  constexpr int P = 1 << LOG2P;
  W stk[LOG2P + 1];
#pragma unroll
  for (int u = 0; u < P; ++u) {
    W val = leaf(bit_reverse(u, LOG2P));
#pragma unroll
    for (int t = 0; t < LOG2P; ++t)
      if (t < trailing_ones(u)) val = add(stk[t], val);
    stk[trailing_ones(u)] = val;
  }
  return stk[LOG2P];
}

// The tree for the runtime P (leaf(v) gives L_v).
template <class W, class Leaf, class Add>
__device__ __forceinline__ W hd_fold(int log2p, const Leaf &leaf, const Add &add) {
  switch (log2p) {
    case 0:
      return hd_tree<0, W>(leaf, add);
    case 1:
      return hd_tree<1, W>(leaf, add);
    case 2:
      return hd_tree<2, W>(leaf, add);
    case 3:
      return hd_tree<3, W>(leaf, add);
    case 4:
      return hd_tree<4, W>(leaf, add);
    case 5:
      return hd_tree<5, W>(leaf, add);
    default:
      return hd_tree<6, W>(leaf, add);
  }
}

// --------------------------------------------------------------------------
// one element, global memory
// --------------------------------------------------------------------------

template <int DT, int WT>
__device__ __forceinline__ typename Scalar<DT, WT>::W fold_group_global(const RingParams &p, int g, int c,
                                                                        unsigned long long i) {
  using S = typename Fmt<DT>::type;
  using SC = Scalar<DT, WT>;
  const int L = p.L;
  int r = c;
  typename SC::W acc = SC::in(load_elem<false, S>(p, g * L + r, i));
  for (int k = 1; k < L; ++k) {
    r = (r + 1 == L) ? 0 : r + 1;
    acc = hop(acc, SC::in(load_elem<false, S>(p, g * L + r, i)));
  }
  return acc;
}

template <int DT, int WT>
__device__ __forceinline__ typename Fmt<DT>::type fold_elem_global(const RingParams &p, unsigned long long i, int c) {
  typename Scalar<DT, WT>::W total = fold_group_global<DT, WT>(p, 0, c, i);
  for (int g = 1; g < p.G; ++g) total = hop(total, fold_group_global<DT, WT>(p, g, c, i));
  return Scalar<DT, WT>::out(total);
}

// The whole collective at element i (every input read, then every output written).
// i is the buffers' (local) index; its chunk is that of the global index first + i.
template <int DT, int WT>
__device__ __forceinline__ typename Fmt<DT>::type hd_elem_global(const RingParams &p, unsigned long long i) {
  using S = typename Fmt<DT>::type;
  using SC = Scalar<DT, WT>;
  using W = typename SC::W;
  const int E = p.hd_extra;
  auto x = [&](int r) { return SC::in(load_elem<false, S>(p, r, i)); };
  auto leaf = [&](int v) { return v < E ? hop(x(2 * v), x(2 * v + 1)) : x(v + E); };
  auto add = [](W a, W b) { return hop(a, b); };
  return SC::out(hd_fold<W>(p.hd_log2p, leaf, add));
}

// HD: the halving-doubling tree instead of the ring / naive fold (a separate
// instantiation, so the ring kernels carry none of its registers).
template <int OP, int DT, int WT, bool HD = false>
__device__ __forceinline__ void element_op(const RingParams &p, unsigned long long i) {
  using S = typename Fmt<DT>::type;
  const int c = start_rank(p, p.first + i);
  if (OP == kOpAllReduce) {
    S v;
    if constexpr (HD)
      v = hd_elem_global<DT, WT>(p, i);
    else
      v = fold_elem_global<DT, WT>(p, i, c);
    for (int r = 0; r < p.R; ++r) store_elem<false, S>(p, r, i, v);
  } else if (OP == kOpReduceScatter) {
    const S v = fold_elem_global<DT, WT>(p, i, c);
    store_elem<true, S>(p, c, i - (unsigned long long)c * p.base, v);
  } else {
    const S v = load_elem<true, S>(p, c, i - (unsigned long long)c * p.base);
    for (int r = 0; r < p.R; ++r) store_elem<false, S>(p, r, i, v);
  }
}

template <int OP, int DT, int WT, bool HD>
__global__ void __launch_bounds__(1024) rr_simple_kernel(const __grid_constant__ RingParams p) {
  grid_dependency_wait();
  grid_dependents_launch();
  const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
  for (unsigned long long i = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; i < p.count; i += stride)
    element_op<OP, DT, WT, HD>(p, i);
}

// --------------------------------------------------------------------------
// tiles in shared memory: slot r of a stage holds rank r's tile
// --------------------------------------------------------------------------

template <class VT>
__device__ __forceinline__ typename VT::W fold_group_vec(const unsigned char *gstage, uint32_t slot_bytes, int L, int c,
                                                         uint32_t off) {
  int r = c;
  typename VT::W acc = VT::in(*reinterpret_cast<const uint4 *>(gstage + (size_t)r * slot_bytes + off));
  for (int k = 1; k < L; ++k) {
    r = (r + 1 == L) ? 0 : r + 1;
    acc = VT::hop(acc, VT::in(*reinterpret_cast<const uint4 *>(gstage + (size_t)r * slot_bytes + off)));
  }
  return acc;
}

// 16 bytes whose elements all lie in chunk c.
template <class VT>
__device__ __forceinline__ uint4 fold_vec_smem(const unsigned char *stage, uint32_t slot_bytes, int L, int G, int c,
                                               uint32_t off) {
  typename VT::W total = fold_group_vec<VT>(stage, slot_bytes, L, c, off);
  for (int g = 1; g < G; ++g)
    total = VT::hop(total, fold_group_vec<VT>(stage + (size_t)g * L * slot_bytes, slot_bytes, L, c, off));
  return VT::out(total);
}

// 16 bytes that straddle a chunk boundary, element by element (i0: global index).
template <int DT, int WT>
__device__ __noinline__ uint4 fold_ragged_smem(const RingParams &p, const unsigned char *stage, uint32_t slot_bytes,
                                               unsigned long long i0, uint32_t off) {
  using S = typename Fmt<DT>::type;
  using SC = Scalar<DT, WT>;
  constexpr int V = 16 / (int)sizeof(S);
  const int L = p.L;
  S res[V];
#pragma unroll
  for (int e = 0; e < V; ++e) {
    const int c = chunk_of(p, i0 + e);
    const uint32_t eo = off + (uint32_t)(e * sizeof(S));
    typename SC::W total;
    for (int g = 0; g < p.G; ++g) {
      const unsigned char *gs = stage + (size_t)g * L * slot_bytes + eo;
      int r = c;
      typename SC::W acc = SC::in(*reinterpret_cast<const S *>(gs + (size_t)r * slot_bytes));
      for (int k = 1; k < L; ++k) {
        r = (r + 1 == L) ? 0 : r + 1;
        acc = hop(acc, SC::in(*reinterpret_cast<const S *>(gs + (size_t)r * slot_bytes)));
      }
      total = (g == 0) ? acc : hop(total, acc);
    }
    res[e] = SC::out(total);
  }
  uint4 out;
  memcpy(&out, res, 16);
  return out;
}

__device__ __forceinline__ unsigned long long tile_begin(const RingParams &p, unsigned long long t) {
  return t * (unsigned long long)p.tile_elems;
}
__device__ __forceinline__ unsigned long long tile_end(const RingParams &p, unsigned long long t) {
  const unsigned long long e = (t + 1) * (unsigned long long)p.tile_elems;
  return e < p.n_bulk ? e : p.n_bulk;
}

// Fold tile t (AllReduce / ReduceScatter); the result replaces slot 0.
template <int DT, int WT, bool HD>
__device__ __forceinline__ void compute_tile(const RingParams &p, unsigned char *stage, uint32_t slot_bytes,
                                             unsigned long long t) {
  using VT = Vec<DT, WT>;
  constexpr int V = VT::V;
  const unsigned long long t0 = tile_begin(p, t), t1 = tile_end(p, t);
  const uint32_t nvec = (uint32_t)((t1 - t0) / V);
  const int L = p.L, G = p.G;
  if constexpr (HD) {  // the same tree for every element
    using W = typename VT::W;
    const int E = p.hd_extra;
    for (uint32_t v = threadIdx.x; v < nvec; v += blockDim.x) {
      const uint32_t off = v * 16u;
      auto x = [&](int r) { return VT::in(*reinterpret_cast<const uint4 *>(stage + (size_t)r * slot_bytes + off)); };
      auto leaf = [&](int u) { return u < E ? VT::hop(x(2 * u), x(2 * u + 1)) : x(u + E); };
      auto add = [](W a, W b) { return VT::hop(a, b); };
      const uint4 res = VT::out(hd_fold<W>(p.hd_log2p, leaf, add));
      *reinterpret_cast<uint4 *>(stage + off) = res;
    }
    return;
  }
  const unsigned long long g0 = p.first + t0;  // global index of the tile's first element
  const int c_first = start_rank(p, g0), c_last = start_rank(p, g0 + (t1 - t0) - 1);
  for (uint32_t v = threadIdx.x; v < nvec; v += blockDim.x) {
    const uint32_t off = v * 16u;
    int c = c_first, c1 = c_last;
    if (c != c1) {
      const unsigned long long i0 = g0 + (unsigned long long)v * V;
      c = chunk_of(p, i0);
      c1 = chunk_of(p, i0 + V - 1);
    }
    uint4 res;
    if (c == c1)
      res = fold_vec_smem<VT>(stage, slot_bytes, L, G, c, off);
    else
      res = fold_ragged_smem<DT, WT>(p, stage, slot_bytes, g0 + (unsigned long long)v * V, off);
    *reinterpret_cast<uint4 *>(stage + off) = res;
  }
}

// Fill a stage with tile t.  AllReduce / ReduceScatter: rank r's tile into
// slot r.  AllGather: the tile of the output vector, gathered chunk by chunk
// from the inputs into slot 0.
template <int OP, int DT>
__device__ __forceinline__ void issue_loads(const RingParams &p, unsigned char *stage, uint32_t slot_bytes,
                                            uint64_t *bar, unsigned long long t, uint64_t pol) {
  constexpr int E = Fmt<DT>::bytes;
  const unsigned long long t0 = tile_begin(p, t), t1 = tile_end(p, t);
  const uint32_t bytes = (uint32_t)((t1 - t0) * E);
  if (OP != kOpAllGather) {
    mbar_arrive_expect_tx(bar, bytes * (uint32_t)p.R);
    for (int r = 0; r < p.R; ++r) bulk_load_in<false, E>(p, r, t0 * E, stage + (size_t)r * slot_bytes, bytes, bar, pol);
  } else {
    mbar_arrive_expect_tx(bar, bytes);
    const int c_lo = chunk_of(p, t0), c_hi = chunk_of(p, t1 - 1);
    for (int c = c_lo; c <= c_hi; ++c) {
      const unsigned long long off = (unsigned long long)c * p.base;
      const unsigned long long end = chunk_end(c, p.base, p.L, p.total);
      const unsigned long long s0 = t0 > off ? t0 : off, s1 = t1 < end ? t1 : end;
      if (s1 > s0) bulk_load_in<true, E>(p, c, (s0 - off) * E, stage + (s0 - t0) * E, (uint32_t)((s1 - s0) * E), bar, pol);
    }
  }
}

// Write slot 0 of a stage (tile t).  AllReduce / AllGather: to every output.
// ReduceScatter: each chunk's part to the output of that chunk.
template <int OP, int DT>
__device__ __forceinline__ void issue_stores(const RingParams &p, const unsigned char *stage, unsigned long long t,
                                             uint64_t pol) {
  constexpr int E = Fmt<DT>::bytes;
  const unsigned long long t0 = tile_begin(p, t), t1 = tile_end(p, t);
  const uint32_t bytes = (uint32_t)((t1 - t0) * E);
  if (OP != kOpReduceScatter) {
    for (int r = 0; r < p.R; ++r) bulk_store_out<false, E>(p, r, t0 * E, stage, bytes, pol);
  } else {
    const int c_lo = chunk_of(p, t0), c_hi = chunk_of(p, t1 - 1);
    for (int c = c_lo; c <= c_hi; ++c) {
      const unsigned long long off = (unsigned long long)c * p.base;
      const unsigned long long end = chunk_end(c, p.base, p.L, p.total);
      const unsigned long long s0 = t0 > off ? t0 : off, s1 = t1 < end ? t1 : end;
      if (s1 > s0) bulk_store_out<true, E>(p, c, (s0 - off) * E, stage + (s0 - t0) * E, (uint32_t)((s1 - s0) * E), pol);
    }
  }
}

template <int OP, int DT, int WT, bool HD>
__global__ void __launch_bounds__(1024) rr_bulk_kernel(const __grid_constant__ RingParams p) {
  grid_dependency_wait();
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int E = Fmt<DT>::bytes;
  const int S = p.stages;
  const uint32_t slot_bytes = (uint32_t)p.tile_elems * E;
  const uint32_t stage_bytes = slot_bytes * (uint32_t)p.slots;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)S * stage_bytes);

  // tiles of this CTA: first, first + step, first + 2 step, ...
  const unsigned long long first = blockIdx.x, step = gridDim.x;
  const long long n_local = first < p.n_tiles ? (long long)((p.n_tiles - 1 - first) / step + 1) : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t pol = l2_evict_first_policy();
  if (threadIdx.x == 0) {
    const long long pro = n_local < S ? n_local : S;
    for (long long j = 0; j < pro; ++j)
      issue_loads<OP, DT>(p, smem + (size_t)j * stage_bytes, slot_bytes, &full[j], first + (unsigned long long)j * step,
                          pol);
  }

  // The ragged end [n_bulk, count) (less than 16 bytes per rank) goes through
  // plain loads and stores in the last CTA, while its first tiles load.
  if (blockIdx.x == gridDim.x - 1)
    for (unsigned long long i = p.n_bulk + threadIdx.x; i < p.count; i += blockDim.x) element_op<OP, DT, WT, HD>(p, i);

  long long j = 0;
  bool ok = true;
  for (; j < n_local; ++j) {
    const int s = (int)(j % S);
    const uint32_t parity = (uint32_t)((j / S) & 1);
    unsigned char *stage = smem + (size_t)s * stage_bytes;
    const unsigned long long t = first + (unsigned long long)j * step;
    const bool got = mbar_wait_bounded(&full[s], parity, kWaitLimitNs);
    if (OP != kOpAllGather && got) compute_tile<DT, WT, HD>(p, stage, slot_bytes, t);
    fence_proxy_async_smem();
    if (!__syncthreads_and(got)) {
      ok = false;
      break;
    }
    if (threadIdx.x == 0) {
      issue_stores<OP, DT>(p, stage, t, pol);
      bulk_commit();
      // refill the stage of tile j-D once its stores have read shared memory
      const int D = p.store_lag;
      if (j >= D && j - D + S < n_local) {
        bulk_wait_read_upto(D);
        const int sp = (int)((j - D) % S);
        issue_loads<OP, DT>(p, smem + (size_t)sp * stage_bytes, slot_bytes, &full[sp],
                            first + (unsigned long long)(j - D + S) * step, pol);
      }
    }
  }
  // Only now may the next kernel be scheduled: its CTAs would fit beside this
  // persistent grid and, while they wait for it, slow it down (measured).
  grid_dependents_launch();
  if (threadIdx.x == 0) {
    if (!ok) {
      atomicOr(p.status, kStatusWaitTimeout);
      // let the loads still in flight land before the shared memory is released
      long long issued_end = (j >= p.store_lag ? j - p.store_lag : 0) + S;
      if (issued_end > n_local) issued_end = n_local;
      for (long long u = j; u < issued_end; ++u)
        mbar_wait_bounded(&full[u % S], (uint32_t)((u / S) & 1), kWaitLimitNs);
    }
    bulk_wait_all();
  }
}

// --------------------------------------------------------------------------
// direct path: every thread takes U 16-byte vectors (a grid-stride apart) per
// iteration, loads them straight from the ranks' buffers in batches of 8 / U
// ranks (so eight 16-byte loads are in flight per thread whatever R is), folds
// them in registers in the ring's order and stores the results straight to
// the outputs: one DRAM round trip per vector, no shared memory, no barriers
// --------------------------------------------------------------------------

constexpr int kDirectThreads = 256;

// The first nbytes bytes of a, the rest of b.
__device__ __forceinline__ uint4 blend_bytes(uint4 a, uint4 b, int nbytes) {
  auto word = [nbytes](uint32_t x, uint32_t y, int w) -> uint32_t {
    const int lo = w * 4;
    if (nbytes >= lo + 4) return x;
    if (nbytes <= lo) return y;
    const uint32_t keep = (1u << (8 * (nbytes - lo))) - 1u;  // the low bytes come from a
    return (x & keep) | (y & ~keep);
  };
  return make_uint4(word(a.x, b.x, 0), word(a.y, b.y, 1), word(a.z, b.z, 2), word(a.w, b.w, 3));
}

// An AllReduce vector whose elements lie in two adjacent chunks c0 and
// c0 + 1: the first ones start the ring at rank c0 (c0, c0+1, ..., c0+L-1),
// the others at c0 + 1 (c0+1, ..., c0+L-1, then c0).  Both folds share one
// pass of 16-byte loads in the first order; the second keeps rank c0's vector
// aside and adds it last.  Vectors over more chunks (chunks shorter than a
// vector) go element by element.
template <int DT, int WT>
__device__ __forceinline__ void straddle_vec(const RingParams &p, unsigned long long v, int c0, int c_last) {
  using VT = Vec<DT, WT>;
  using W = typename VT::W;
  constexpr int V = VT::V;
  constexpr int E = Fmt<DT>::bytes;
  const unsigned long long i0 = v * V, boff = i0 * E;
  const int L = p.L;
  if (c_last != c0 + 1) {
    for (int e = 0; e < V; ++e) element_op<kOpAllReduce, DT, WT>(p, i0 + e);
    return;
  }
  const int split = (int)(chunk_end(c0, p.base, L, p.total) - (p.first + i0));  // elements starting at c0
  W total_a, total_b;
  for (int g = 0; g < p.G; ++g) {
    W a, b;
    uint4 first;
    for (int k0 = 0; k0 < L; k0 += 4) {  // rare: a short batch keeps its registers few
      uint4 x[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (k0 + j < L) {
          int r = c0 + k0 + j;
          r -= (r >= L) ? L : 0;
          x[j] = load_in<false, E>(p, g * L + r, boff);
        }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int k = k0 + j;
        if (k >= L) break;
        const W w = VT::in(x[j]);
        if (k == 0) {
          a = w;
          first = x[j];
        } else {
          a = VT::hop(a, w);
          b = (k == 1) ? w : VT::hop(b, w);
        }
      }
    }
    b = VT::hop(b, VT::in(first));
    total_a = (g == 0) ? a : VT::hop(total_a, a);
    total_b = (g == 0) ? b : VT::hop(total_b, b);
  }
  const uint4 res = blend_bytes(VT::out(total_a), VT::out(total_b), split * E);
  for (int r = 0; r < p.R; ++r) store_out<false, E>(p, r, boff, res);
}

// The AllReduce vectors that straddle a chunk boundary, done by one extra CTA
// of the direct grid (the other CTAs skip them): at most one per boundary b
// (chunk b starts at global index b * base), taken by the boundary that falls
// first inside it.
template <int DT, int WT>
__device__ __forceinline__ void straddle_pass(const RingParams &p) {
  constexpr int V = Vec<DT, WT>::V;
  for (int b = 1 + threadIdx.x; b < p.L; b += blockDim.x) {
    const unsigned long long gb = (unsigned long long)b * p.base;
    if (gb <= p.first || gb - p.first >= p.n_bulk || (gb - p.first) % V == 0) continue;
    const unsigned long long v = (gb - p.first) / V, g0 = p.first + v * V;
    if ((unsigned long long)(b - 1) * p.base > g0) continue;  // an earlier boundary lies inside this vector
    const int c0 = start_rank(p, g0), c_last = start_rank(p, g0 + V - 1);
    if (c0 != c_last) straddle_vec<DT, WT>(p, v, c0, c_last);
  }
}

// OCC: 256-thread CTAs per SM the registers are budgeted for (2: up to 128
// registers a thread, 3: up to 85).
// L2 prefetch of the inputs of the U vectors v0, v0 + T, ... (those below nvec).
template <int OP, int DT, int U>
__device__ __forceinline__ void prefetch_vectors(const RingParams &p, unsigned long long v0, unsigned long long T,
                                                 unsigned long long nvec) {
  constexpr int E = Fmt<DT>::bytes;
  constexpr int V = 16 / E;
#pragma unroll
  for (int k = 0; k < U; ++k) {
    const unsigned long long v = v0 + (unsigned long long)k * T;
    if (v >= nvec) break;
    if constexpr (OP == kOpAllGather) {
      const unsigned long long g0 = v * V;
      const int c = chunk_of(p, g0);
      if (c == chunk_of(p, g0 + V - 1)) prefetch_in<true, E>(p, c, (g0 - (unsigned long long)c * p.base) * E);
    } else {
      for (int r = 0; r < p.R; ++r) prefetch_in<false, E>(p, r, v * 16);
    }
  }
}

// CACHE: folds of two or more vectors a thread look their chunk up through
// the per-thread cache (false: the plain division, for AllReduce groups of
// three or more ranks, where the division measured faster).
template <int OP, int DT, int WT, int U, int OCC, bool CACHE = true>
__global__ void __launch_bounds__(kDirectThreads, OCC) rr_direct_kernel(const __grid_constant__ RingParams p) {
  using VT = Vec<DT, WT>;
  using W = typename VT::W;
  constexpr int V = VT::V;
  constexpr int E = Fmt<DT>::bytes;
  constexpr int NB = direct_batch_ranks(U);  // ranks per batch of loads
  const unsigned long long nvec = p.n_bulk / V;
  const unsigned long long T = (unsigned long long)(gridDim.x - p.straddle_cta) * blockDim.x;
  const unsigned long long first_v = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
  const bool main_cta = !(OP == kOpAllReduce && p.straddle_cta && blockIdx.x == gridDim.x - 1);
  if ((p.prefetch & kPrefetchHead) && main_cta) prefetch_vectors<OP, DT, U>(p, first_v, T, nvec);
  // The next kernel may be scheduled at once: a large grid fills the SMs'
  // registers or thread slots, so its CTAs take SMs only as this grid's leave.
  grid_dependency_wait();
  grid_dependents_launch();
  if constexpr (OP == kOpAllReduce) {
    if (!main_cta) {
      straddle_pass<DT, WT>(p);
      return;
    }
  }
  const bool naive = p.algo == kAlgoNaive;
  ChunkCache cc;
  for (unsigned long long v0 = first_v; v0 < nvec; v0 += T * U) {
    if (p.prefetch & kPrefetchAhead) prefetch_vectors<OP, DT, U>(p, v0 + T * U, T, nvec);
    if constexpr (OP == kOpAllGather) {
      // all U loads first, then the stores: U loads in flight per thread
      uint4 val[U];
      bool live[U];
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const unsigned long long v = v0 + (unsigned long long)k * T;
        live[k] = v < nvec;
        if (!live[k]) continue;
        const unsigned long long i0 = v * V, g0 = p.first + i0;
        const int c = cached_chunk(cc, p, g0);
        if (!p.chunks_on_grid && g0 + V - 1 >= cc.hi) {  // over a chunk boundary: element by element
          for (int e = 0; e < V; ++e) element_op<OP, DT, WT>(p, i0 + e);
          live[k] = false;
          continue;
        }
        val[k] = load_in<true, E>(p, c, (i0 - (unsigned long long)c * p.base) * E);
      }
#pragma unroll
      for (int k = 0; k < U; ++k) {
        if (!live[k]) continue;
        const unsigned long long boff = (v0 + (unsigned long long)k * T) * V * E;
        for (int r = 0; r < p.R; ++r) store_out<false, E>(p, r, boff, val[k]);
      }
    } else {  // ring / naive fold, AllReduce or ReduceScatter
      unsigned long long boff[U];
      int c[U];
      bool live[U];
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const unsigned long long v = v0 + (unsigned long long)k * T;
        live[k] = v < nvec;
        boff[k] = v * V * E;
        c[k] = 0;
        if (live[k] && !naive) {  // the naive order starts every element at rank 0
          const unsigned long long g0 = p.first + v * V;
          // one vector a thread (five or more ranks a group), and AllReduce
          // kernels built without the cache: the plain lookup, which measured
          // faster there than the cache, whose state costs registers
          constexpr bool cached = U > 1 && CACHE;
          c[k] = cached ? cached_chunk(cc, p, g0) : chunk_of(p, g0);
          if (!p.chunks_on_grid && (cached ? g0 + V - 1 >= cc.hi : c[k] != chunk_of(p, g0 + V - 1))) {
            if (!p.straddle_cta)
              for (int e = 0; e < V; ++e) element_op<OP, DT, WT>(p, v * V + e);
            live[k] = false;
          }
        }
      }
      const int L = p.L;
      W total[U];
      for (int g = 0; g < p.G; ++g) {
        W acc[U];
        for (int k0 = 0; k0 < L; k0 += NB) {
          uint4 x[U][NB];
#pragma unroll
          for (int k = 0; k < U; ++k)
#pragma unroll
            for (int j = 0; j < NB; ++j)
              if (live[k] && k0 + j < L) {
                int r = c[k] + k0 + j;
                r -= (r >= L) ? L : 0;
                x[k][j] = load_in<false, E>(p, g * L + r, boff[k]);
              }
#pragma unroll
          for (int k = 0; k < U; ++k)
#pragma unroll
            for (int j = 0; j < NB; ++j)
              if (live[k] && k0 + j < L) acc[k] = (k0 + j == 0) ? VT::in(x[k][j]) : VT::hop(acc[k], VT::in(x[k][j]));
        }
#pragma unroll
        for (int k = 0; k < U; ++k) total[k] = (g == 0) ? acc[k] : VT::hop(total[k], acc[k]);
      }
#pragma unroll
      for (int k = 0; k < U; ++k) {
        if (!live[k]) continue;
        const uint4 res = VT::out(total[k]);
        if constexpr (OP == kOpAllReduce) {
          for (int r = 0; r < p.R; ++r) store_out<false, E>(p, r, boff[k], res);
        } else {  // ReduceScatter: the vector lies in chunk c[k]
          const unsigned long long i0 = boff[k] / E;
          store_out<true, E>(p, c[k], (i0 - (unsigned long long)c[k] * p.base) * E, res);
        }
      }
    }
  }
  // the ragged end (under 16 bytes per rank)
  for (unsigned long long i = p.n_bulk + (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; i < p.count; i += T)
    element_op<OP, DT, WT>(p, i);
}

// --------------------------------------------------------------------------
// ReduceScatter / AllGather (and AllReduce, chunks on the grid) chunk by
// chunk.  Where the chunk boundaries are off the 16-byte grid, the chunk-local buffers (the ReduceScatter outputs,
// the AllGather inputs) are shifted against the rank vectors by (c * base)
// mod V elements, and each 16-byte vector aligned in the shifted buffer is
// built from two aligned blocks of the other side; on the grid the shift is
// zero and each vector is one block.
// --------------------------------------------------------------------------

// US: rows of output vectors a warp takes at once (ReduceScatter, and
// AllGather over at most four ranks) or vectors a thread takes at once
// (AllGather over more ranks); more rows keep more loads in flight.
template <int OP, int DT, int WT, int US>
__global__ void __launch_bounds__(kDirectThreads, shift_occupancy(US)) rr_shift_kernel(const __grid_constant__ RingParams p) {
  using VT = Vec<DT, WT>;
  using W = typename VT::W;
  constexpr int V = VT::V;
  constexpr int E = Fmt<DT>::bytes;
  const int L = p.L;
  const unsigned long long base = p.base, N = p.total;
  const unsigned long long T = (unsigned long long)gridDim.x * blockDim.x;
  const unsigned long long tid = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
  if constexpr (OP == kOpReduceScatter) {
    // Chunk by chunk (the shift is the chunk's), each warp takes US rows of
    // 31 consecutive output vectors.  In a row, lane t loads every rank's
    // aligned block under output vector t's start and folds them as they are,
    // in the ring order of the chunk (the fold is element-wise, and every
    // element of the chunk starts at rank c; the block's elements outside the
    // chunk are folded too and dropped); the folded block is also the upper
    // half lane t - 1 needs, so one shuffle and one funnel shift of the
    // result build each output vector, whatever R is.  Lane 31 only supplies
    // its block.  Every work item but a chunk's last lies wholly inside the
    // chunk and the rank vectors, so it loads and stores without a check;
    // the last items go first, a row to a warp.  A vector whose upper block
    // would pass the end of the rank vectors goes element by element, and so
    // do the elements past a chunk's last full vector.
    constexpr int NB = direct_batch_ranks(US);  // ranks per batch: 8 (US = 3: 9) loads in flight a lane
    constexpr unsigned long long VB = (unsigned long long)V * E;  // bytes of a vector (16)
    const unsigned lane = threadIdx.x & 31u;
    const unsigned long long warp = tid >> 5, n_warps = T >> 5;
    const unsigned long long len_last = N - (unsigned long long)(L - 1) * base;
    // work items: one per 31 * US output vectors of a chunk
    constexpr unsigned long long per_item = 31ull * US;
    const unsigned long long ipc = (base / V + per_item - 1) / per_item;      // items in chunks 0..L-2
    const unsigned long long ipl = (len_last / V + per_item - 1) / per_item;  // items in the last chunk
    // inner items (all but each chunk's last), numbered across the chunks so
    // that every warp's items spread over them
    const unsigned long long inc = ipc ? ipc - 1 : 0, inl = ipl ? ipl - 1 : 0;
    const unsigned long long n_inner = (unsigned long long)(L - 1) * inc + inl;
    // the blocks lane `lane` loads for item `item` of chunk c, into L2
    auto prefetch_item = [&](int c, unsigned long long item) {
      const unsigned long long g0 = (unsigned long long)c * base, a0 = g0 - g0 % V;
      const unsigned long long off = (a0 + (item * per_item + lane) * V) * E;
#pragma unroll
      for (int k = 0; k < US; ++k)
        for (int r = 0; r < L; ++r) prefetch_in<false, E>(p, r, off + 31ull * VB * k);
    };
    // the inner item n_warps on: across chunk ends one at a time (at most L - 1 steps)
    auto advance = [&](int &c, unsigned long long &item) {
      item += n_warps;
      while (c < L - 1 && item >= inc) {
        item -= inc;
        ++c;
      }
    };
    // work units, dealt to the warps in turn: first the rows of each chunk's
    // last item (L * US units), then the inner items; w0 is this warp's
    // first inner item
    const unsigned long long n_edge = (unsigned long long)L * US;
    const unsigned long long w0 =
        warp < n_edge ? warp + (n_edge - warp + n_warps - 1) / n_warps * n_warps - n_edge : warp - n_edge;
    int c = L - 1;
    unsigned long long item = 0;
    if (w0 < n_inner) {
      if (w0 < (unsigned long long)(L - 1) * inc) {
        c = (int)(w0 / inc);
        item = w0 - (unsigned long long)c * inc;
      } else {
        item = w0 - (unsigned long long)(L - 1) * inc;
      }
      if (p.prefetch & kPrefetchHead) prefetch_item(c, item);
    }
    grid_dependency_wait();
    grid_dependents_launch();
    // the rows of each chunk's last item, one to a warp
    for (unsigned long long e = warp; e < n_edge; e += n_warps) {  // warp-uniform
      const int ce = (int)(e / US), k = (int)(e % US);
      const unsigned long long len = ce < L - 1 ? base : len_last, nv = len / V, n_c = ce < L - 1 ? ipc : ipl;
      if (n_c == 0) continue;
      const unsigned long long g0 = (unsigned long long)ce * base;
      const int shift = (int)(g0 % V), sh = shift * E;
      const unsigned long long u = (n_c - 1) * per_item + 31ull * k + lane, ga = g0 - (unsigned long long)shift + u * V;
      const bool load = u <= nv && ga + V <= N;  // the block under vector u's start
      const bool act = lane < 31u && u < nv;
      const bool tail = act && sh != 0 && ga + 2 * V > N;  // no upper block to shift in
      W acc;
      for (int k0 = 0; k0 < L; k0 += NB) {
        uint4 blk[NB];
#pragma unroll
        for (int j = 0; j < NB; ++j)
          if (k0 + j < L) {
            int r = ce + k0 + j;
            r -= (r >= L) ? L : 0;
            blk[j] = load ? load_in<false, E>(p, r, ga * E) : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
        for (int j = 0; j < NB; ++j)
          if (k0 + j < L) {
            const W x = VT::in(blk[j]);
            acc = (k0 + j == 0) ? x : VT::hop(acc, x);
          }
      }
      const uint4 res = VT::out(acc);
      const uint4 up = make_uint4(__shfl_down_sync(0xffffffffu, res.x, 1), __shfl_down_sync(0xffffffffu, res.y, 1),
                                  __shfl_down_sync(0xffffffffu, res.z, 1), __shfl_down_sync(0xffffffffu, res.w, 1));
      if (tail) {
        for (int e2 = 0; e2 < V; ++e2) element_op<OP, DT, WT>(p, g0 + u * V + e2);
      } else if (act) {
        store_out<true, E>(p, ce, u * VB, sh ? funnel16(res, up, sh) : res);
      }
    }
    for (unsigned long long w = w0; w < n_inner; w += n_warps) {  // warp-uniform
      if (p.prefetch & kPrefetchAhead) {
        int c2 = c;
        unsigned long long item2 = item;
        advance(c2, item2);
        if (w + n_warps < n_inner) prefetch_item(c2, item2);
      }
      const unsigned long long g0 = (unsigned long long)c * base;
      const int sh = (int)(g0 % V) * E;  // bytes the chunk's vectors start into their aligned blocks
      // row 0's block of this lane; row k's sits 31 k vectors further on
      const unsigned long long u = item * per_item + lane, off = (g0 - g0 % V + u * V) * E;
      W acc[US];
      for (int k0 = 0; k0 < L; k0 += NB) {
        uint4 blk[US][NB];
#pragma unroll
        for (int k = 0; k < US; ++k)
#pragma unroll
          for (int j = 0; j < NB; ++j)
            if (k0 + j < L) {
              int r = c + k0 + j;
              r -= (r >= L) ? L : 0;
              blk[k][j] = load_in<false, E>(p, r, off + 31ull * VB * k);
            }
#pragma unroll
        for (int k = 0; k < US; ++k)
#pragma unroll
          for (int j = 0; j < NB; ++j)
            if (k0 + j < L) {
              const W x = VT::in(blk[k][j]);
              acc[k] = (k0 + j == 0) ? x : VT::hop(acc[k], x);
            }
      }
#pragma unroll
      for (int k = 0; k < US; ++k) {
        const uint4 res = VT::out(acc[k]);  // the folded block under output vector u + 31 k's start
        const uint4 up = make_uint4(__shfl_down_sync(0xffffffffu, res.x, 1), __shfl_down_sync(0xffffffffu, res.y, 1),
                                    __shfl_down_sync(0xffffffffu, res.z, 1), __shfl_down_sync(0xffffffffu, res.w, 1));
        if (lane < 31u) store_out<true, E>(p, c, (u + 31ull * k) * VB, sh ? funnel16(res, up, sh) : res);
      }
      advance(c, item);
    }
    for (unsigned long long t = tid; t < (unsigned long long)L * V; t += T) {
      const int c = (int)(t / V), e = (int)(t % V);
      const unsigned long long len = c < L - 1 ? base : len_last, full = len / V * V;
      if (full + e < len) element_op<OP, DT, WT>(p, (unsigned long long)c * base + full + e);
    }
  } else if constexpr (OP == kOpAllReduce) {
    // AllReduce over a flat ring of few ranks with every chunk boundary on the
    // 16-byte grid and whole rank vectors (no range): chunk by chunk in rows of
    // 32 vectors; lane t folds every rank's vector t of a row in the chunk's
    // ring order and stores the sum to every output.  As in the
    // ReduceScatter, every item but a chunk's last holds only whole vectors of
    // the chunk, so it loads and stores without a check; the last items go
    // first, a row to a warp; the elements past the last chunk's last whole
    // vector go one by one.
    constexpr int NB = direct_batch_ranks(US);
    constexpr unsigned long long VB = (unsigned long long)V * E;
    const unsigned lane = threadIdx.x & 31u;
    const unsigned long long warp = tid >> 5, n_warps = T >> 5;
    const unsigned long long len_last = N - (unsigned long long)(L - 1) * base;
    constexpr unsigned long long per_item = 32ull * US;
    const unsigned long long nvc = base / V, nvl = len_last / V;  // whole vectors of a chunk, of the last
    const unsigned long long ipc = (nvc + per_item - 1) / per_item, ipl = (nvl + per_item - 1) / per_item;
    const unsigned long long inc = ipc ? ipc - 1 : 0, inl = ipl ? ipl - 1 : 0;
    const unsigned long long n_inner = (unsigned long long)(L - 1) * inc + inl;
    const unsigned long long n_edge = (unsigned long long)L * US;
    auto advance = [&](int &c, unsigned long long &item) {
      item += n_warps;
      while (c < L - 1 && item >= inc) {
        item -= inc;
        ++c;
      }
    };
    auto prefetch_item = [&](int c, unsigned long long item) {
      const unsigned long long off = ((unsigned long long)c * base + (item * per_item + lane) * V) * E;
#pragma unroll
      for (int k = 0; k < US; ++k)
        for (int r = 0; r < L; ++r) prefetch_in<false, E>(p, r, off + 32ull * VB * k);
    };
    const unsigned long long w0 =
        warp < n_edge ? warp + (n_edge - warp + n_warps - 1) / n_warps * n_warps - n_edge : warp - n_edge;
    int c = L - 1;
    unsigned long long item = 0;
    if (w0 < n_inner) {
      if (w0 < (unsigned long long)(L - 1) * inc) {
        c = (int)(w0 / inc);
        item = w0 - (unsigned long long)c * inc;
      } else {
        item = w0 - (unsigned long long)(L - 1) * inc;
      }
      if (p.prefetch & kPrefetchHead) prefetch_item(c, item);
    }
    grid_dependency_wait();
    grid_dependents_launch();
    for (unsigned long long e = warp; e < n_edge; e += n_warps) {  // a chunk's last item, a row to a warp
      const int ce = (int)(e / US), k = (int)(e % US);
      const unsigned long long nv = ce < L - 1 ? nvc : nvl, n_c = ce < L - 1 ? ipc : ipl;
      if (n_c == 0) continue;
      const unsigned long long u = (n_c - 1) * per_item + 32ull * k + lane;
      if (u >= nv) continue;
      const unsigned long long off = ((unsigned long long)ce * base + u * V) * E;
      W acc;
      for (int k0 = 0; k0 < L; k0 += NB) {
        uint4 blk[NB];
#pragma unroll
        for (int j = 0; j < NB; ++j)
          if (k0 + j < L) {
            int r = ce + k0 + j;
            r -= (r >= L) ? L : 0;
            blk[j] = load_in<false, E>(p, r, off);
          }
#pragma unroll
        for (int j = 0; j < NB; ++j)
          if (k0 + j < L) {
            const W x = VT::in(blk[j]);
            acc = (k0 + j == 0) ? x : VT::hop(acc, x);
          }
      }
      const uint4 res = VT::out(acc);
      for (int r = 0; r < p.R; ++r) store_out<false, E>(p, r, off, res);
    }
    for (unsigned long long w = w0; w < n_inner; w += n_warps) {  // warp-uniform
      if (p.prefetch & kPrefetchAhead) {
        int c2 = c;
        unsigned long long item2 = item;
        advance(c2, item2);
        if (w + n_warps < n_inner) prefetch_item(c2, item2);
      }
      const unsigned long long off = ((unsigned long long)c * base + (item * per_item + lane) * V) * E;
      W acc[US];
      for (int k0 = 0; k0 < L; k0 += NB) {
        uint4 blk[US][NB];
#pragma unroll
        for (int j = 0; j < NB; ++j)
          if (k0 + j < L) {
            int r = c + k0 + j;
            r -= (r >= L) ? L : 0;
#pragma unroll
            for (int k = 0; k < US; ++k) blk[k][j] = load_in<false, E>(p, r, off + 32ull * VB * k);
          }
#pragma unroll
        for (int k = 0; k < US; ++k)
#pragma unroll
          for (int j = 0; j < NB; ++j)
            if (k0 + j < L) {
              const W x = VT::in(blk[k][j]);
              acc[k] = (k0 + j == 0) ? x : VT::hop(acc[k], x);
            }
      }
#pragma unroll
      for (int k = 0; k < US; ++k) {
        const uint4 res = VT::out(acc[k]);
        for (int r = 0; r < p.R; ++r) store_out<false, E>(p, r, off + 32ull * VB * k, res);
      }
      advance(c, item);
    }
    for (unsigned long long i = (unsigned long long)(L - 1) * base + nvl * V + tid; i < N; i += T)
      element_op<OP, DT, WT>(p, i);
  } else if (p.shift_rows) {
    // AllGather over up to four ranks (where the loads weigh most), and over
    // more from 12 MiB per rank (also with the chunks on the grid, unshifted,
    // from 12 MiB, two ranks from 64 MiB): rows of 32 output vectors aligned
    // to 32 vectors (512-byte store segments), clipped to one chunk; a warp's
    // work item is US consecutive rows of one chunk.  Lane t
    // loads the aligned source block under vector t's start, which is also
    // the upper block lane t - 1 needs (a shuffle), and lane 31 loads its
    // upper block itself; every row's loads are issued before any store.
    // Output vector v of chunk c (first vector wholly inside it: vf) starts
    // (v - vf) V + s elements into the chunk's buffer, s = vf V - c base.
    // With m = floor(len / V) for a chunk of len elements, every vector from
    // vf to vf + m - 2 lies wholly in the chunk with both its source blocks
    // inside the buffer, and the chunk has n = ceil((floor(m / 32) + 2) / US)
    // items: the items from the second to the fourth last hold only such
    // vectors (at most three items lie past vf + m - 2, one before vf), so
    // they load and store without a check, and each chunk's first item and
    // last three go first, a row to a warp, with the checks.  Vectors over a
    // chunk boundary (at most one per boundary, taken by the first boundary
    // inside it), vectors whose upper block would pass the end of the chunk's
    // buffer and the ragged end go element by element.
    const unsigned lane = threadIdx.x & 31u;
    const unsigned long long warp = tid >> 5, n_warps = T >> 5;
    const unsigned long long nvec = p.n_bulk / V;  // output vectors wholly before the ragged end
    const unsigned long long len_last = N - (unsigned long long)(L - 1) * base;
    const unsigned long long rpc = (base / V + 64) / 32, rpl = (len_last / V + 64) / 32;  // rows per chunk, at most
    const unsigned long long ipc = (rpc + US - 1) / US, ipl = (rpl + US - 1) / US;        // items per chunk
    const unsigned long long inc = ipc > 4 ? ipc - 4 : 0, inl = ipl > 4 ? ipl - 4 : 0;    // inner items
    const unsigned long long epc = (ipc - inc) * US, epl = (ipl - inl) * US;              // checked rows
    const unsigned long long n_edge = (unsigned long long)(L - 1) * epc + epl;
    const unsigned long long n_inner = (unsigned long long)(L - 1) * inc + inl;
    // chunk c: its buffer's length, its first and (one past) last output
    // vectors wholly inside it, the shift
    struct Chunk {
      unsigned long long len, vf, ve;
      int sh;  // bytes a vector's source starts into its aligned block
    };
    auto chunk = [&](int c) {
      Chunk k;
      const unsigned long long cb = (unsigned long long)c * base;
      k.len = c < L - 1 ? base : len_last;
      k.vf = (cb + V - 1) / V;
      k.ve = (cb + k.len) / V < nvec ? (cb + k.len) / V : nvec;
      k.sh = (int)(k.vf * V - cb) * E;
      return k;
    };
    // the inner item n_warps on (i counts a chunk's inner items): across
    // chunk ends one at a time
    auto advance = [&](int &c, unsigned long long &i) {
      i += n_warps;
      while (c < L - 1 && i >= inc) {
        i -= inc;
        ++c;
      }
    };
    // the source blocks lane `lane` loads for inner item i of chunk c, into L2
    auto prefetch_item = [&](int c, unsigned long long i) {
      const Chunk k = chunk(c);
#pragma unroll
      for (int r = 0; r < US; ++r) {
        const unsigned long long v = (k.vf / 32 + (1 + i) * US + r) * 32 + lane;
        prefetch_in<true, E>(p, c, (v - k.vf) * V * E);
      }
    };
    // work units, dealt to the warps in turn: first the checked rows, then
    // the inner items; w0 is this warp's first inner item
    const unsigned long long w0 =
        warp < n_edge ? warp + (n_edge - warp + n_warps - 1) / n_warps * n_warps - n_edge : warp - n_edge;
    int c = L - 1;
    unsigned long long item = 0;
    if (w0 < n_inner) {
      if (w0 < (unsigned long long)(L - 1) * inc) {
        c = (int)(w0 / inc);
        item = w0 - (unsigned long long)c * inc;
      } else {
        item = w0 - (unsigned long long)(L - 1) * inc;
      }
      if (p.prefetch & kPrefetchHead) prefetch_item(c, item);
    }
    grid_dependency_wait();
    grid_dependents_launch();
    for (unsigned long long e = warp; e < n_edge; e += n_warps) {  // warp-uniform
      // checked row e: chunk ce's first item, then its last ones
      const int ce = e < (unsigned long long)(L - 1) * epc ? (int)(e / epc) : L - 1;
      const unsigned long long u = e - (unsigned long long)ce * epc, j = u / US;
      const unsigned long long in_c = ce < L - 1 ? inc : inl;
      const unsigned long long it = (j == 0 || in_c == 0) ? j : j + in_c;  // the item
      const Chunk k = chunk(ce);
      const unsigned long long v = (k.vf / 32 + it * US + u % US) * 32 + lane;
      const bool act = v >= k.vf && v < k.ve;
      const unsigned long long oa = v >= k.vf ? (v - k.vf) * V : 0;  // the aligned source block under v's start
      const bool load = v >= k.vf && v <= k.ve && oa + V <= k.len;
      const bool tail = act && k.sh != 0 && oa + 2 * V > k.len;
      const uint4 blk = load ? load_in<true, E>(p, ce, oa * E) : make_uint4(0u, 0u, 0u, 0u);
      uint4 nxt = (lane == 31u && act && k.sh != 0 && !tail) ? load_in<true, E>(p, ce, (oa + V) * E)
                                                             : make_uint4(0u, 0u, 0u, 0u);
      const uint4 up = make_uint4(__shfl_down_sync(0xffffffffu, blk.x, 1), __shfl_down_sync(0xffffffffu, blk.y, 1),
                                  __shfl_down_sync(0xffffffffu, blk.z, 1), __shfl_down_sync(0xffffffffu, blk.w, 1));
      if (lane != 31u) nxt = up;
      if (tail) {
        for (int e2 = 0; e2 < V; ++e2) element_op<OP, DT, WT>(p, v * V + e2);
      } else if (act) {
        const uint4 x = k.sh ? funnel16(blk, nxt, k.sh) : blk;
        for (int r = 0; r < p.R; ++r) store_out<false, E>(p, r, v * V * E, x);
      }
    }
    for (unsigned long long w = w0; w < n_inner; w += n_warps) {  // warp-uniform
      if (p.prefetch & kPrefetchAhead) {
        int c2 = c;
        unsigned long long item2 = item;
        advance(c2, item2);
        if (w + n_warps < n_inner) prefetch_item(c2, item2);
      }
      const Chunk k = chunk(c);
      const unsigned long long v0 = (k.vf / 32 + (1 + item) * US) * 32 + lane;  // row 0's vector
      const unsigned long long oa0 = (v0 - k.vf) * V;  // its source block, elements into the buffer
      uint4 blk[US], nxt[US];
#pragma unroll
      for (int r = 0; r < US; ++r) {
        blk[r] = load_in<true, E>(p, c, (oa0 + 32ull * V * r) * E);
        nxt[r] = (lane == 31u && k.sh != 0) ? load_in<true, E>(p, c, (oa0 + 32ull * V * r + V) * E)
                                            : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int r = 0; r < US; ++r) {
        const uint4 up = make_uint4(__shfl_down_sync(0xffffffffu, blk[r].x, 1), __shfl_down_sync(0xffffffffu, blk[r].y, 1),
                                    __shfl_down_sync(0xffffffffu, blk[r].z, 1), __shfl_down_sync(0xffffffffu, blk[r].w, 1));
        if (lane != 31u) nxt[r] = up;
      }
#pragma unroll
      for (int r = 0; r < US; ++r) {
        const uint4 x = k.sh ? funnel16(blk[r], nxt[r], k.sh) : blk[r];
        for (int q = 0; q < p.R; ++q) store_out<false, E>(p, q, (v0 + 32ull * r) * V * E, x);
      }
      advance(c, item);
    }
    for (unsigned long long b = 1 + tid; b < (unsigned long long)L; b += T) {  // vectors over a boundary
      const unsigned long long gb = b * base, vb = gb / V;
      if (gb % V == 0 || vb >= nvec) continue;
      if ((b - 1) * base > vb * V) continue;  // an earlier boundary lies inside this vector
      for (int e = 0; e < V; ++e) element_op<OP, DT, WT>(p, vb * V + e);
    }
    for (unsigned long long i = p.n_bulk + tid; i < p.count; i += T) element_op<OP, DT, WT>(p, i);
  } else {
    // AllGather over five or more ranks below 12 MiB per rank: each thread
    // takes US output vectors a grid-stride apart and builds each from the
    // two aligned blocks of its chunk's input under it (the second served by
    // L1); all loads before the stores
    const unsigned long long nvec = p.n_bulk / V;
    // L2 prefetch of the lower source blocks of vectors v0, v0 + T, ...
    auto prefetch_vecs = [&](unsigned long long v0) {
#pragma unroll
      for (int k = 0; k < US; ++k) {
        const unsigned long long v = v0 + (unsigned long long)k * T;
        if (v >= nvec) break;
        const unsigned long long gs = v * V;
        const int c = chunk_of(p, gs);
        const unsigned long long o = gs - (unsigned long long)c * base, oa = o / V * V;
        if (oa + V <= chunk_end(c, base, L, N) - (unsigned long long)c * base) prefetch_in<true, E>(p, c, oa * E);
      }
    };
    if (p.prefetch & kPrefetchHead) prefetch_vecs(tid);
    grid_dependency_wait();
    grid_dependents_launch();
    for (unsigned long long v0 = tid; v0 < nvec; v0 += T * US) {
      if (p.prefetch & kPrefetchAhead) prefetch_vecs(v0 + T * US);
      uint4 lo[US], hi[US];
      int sh[US];
      bool live[US];
#pragma unroll
      for (int k = 0; k < US; ++k) {
        const unsigned long long v = v0 + (unsigned long long)k * T;
        live[k] = v < nvec;
        if (!live[k]) continue;
        const unsigned long long gs = v * V;
        const int c = chunk_of(p, gs);
        const unsigned long long o = gs - (unsigned long long)c * base;  // offset in chunk c's buffer
        const unsigned long long oa = o / V * V, len = chunk_end(c, base, L, N) - (unsigned long long)c * base;
        sh[k] = (int)(o - oa) * E;
        if (c != chunk_of(p, gs + V - 1) || (sh[k] != 0 && oa + 2 * V > len)) {
          for (int e = 0; e < V; ++e) element_op<OP, DT, WT>(p, gs + e);
          live[k] = false;
          continue;
        }
        lo[k] = load_in_l1<true, E>(p, c, oa * E);
        hi[k] = sh[k] ? load_in_l1<true, E>(p, c, oa * E + 16) : lo[k];
      }
#pragma unroll
      for (int k = 0; k < US; ++k) {
        if (!live[k]) continue;
        const uint4 x = sh[k] ? funnel16(lo[k], hi[k], sh[k]) : lo[k];
        const unsigned long long gs = (v0 + (unsigned long long)k * T) * V;
        for (int r = 0; r < p.R; ++r) store_out<false, E>(p, r, gs * E, x);
      }
    }
    for (unsigned long long i = p.n_bulk + tid; i < p.count; i += T) element_op<OP, DT, WT>(p, i);
  }
}

// --------------------------------------------------------------------------
// host side: one launch of (OP, DT, WT)
// --------------------------------------------------------------------------

// One launch of kernel k on the plan's grid, with programmatic stream
// serialisation when the plan asks for it.
inline cudaError_t launch_kernel(void (*k)(RingParams), const Launch &l, size_t smem, cudaStream_t s,
                                 const RingParams &p) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t c = {};
  c.gridDim = dim3((unsigned)l.grid);
  c.blockDim = dim3((unsigned)l.threads);
  c.dynamicSmemBytes = smem;
  c.stream = s;
  c.attrs = attr;
  c.numAttrs = l.early_launch ? 1 : 0;
  return cudaLaunchKernelEx(&c, k, p);
}

// The direct kernel of the plan's (U, OCC); the planner picks only variants
// for which direct_variant_exists holds.
template <int OP, int DT, int WT>
cudaError_t launch_direct(const RingParams &p, const Launch &l, cudaStream_t s) {
  constexpr bool wide = DT != kF32 && WT == kF32;
  const int U = p.direct_u, occ = l.direct_occ;
  if constexpr (OP == kOpAllGather) {
    switch (U) {
      case 1: return launch_kernel(rr_direct_kernel<OP, DT, WT, 1, 2>, l, 0, s, p);
      case 2: return launch_kernel(rr_direct_kernel<OP, DT, WT, 2, 2>, l, 0, s, p);
      case 4: return launch_kernel(rr_direct_kernel<OP, DT, WT, 4, 2>, l, 0, s, p);
    }
  } else if constexpr (wide) {
    if (U == 1) return launch_kernel(rr_direct_kernel<OP, DT, WT, 1, 2>, l, 0, s, p);
    if (U == 2) return launch_kernel(rr_direct_kernel<OP, DT, WT, 2, 2>, l, 0, s, p);
  } else {
    // AllReduce over groups of three or more ranks at two vectors a thread:
    // the kernels without the lookup cache (same-box A/B at 256 MiB per rank,
    // binary16: R = 3 254 -> 242 us, R = 4 326 -> 321 us)
    if constexpr (OP == kOpAllReduce) {
      if (U == 2 && p.L >= 3 && p.algo == kAlgoRing) {
        if (occ == 3) return launch_kernel(rr_direct_kernel<OP, DT, WT, 2, 3, false>, l, 0, s, p);
        if (occ == 2) return launch_kernel(rr_direct_kernel<OP, DT, WT, 2, 2, false>, l, 0, s, p);
      }
    }
    switch (U * 8 + occ) {
      case 1 * 8 + 2: return launch_kernel(rr_direct_kernel<OP, DT, WT, 1, 2>, l, 0, s, p);
      case 1 * 8 + 3: return launch_kernel(rr_direct_kernel<OP, DT, WT, 1, 3>, l, 0, s, p);
      case 2 * 8 + 2: return launch_kernel(rr_direct_kernel<OP, DT, WT, 2, 2>, l, 0, s, p);
      case 2 * 8 + 3: return launch_kernel(rr_direct_kernel<OP, DT, WT, 2, 3>, l, 0, s, p);
      case 3 * 8 + 2: return launch_kernel(rr_direct_kernel<OP, DT, WT, 3, 2>, l, 0, s, p);
      case 4 * 8 + 2: return launch_kernel(rr_direct_kernel<OP, DT, WT, 4, 2>, l, 0, s, p);
    }
  }
  return cudaErrorInvalidConfiguration;  // not a variant the planner picks
}

// The shifted kernel of the plan's rows per work item (shift_variant_exists).
template <int OP, int DT, int WT>
cudaError_t launch_shift(const RingParams &p, const Launch &l, cudaStream_t s) {
  constexpr bool wide = DT != kF32 && WT == kF32;
  if constexpr (OP == kOpAllReduce) {  // two or four rows, accumulators of the fold's own type
    if constexpr (!wide) {
      if (p.direct_u == 2) return launch_kernel(rr_shift_kernel<OP, DT, WT, 2>, l, 0, s, p);
      if (p.direct_u == 4) return launch_kernel(rr_shift_kernel<OP, DT, WT, 4>, l, 0, s, p);
    }
  } else {
    switch (p.direct_u) {
      case 1: return launch_kernel(rr_shift_kernel<OP, DT, WT, 1>, l, 0, s, p);
      case 2: return launch_kernel(rr_shift_kernel<OP, DT, WT, 2>, l, 0, s, p);
      case 3:
        if constexpr (OP == kOpReduceScatter && !wide)
          return launch_kernel(rr_shift_kernel<OP, DT, WT, 3>, l, 0, s, p);
        break;
      case 4:
        if constexpr (!wide) return launch_kernel(rr_shift_kernel<OP, DT, WT, 4>, l, 0, s, p);
        break;
    }
  }
  return cudaErrorInvalidConfiguration;  // not a variant the planner picks
}

template <int OP, int DT, int WT, bool HD>
cudaError_t launch_variant(const RingParams &p, const Launch &l, cudaStream_t s) {
  if (l.path == RR_PATH_BULK) {
    // Largest dynamic shared memory opted in, per device.  The attribute is
    // only ever raised, and the raise and its record happen under one lock, so
    // a thread that finds a size recorded knows the attribute is at least that.
    static std::mutex smem_mu;
    static int smem_set[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (l.smem > 48 * 1024) {
      std::lock_guard<std::mutex> lock(smem_mu);
      if (dev >= 64 || smem_set[dev] < (int)l.smem) {
        e = cudaFuncSetAttribute(rr_bulk_kernel<OP, DT, WT, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)l.smem);
        if (e != cudaSuccess) return e;
        if (dev < 64) smem_set[dev] = (int)l.smem;
      }
    }
    return launch_kernel(rr_bulk_kernel<OP, DT, WT, HD>, l, l.smem, s, p);
  } else if (l.path == RR_PATH_DIRECT) {
    if constexpr (HD) {
      return launch_hd_direct(DT, WT, p, l, s);
    } else {
      if (p.shifted) return launch_shift<OP, DT, WT>(p, l, s);
      return launch_direct<OP, DT, WT>(p, l, s);
    }
  }
  return launch_kernel(rr_simple_kernel<OP, DT, WT, HD>, l, 0, s, p);
}

template <int OP, int DT, int WT>
cudaError_t launch_one(const RingParams &p, const Launch &l, cudaStream_t s) {
  if constexpr (OP == kOpAllReduce)
    if (p.algo == kAlgoHalvingDoubling) return launch_variant<OP, DT, WT, true>(p, l, s);
  return launch_variant<OP, DT, WT, false>(p, l, s);
}

}  // namespace rr
