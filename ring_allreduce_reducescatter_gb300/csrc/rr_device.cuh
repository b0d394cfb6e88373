// rr_device.cuh -- device building blocks of libringred (sm_103a).
//
//  * element formats and one ring hop: the binary32 sum of two wire values
//    rounded once to the wire format (page hwcomputing.csdn.net/6a0dc11a...,
//    section "大模型训练中的通信优化": gradients travel in FP16).  binary16 and
//    bfloat16 hops use the hardware's correctly rounded 16-bit adds: because
//    binary32 carries at least 2p+2 significand bits for p = 11 and p = 8, one
//    correctly rounded 16-bit add equals the binary32 sum rounded once.
//  * 16-byte vector forms of ingress (storage -> wire), hop and egress, for
//    every supported (storage, wire) pair, including 16-bit storage summed in
//    binary32 (the same section's FP16 / FP32 mixed precision).
//  * chunk lookup of the partition of N elements into L chunks (page
//    ai6s.net/6a157e65..., section "自定义通信模式": floor(N/L) per chunk, the
//    last chunk takes the rest).
//  * PTX wrappers: mbarrier, bulk asynchronous copies global <-> shared, L2
//    eviction policy, and a bounded mbarrier wait.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <string.h>

#include "rr_params.h"

namespace rr {

// --------------------------------------------------------------------------
// formats
// --------------------------------------------------------------------------

template <int T>
struct Fmt;
template <>
struct Fmt<kF32> {
  using type = float;
  static constexpr int bytes = 4;
};
template <>
struct Fmt<kF16> {
  using type = __half;
  static constexpr int bytes = 2;
};
template <>
struct Fmt<kBF16> {
  using type = __nv_bfloat16;
  static constexpr int bytes = 2;
};

__device__ __forceinline__ float hop(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ __half hop(__half a, __half b) { return __hadd(a, b); }
__device__ __forceinline__ __nv_bfloat16 hop(__nv_bfloat16 a, __nv_bfloat16 b) { return __hadd(a, b); }

// Scalar ingress (storage -> wire) and egress (wire -> storage).
template <int DT, int WT>
struct Scalar {
  using S = typename Fmt<DT>::type;
  using W = typename Fmt<WT>::type;
  static __device__ __forceinline__ W in(S x);
  static __device__ __forceinline__ S out(W w);
};
template <>
__device__ __forceinline__ float Scalar<kF32, kF32>::in(float x) { return x; }
template <>
__device__ __forceinline__ float Scalar<kF32, kF32>::out(float w) { return w; }
template <>
__device__ __forceinline__ __half Scalar<kF16, kF16>::in(__half x) { return x; }
template <>
__device__ __forceinline__ __half Scalar<kF16, kF16>::out(__half w) { return w; }
template <>
__device__ __forceinline__ __nv_bfloat16 Scalar<kBF16, kBF16>::in(__nv_bfloat16 x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 Scalar<kBF16, kBF16>::out(__nv_bfloat16 w) { return w; }
template <>
__device__ __forceinline__ __nv_bfloat16 Scalar<kF32, kBF16>::in(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ float Scalar<kF32, kBF16>::out(__nv_bfloat16 w) { return __bfloat162float(w); }
template <>
__device__ __forceinline__ __half Scalar<kF32, kF16>::in(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ float Scalar<kF32, kF16>::out(__half w) { return __half2float(w); }
// 16-bit storage accumulated in binary32: exact widening, one rounding at the end
template <>
__device__ __forceinline__ float Scalar<kF16, kF32>::in(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ __half Scalar<kF16, kF32>::out(float w) { return __float2half_rn(w); }
template <>
__device__ __forceinline__ float Scalar<kBF16, kF32>::in(__nv_bfloat16 x) { return __bfloat162float(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 Scalar<kBF16, kF32>::out(float w) { return __float2bfloat16_rn(w); }

// --------------------------------------------------------------------------
// 16-byte vectors: V storage elements, held in the wire format as W
// --------------------------------------------------------------------------

__device__ __forceinline__ __half2 as_h2(uint32_t u) {
  __half2 h;
  memcpy(&h, &u, 4);
  return h;
}
__device__ __forceinline__ __nv_bfloat162 as_b2(uint32_t u) {
  __nv_bfloat162 h;
  memcpy(&h, &u, 4);
  return h;
}
template <class T2>
__device__ __forceinline__ uint32_t as_u32(T2 h) {
  uint32_t u;
  memcpy(&u, &h, 4);
  return u;
}

template <int DT, int WT>
struct Vec;

template <>
struct Vec<kF32, kF32> {
  static constexpr int V = 4;
  using W = float4;
  static __device__ __forceinline__ W in(uint4 r) {
    return make_float4(__uint_as_float(r.x), __uint_as_float(r.y), __uint_as_float(r.z), __uint_as_float(r.w));
  }
  static __device__ __forceinline__ W hop(W a, W b) {
    return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
  }
  static __device__ __forceinline__ uint4 out(W w) {
    return make_uint4(__float_as_uint(w.x), __float_as_uint(w.y), __float_as_uint(w.z), __float_as_uint(w.w));
  }
};

template <>
struct Vec<kF16, kF16> {
  static constexpr int V = 8;
  using W = uint4;  // four __half2
  static __device__ __forceinline__ W in(uint4 r) { return r; }
  static __device__ __forceinline__ W hop(W a, W b) {
    return make_uint4(as_u32(__hadd2(as_h2(a.x), as_h2(b.x))), as_u32(__hadd2(as_h2(a.y), as_h2(b.y))),
                      as_u32(__hadd2(as_h2(a.z), as_h2(b.z))), as_u32(__hadd2(as_h2(a.w), as_h2(b.w))));
  }
  static __device__ __forceinline__ uint4 out(W w) { return w; }
};

template <>
struct Vec<kBF16, kBF16> {
  static constexpr int V = 8;
  using W = uint4;  // four __nv_bfloat162
  static __device__ __forceinline__ W in(uint4 r) { return r; }
  static __device__ __forceinline__ W hop(W a, W b) {
    return make_uint4(as_u32(__hadd2(as_b2(a.x), as_b2(b.x))), as_u32(__hadd2(as_b2(a.y), as_b2(b.y))),
                      as_u32(__hadd2(as_b2(a.z), as_b2(b.z))), as_u32(__hadd2(as_b2(a.w), as_b2(b.w))));
  }
  static __device__ __forceinline__ uint4 out(W w) { return w; }
};

template <>
struct Vec<kF32, kBF16> {
  static constexpr int V = 4;
  using W = uint2;  // two __nv_bfloat162
  static __device__ __forceinline__ W in(uint4 r) {
    return make_uint2(as_u32(__floats2bfloat162_rn(__uint_as_float(r.x), __uint_as_float(r.y))),
                      as_u32(__floats2bfloat162_rn(__uint_as_float(r.z), __uint_as_float(r.w))));
  }
  static __device__ __forceinline__ W hop(W a, W b) {
    return make_uint2(as_u32(__hadd2(as_b2(a.x), as_b2(b.x))), as_u32(__hadd2(as_b2(a.y), as_b2(b.y))));
  }
  static __device__ __forceinline__ uint4 out(W w) {
    float2 lo = __bfloat1622float2(as_b2(w.x)), hi = __bfloat1622float2(as_b2(w.y));
    return make_uint4(__float_as_uint(lo.x), __float_as_uint(lo.y), __float_as_uint(hi.x), __float_as_uint(hi.y));
  }
};

template <>
struct Vec<kF32, kF16> {
  static constexpr int V = 4;
  using W = uint2;  // two __half2
  static __device__ __forceinline__ W in(uint4 r) {
    return make_uint2(as_u32(__floats2half2_rn(__uint_as_float(r.x), __uint_as_float(r.y))),
                      as_u32(__floats2half2_rn(__uint_as_float(r.z), __uint_as_float(r.w))));
  }
  static __device__ __forceinline__ W hop(W a, W b) {
    return make_uint2(as_u32(__hadd2(as_h2(a.x), as_h2(b.x))), as_u32(__hadd2(as_h2(a.y), as_h2(b.y))));
  }
  static __device__ __forceinline__ uint4 out(W w) {
    float2 lo = __half22float2(as_h2(w.x)), hi = __half22float2(as_h2(w.y));
    return make_uint4(__float_as_uint(lo.x), __float_as_uint(lo.y), __float_as_uint(hi.x), __float_as_uint(hi.y));
  }
};

// Eight binary32 lanes: 16 bytes of 16-bit storage accumulated in binary32.
struct F8 {
  float4 lo, hi;
};

__device__ __forceinline__ F8 add_f8(const F8 &a, const F8 &b) {
  F8 r;
  r.lo = make_float4(__fadd_rn(a.lo.x, b.lo.x), __fadd_rn(a.lo.y, b.lo.y), __fadd_rn(a.lo.z, b.lo.z),
                     __fadd_rn(a.lo.w, b.lo.w));
  r.hi = make_float4(__fadd_rn(a.hi.x, b.hi.x), __fadd_rn(a.hi.y, b.hi.y), __fadd_rn(a.hi.z, b.hi.z),
                     __fadd_rn(a.hi.w, b.hi.w));
  return r;
}

template <>
struct Vec<kF16, kF32> {
  static constexpr int V = 8;
  using W = F8;
  static __device__ __forceinline__ W in(uint4 r) {
    float2 a = __half22float2(as_h2(r.x)), b = __half22float2(as_h2(r.y)), c = __half22float2(as_h2(r.z)),
           d = __half22float2(as_h2(r.w));
    return F8{make_float4(a.x, a.y, b.x, b.y), make_float4(c.x, c.y, d.x, d.y)};
  }
  static __device__ __forceinline__ W hop(W a, W b) { return add_f8(a, b); }
  static __device__ __forceinline__ uint4 out(W w) {
    return make_uint4(as_u32(__floats2half2_rn(w.lo.x, w.lo.y)), as_u32(__floats2half2_rn(w.lo.z, w.lo.w)),
                      as_u32(__floats2half2_rn(w.hi.x, w.hi.y)), as_u32(__floats2half2_rn(w.hi.z, w.hi.w)));
  }
};

template <>
struct Vec<kBF16, kF32> {
  static constexpr int V = 8;
  using W = F8;
  static __device__ __forceinline__ W in(uint4 r) {
    float2 a = __bfloat1622float2(as_b2(r.x)), b = __bfloat1622float2(as_b2(r.y)),
           c = __bfloat1622float2(as_b2(r.z)), d = __bfloat1622float2(as_b2(r.w));
    return F8{make_float4(a.x, a.y, b.x, b.y), make_float4(c.x, c.y, d.x, d.y)};
  }
  static __device__ __forceinline__ W hop(W a, W b) { return add_f8(a, b); }
  static __device__ __forceinline__ uint4 out(W w) {
    return make_uint4(as_u32(__floats2bfloat162_rn(w.lo.x, w.lo.y)), as_u32(__floats2bfloat162_rn(w.lo.z, w.lo.w)),
                      as_u32(__floats2bfloat162_rn(w.hi.x, w.hi.y)), as_u32(__floats2bfloat162_rn(w.hi.z, w.hi.w)));
  }
};

// --------------------------------------------------------------------------
// chunk table of (N, L): chunk c covers [c*base, c*base + len_c)
// --------------------------------------------------------------------------

// The chunk holding element i (p.base = floor(N / L)).
__device__ __forceinline__ int chunk_of(const RingParams &p, unsigned long long i) {
  if (p.base == 0) return p.L - 1;  // N < L: chunks 0..L-2 are empty
  const unsigned long long c = i / p.base;
  return c >= (unsigned long long)(p.L - 1) ? p.L - 1 : (int)c;
}

__device__ __forceinline__ unsigned long long chunk_end(int c, unsigned long long base, int L,
                                                        unsigned long long N) {
  return c == L - 1 ? N : (unsigned long long)(c + 1) * base;
}

// --------------------------------------------------------------------------
// 16-byte global accesses of the direct path: loads through the read-only
// path without an L1 allocation (every byte is read once), stores marked as
// streaming.  A thread only ever rereads what it wrote itself.
// --------------------------------------------------------------------------

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 16-byte load that allocates in L1: the shifted ReduceScatter / AllGather
// read each aligned block twice (as one thread's upper and the next thread's
// lower half).
__device__ __forceinline__ uint4 ldg_l1(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// The 16 bytes that start sh bytes into the 32 bytes lo:hi (0 <= sh < 16).
__device__ __forceinline__ uint4 funnel16(uint4 lo, uint4 hi, int sh) {
  const unsigned b = (unsigned)(sh & 3) * 8u;
  uint32_t a0, a1, a2, a3, a4;
  switch (sh >> 2) {
    case 0:
      a0 = lo.x, a1 = lo.y, a2 = lo.z, a3 = lo.w, a4 = hi.x;
      break;
    case 1:
      a0 = lo.y, a1 = lo.z, a2 = lo.w, a3 = hi.x, a4 = hi.y;
      break;
    case 2:
      a0 = lo.z, a1 = lo.w, a2 = hi.x, a3 = hi.y, a4 = hi.z;
      break;
    default:
      a0 = lo.w, a1 = hi.x, a2 = hi.y, a3 = hi.z, a4 = hi.w;
      break;
  }
  return make_uint4(__funnelshift_r(a0, a1, b), __funnelshift_r(a1, a2, b), __funnelshift_r(a2, a3, b),
                    __funnelshift_r(a3, a4, b));
}

// Brings the line holding p into L2 (a hint: no data reaches the SM).
__device__ __forceinline__ void prefetch_l2(const void *p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

__device__ __forceinline__ void stg_stream(void *p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may start while the kernel before it on the stream still
// runs.  grid_dependency_wait() blocks until that kernel has completed and its
// writes are visible (at once for a kernel launched in plain stream order); it
// comes first in every kernel, before any global memory access.
// grid_dependents_launch() lets the next kernel on the stream be scheduled
// once every CTA of this grid has executed it or exited.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// --------------------------------------------------------------------------
// PTX: mbarrier, bulk asynchronous copies, L2 policy, timer
// --------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes the barrier initialisation visible to the async proxy (bulk copies).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Counts `bytes` of the barrier's expected transaction as arrived without a
// copy (the debug build's checks retire the bytes of a copy they skipped).
__device__ __forceinline__ void mbar_complete_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits until the phase of `bar` with this parity has completed.  Gives up
// after limit_ns of wall time (%globaltimer) or 2^26 polls, whichever comes
// first, and returns false then.  Every poll is a try_wait, which suspends
// for a bounded, hardware-defined time, so the loop always ends.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 0; it < (1u << 26); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 15u && global_ns() - t0 > limit_ns) return false;
  }
  return false;
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk copy global -> shared, completion counted on `bar` (bytes: multiple of
// 16; both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gmem_src, uint32_t bytes, uint64_t *bar,
                                          uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

// Bulk copy shared -> global in the current bulk group.
__device__ __forceinline__ void bulk_store(void *gmem_dst, const void *smem_src, uint32_t bytes, uint64_t pol) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(gmem_dst),
               "r"(smem_addr(smem_src)), "r"(bytes), "l"(pol)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until at most N bulk groups still read their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// bulk_wait_read<N> for a runtime N in 0..8.
__device__ __forceinline__ void bulk_wait_read_upto(int n) {
  switch (n) {
    case 0: bulk_wait_read<0>(); break;
    case 1: bulk_wait_read<1>(); break;
    case 2: bulk_wait_read<2>(); break;
    case 3: bulk_wait_read<3>(); break;
    case 4: bulk_wait_read<4>(); break;
    case 5: bulk_wait_read<5>(); break;
    case 6: bulk_wait_read<6>(); break;
    case 7: bulk_wait_read<7>(); break;
    default: bulk_wait_read<8>(); break;
  }
}

// Waits until every bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) reads of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace rr
