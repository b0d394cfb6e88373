// rr_api.cu -- the C ABI of libringred (include/ringred.h): argument
// validation, the chunk table, launch planning and dispatch.
//
// Validation runs entirely on the host and before any CUDA call, so every
// argument error returns without touching the device.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "ringred.h"
#include "rr_params.h"

namespace {

// Debug builds: bytes the device-side bounds checks take off every buffer's
// extent (ring_debug_set_margin); 0 checks the true extents.
std::atomic<unsigned long long> g_debug_margin{0};

// Sticky device status word (bit rr::kStatusWaitTimeout).  Kernels get its
// device address, taken with cudaGetSymbolAddress for each device.
__device__ unsigned int g_rr_status_word;

struct DeviceInfo {
  int sms = 0;
  int smem_per_sm = 0;
  int smem_optin = 0;
  unsigned int *status = nullptr;
  bool valid = false;
};

constexpr int kMaxDevices = 64;

// The CUDA runtime error behind the calling thread's last RR_ERR_CUDA.
thread_local int g_last_cuda_error = 0;
bool cuda_ok(cudaError_t e) {
  if (e == cudaSuccess) return true;
  g_last_cuda_error = (int)e;
  return false;
}

DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mu;

rr_status current_device(DeviceInfo *out) {
  int dev = 0;
  if (!cuda_ok(cudaGetDevice(&dev)) || dev < 0 || dev >= kMaxDevices) return RR_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_devices_mu);
  DeviceInfo &d = g_devices[dev];
  if (!d.valid) {
    void *addr = nullptr;
    if (!cuda_ok(cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) ||
        !cuda_ok(cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) ||
        !cuda_ok(cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) ||
        !cuda_ok(cudaGetSymbolAddress(&addr, g_rr_status_word)))
      return RR_ERR_CUDA;
    d.status = static_cast<unsigned int *>(addr);
    d.valid = true;
  }
  *out = d;
  return RR_OK;
}

constexpr int kMaxStages = 16;  // pipeline depth limit of the bulk path
// Programmatic dependent launch by default: a kernel's launch overlaps the
// previous kernel on the stream; it waits for that kernel before any access.
constexpr bool kEarlyLaunchDefault = true;

size_t elem_bytes(int t) { return t == RR_FP32 ? 4 : 2; }
bool valid_type(int t) { return t == RR_FP32 || t == RR_FP16 || t == RR_BF16; }

size_t chunk_len(size_t count, int R, int c) {
  const size_t base = count / (size_t)R;
  return c < R - 1 ? base : count - (size_t)(R - 1) * base;
}

struct Buf {
  uintptr_t lo, hi;  // [lo, hi)
  bool written;
  int rank;
  bool is_in;
};

// Everything that can be checked without the device.
struct Checked {
  int op, R, L, dtype, wire;
  size_t count;  // N, elements of the whole rank vector
  size_t first;  // AllReduce ranges: the buffers hold elements [first, first + n)
  size_t n;
  size_t E;
  bool all_16b_aligned;
  int algo;  // AllReduce summation order (rr_algo)
};

// Checks of everything but the buffers.
rr_status check_scalars(int op, int R, size_t count, int dtype, int wire, int group_size, const rr_launch_cfg *cfg,
                        Checked *ck) {
  if (op != RR_OP_ALLREDUCE && op != RR_OP_REDUCE_SCATTER && op != RR_OP_ALLGATHER) return RR_ERR_INVALID_ARG;
  if (R < 1 || R > RR_MAX_RANKS) return RR_ERR_INVALID_ARG;
  if (!valid_type(dtype) || !valid_type(wire)) return RR_ERR_INVALID_ARG;
  if (!(dtype == wire || dtype == RR_FP32 || wire == RR_FP32)) return RR_ERR_UNSUPPORTED;
  if (op == RR_OP_ALLGATHER && wire != dtype) return RR_ERR_UNSUPPORTED;
  const int L = group_size == 0 ? R : group_size;
  if (L < 1 || L > R || R % L != 0) return RR_ERR_INVALID_ARG;
  if (op != RR_OP_ALLREDUCE && L != R) return RR_ERR_INVALID_ARG;
  if (cfg) {
    if (cfg->path < RR_PATH_AUTO || cfg->path > RR_PATH_DIRECT) return RR_ERR_INVALID_ARG;
    if (cfg->tile_bytes != 0 && (cfg->tile_bytes < 16 || cfg->tile_bytes % 16 != 0 || cfg->tile_bytes > (1 << 20)))
      return RR_ERR_INVALID_ARG;
    if (cfg->stages != 0 && (cfg->stages < 2 || cfg->stages > kMaxStages)) return RR_ERR_INVALID_ARG;
    if (cfg->ctas_per_sm != 0 && (cfg->ctas_per_sm < 1 || cfg->ctas_per_sm > 4)) return RR_ERR_INVALID_ARG;
    if (cfg->threads != 0 && (cfg->threads < 64 || cfg->threads > 1024 || cfg->threads % 32 != 0))
      return RR_ERR_INVALID_ARG;
    if (cfg->max_ctas < 0) return RR_ERR_INVALID_ARG;
    if (cfg->early_launch < 0 || cfg->early_launch > 2) return RR_ERR_INVALID_ARG;
    if (cfg->vectors < 0 || cfg->vectors > 4) return RR_ERR_INVALID_ARG;
    if (cfg->beside_compute < 0 || cfg->beside_compute > 1) return RR_ERR_INVALID_ARG;
    if (cfg->prefetch < 0 || cfg->prefetch > 4) return RR_ERR_INVALID_ARG;
  }
  ck->op = op;
  ck->R = R;
  ck->L = L;
  ck->dtype = dtype;
  ck->wire = wire;
  ck->count = count;
  ck->first = 0;
  ck->n = count;
  ck->algo = RR_ALGO_RING;
  ck->E = elem_bytes(dtype);
  ck->all_16b_aligned = true;
  if (count > (SIZE_MAX / 4) / ck->E) return RR_ERR_INVALID_ARG;
  return RR_OK;
}

// Buffer checks: sizes, NULL, element alignment, address wrap, aliasing.
rr_status check_buffers(const void *const *in, void *const *out, Checked *ck);

rr_status check_args(int op, const void *const *in, void *const *out, int R, size_t count, int dtype, int wire,
                     int group_size, const rr_launch_cfg *cfg, Checked *ck) {
  rr_status st = check_scalars(op, R, count, dtype, wire, group_size, cfg, ck);
  if (st != RR_OK) return st;
  return check_buffers(in, out, ck);
}

rr_status check_buffers(const void *const *in, void *const *out, Checked *ck) {
  if (!in || !out) return RR_ERR_INVALID_ARG;
  if (ck->n == 0) return RR_OK;
  const size_t E = ck->E;
  const int R = ck->R, op = ck->op;
  const size_t count = ck->count;

  // sizes, pointers, alignment
  Buf bufs[2 * RR_MAX_RANKS];
  int nb = 0;
  for (int r = 0; r < R; ++r) {
    const size_t n_in = (op == RR_OP_ALLGATHER) ? chunk_len(count, R, r) : ck->n;
    const size_t n_out = (op == RR_OP_REDUCE_SCATTER) ? chunk_len(count, R, r) : ck->n;
    for (int side = 0; side < 2; ++side) {
      const void *ptr = side == 0 ? in[r] : out[r];
      const size_t bytes = (side == 0 ? n_in : n_out) * E;
      if (bytes == 0) continue;
      const uintptr_t a = reinterpret_cast<uintptr_t>(ptr);
      if (a == 0 || a % E != 0) return RR_ERR_INVALID_ARG;
      if (a > UINTPTR_MAX - bytes) return RR_ERR_INVALID_ARG;
      if (a % 16 != 0) ck->all_16b_aligned = false;
      bufs[nb++] = Buf{a, a + bytes, side == 1, r, side == 0};
    }
  }
  // an output may overlap nothing, except its own input in an in-place AllReduce
  for (int x = 0; x < nb; ++x) {
    if (!bufs[x].written) continue;
    for (int y = 0; y < nb; ++y) {
      if (y == x) continue;
      const Buf &o = bufs[x], &b = bufs[y];
      if (o.lo >= b.hi || b.lo >= o.hi) continue;
      const bool in_place = op == RR_OP_ALLREDUCE && b.is_in && b.rank == o.rank && b.lo == o.lo && b.hi == o.hi;
      if (!in_place) return RR_ERR_ALIAS;
    }
  }
  return RR_OK;
}

int clamp_int(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

unsigned round16_down(unsigned long long x) { return (unsigned)(x & ~15ull); }

// Which of the two 16-byte-aligned paths is faster, from a measured sweep of
// both (bench.py --path-sweep; CUDA-graph replay over inputs colder than L2).
// The direct path keeps about eight loads in flight per thread (plus its L2
// prefetches) and needs no barriers: it wins for every AllGather, every
// ReduceScatter, every two-level ring and every flat AllReduce but one case.
// (Two ranks moved to it once the chunk lookup lost its 64-bit division: at
// 256 MiB per rank, binary16, 0.94 of the copy bandwidth against the tile
// pipeline's 0.90; ReduceScatter 0.89 against 0.78.)  The tile pipeline wins
// for a flat ring of 16 ranks from 64 MiB per rank (two CTAs of three 32 KiB
// stages fit an SM exactly), and for capped grids (each CTA then owns an SM and
// moves 8 KB per bulk copy).
bool prefer_direct(int op, int R, int L, unsigned long long msg_bytes, int max_ctas) {
  const unsigned long long MiB = 1ull << 20;
  if (max_ctas > 0) return false;                       // capped grids: one tile pipeline per SM
  if (op != RR_OP_ALLREDUCE || L < R) return true;      // ReduceScatter, AllGather, two-level
  if (R == 16) return msg_bytes < 64 * MiB;             // two CTAs of three 32 KiB stages per SM
  return true;
}

// Resolve the launch: path, tiles, stages, grid.  Fills every field of *p
// except the buffer pointers and the status word.  Every tile size it picks is
// a multiple of 16 bytes (the bulk copies and the 16-byte shared-memory
// vectors need it) and every shared-memory size fits the device.
rr_status plan_launch(const Checked &ck, const rr_launch_cfg *cfg, int sms, int smem_per_sm, int smem_optin,
                      rr::RingParams *p, rr::Launch *l) {
  const rr_launch_cfg zero = {};
  rr_launch_cfg c = cfg ? *cfg : zero;
  const size_t E = ck.E;
  const unsigned long long N = ck.n;  // elements of this launch
  if (sms < 1 || smem_per_sm < 1 || smem_optin < 1) return RR_ERR_INVALID_ARG;
  // beside compute kernels: a share of the SMs, one CTA each (a tile pipeline
  // per SM), unless the caller gave the cap itself
  if (c.beside_compute && c.max_ctas == 0) {
    c.max_ctas = (int)((long long)sms * RR_BESIDE_COMPUTE_SM_EIGHTHS / 8);
    if (c.max_ctas < 1) c.max_ctas = 1;
  }
  auto capped = [&](int grid) { return (c.max_ctas > 0 && grid > c.max_ctas) ? c.max_ctas : grid; };

  p->count = N;
  p->first = ck.first;
  p->total = ck.count;
  p->R = ck.R;
  p->L = ck.L;
  p->G = ck.R / ck.L;
  p->base = (unsigned long long)ck.count / (unsigned long long)ck.L;
  {  // no 16-byte vector of this launch holds elements of two chunks
    const unsigned long long V = 16 / ck.E;
    p->chunks_on_grid = (p->base == 0 || (p->base % V == 0 && (unsigned long long)ck.first % V == 0)) ? 1 : 0;
  }
  p->algo = ck.algo;
  int P = 1, log2p = 0;
  while (P * 2 <= ck.R) {
    P *= 2;
    ++log2p;
  }
  p->hd_log2p = log2p;
  p->hd_extra = ck.R - P;

  // the 16-byte paths need 16-byte aligned buffers; the tile pipeline also
  // needs ReduceScatter / AllGather chunk boundaries on 16-byte multiples
  // (segments are copied per chunk), the direct path's shifted kernel not
  const bool chunks_aligned = ck.op == RR_OP_ALLREDUCE || (p->base * E) % 16 == 0;
  const unsigned long long n_bulk = (N * E / 16) * 16 / E;
  const bool vec_ok = ck.all_16b_aligned && n_bulk > 0;
  const bool bulk_ok = vec_ok && chunks_aligned;
  int path = c.path;
  if (path == RR_PATH_BULK && !bulk_ok) return RR_ERR_UNSUPPORTED;
  if (path == RR_PATH_DIRECT && !vec_ok) return RR_ERR_UNSUPPORTED;
  if (path == RR_PATH_AUTO) {
    if (!vec_ok)
      path = RR_PATH_SIMPLE;
    else if (!chunks_aligned)  // ReduceScatter / AllGather with chunk boundaries off the 16-byte grid
      path = RR_PATH_DIRECT;
    else
      path = prefer_direct(ck.op, ck.R, ck.L, (unsigned long long)ck.count * E, c.max_ctas) ? RR_PATH_DIRECT
                                                                                             : RR_PATH_BULK;
  }
  p->shifted = (path == RR_PATH_DIRECT && !chunks_aligned) ? 1 : 0;
  // The chunk-by-chunk rows on aligned chunks (below) are taken when no
  // register budget is asked for and the vectors asked for, if any, are a row
  // count the rows are built for; otherwise the direct kernel runs.
  const bool rows_ok = c.ctas_per_sm == 0 &&
                       (c.vectors == 0 || rr::shift_variant_exists(ck.op, ck.dtype != RR_FP32 && ck.wire == RR_FP32,
                                                                   c.vectors));
  // ReduceScatter over two ranks from 32 MiB per rank: the chunk-by-chunk
  // (shifted) kernel also where the chunks sit on the 16-byte grid (it then
  // shifts by nothing).  It knows each work item's chunk, where the direct
  // kernel looks up every vector's, and its four rows keep eight loads in
  // flight a lane.  Measured, binary16, of the copy bandwidth, at 16 / 32 /
  // 64 / 256 MiB per rank: direct 0.70 / 0.74 / 0.84 / 0.89, chunk by chunk
  // 0.70 / 0.80 / 0.88 / 0.96; over three or more ranks the direct kernel is
  // as fast or faster.
  if (path == RR_PATH_DIRECT && ck.op == RR_OP_REDUCE_SCATTER && ck.algo == RR_ALGO_RING && ck.L == 2 &&
      (unsigned long long)ck.count * E >= (32ull << 20) && rows_ok)
    p->shifted = 1;
  // AllGather from 12 MiB per rank (two ranks: 64 MiB) likewise, in rows of 32
  // vectors of one chunk that end on 512-byte store segments.  Measured,
  // binary16, of the copy bandwidth, direct -> rows on aligned chunks at 16 /
  // 64 / 256 MiB per rank: R = 4 0.87 / 0.89 / 0.93 -> 0.94 / 0.95 / 0.95, R =
  // 8 0.89 / 0.91 / 0.92 -> 0.96 / 0.95 / 0.94, R = 16 0.90 / 0.90 / 0.90 ->
  // 0.96 / 0.95 / 0.94; R = 3 / 5 at 64 MiB 0.88 / 0.91 -> 0.93 / 0.94; R = 2
  // at 64 / 256 MiB 0.88 / 0.92 -> 0.92 / 0.96 (at 16 MiB 0.80 -> 0.77); at
  // 12 MiB R = 8 / 16 0.88 / 0.89 -> 0.95 / 0.96; at 8 MiB rows lost up to 6 %,
  // at 4 MiB up to 35 %.
  if (path == RR_PATH_DIRECT && ck.op == RR_OP_ALLGATHER && ck.algo == RR_ALGO_RING &&
      (unsigned long long)ck.count * E >= (ck.L == 2 ? (64ull << 20) : (12ull << 20)) && rows_ok)
    p->shifted = 1;
  // AllReduce over flat rings of two to four ranks from 16 MiB per rank, the
  // chunks on the grid and the whole rank vectors in one call (no range): the
  // same chunk-by-chunk rows, folding each row's vectors and storing the sum
  // to every output.  Measured, binary16, of the copy bandwidth, direct ->
  // rows at 16 / 32 / 128 / 256 MiB per rank: R = 2 0.82 / 0.88 / 0.94 / 0.93
  // -> 0.87 / 0.90 / 0.99 / 0.98, R = 3 (24 / 32 / 128 / 256 MiB) 0.93 / 0.91
  // / 0.96 / 0.96 -> 0.94 / 0.95 / 1.00 / 1.00, R = 4 0.94 / 0.98 / 0.97 /
  // 0.97 -> 0.97 / 0.97 / 1.00 / 0.99; binary32 at 64 MiB R = 2 / 4 0.94 /
  // 0.96 -> 0.95 / 0.99.  (R = 2 at 24 MiB lost 2-3 %.)
  if (path == RR_PATH_DIRECT && ck.op == RR_OP_ALLREDUCE && ck.algo == RR_ALGO_RING && ck.L == ck.R && ck.L >= 2 &&
      ck.L <= 4 && ck.first == 0 && ck.n == ck.count && (p->base * E) % 16 == 0 &&
      !(ck.dtype != RR_FP32 && ck.wire == RR_FP32) && (unsigned long long)ck.count * E >= (16ull << 20) && rows_ok)
    p->shifted = 1;

  l->path = path;
  // 128-thread CTAs on the direct path: finer grid granularity, measured 1-5 %
  // faster than 256 up to 16 MiB per rank and the same above
  l->threads = c.threads ? c.threads : (path == RR_PATH_DIRECT ? 128 : 256);
  l->early_launch = c.early_launch == 0 ? kEarlyLaunchDefault : c.early_launch == 1;
  if (path == RR_PATH_DIRECT) {  // U 16-byte vectors per thread
    if (l->threads > 256) return RR_ERR_UNSUPPORTED;
    const bool wide = ck.dtype != RR_FP32 && ck.wire == RR_FP32;  // eight binary32 accumulators: 128 registers
    const unsigned long long msg_bytes = (unsigned long long)ck.count * E;
    // About eight loads in flight per thread: few ranks per group take several
    // vectors (two vectors for up to four ranks per group: for two ranks, four
    // vectors a thread reached 0.61 of the copy bandwidth and two vectors at
    // three CTAs per SM 0.78, at 256 MiB).
    int U = (ck.op == RR_OP_ALLGATHER || ck.algo == RR_ALGO_HALVING_DOUBLING) ? 1 : (ck.L <= 4 ? 2 : 1);
    // ReduceScatter stores one vector per R loads, so nearly all its traffic
    // is loads and it wants more of them in flight: two vectors a thread
    // (batches of four ranks) from 64 MiB per rank.  Measured at 256 MiB per
    // rank, binary32, of the copy bandwidth: R = 5 0.79 -> 0.90, R = 8 0.95 ->
    // 1.04, R = 9 0.87 -> 1.00, R = 16 0.99 -> 1.04 (results bit-identical);
    // R = 9 at 4 MiB lost 3 %.  (Three ranks at three vectors, nine loads but
    // two CTAs per SM: 0.60 against 0.875 at 256 MiB, binary16.)
    if (ck.op == RR_OP_REDUCE_SCATTER && ck.algo == RR_ALGO_RING && msg_bytes >= (64ull << 20)) U = 2;
    // AllGather from 4 MiB per rank: two vectors a thread over up to five
    // ranks below 16 MiB, and over two ranks below 64 MiB on two waves of two
    // 256-thread CTAs per SM (below).  Measured, of the copy bandwidth, median
    // of two buffer layouts: binary32 at 4 / 8 MiB per rank R = 3 0.61 / 0.73
    // -> 0.64 / 0.75, R = 4 0.68 / 0.82 -> 0.71 / 0.83, R = 5 0.72 / 0.84 ->
    // 0.74 / 0.88; binary16 R = 2 at 8 / 16 / 32 MiB 0.65 / 0.75 / 0.86 -> 0.70
    // / 0.81 / 0.88.  Not below 4 MiB (R = 2 at 1 MiB lost 14 %; grids of 1.3
    // waves at two vectors lost 7-16 % at 3 MiB), nor over eight ranks or
    // more (R = 8 at 4 MiB lost 3 %, R = 16 12 %), nor for three ranks from 16
    // MiB (0-1 % either way).
    const bool ag_pair = ck.op == RR_OP_ALLGATHER && ck.algo == RR_ALGO_RING && ck.R == 2 &&
                         msg_bytes >= (4ull << 20) && msg_bytes < (64ull << 20);
    if (ag_pair || (ck.op == RR_OP_ALLGATHER && ck.algo == RR_ALGO_RING && ck.R <= 5 && msg_bytes >= (4ull << 20) &&
                    msg_bytes < (16ull << 20)))
      U = 2;
    if (p->shifted) {
      // rows a warp takes at once.  ReduceScatter, measured, binary16, of the
      // copy bandwidth, median of two buffer layouts: two rows, but four for
      // two ranks from 8 MiB per rank (R = 2 at 16 / 64 / 256 MiB: two 0.68 /
      // 0.83 / 0.90, four 0.70 / 0.88 / 0.96; at 4 MiB two 0.31, four 0.28),
      // one for four or more ranks below 8 MiB (4 MiB: R = 4 0.38 -> 0.39, R =
      // 5 0.40 -> 0.47, R = 8 0.66 -> 0.71, R = 16 0.72 -> 0.82; at 16 MiB
      // one row lost 1-18 %), four for eight or more ranks from 128 MiB (256
      // MiB: R = 8 0.95 -> 0.98, R = 16 0.97 -> 1.00; at 64 MiB 0-1 % lost).
      // AllGather: rows of 32 vectors for up to four ranks (two rows; R = 2
      // at 16 / 256 MiB: two 0.68 / 0.82, four 0.63 / 0.83) and for more from
      // 12 MiB per rank, two rows, four for eight or more ranks from 64 MiB;
      // below that five or more ranks take one vector a thread a grid-stride
      // apart.  Measured, binary16, of the copy bandwidth, against vectors a
      // thread at 12 / 16 / 64 / 256 MiB: R = 5 0.83 / 0.82 / 0.91 / 0.91 ->
      // 0.86 / 0.94 / 0.94 / 0.95, R = 8 0.85 / 0.88 / 0.92 / 0.93 -> 0.92 /
      // 0.96 / 0.95 / 0.93, R = 16 0.92 / 0.94 / 0.94 / 0.94 -> 0.95 / 0.96 /
      // 0.95 / 0.94; at 8 MiB rows lost up to 4 %, at 1 and 4 MiB 7-25 %, and
      // one vector a thread beat two by 1-13 %.
      if (ck.op == RR_OP_ALLREDUCE) {  // four rows for two ranks from 64 MiB, for more from 128 MiB
        U = ((ck.L == 2 && msg_bytes >= (64ull << 20)) || msg_bytes >= (128ull << 20)) ? 4 : 2;
      } else if (ck.op == RR_OP_REDUCE_SCATTER) {
        U = 2;
        if (ck.L == 2 && msg_bytes >= (8ull << 20)) U = 4;
        if (ck.L >= 4 && msg_bytes < (8ull << 20)) U = 1;
        if (ck.L >= 8 && msg_bytes >= (128ull << 20)) U = 4;
      } else {
        p->shift_rows = (ck.L <= 4 || msg_bytes >= (12ull << 20)) ? 1 : 0;
        U = !p->shift_rows ? 1 : (ck.L >= 8 && msg_bytes >= (64ull << 20)) ? 4 : 2;
      }
    }
    if (wide && U > 2) U = 2;
    // Flat rings of up to four ranks under 32 MiB per rank (ring order,
    // AllReduce below the chunk-by-chunk rows' 16 MiB and ReduceScatter,
    // chunks on the grid): one wave of resident CTAs whose threads loop, with
    // the L2 prefetch of the first and the next iteration, instead of several
    // waves with a partial last one.  One vector
    // a thread where two would leave SMs idle (under two vectors per thread of
    // a wave of two 256-thread CTAs per SM); two CTAs per SM up to 8 MiB, three
    // above.  Measured (binary16 unless stated, of the copy bandwidth, median of
    // two buffer layouts): 1 MiB AllReduce R = 2 / 3 / 4 0.24 / 0.34 / 0.41 ->
    // 0.29 / 0.40 / 0.48; 4 MiB AllReduce R = 4 binary32 0.67 -> 0.76,
    // ReduceScatter 0.57 -> 0.60; 16 MiB AllReduce R = 2 / 3 0.78 / 0.91 ->
    // 0.81 / 0.94, ReduceScatter R = 3 / 4 0.79 / 0.83 -> 0.87 / 0.92.
    const unsigned long long vecs_here = n_bulk * E / 16;
    const bool one_wave = ck.algo == RR_ALGO_RING && !p->shifted && ck.op != RR_OP_ALLGATHER && ck.L == ck.R &&
                          ck.L <= 4 && msg_bytes < (32ull << 20) && !wide && c.max_ctas == 0;
    if (one_wave) U = vecs_here < 2ull * 128ull * 4ull * (unsigned long long)sms ? 1 : 2;
    if (c.vectors) U = c.vectors;
    p->direct_u = U;
    // L2 prefetch (kPrefetch* bits; only the ring / naive kernels on 16-byte
    // chunk boundaries prefetch).  Measured, binary16, of the copy bandwidth,
    // median over buffer layouts:
    //  - before the launch wait (its DRAM latency overlaps the previous
    //    kernel): AllReduce R = 8 1 MiB 0.55 -> 0.64, 4 MiB 0.84 -> 0.87;
    //    R = 4 binary32 ReduceScatter 4 MiB 0.51 -> 0.58; little effect from
    //    64 MiB, where R = 8 lost 1 % and groups of up to four ranks gained
    //    0-3 %: below 64 MiB, or up to four ranks a group;
    //  - one iteration ahead (twice the requests in flight): where threads
    //    have few loads each, R = 2 (AllReduce 256 MiB 0.90 -> 0.94), every
    //    AllGather (R = 2 256 MiB 0.88 -> 0.93), ReduceScatter over three
    //    ranks (0.94 -> 1.00); and from 8 to 64 MiB (AllReduce R = 3 / 4 / 8
    //    at 16 MiB 0.82 / 0.88 / 0.96 -> 0.91 / 0.94 / 0.99 with both); not
    //    for ReduceScatter over five or more ranks (R = 8, 16 MiB: 0.99 -> 0.91)
    //    nor above 64 MiB otherwise (AllReduce R = 8 256 MiB: 0.99 -> 0.95).
    {
      const bool small = msg_bytes < (64ull << 20), mid = small && msg_bytes >= (8ull << 20);
      const bool rs_many = ck.op == RR_OP_REDUCE_SCATTER && ck.L >= 5;
      int pf = 0;
      if (small || ck.L <= 4) pf |= rr::kPrefetchHead;
      if (ck.R == 2 || ck.op == RR_OP_ALLGATHER || (ck.op == RR_OP_REDUCE_SCATTER && ck.L == 3) || (mid && !rs_many))
        pf |= rr::kPrefetchAhead;
      if (one_wave) pf = rr::kPrefetchHead | rr::kPrefetchAhead;
      p->prefetch = c.prefetch ? c.prefetch - 1 : pf;
    }
    // The shifted kernels: the AllGather prefetches its first work item and
    // the next one (binary16, of the copy bandwidth: R = 2 at 256 MiB 0.80 ->
    // 0.86, R = 8 at 16 MiB 0.83 -> 0.88); the ReduceScatter its first item,
    // over three to five ranks below 32 MiB per rank (4 / 16 MiB: R = 3 0.32 /
    // 0.77 -> 0.35 / 0.82, R = 4 0.38 / 0.84 -> 0.39 / 0.87, R = 5 0.40 / 0.78
    // -> 0.42 / 0.85; two ranks lost 1-3 %, eight or more 10-14 %; one item
    // ahead lost 2-20 % everywhere).
    if (p->shifted && c.prefetch == 0) {
      if (ck.op == RR_OP_ALLGATHER)
        p->prefetch = rr::kPrefetchHead | rr::kPrefetchAhead;
      else if (ck.op == RR_OP_ALLREDUCE)  // the first item below 24 MiB (16 MiB: R = 2 0.84 -> 0.87, R = 4
        p->prefetch = msg_bytes < (24ull << 20) ? rr::kPrefetchHead : 0;  // 0.94 -> 0.97), none above (1-3 %)
      else
        p->prefetch = (ck.L >= 3 && ck.L <= 5 && msg_bytes < (32ull << 20)) ? rr::kPrefetchHead : 0;
    }
    if (ck.algo == RR_ALGO_HALVING_DOUBLING) p->prefetch = 0;
    // A third CTA per SM (registers capped at 85) keeps more loads in flight
    // once threads loop (measured at 256 MiB, of the copy bandwidth: R = 5
    // 0.88 -> 0.98, R = 9 0.93 -> 0.99, R = 3 0.85 -> 0.96).  A grid that
    // two CTAs per SM cover in one wave (twice that for 16 or more ranks)
    // finishes sooner with the 128-register code (1 MiB: 3-10 %).  Threads
    // whose group is exactly one batch of seven or eight loads (R = 7 or 8;
    // two-level rings of 4- or 8-rank groups) keep DRAM busy with two, which
    // did better from 64 MiB (R = 8, 256 MiB: 1.006 against 0.991); flat rings
    // of three or four ranks (two vectors a thread) do not.
    const unsigned long long vecs = n_bulk * E / 16;
    const int batch = U * ck.L;  // loads of one group a thread issues together
    const bool full_batch = (batch == 7 || batch == 8) && msg_bytes >= (64ull << 20) && !(U == 2 && ck.L == ck.R);
    const bool looping = vecs > (unsigned long long)sms * 512ull * (unsigned long long)U * (ck.L >= 16 ? 2ull : 1ull);
    l->direct_occ = (U <= 3 && ck.op != RR_OP_ALLGATHER && looping && !full_batch && !wide) ? 3 : 2;
    // Halving-doubling loads a whole tree (up to 16 vectors) per batch: a third
    // CTA helped only below seven ranks (R = 5: 0.85 -> 1.00 at 256 MiB; R = 12:
    // 1.01 -> 0.99).
    if (ck.algo == RR_ALGO_HALVING_DOUBLING)
      l->direct_occ = (ck.R < 7 && looping && !wide) ? 3 : 2;
    if (one_wave) l->direct_occ = (U == 1 || msg_bytes <= (8ull << 20)) ? 2 : 3;
    if (U >= 3 && !p->shifted) l->direct_occ = 2;  // three or four vectors: 128 registers
    if (p->shifted) l->direct_occ = rr::shift_occupancy(U);  // fixed per row count
    // ctas_per_sm asks for a register budget (2 or 3 CTAs per SM).  It applies
    // when a kernel of that budget exists for this plan; otherwise (1 or 4,
    // tile-pipeline shapes, or a budget the kernel is not built for) it is
    // ignored, unless the direct path was forced.
    if (c.ctas_per_sm != 0) {
      const int want = c.ctas_per_sm;
      bool ok = want == 2 || want == 3;
      if (ok) {
        if (ck.algo == RR_ALGO_HALVING_DOUBLING)
          ok = want == 2 || (!wide && ck.R < 8);
        else if (p->shifted)
          ok = want == rr::shift_occupancy(U);
        else
          ok = rr::direct_variant_exists(ck.op, wide, U, want);
      }
      if (ok)
        l->direct_occ = want;
      else if (c.path == RR_PATH_DIRECT)
        return RR_ERR_UNSUPPORTED;
    }
    // only kernels that exist (a forced configuration may ask for others)
    if (ck.algo == RR_ALGO_HALVING_DOUBLING) {
      if (U != 1 || (l->direct_occ != 2 && !(l->direct_occ == 3 && !wide && ck.R < 8))) return RR_ERR_UNSUPPORTED;
    } else if (p->shifted) {
      if (!rr::shift_variant_exists(ck.op, wide, U)) return RR_ERR_UNSUPPORTED;
    } else if (!rr::direct_variant_exists(ck.op, wide, U, l->direct_occ)) {
      return RR_ERR_UNSUPPORTED;
    }
    const unsigned long long blocks = (vecs + (unsigned long long)l->threads * U - 1) / ((unsigned long long)l->threads * U);
    unsigned long long cap = (unsigned long long)sms * (2048 / l->threads);
    // ReduceScatter, and ring AllReduce over groups of at most three ranks, do
    // better on two whole waves of the resident CTAs than on sixteen 128-thread
    // CTAs per SM (2.67 waves at three CTAs per SM).  Measured at 256 MiB per
    // rank, of the copy bandwidth: ReduceScatter R = 4 0.95 -> 0.99, R = 5
    // 0.74 -> 0.79, R = 16 0.96 -> 0.99; AllReduce R = 3 0.96 -> 0.99; two-level
    // 4 x 2 at 64 MiB 0.90 -> 0.95.  AllReduce over four or more ranks a group
    // and AllGather lost 1-9 % on any whole number of waves from one to four.
    if (ck.algo == RR_ALGO_RING && !p->shifted &&
        (ck.op == RR_OP_REDUCE_SCATTER || (ck.op == RR_OP_ALLREDUCE && ck.L <= 3)))
      cap = (unsigned long long)sms * (unsigned long long)l->direct_occ * (256ull / l->threads) * 2ull;
    if (one_wave)  // one wave of the CTAs the registers let reside
      cap = (unsigned long long)sms * (unsigned long long)l->direct_occ * (256ull / l->threads);
    if (ag_pair && !p->shifted)
      cap = (unsigned long long)sms * (unsigned long long)l->direct_occ * (256ull / l->threads) * 2ull;
    // The shifted ReduceScatter: twelve 128-thread CTAs per SM (two whole waves
    // of the two- and three-row kernels, three of the four-row one) instead of
    // sixteen, over groups of up to four ranks and, for more, from 32 MiB per
    // rank.  Measured, binary16, of the copy bandwidth, median of two buffer
    // layouts, at 16 / 64 / 256 MiB per rank: R = 2 0.59 / 0.75 / 0.85 ->
    // 0.60 / 0.76 / 0.84; R = 3 0.64 / 0.80 / 0.87 -> 0.69 / 0.84 / 0.87; R = 4
    // 0.73 / 0.88 / 0.91 -> 0.77 / 0.92 / 0.93; R = 5 (64 / 256) 0.79 / 0.85 ->
    // 0.83 / 0.89; R = 9 0.91 / 0.92 -> 0.94 / 0.95; R = 16 0.98 / 0.97 ->
    // 0.98 / 0.98.  At 16 MiB five or more ranks lost 2-5 %.
    if (p->shifted && ck.op == RR_OP_REDUCE_SCATTER && (ck.L <= 4 || msg_bytes >= (32ull << 20)))
      cap = (unsigned long long)sms * 1536ull / (unsigned long long)l->threads;
    // Vectors over a chunk boundary (ring order, boundaries off the 16-byte
    // grid): one extra CTA folds them, so the main loop stays lean.
    const unsigned long long V = 16 / E;
    p->straddle_cta = (ck.op == RR_OP_ALLREDUCE && ck.algo == RR_ALGO_RING && ck.L > 1 && p->base > 0 &&
                       (p->base % V != 0 || ck.first % V != 0))
                          ? 1
                          : 0;
    l->grid = capped((int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap));
    if (p->straddle_cta) {
      if (!(c.max_ctas > 0 && l->grid >= c.max_ctas))
        l->grid += 1;                      // one more CTA
      else if (l->grid < 2)
        p->straddle_cta = 0;               // a one-CTA cap: the main loop folds them element by element
    }
    l->smem = 0;
    l->ctas_per_sm = 0;
    p->n_bulk = n_bulk;
    p->n_tiles = 0;
    p->tile_elems = 0;
    p->stages = 0;
    p->slots = 0;
    p->store_lag = 0;
    return RR_OK;
  }
  if (path == RR_PATH_SIMPLE) {
    const unsigned long long blocks = (N + l->threads - 1) / l->threads;
    const unsigned long long cap = (unsigned long long)sms * 8;
    l->grid = capped((int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap));
    l->smem = 0;
    l->ctas_per_sm = 0;
    p->n_bulk = 0;
    p->n_tiles = 0;
    p->tile_elems = 0;
    p->stages = 0;
    p->slots = 0;
    return RR_OK;
  }

  const int slots = ck.op == RR_OP_ALLGATHER ? 1 : ck.R;
  const unsigned long long total_bytes = n_bulk * E;
  // shared memory one CTA may use when `ctas` CTAs share an SM (the runtime keeps 1 KB per CTA)
  auto budget_for = [&](int ctas) {
    long long b = (long long)smem_per_sm / ctas - 1024;
    return b > smem_optin ? (long long)smem_optin : b;
  };

  // A grid capped below 3 CTAs per SM (say, beside compute kernels) gives every
  // CTA its own SM; one issuing thread per SM then needs larger bulk copies to
  // keep its SM's bandwidth (measured: 96 capped CTAs reached 0.77 of the full
  // bandwidth with 8 KB tiles, 0.46 with 2 KB tiles).
  const bool few_ctas = c.max_ctas > 0 && (unsigned long long)c.max_ctas < 3ull * (unsigned long long)sms &&
                        c.ctas_per_sm == 0 && c.stages == 0;

  // Tile: 16 KB per stage across the slots, at least 2 KB per rank (smaller
  // bulk copies lose bandwidth), shrunk only when two stages do not fit one CTA.
  unsigned long long tile = (unsigned long long)c.tile_bytes;
  if (tile == 0 && few_ctas) {
    tile = 8192;
    while (tile > 2048 && 3ull * (tile * slots + 8) > (unsigned long long)budget_for(1)) tile /= 2;
    while (tile > 16 && 2ull * (tile * slots + 8) > (unsigned long long)budget_for(1)) tile = round16_down(tile / 2);
  }
  if (tile == 0) {
    tile = round16_down(16384 / slots);
    if (tile < 2048) tile = 2048;
    if (tile > 16384) tile = 16384;
    const long long fit = budget_for(c.ctas_per_sm ? c.ctas_per_sm : 1);
    while (tile > 16 && 2ull * (tile * slots + 8) > (unsigned long long)fit) tile = round16_down(tile / 2);
  }
  if (tile < 16 || tile % 16 != 0 || tile % E != 0) return RR_ERR_INVALID_ARG;
  const unsigned long long stage_bytes = tile * slots;
  const unsigned long long n_tiles = (total_bytes + tile - 1) / tile;

  // CTAs per SM and stages.  Several independent CTA pipelines per SM keep
  // more bulk copies in flight than one deep pipeline: prefer 3 CTAs of 3
  // stages.  A message with at most 4 tiles per SM gets one CTA per tile.
  int ctas = c.ctas_per_sm, stages = c.stages;
  if (few_ctas) {
    ctas = 1;
    stages = clamp_int((int)((unsigned long long)budget_for(1) / (stage_bytes + 8)), 2, 3);
  } else if (ctas == 0 && stages == 0 && n_tiles <= 4ull * (unsigned long long)sms) {
    ctas = (int)((n_tiles + sms - 1) / sms);
    if (ctas < 1) ctas = 1;
    while (ctas > 1 && 2ull * (stage_bytes + 8) > (unsigned long long)budget_for(ctas)) --ctas;
    stages = 2;
  }
  if (ctas == 0) {
    const int want_stages = stages ? stages : 3;
    ctas = 1;
    for (int cand = 3; cand >= 1; --cand)
      if ((unsigned long long)want_stages * (stage_bytes + 8) <= (unsigned long long)budget_for(cand)) {
        ctas = cand;
        break;
      }
  }
  const long long budget = budget_for(ctas);
  if (budget < 64) return RR_ERR_UNSUPPORTED;
  if (stages == 0) stages = clamp_int((int)((unsigned long long)budget / (stage_bytes + 8)), 2, 3);
  const unsigned long long smem = (unsigned long long)stages * (stage_bytes + 8);
  if (smem > (unsigned long long)budget) return RR_ERR_UNSUPPORTED;

  p->tile_elems = (int)(tile / E);
  // store groups left in flight before a stage is refilled: deep pipelines
  // split their stages between loads and stores
  p->store_lag = stages >= 5 ? (stages - 1) / 2 : 1;
  if (p->store_lag > 8) p->store_lag = 8;
  p->n_bulk = n_bulk;
  p->n_tiles = (n_bulk + p->tile_elems - 1) / p->tile_elems;
  p->stages = stages;
  p->slots = slots;
  const unsigned long long cap = (unsigned long long)sms * ctas;
  l->grid = capped((int)(p->n_tiles < cap ? p->n_tiles : cap));
  l->smem = (size_t)smem;
  l->ctas_per_sm = ctas;
  return RR_OK;
}

// Plan for the current device and fill the buffer pointers.
rr_status plan(const Checked &ck, const void *const *in, void *const *out, const rr_launch_cfg *cfg,
               const DeviceInfo &dev, rr::RingParams *p, rr::Launch *l) {
  *p = rr::RingParams{};
  for (int r = 0; r < ck.R; ++r) {
    p->in[r] = in[r];
    p->out[r] = out[r];
  }
  p->status = dev.status;
  p->debug_margin = g_debug_margin.load(std::memory_order_relaxed);
  return plan_launch(ck, cfg, dev.sms, dev.smem_per_sm, dev.smem_optin, p, l);
}

void export_plan(const rr::RingParams &p, const rr::Launch &l, size_t E, bool beside_compute,
                 rr_launch_cfg *chosen) {
  chosen->path = l.path;
  chosen->tile_bytes = l.path == RR_PATH_BULK ? p.tile_elems * (int)E : 0;
  chosen->stages = l.path == RR_PATH_BULK ? p.stages : 0;
  chosen->ctas_per_sm = l.path == RR_PATH_DIRECT ? l.direct_occ : l.ctas_per_sm;
  chosen->threads = l.threads;
  chosen->max_ctas = l.grid;
  chosen->early_launch = l.early_launch ? 1 : 2;
  chosen->vectors = l.path == RR_PATH_DIRECT ? p.direct_u : 0;
  chosen->prefetch = l.path == RR_PATH_DIRECT ? p.prefetch + 1 : 0;
  chosen->beside_compute = beside_compute ? 1 : 0;
}

// Plan and launch a validated collective on the current device.
rr_status launch_checked(const Checked &ck, const void *const *in, void *const *out, const rr_launch_cfg *cfg,
                         cudaStream_t stream) {
  DeviceInfo dev;
  rr_status st = current_device(&dev);
  if (st != RR_OK) return st;
  rr::RingParams p;
  rr::Launch l;
  st = plan(ck, in, out, cfg, dev, &p, &l);
  if (st != RR_OK) return st;
  const cudaError_t e = rr::launch_collective(ck.op, ck.dtype, ck.wire, p, l, stream);
  return cuda_ok(e) ? RR_OK : RR_ERR_CUDA;
}

rr_status run(int op, const void *const *in, void *const *out, int R, size_t count, int dtype, int wire,
              int group_size, const rr_launch_cfg *cfg, cudaStream_t stream) {
  Checked ck;
  rr_status st = check_args(op, in, out, R, count, dtype, wire, group_size, cfg, &ck);
  if (st != RR_OK || count == 0) return st;
  return launch_checked(ck, in, out, cfg, stream);
}

// --------------------------------------------------------------------------
// AllReduce of host buffers through a device workspace, pipelined in pieces
// --------------------------------------------------------------------------

constexpr int kHostSlots = 3;           // workspace slots: copy-in, fold, copy-out overlap
constexpr size_t kPieceAlign = 256;     // piece length granularity (elements)

struct Pipe {
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t copied_in[kHostSlots] = {}, folded[kHostSlots] = {}, copied_out[kHostSlots] = {};
  bool valid = false;
  std::mutex mu;
};
Pipe g_pipes[kMaxDevices];

rr_status pipe_for_current_device(Pipe **out) {
  int dev = 0;
  if (!cuda_ok(cudaGetDevice(&dev)) || dev < 0 || dev >= kMaxDevices) return RR_ERR_CUDA;
  Pipe &pp = g_pipes[dev];
  std::lock_guard<std::mutex> lock(g_devices_mu);
  if (!pp.valid) {
    if (!cuda_ok(cudaStreamCreateWithFlags(&pp.h2d, cudaStreamNonBlocking)) ||
        !cuda_ok(cudaStreamCreateWithFlags(&pp.d2h, cudaStreamNonBlocking)) ||
        !cuda_ok(cudaEventCreateWithFlags(&pp.start, cudaEventDisableTiming)))
      return RR_ERR_CUDA;
    for (int k = 0; k < kHostSlots; ++k)
      if (!cuda_ok(cudaEventCreateWithFlags(&pp.copied_in[k], cudaEventDisableTiming)) ||
          !cuda_ok(cudaEventCreateWithFlags(&pp.folded[k], cudaEventDisableTiming)) ||
          !cuda_ok(cudaEventCreateWithFlags(&pp.copied_out[k], cudaEventDisableTiming)))
        return RR_ERR_CUDA;
    pp.valid = true;
  }
  *out = &pp;
  return RR_OK;
}

// copy_mode RR_HOST_COPIES_OVERLAP: piece k+1 copied in on one internal
// stream while piece k-1 is copied out on the other (both directions of the
// host link at once).  RR_HOST_COPIES_ONE_WAY: both directions on one copy
// stream, in the order copy-in k+1, copy-out k, so the link carries one
// direction at a time and the fold of piece k still overlaps the copies.
rr_status host_pipeline(const void *const *host_in, void *const *host_out, int R, size_t count, int dtype, int wire,
                        int group_size, void *ws, size_t ws_bytes, int copy_mode, cudaStream_t stream) {
  Checked ck;
  rr_status st = check_scalars(RR_OP_ALLREDUCE, R, count, dtype, wire, group_size, nullptr, &ck);
  if (st != RR_OK) return st;
  st = check_buffers(host_in, host_out, &ck);  // the host buffers: sizes, NULL, aliasing
  if (st != RR_OK || count == 0) return st;
  const size_t E = ck.E;
  const uintptr_t wsa = reinterpret_cast<uintptr_t>(ws);
  if (!ws || wsa % 16 != 0) return RR_ERR_INVALID_ARG;
  size_t piece = ws_bytes / ((size_t)kHostSlots * R * E) / kPieceAlign * kPieceAlign;
  if (piece == 0) return RR_ERR_INVALID_ARG;
  if (piece > count) piece = (count + kPieceAlign - 1) / kPieceAlign * kPieceAlign;
  const size_t slot_bytes = (size_t)R * piece * E;
  // the workspace must not overlap the host buffers (they may be device-visible)
  for (int r = 0; r < R; ++r) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(host_in[r]), b = reinterpret_cast<uintptr_t>(host_out[r]);
    const uintptr_t lo = wsa, hi = wsa + (size_t)kHostSlots * slot_bytes;
    if ((a < hi && lo < a + count * E) || (b < hi && lo < b + count * E)) return RR_ERR_ALIAS;
  }

  Pipe *pp = nullptr;
  st = pipe_for_current_device(&pp);
  if (st != RR_OK) return st;
  std::lock_guard<std::mutex> lock(pp->mu);
  auto ok = [](cudaError_t e) { return cuda_ok(e); };
  // the copies start after the work already enqueued on `stream`
  if (!ok(cudaEventRecord(pp->start, stream)) || !ok(cudaStreamWaitEvent(pp->h2d, pp->start, 0))) return RR_ERR_CUDA;
  const size_t pieces = (count + piece - 1) / piece;
  if (copy_mode == RR_HOST_COPIES_ONE_WAY) {
    // one copy stream (h2d) for both directions: in k+1, then out k
    auto slot_ptr = [&](size_t k) { return static_cast<unsigned char *>(ws) + (k % kHostSlots) * slot_bytes; };
    auto copy_in = [&](size_t k) -> bool {
      const size_t first = k * piece, n = (count - first < piece) ? count - first : piece;
      for (int r = 0; r < R; ++r)
        if (!ok(cudaMemcpyAsync(slot_ptr(k) + (size_t)r * piece * E, static_cast<const unsigned char *>(host_in[r]) + first * E,
                                n * E, cudaMemcpyHostToDevice, pp->h2d)))
          return false;
      return ok(cudaEventRecord(pp->copied_in[k % kHostSlots], pp->h2d));
    };
    if (!copy_in(0)) return RR_ERR_CUDA;
    for (size_t k = 0; k < pieces; ++k) {
      const int sl = (int)(k % kHostSlots);
      const size_t first = k * piece, n = (count - first < piece) ? count - first : piece;
      if (k + 1 < pieces && !copy_in(k + 1)) return RR_ERR_CUDA;  // its slot's copy-out (k - 2) is earlier on h2d
      if (!ok(cudaStreamWaitEvent(stream, pp->copied_in[sl], 0))) return RR_ERR_CUDA;
      const void *dev_in[RR_MAX_RANKS];
      void *dev_out[RR_MAX_RANKS];
      for (int r = 0; r < R; ++r) dev_in[r] = dev_out[r] = slot_ptr(k) + (size_t)r * piece * E;
      Checked pk = ck;
      pk.first = first;
      pk.n = n;
      pk.all_16b_aligned = true;
      st = launch_checked(pk, dev_in, dev_out, nullptr, stream);
      if (st != RR_OK) return st;
      if (!ok(cudaEventRecord(pp->folded[sl], stream)) || !ok(cudaStreamWaitEvent(pp->h2d, pp->folded[sl], 0)))
        return RR_ERR_CUDA;
      for (int r = 0; r < R; ++r)
        if (!ok(cudaMemcpyAsync(static_cast<unsigned char *>(host_out[r]) + first * E, slot_ptr(k) + (size_t)r * piece * E,
                                n * E, cudaMemcpyDeviceToHost, pp->h2d)))
          return RR_ERR_CUDA;
    }
    // work enqueued on `stream` after this call sees every output copied
    if (!ok(cudaEventRecord(pp->copied_out[0], pp->h2d)) || !ok(cudaStreamWaitEvent(stream, pp->copied_out[0], 0)))
      return RR_ERR_CUDA;
    return RR_OK;
  }
  for (size_t k = 0; k < pieces; ++k) {
    const int sl = (int)(k % kHostSlots);
    const size_t first = k * piece, n = (count - first < piece) ? count - first : piece;
    unsigned char *slot = static_cast<unsigned char *>(ws) + (size_t)sl * slot_bytes;
    const void *dev_in[RR_MAX_RANKS];
    void *dev_out[RR_MAX_RANKS];
    // copy in once the slot's previous copy-out has finished
    if (!ok(cudaStreamWaitEvent(pp->h2d, pp->copied_out[sl], 0))) return RR_ERR_CUDA;
    for (int r = 0; r < R; ++r) {
      unsigned char *d = slot + (size_t)r * piece * E;
      dev_in[r] = d;
      dev_out[r] = d;
      if (!ok(cudaMemcpyAsync(d, static_cast<const unsigned char *>(host_in[r]) + first * E, n * E,
                              cudaMemcpyHostToDevice, pp->h2d)))
        return RR_ERR_CUDA;
    }
    if (!ok(cudaEventRecord(pp->copied_in[sl], pp->h2d)) || !ok(cudaStreamWaitEvent(stream, pp->copied_in[sl], 0)))
      return RR_ERR_CUDA;
    // fold the piece in place: elements [first, first + n) of the count-element AllReduce
    Checked pk = ck;
    pk.first = first;
    pk.n = n;
    pk.all_16b_aligned = true;  // slot buffers start on 512-byte multiples of a 16-byte aligned workspace
    st = launch_checked(pk, dev_in, dev_out, nullptr, stream);
    if (st != RR_OK) return st;
    if (!ok(cudaEventRecord(pp->folded[sl], stream)) || !ok(cudaStreamWaitEvent(pp->d2h, pp->folded[sl], 0)))
      return RR_ERR_CUDA;
    for (int r = 0; r < R; ++r)
      if (!ok(cudaMemcpyAsync(static_cast<unsigned char *>(host_out[r]) + first * E, slot + (size_t)r * piece * E,
                              n * E, cudaMemcpyDeviceToHost, pp->d2h)))
        return RR_ERR_CUDA;
    if (!ok(cudaEventRecord(pp->copied_out[sl], pp->d2h))) return RR_ERR_CUDA;
  }
  // work enqueued on `stream` after this call sees every output copied
  const int used = pieces < (size_t)kHostSlots ? (int)pieces : kHostSlots;
  for (int sl = 0; sl < used; ++sl)
    if (!ok(cudaStreamWaitEvent(stream, pp->copied_out[sl], 0))) return RR_ERR_CUDA;
  return RR_OK;
}

// --------------------------------------------------------------------------
// Staging memory for callers that cannot allocate: a fixed array in the
// library's own device image.  Host code only ever holds its address as
// returned by cudaGetSymbolAddress for the current device; the symbol itself
// is a host-side stand-in, not a device address.
// --------------------------------------------------------------------------

static __device__ __align__(256) unsigned char g_rr_static_scratch[RR_STATIC_SCRATCH_BYTES];

unsigned char *g_static_scratch_addr[kMaxDevices];
std::mutex g_static_scratch_mu;

// Once per device, with that device current: look up the array's device address.
rr_status static_scratch_for_current_device(unsigned char **out) {
  int dev = 0;
  if (!cuda_ok(cudaGetDevice(&dev)) || dev < 0 || dev >= kMaxDevices) return RR_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_static_scratch_mu);
  if (!g_static_scratch_addr[dev]) {
    void *addr = nullptr;
    if (!cuda_ok(cudaGetSymbolAddress(&addr, g_rr_static_scratch)) || !addr) return RR_ERR_CUDA;
    g_static_scratch_addr[dev] = static_cast<unsigned char *>(addr);
  }
  *out = g_static_scratch_addr[dev];
  return RR_OK;
}

}  // namespace

extern "C" {

rr_status ring_collective(rr_op op, const void *const *in_bufs, void *const *out_bufs, int R, size_t count,
                          rr_dtype dtype, rr_dtype wire, int group_size, const rr_launch_cfg *cfg,
                          cudaStream_t stream) {
  return run(op, in_bufs, out_bufs, R, count, dtype, wire, group_size, cfg, stream);
}

rr_status ring_allreduce(const void *const *in_bufs, void *const *out_bufs, int R, size_t count, rr_dtype dtype,
                         cudaStream_t stream) {
  return run(RR_OP_ALLREDUCE, in_bufs, out_bufs, R, count, dtype, dtype, 0, nullptr, stream);
}

rr_status ring_allreduce_ex(const void *const *in_bufs, void *const *out_bufs, int R, size_t count,
                            rr_dtype dtype, rr_dtype wire, int group_size, cudaStream_t stream) {
  return run(RR_OP_ALLREDUCE, in_bufs, out_bufs, R, count, dtype, wire, group_size, nullptr, stream);
}

rr_status ring_reduce_scatter(const void *const *in_bufs, void *const *out_bufs, int R, size_t count,
                              rr_dtype dtype, cudaStream_t stream) {
  return run(RR_OP_REDUCE_SCATTER, in_bufs, out_bufs, R, count, dtype, dtype, 0, nullptr, stream);
}

rr_status ring_reduce_scatter_ex(const void *const *in_bufs, void *const *out_bufs, int R, size_t count,
                                 rr_dtype dtype, rr_dtype wire, cudaStream_t stream) {
  return run(RR_OP_REDUCE_SCATTER, in_bufs, out_bufs, R, count, dtype, wire, 0, nullptr, stream);
}

rr_status ring_allgather(const void *const *in_bufs, void *const *out_bufs, int R, size_t count, rr_dtype dtype,
                         cudaStream_t stream) {
  return run(RR_OP_ALLGATHER, in_bufs, out_bufs, R, count, dtype, dtype, 0, nullptr, stream);
}

rr_status ring_plan(rr_op op, const void *const *in_bufs, void *const *out_bufs, int R, size_t count,
                    rr_dtype dtype, rr_dtype wire, int group_size, const rr_launch_cfg *cfg,
                    rr_launch_cfg *chosen) {
  if (!chosen) return RR_ERR_INVALID_ARG;
  Checked ck;
  rr_status st = check_args(op, in_bufs, out_bufs, R, count, dtype, wire, group_size, cfg, &ck);
  if (st != RR_OK) return st;
  *chosen = rr_launch_cfg{};
  chosen->path = RR_PATH_SIMPLE;
  if (count == 0) return RR_OK;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != RR_OK) return st;
  rr::RingParams p;
  rr::Launch l;
  st = plan(ck, in_bufs, out_bufs, cfg, dev, &p, &l);
  if (st != RR_OK) return st;
  export_plan(p, l, ck.E, cfg && cfg->beside_compute, chosen);
  return RR_OK;
}

rr_status ring_plan_device(rr_op op, int R, size_t count, rr_dtype dtype, rr_dtype wire, int group_size,
                           int buffers_16b_aligned, int sm_count, int smem_per_sm, int smem_per_block_optin,
                           const rr_launch_cfg *cfg, rr_launch_cfg *chosen, int *grid, size_t *smem_bytes) {
  if (!chosen || !grid || !smem_bytes) return RR_ERR_INVALID_ARG;
  Checked ck;
  rr_status st = check_scalars(op, R, count, dtype, wire, group_size, cfg, &ck);
  if (st != RR_OK) return st;
  if (count == 0) return RR_ERR_INVALID_ARG;
  ck.all_16b_aligned = buffers_16b_aligned != 0;
  rr::RingParams p = rr::RingParams{};
  rr::Launch l;
  st = plan_launch(ck, cfg, sm_count, smem_per_sm, smem_per_block_optin, &p, &l);
  if (st != RR_OK) return st;
  export_plan(p, l, ck.E, cfg && cfg->beside_compute, chosen);
  *grid = l.grid;
  *smem_bytes = l.smem;
  return RR_OK;
}

size_t ring_chunk_count(size_t count, int R, int c) {
  if (R < 1 || c < 0 || c >= R) return 0;
  return chunk_len(count, R, c);
}

size_t ring_chunk_offset(size_t count, int R, int c) {
  if (R < 1 || c < 0 || c >= R) return 0;
  return (size_t)c * (count / (size_t)R);
}

const char *ring_status_string(rr_status status) {
  switch (status) {
    case RR_OK:
      return "success";
    case RR_ERR_INVALID_ARG:
      return "invalid argument";
    case RR_ERR_UNSUPPORTED:
      return "unsupported dtype/wire combination or launch path";
    case RR_ERR_ALIAS:
      return "an output buffer overlaps another buffer";
    case RR_ERR_CUDA:
      return "CUDA runtime error";
    case RR_ERR_TIMEOUT:
      return "a bounded device-side wait timed out";
  }
  return "unknown status";
}

rr_status ring_device_status(unsigned int *flags) {
  if (!flags) return RR_ERR_INVALID_ARG;
  DeviceInfo dev;
  rr_status st = current_device(&dev);
  if (st != RR_OK) return st;
  unsigned int v = 0, zero = 0;
  if (!cuda_ok(cudaDeviceSynchronize())) return RR_ERR_CUDA;
  if (!cuda_ok(cudaMemcpyFromSymbol(&v, g_rr_status_word, sizeof(v)))) return RR_ERR_CUDA;
  if (v != 0 && !cuda_ok(cudaMemcpyToSymbol(g_rr_status_word, &zero, sizeof(zero)))) return RR_ERR_CUDA;
  *flags = v;
  return RR_OK;
}

rr_status ring_selftest_bounded_wait(unsigned long long limit_ns, cudaStream_t stream) {
  if (limit_ns < 1000ull || limit_ns > 10000000000ull) return RR_ERR_INVALID_ARG;
  DeviceInfo dev;
  rr_status st = current_device(&dev);
  if (st != RR_OK) return st;
  if (!cuda_ok(rr::launch_wait_probe(dev.status, limit_ns, stream))) return RR_ERR_CUDA;
  if (!cuda_ok(cudaStreamSynchronize(stream))) return RR_ERR_CUDA;
  unsigned int flags = 0;
  st = ring_device_status(&flags);
  if (st != RR_OK) return st;
  return (flags & rr::kStatusWaitTimeout) ? RR_ERR_TIMEOUT : RR_OK;
}

int ring_abi_version(void) { return RR_ABI_VERSION; }

int ring_debug_checks(void) {
#ifdef RR_DEBUG_CHECKS
  return 1;
#else
  return 0;
#endif
}

rr_status ring_debug_set_margin(size_t bytes) {
#ifdef RR_DEBUG_CHECKS
  g_debug_margin.store((unsigned long long)bytes, std::memory_order_relaxed);
  return RR_OK;
#else
  (void)bytes;
  return RR_ERR_UNSUPPORTED;
#endif
}

int ring_last_cuda_error(void) { return g_last_cuda_error; }

const char *ring_last_cuda_error_string(void) {
  return g_last_cuda_error ? cudaGetErrorString((cudaError_t)g_last_cuda_error) : "no CUDA error";
}

rr_status ring_allreduce_algo(const void *const *in_bufs, void *const *out_bufs, int R, size_t count, rr_dtype dtype,
                              rr_dtype wire, rr_algo algo, const rr_launch_cfg *cfg, cudaStream_t stream) {
  if (algo != RR_ALGO_RING && algo != RR_ALGO_HALVING_DOUBLING && algo != RR_ALGO_NAIVE) return RR_ERR_INVALID_ARG;
  Checked ck;
  rr_status st = check_scalars(RR_OP_ALLREDUCE, R, count, dtype, wire, 0, cfg, &ck);
  if (st != RR_OK) return st;
  ck.algo = algo;
  st = check_buffers(in_bufs, out_bufs, &ck);
  if (st != RR_OK || count == 0) return st;
  return launch_checked(ck, in_bufs, out_bufs, cfg, stream);
}

rr_status ring_allreduce_range(const void *const *in_bufs, void *const *out_bufs, int R, size_t count, size_t first,
                               size_t n, rr_dtype dtype, rr_dtype wire, int group_size, const rr_launch_cfg *cfg,
                               cudaStream_t stream) {
  Checked ck;
  rr_status st = check_scalars(RR_OP_ALLREDUCE, R, count, dtype, wire, group_size, cfg, &ck);
  if (st != RR_OK) return st;
  if (first > count || n > count - first) return RR_ERR_INVALID_ARG;
  ck.first = first;
  ck.n = n;
  st = check_buffers(in_bufs, out_bufs, &ck);
  if (st != RR_OK || n == 0) return st;
  return launch_checked(ck, in_bufs, out_bufs, cfg, stream);
}

size_t ring_allreduce_host_workspace(int R, size_t piece_count, rr_dtype dtype) {
  if (R < 1 || R > RR_MAX_RANKS || !valid_type(dtype) || piece_count == 0) return 0;
  const size_t piece = (piece_count + kPieceAlign - 1) / kPieceAlign * kPieceAlign;
  return (size_t)kHostSlots * (size_t)R * piece * elem_bytes(dtype);
}

rr_status ring_allreduce_host(const void *const *host_in, void *const *host_out, int R, size_t count,
                              rr_dtype dtype, rr_dtype wire, int group_size, void *dev_workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  return host_pipeline(host_in, host_out, R, count, dtype, wire, group_size, dev_workspace, workspace_bytes,
                       RR_HOST_COPIES_OVERLAP, stream);
}

rr_status ring_allreduce_host_ex(const void *const *host_in, void *const *host_out, int R, size_t count,
                                 rr_dtype dtype, rr_dtype wire, int group_size, void *dev_workspace,
                                 size_t workspace_bytes, rr_host_copies copy_mode, cudaStream_t stream) {
  if (copy_mode != RR_HOST_COPIES_OVERLAP && copy_mode != RR_HOST_COPIES_ONE_WAY) return RR_ERR_INVALID_ARG;
  return host_pipeline(host_in, host_out, R, count, dtype, wire, group_size, dev_workspace, workspace_bytes,
                       copy_mode, stream);
}

rr_status ring_allreduce_host_static(const void *const *host_in, void *const *host_out, int R, size_t count,
                                     rr_dtype dtype, rr_dtype wire, int group_size, size_t piece_count,
                                     cudaStream_t stream) {
  // size checks first: nothing is touched when the request does not fit
  if (R < 1 || R > RR_MAX_RANKS || !valid_type(dtype)) return RR_ERR_INVALID_ARG;
  const size_t per_slot_elem = (size_t)kHostSlots * (size_t)R * elem_bytes(dtype);
  const size_t largest = RR_STATIC_SCRATCH_BYTES / per_slot_elem / kPieceAlign * kPieceAlign;
  if (largest == 0 || piece_count > largest) return RR_ERR_INVALID_ARG;
  const size_t piece = piece_count == 0 ? largest : (piece_count + kPieceAlign - 1) / kPieceAlign * kPieceAlign;
  unsigned char *scratch = nullptr;
  rr_status st = static_scratch_for_current_device(&scratch);
  if (st != RR_OK) return st;
  // the pipeline never reads a slot it has not first filled, so nothing needs clearing
  return host_pipeline(host_in, host_out, R, count, dtype, wire, group_size, scratch, piece * per_slot_elem,
                       RR_HOST_COPIES_OVERLAP, stream);
}

}  // extern "C"
