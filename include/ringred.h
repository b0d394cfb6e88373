/*
 * ringred.h -- C ABI of libringred.
 *
 * libringred computes the ring AllReduce, ReduceScatter and AllGather of R
 * "ranks" whose buffers all live in the memory of one GPU.  It reproduces the
 * data semantics of the ring collective described on these pages:
 *
 *   [p3] ai6s.net/6a102b5410ee7a33f2746c06.html, section "hcomm 与 HCCL 的关系":
 *        AllReduce = ReduceScatter + AllGather; the ReduceScatter runs N-1 steps
 *        in which every rank passes one chunk to the next rank, which adds it
 *        element-wise to its own copy of that chunk.
 *   [p5] hwcomputing.csdn.net/6a0dc11a10ee7a33f273f7fd.html, section
 *        "Ring 通信为什么常见": block c starts on card c and is passed around
 *        the ring; after the reduce-scatter phase each card holds one summed
 *        block, and the AllGather phase hands the summed blocks to all cards.
 *   [p2] ai6s.net/6a157e6510ee7a33f27553e9.html, section "自定义通信模式":
 *        chunk c has floor(count / R) elements, the last chunk takes the rest.
 *   [p5] section "大模型训练中的通信优化": gradients travel in FP16.
 *   [p5] section "通信拓扑与带宽利用率": one exchange between nodes per
 *        AllReduce (the two-level ring).
 *
 * Result, element by element.  With L ranks per group (L = R for the flat
 * ring), G = R / L groups, and c = the chunk of element i in the partition of
 * `count` into L chunks:
 *     S_g[i] = x_{gL+c}[i] (+) x_{gL+c+1}[i] (+) ... (+) x_{gL+c+L-1}[i]
 *              (ranks taken mod L inside group g, folded left to right)
 *     y[i]   = S_0[i] (+) S_1[i] (+) ... (+) S_{G-1}[i]
 * where (+) is one hop: the binary32 sum of its two operands rounded once to
 * the wire format (round to nearest even; no fused multiply-add; subnormals
 * kept).  With a binary32 wire the hop is the binary32 addition.  On a 16-bit
 * wire with binary32 storage, every input is first rounded to the wire format
 * and the result is widened back exactly; with 16-bit storage on a binary32
 * wire, every input is widened exactly and the result rounded once.  The
 * result is the same on every
 * GPU and every launch configuration: it depends only on the inputs, R, L,
 * count and the formats.
 *
 * Common rules for every collective below:
 *   - in_bufs and out_bufs are HOST arrays of R DEVICE pointers (current
 *     device).  The library reads the arrays during the call only.
 *   - The caller owns every buffer and the stream.  The library allocates no
 *     memory and keeps no pointer after the call returns (ring_allreduce_host
 *     creates two streams and ten events per device on first use and keeps
 *     them until exit).
 *   - The call is asynchronous: it validates its arguments, enqueues work on
 *     `stream` and returns.  Errors of the enqueued work surface when the
 *     caller synchronizes the stream; a bounded wait inside a kernel that gave
 *     up is recorded in the device status word (ring_device_status).
 *   - Argument errors are detected before anything is enqueued and return
 *     RR_ERR_INVALID_ARG / RR_ERR_UNSUPPORTED / RR_ERR_ALIAS; nothing is
 *     written then.  A failed launch returns RR_ERR_CUDA (and
 *     ring_last_cuda_error names the runtime error).
 *   - Kernels are launched with programmatic stream serialisation by default
 *     (rr_launch_cfg.early_launch): a launch may be scheduled while the kernel
 *     before it on the stream runs, but every kernel waits for that kernel's
 *     completion and writes before touching memory, so stream order holds.
 *   - count == 0 returns RR_OK and enqueues nothing.  A buffer of zero
 *     elements may be NULL.  Every other buffer must be non-NULL and aligned
 *     to its element size; 16-byte aligned buffers take the fast path.
 *   - A buffer written by the call (an output) must not overlap any other
 *     buffer, with one exception: ring_allreduce* accepts out_bufs[r] ==
 *     in_bufs[r] (in place).  Inputs may overlap one another.
 *   - 1 <= R <= RR_MAX_RANKS.
 * Layout (speed only): the kernels access element i of every rank's vector
 * at about the same time.  Vectors whose start addresses agree modulo a large
 * power of two (separate allocations of one power-of-two size, rows of an
 * unpadded [R][N] array) then load the same memory channels together; the
 * R = 8, 512 MiB AllReduce measured about 2 % slower on them than on vectors
 * staggered by 1-17 MiB (the Python binding's rank_buffers lays them out so).
 */
#ifndef RINGRED_H
#define RINGRED_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's stream handle (the same declaration as the runtime's). */
typedef struct CUstream_st *cudaStream_t;

#define RR_MAX_RANKS 64
#define RR_ABI_VERSION 3

typedef enum { RR_FP32 = 0, RR_FP16 = 1, RR_BF16 = 2 } rr_dtype;

typedef enum {
  RR_OK = 0,
  RR_ERR_INVALID_ARG = 1, /* bad R, count, group size, NULL or misaligned pointer */
  RR_ERR_UNSUPPORTED = 2, /* (storage, wire) pair or forced path not available */
  RR_ERR_ALIAS = 3,       /* an output overlaps another buffer */
  RR_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  RR_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up */
} rr_status;

typedef enum { RR_OP_ALLREDUCE = 0, RR_OP_REDUCE_SCATTER = 1, RR_OP_ALLGATHER = 2 } rr_op;

/*
 * ring_allreduce -- [p3] AllReduce = ReduceScatter + AllGather; [p5] ring walkthrough.
 * in_bufs[r], out_bufs[r]: `count` elements of `dtype` each.  Every out_bufs[r]
 * receives y (above) with L = R and the wire format equal to `dtype`.
 */
rr_status ring_allreduce(const void *const *in_bufs, void *const *out_bufs, int R, size_t count,
                         rr_dtype dtype, cudaStream_t stream);

/*
 * ring_allreduce_ex -- ring_allreduce with a wire format and a two-level ring.
 * wire: the storage type itself; a 16-bit wire under RR_FP32 storage ([p5]
 *   FP16 communication: inputs rounded to the wire, every hop rounded); or
 *   RR_FP32 under 16-bit storage ([p5] FP16/FP32 mixed precision: inputs
 *   widened exactly, hops in binary32, one rounding to the storage format at
 *   the end).  Supported (dtype, wire): (FP32,FP32) (FP16,FP16) (BF16,BF16)
 *   (FP32,BF16) (FP32,FP16) (FP16,FP32) (BF16,FP32).
 * group_size: L, ranks per group ([p5] "通信拓扑与带宽利用率"); 0 or R = the
 *   flat ring; otherwise L must divide R, and group g holds ranks gL..gL+L-1.
 */
rr_status ring_allreduce_ex(const void *const *in_bufs, void *const *out_bufs, int R, size_t count,
                            rr_dtype dtype, rr_dtype wire, int group_size, cudaStream_t stream);

/*
 * ring_reduce_scatter -- [p3] the simplified ReduceScatter code.
 * in_bufs[r]: `count` elements.  out_bufs[r]: ring_chunk_count(count, R, r)
 * elements, receiving chunk r of y (the NCCL placement: rank r gets chunk r).
 * count is the full per-rank input length, not the per-rank output length.
 */
rr_status ring_reduce_scatter(const void *const *in_bufs, void *const *out_bufs, int R,
                              size_t count, rr_dtype dtype, cudaStream_t stream);

/* ring_reduce_scatter_ex -- ring_reduce_scatter with a wire format (pairs as above). */
rr_status ring_reduce_scatter_ex(const void *const *in_bufs, void *const *out_bufs, int R,
                                 size_t count, rr_dtype dtype, rr_dtype wire, cudaStream_t stream);

/*
 * ring_allgather -- [p5] the AllGather phase; [p3] "分布式推理中的通信".
 * in_bufs[c]: ring_chunk_count(count, R, c) elements (chunk c).  out_bufs[r]:
 * `count` elements; every output receives all chunks in order:
 *   out_bufs[r][ring_chunk_offset(count, R, c) + j] = in_bufs[c][j].
 * Every AllGather schedule on the pages (the ring, the tree of recursive
 * doubling, gather to one rank then broadcast) delivers exactly these copies;
 * with all ranks in one GPU's memory the kernel is the copy itself, so this
 * one entry point stands for all of them.
 */
rr_status ring_allgather(const void *const *in_bufs, void *const *out_bufs, int R, size_t count,
                         rr_dtype dtype, cudaStream_t stream);

/* Launch paths: RR_PATH_BULK stages tiles through shared memory with bulk
 * asynchronous copies (needs 16-byte aligned buffers, and for ReduceScatter /
 * AllGather chunk offsets that are multiples of 16 bytes); RR_PATH_DIRECT has
 * every thread load its ranks' 16-byte vectors straight from global memory
 * and store the results straight back (16-byte aligned buffers, at most 256
 * threads per CTA; chunk offsets off the 16-byte grid are handled by building
 * each vector from two aligned loads, chunk by chunk in rows of vectors, the
 * form larger calls over few ranks also take); RR_PATH_SIMPLE is one element per
 * thread with plain loads and stores (any alignment). */
typedef enum { RR_PATH_AUTO = 0, RR_PATH_BULK = 1, RR_PATH_SIMPLE = 2, RR_PATH_DIRECT = 3 } rr_path;

/* Optional launch configuration; zero fields mean "choose automatically".
 * A configuration never changes the result, only the speed. */
typedef struct {
  int path;        /* rr_path */
  int tile_bytes;  /* bulk path: bytes per rank per tile, a multiple of 16 */
  int stages;      /* bulk path: tiles in flight per CTA, 2..16 */
  int ctas_per_sm; /* bulk path: 1..4.  Direct path: 2 or 3, the 256-thread
                      CTAs per SM its registers are budgeted for (3: at most
                      85 registers a thread, more CTAs resident).  A value
                      the direct kernel is not built for is ignored, or
                      RR_ERR_UNSUPPORTED when path is RR_PATH_DIRECT. */
  int threads;     /* threads per CTA: 64..1024, a multiple of 32 */
  int max_ctas;    /* at most this many CTAs (0: no limit); a chunked AllReduce
                      that runs beside compute kernels can leave them SMs.
                      With fewer CTAs than 3 per SM and no stages / CTAs-per-SM
                      given, each CTA takes a whole SM with larger tiles. */
  int early_launch; /* 0: the library's choice; 1: the kernel may be scheduled
                      while the previous kernel on the stream is still
                      running (programmatic dependent launch: it waits for that
                      kernel's completion and writes before touching memory);
                      2: plain stream order. */
  int vectors;     /* direct path: 16-byte vectors a thread takes at once,
                      1..4 (AllGather 1, 2 or 4; 16-bit storage summed in
                      binary32 1 or 2); where the direct path works chunk by
                      chunk (chunk boundaries off the 16-byte grid; on it,
                      AllGather from 12 MiB per rank, two-rank ReduceScatter
                      from 32 MiB and AllReduce over two to four ranks from
                      16 MiB, unless ctas_per_sm is given or vectors is not a
                      row count below), rows of 31-32 vectors a warp takes at
                      once (ReduceScatter 1..4, AllGather 1, 2 or 4,
                      AllReduce 2 or 4; 16-bit storage summed in binary32: 1
                      or 2, AllReduce none).  A value outside these is
                      RR_ERR_UNSUPPORTED. */
  int beside_compute; /* 1: the call runs beside compute kernels on other
                      streams; unless max_ctas is given, the grid is capped at
                      RR_BESIDE_COMPUTE_SM_EIGHTHS eighths of the SMs (one CTA each),
                      leaving the rest to the compute.  0: the whole GPU. */
  int prefetch;    /* direct path, L2 prefetch of the inputs: 0 the library's
                      choice (by message size and ranks); 1 none; 2 each
                      thread's first vectors before the wait for the previous
                      kernel (safe: a prefetch never changes what is read after
                      the wait); 3 the next iteration's vectors while the
                      current ones load; 4 both.  Ignored by the halving-
                      doubling order. */
} rr_launch_cfg;

/* Share of the SMs (numerator / 8) a call with beside_compute = 1 takes
 * (measured: eight binary16 GEMMs of 8192^3 with the ranges of a 512 MiB
 * eight-rank AllReduce between them took least time together at 7/8). */
#define RR_BESIDE_COMPUTE_SM_EIGHTHS 7

/*
 * ring_collective -- every collective through one entry point with an
 * explicit launch configuration (cfg may be NULL).  op selects the
 * collective; buffer layouts are those of the named entry points; wire and
 * group_size as for ring_allreduce_ex (ReduceScatter: group_size 0 or R;
 * AllGather: wire == dtype, group_size 0 or R).  The launch configuration
 * never changes the result, only the speed.  A forced RR_PATH_BULK that the
 * buffers do not allow returns RR_ERR_UNSUPPORTED.
 */
rr_status ring_collective(rr_op op, const void *const *in_bufs, void *const *out_bufs, int R,
                          size_t count, rr_dtype dtype, rr_dtype wire, int group_size,
                          const rr_launch_cfg *cfg, cudaStream_t stream);

/* AllReduce algorithms: the summation order of the result. */
typedef enum { RR_ALGO_RING = 0, RR_ALGO_HALVING_DOUBLING = 1, RR_ALGO_NAIVE = 2 } rr_algo;

/*
 * ring_allreduce_algo -- the AllReduce of another algorithm on the topology
 * switch of the page ai6s.net/6a0dd5b5662f9a54cb75ef90.html
 * (TpAllReduceOp::Execute): same buffers, same bytes moved, a different
 * summation order and so different bits.
 *   RR_ALGO_RING: ring_allreduce_ex with group_size 0.
 *   RR_ALGO_NAIVE (Reduce + Broadcast; the collector of the page
 *     hwcomputing.csdn.net/6a0dc11a10ee7a33f273f7fd.html, section
 *     "为什么大模型训练离不开通信"): y = ((x_0 (+) x_1) (+) x_2) ... (+) x_{R-1}.
 *   RR_ALGO_HALVING_DOUBLING (full mesh, logarithmic steps; the pages give
 *     no steps, the textbook recursive-halving / recursive-doubling algorithm
 *     is taken): with P the largest power of two <= R and E = R - P, leaves
 *     L_v = x_{2v} (+) x_{2v+1} for v < E and x_{v+E} otherwise, then
 *     L_v = L_v (+) L_{v+d} for d = P/2, P/4, ..., 1; y = L_0.
 * Arguments as for ring_allreduce_ex without group_size (flat ranks only);
 * cfg as for ring_collective.
 */
rr_status ring_allreduce_algo(const void *const *in_bufs, void *const *out_bufs, int R, size_t count,
                              rr_dtype dtype, rr_dtype wire, rr_algo algo, const rr_launch_cfg *cfg,
                              cudaStream_t stream);

/*
 * ring_allreduce_range -- elements [first, first + n) of the AllReduce of
 * count-element rank vectors: the building block of a chunked AllReduce that
 * overlaps compute (page bjdmk.com.cn/news/5966809, sections 4.2-4.3: the big
 * tensor is cut into pieces and each piece is reduced on a communication
 * stream as soon as it is ready).
 * in_bufs[r], out_bufs[r]: n elements each, holding elements first .. first+n-1
 * of rank r's vector (out_bufs[r] == in_bufs[r] allowed).  Every element is
 * reduced exactly as ring_allreduce_ex would reduce it: its chunk (hence its
 * start rank) comes from its global index in the count-element vector, so
 * any split of [0, count) into ranges gives the same bits as one call.
 * Requires first + n <= count.  group_size, wire and cfg as for
 * ring_collective.
 */
rr_status ring_allreduce_range(const void *const *in_bufs, void *const *out_bufs, int R, size_t count,
                               size_t first, size_t n, rr_dtype dtype, rr_dtype wire, int group_size,
                               const rr_launch_cfg *cfg, cudaStream_t stream);

/*
 * ring_allreduce_host -- the AllReduce of vectors held in HOST memory
 * (host_in[r], host_out[r]: `count` elements each; host_out[r] == host_in[r]
 * allowed; page-locked memory lets the copies overlap).  The vectors stream
 * through the caller's device workspace in pieces: while piece k is reduced
 * on `stream`, piece k+1 is copied in and piece k-1 copied out on two
 * internal streams (created once per device, with their events), the
 * pipelining of page bjdmk.com.cn/news/5966809, section 4.3.
 * dev_workspace: device memory, 16-byte aligned, workspace_bytes long, used
 * by this call until `stream` reaches the point where the call returns; the
 * piece length is the largest multiple of 256 elements whose three slots of R
 * pieces fit (ring_allreduce_host_workspace gives the size for a piece
 * length).  The result equals ring_allreduce_ex on device copies, bit for
 * bit.  Work enqueued on `stream` after the call sees host_out complete.
 * Calls from several host threads on one device are serialised.
 * Errors: as above; RR_ERR_INVALID_ARG if the workspace cannot hold 256
 * elements per slot; RR_ERR_ALIAS if it overlaps a host buffer.
 */
rr_status ring_allreduce_host(const void *const *host_in, void *const *host_out, int R, size_t count,
                              rr_dtype dtype, rr_dtype wire, int group_size, void *dev_workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/* How ring_allreduce_host_ex schedules its copies.  OVERLAP (what
 * ring_allreduce_host does): piece k+1 is copied in while piece k-1 is copied
 * out, so the host link carries both directions at once.  ONE_WAY: both
 * directions take turns on one internal stream (copy-in k+1, copy-out k) and
 * only the reduction overlaps them.  Which is faster depends on the machine:
 * on one GB300 node 4 GiB each way took 25 ms with both directions at once,
 * on others 58-104 ms, against 42.5 ms one after the other; time both on the
 * caller's own buffers and keep the faster. */
typedef enum { RR_HOST_COPIES_OVERLAP = 0, RR_HOST_COPIES_ONE_WAY = 1 } rr_host_copies;

/*
 * ring_allreduce_host_ex -- ring_allreduce_host with the copy schedule
 * chosen by the caller (copy_mode, above).  Same arguments, result, ordering
 * and errors otherwise; an unknown copy_mode is RR_ERR_INVALID_ARG.
 */
rr_status ring_allreduce_host_ex(const void *const *host_in, void *const *host_out, int R, size_t count,
                                 rr_dtype dtype, rr_dtype wire, int group_size, void *dev_workspace,
                                 size_t workspace_bytes, rr_host_copies copy_mode, cudaStream_t stream);

/* Workspace bytes ring_allreduce_host needs for pieces of piece_count
 * elements (rounded up to 256); 0 for invalid arguments. */
size_t ring_allreduce_host_workspace(int R, size_t piece_count, rr_dtype dtype);

/* Size of the staging array that ring_allreduce_host_static uses instead of a
 * caller workspace: 32 MiB, held on every GPU that loads the library until the
 * process exits. */
#define RR_STATIC_SCRATCH_BYTES (32u << 20)

/*
 * ring_allreduce_host_static -- ring_allreduce_host without a workspace
 * argument, for callers that cannot hand the library device memory: plugin
 * code whose host program's allocator owns all device memory and offers no
 * raw buffer, or a path that must not risk an allocation failing or blocking
 * at run time.  The pages have no counterpart; it exists for such callers.
 * It allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * routine.  The pieces go through RR_STATIC_SCRATCH_BYTES of device memory
 * compiled into the library.  The first call on a device looks up that
 * memory's device address (cudaGetSymbolAddress, with the device current) and
 * creates the two internal streams and ten events of the pipelined copies;
 * make that first call before any stream capture.
 * host_in, host_out, R, count, dtype, wire, group_size, stream: as for
 * ring_allreduce_host, with the same result bit for bit.  piece_count:
 * elements per rank per piece, rounded up to 256; 0 picks the largest that
 * fits.  A piece whose three slots of R pieces would exceed
 * RR_STATIC_SCRATCH_BYTES is rejected with RR_ERR_INVALID_ARG before any CUDA
 * call; the message length itself is not limited.
 * Every call on a device shares the one array and leaves its last contents in
 * it; nothing in it needs to start at zero, since a slot is always filled
 * before it is read.  The library chains its own calls through per-device
 * events and a lock so their pieces take turns in the array; GPU work that
 * overlapped one of these calls while using the array would race with it.
 */
rr_status ring_allreduce_host_static(const void *const *host_in, void *const *host_out, int R, size_t count,
                                     rr_dtype dtype, rr_dtype wire, int group_size, size_t piece_count,
                                     cudaStream_t stream);

/*
 * ring_plan -- the launch configuration ring_collective would use for these
 * arguments (after validation; nothing is enqueued).  *chosen receives the
 * path and the resolved tile / stage / CTA-per-SM / thread counts (0 where
 * the path has none), max_ctas = the grid's CTA count, and early_launch = 1
 * (programmatic launch) or 2 (plain stream order).
 */
rr_status ring_plan(rr_op op, const void *const *in_bufs, void *const *out_bufs, int R,
                    size_t count, rr_dtype dtype, rr_dtype wire, int group_size,
                    const rr_launch_cfg *cfg, rr_launch_cfg *chosen);

/*
 * ring_plan_device -- the planner of ring_collective for a described device
 * instead of the current one: sm_count SMs, smem_per_sm bytes of shared
 * memory per SM, smem_per_block_optin bytes per CTA at most, and buffers that
 * are (buffers_16b_aligned != 0) or are not all 16-byte aligned.  Pure host
 * computation, no CUDA call.  *chosen as for ring_plan; *grid receives the
 * CTA count and *smem_bytes the dynamic shared memory of one CTA.  count must
 * be positive.
 */
rr_status ring_plan_device(rr_op op, int R, size_t count, rr_dtype dtype, rr_dtype wire, int group_size,
                           int buffers_16b_aligned, int sm_count, int smem_per_sm, int smem_per_block_optin,
                           const rr_launch_cfg *cfg, rr_launch_cfg *chosen, int *grid, size_t *smem_bytes);

/* [p2] chunk table: length and offset of chunk c of `count` elements split
 * over R ranks (0 when R < 1 or c is out of range). */
size_t ring_chunk_count(size_t count, int R, int c);
size_t ring_chunk_offset(size_t count, int R, int c);

/* A static English description of a status code. */
const char *ring_status_string(rr_status status);

/*
 * ring_device_status -- reads and clears the current device's sticky status
 * word.  Bit 0 set: a bounded wait inside a kernel gave up (its collective
 * did not complete).  Synchronizes the current device first.  Returns RR_OK,
 * or RR_ERR_CUDA if the CUDA runtime reported an error.
 */
rr_status ring_device_status(unsigned int *flags);

/*
 * ring_selftest_bounded_wait -- launches one CTA that waits on a shared-memory
 * barrier no one completes, with a limit of limit_ns nanoseconds (1e3..1e10),
 * then synchronizes `stream`.  Returns RR_ERR_TIMEOUT when the wait gave up and
 * set the status bit (the expected outcome, which the call then clears), RR_OK
 * if it did not, RR_ERR_CUDA on a runtime error.  It exercises the bounded
 * wait that every pipelined kernel in the library uses.
 */
rr_status ring_selftest_bounded_wait(unsigned long long limit_ns, cudaStream_t stream);

/*
 * Debug builds.  The library can be built with device-side bounds checks
 * (the build script's debug mode, -DRR_DEBUG_CHECKS): every load, store,
 * bulk copy and prefetch a kernel makes of a rank buffer is checked against
 * that buffer's extent in the launch (count elements, or one chunk for a
 * ReduceScatter output / AllGather input).  An access outside is skipped
 * instead of made, and bit 1 (value 2) of the device status word is set
 * (ring_device_status); nothing faults.  Results are otherwise bit-identical.
 * ring_debug_checks returns 1 for such a build, 0 for a release build.
 * ring_debug_set_margin(bytes) makes the checks treat every buffer as `bytes`
 * shorter than it is (process-wide, for later launches), so a test can see
 * the checks fire on accesses that are in fact valid; 0 restores the true
 * extents.  A release build returns RR_ERR_UNSUPPORTED.
 */
int ring_debug_checks(void);
rr_status ring_debug_set_margin(size_t bytes);

/* RR_ABI_VERSION of the library. */
int ring_abi_version(void);

/*
 * The CUDA runtime error (a cudaError_t value) behind the calling thread's
 * most recent RR_ERR_CUDA, or 0 if it has had none, and the runtime's
 * description of it ("no CUDA error" for 0; a static string).
 */
int ring_last_cuda_error(void);
const char *ring_last_cuda_error_string(void);

#ifdef __cplusplus
}
#endif
#endif /* RINGRED_H */
