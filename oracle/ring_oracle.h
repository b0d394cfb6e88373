/*
 * ring_oracle.h -- CPU oracle for the ring AllReduce / ReduceScatter / AllGather.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this code: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; the two agree only because both follow the same published
 * method.
 *
 * Sources (page address, section heading):
 *   [p3] ai6s.net/6a102b5410ee7a33f2746c06.html, "hcomm 与 HCCL 的关系" --
 *        HCCL's AllReduce is ReduceScatter followed by AllGather; the simplified
 *        ReduceScatter code: N-1 steps, at each step a rank sends one chunk to
 *        the next rank, receives one chunk from the previous rank and adds it
 *        element-wise; the chunk indices move back by one each step.
 *   [p5] hwcomputing.csdn.net/6a0dc11a10ee7a33f273f7fd.html, "Ring 通信为什么常见"
 *        -- the 4-card walkthrough: in step 1 card r sends block r to card r+1;
 *        after the reduce-scatter phase every card holds one fully summed
 *        block; the AllGather phase circulates the summed blocks; total traffic
 *        2(N-1)*S/N per card.
 *   [p2] ai6s.net/6a157e6510ee7a33f27553e9.html, "自定义通信模式" -- the chunk
 *        partition: floor(count/ranks) per chunk, the last chunk takes the rest.
 *   [p5] "大模型训练中的通信优化" -- gradients communicated in FP16; mixed
 *        FP16 / FP32 precision (read here both ways: binary32 values on a
 *        16-bit wire, and 16-bit values accumulated in binary32).
 *   [p5] "通信拓扑与带宽利用率" -- across nodes, one inter-node exchange per
 *        AllReduce (the two-level ring).
 *
 * Readings where the pages are silent or garbled (each one is tested):
 *   - the element-wise add goes into the RECEIVED chunk (the snippet's loop adds
 *     into the send chunk, but its own index updates and the walkthrough show the
 *     received chunk is the one that accumulates);
 *   - rounding is IEEE round-to-nearest-even; a hop on a 16-bit wire is the
 *     binary32 sum of the two operands rounded once to the wire format;
 *   - a standalone ReduceScatter leaves chunk r on output r (NCCL placement);
 *   - two-level: groups are contiguous (rank r is in group r / L), each group
 *     runs the flat ring with the chunk table of (count, L), the group partial
 *     sums of a chunk are folded in group order 0..G-1 by a chain of sends
 *     between the chunk's owners, and the total is sent back along the chain.
 *
 * Parity unpinned: the group order of the two-level fold when there are more
 * than two groups (the pages fix nothing there; with two groups every order
 * gives the same bits, which the tests check); the steps of halving-doubling
 * and the collector's order in the naive AllReduce (the pages name both
 * algorithms but give no steps; the readings are stated at
 * orc_allreduce_algo).
 *
 * Element storage: ORC_F32 elements are IEEE binary32; ORC_F16 and ORC_BF16
 * elements are 16-bit encodings held in uint16_t.
 */
#ifndef RING_ORACLE_H
#define RING_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

enum {
  ORC_OK = 0,
  ORC_EINVAL = 1,       /* bad R, group size, null pointer */
  ORC_EUNSUPPORTED = 2, /* (storage, wire) pair not supported */
  ORC_ENOMEM = 3,
  ORC_EPROTO = 4,       /* a message arrived twice or with the wrong chunk */
  ORC_ETIMEOUT = 5      /* a receive found no message within its poll limit */
};

/* Phases of a message in the trace.  ORC_PHASE_RS / ORC_PHASE_AG are the
 * reduce and distribute halves of every algorithm; PRE / POST are the folding
 * of the extra ranks of halving-doubling when R is not a power of two. */
enum {
  ORC_PHASE_RS = 0,
  ORC_PHASE_XCHG = 1,
  ORC_PHASE_XBCAST = 2,
  ORC_PHASE_AG = 3,
  ORC_PHASE_PRE = 4,
  ORC_PHASE_POST = 5
};

/* AllReduce algorithms (page ai6s.net/6a0dd5b5662f9a54cb75ef90.html, the
 * topology switch of TpAllReduceOp::Execute: ring for a ring topology,
 * halving-doubling with logarithmic steps for a full mesh, naive Reduce +
 * Broadcast otherwise; page hwcomputing.csdn.net/6a0dc11a..., section
 * "为什么大模型训练离不开通信": without a library every card sends its
 * gradients to a collector, which adds them and sends the sum back). */
enum { ORC_ALGO_RING = 0, ORC_ALGO_HALVING_DOUBLING = 1, ORC_ALGO_NAIVE = 2 };

/* One simulated message. */
typedef struct {
  int32_t phase, step, src, dst, chunk;
  int32_t pad;
  uint64_t bytes;
} orc_msg;

/* Host-side fault injection into the simulated transport. */
enum { ORC_FAULT_NONE = 0, ORC_FAULT_DROP = 1, ORC_FAULT_DUP = 2, ORC_FAULT_SILENT = 3 };
typedef struct {
  int32_t kind;  /* ORC_FAULT_* */
  int32_t rank;  /* the sending rank the fault applies to */
  int32_t phase; /* ORC_PHASE_* of the affected send (SILENT: from this phase on) */
  int32_t step;  /* step of the affected send (SILENT: from this step on) */
} orc_fault;

/* Optional outputs and fault injection of one simulated collective. */
typedef struct {
  uint64_t *sent_bytes; /* [R] bytes each rank sent, or NULL */
  orc_msg *trace;       /* message log, or NULL */
  size_t trace_cap;     /* capacity of trace */
  size_t trace_len;     /* out: messages logged (may exceed trace_cap) */
  orc_fault fault;      /* kind = ORC_FAULT_NONE for a clean run */
  int32_t poll_limit;   /* receive polls before ORC_ETIMEOUT (<= 0: 16) */
} orc_opts;

/* IEEE 754 encodings, round-to-nearest-even, subnormals kept. */
uint16_t orc_f32_to_f16(float x);
uint16_t orc_f32_to_bf16(float x);
float orc_f16_to_f32(uint16_t h);
float orc_bf16_to_f32(uint16_t b);
/* One ring hop on the wire: a + b rounded to `wire`; operands and result are
 * encodings (binary32 bits for ORC_F32). */
uint32_t orc_wire_add(int wire, uint32_t a, uint32_t b);
/* Batch conversions (for the tests). */
void orc_f32_to_wire_batch(int wire, const float *x, uint16_t *out, size_t n);
void orc_wire_add_batch(int wire, const uint16_t *a, const uint16_t *b, uint16_t *out, size_t n);

/* Chunk table of the partition of `count` elements into R chunks. */
size_t orc_chunk_len(size_t count, int R, int c);
size_t orc_chunk_off(size_t count, int R, int c);

/*
 * AllReduce over R simulated ranks: in[r] and out[r] hold `count` elements of
 * `dtype`; values travel and are summed in `wire`.  group_size L (0 = R) splits
 * the ranks into R/L contiguous groups (the two-level ring).  out[r] may equal
 * in[r].  Returns ORC_OK or an error code; opts may be NULL.
 */
int orc_allreduce(const void *const *in, void *const *out, int R, size_t count, int dtype,
                  int wire, int group_size, orc_opts *opts);

/* ReduceScatter: in[r] has `count` elements, out[r] receives chunk r
 * (orc_chunk_len(count, R, r) elements). */
int orc_reduce_scatter(const void *const *in, void *const *out, int R, size_t count, int dtype,
                       int wire, orc_opts *opts);

/* AllGather: in[c] holds chunk c (orc_chunk_len(count, R, c) elements), every
 * out[r] receives all `count` elements. */
int orc_allgather(const void *const *in, void *const *out, int R, size_t count, int dtype,
                  orc_opts *opts);

/*
 * AllReduce by algorithm (flat: one group).  ORC_ALGO_RING is orc_allreduce.
 * ORC_ALGO_NAIVE: ranks 1..R-1 send their vectors to rank 0 in rank order,
 * rank 0 adds each as it arrives (((x0 + x1) + x2) + ...), then sends the sum
 * to ranks 1..R-1.
 * ORC_ALGO_HALVING_DOUBLING (reading: the textbook recursive-halving
 * reduce-scatter and recursive-doubling allgather, the pages give no steps):
 * with P the largest power of two <= R and E = R - P, rank 2k (k < E) first
 * sends its vector to rank 2k+1, which adds it; the remaining P ranks (virtual
 * rank v is rank 2v+1 for v < E, rank v+E otherwise) split the vector into P
 * blocks (the chunk table of (count, P)); at step t = 0..log2(P)-1, virtual
 * ranks v and v ^ (P >> (t+1)) swap halves of their current block range, the
 * lower rank keeping the lower half, and each adds the half it keeps; the
 * allgather reverses the steps with copies; rank 2k+1 finally sends the result
 * to rank 2k.
 */
int orc_allreduce_algo(const void *const *in, void *const *out, int R, size_t count, int dtype, int wire,
                       int algo, orc_opts *opts);

/*
 * AllGather by schedule (in/out as orc_allgather; every schedule delivers the
 * same copies, only the messages differ).  ORC_ALGO_RING is orc_allgather.
 * ORC_ALGO_NAIVE (gather, then broadcast): ranks 1..R-1 send their chunks to
 * rank 0 in rank order, then rank 0 sends the whole vector to ranks 1..R-1.
 * ORC_ALGO_HALVING_DOUBLING (the tree AllGather, recursive doubling; reading:
 * the textbook schedule, the pages give no steps): with P the largest power
 * of two <= R and E = R - P, rank 2k (k < E) first sends its chunk to rank
 * 2k+1; virtual rank v (rank 2v+1 for v < E, rank v+E otherwise) then holds
 * a contiguous run of chunks, and at step t = 0..log2(P)-1 virtual ranks v and
 * v ^ 2^t swap everything they hold; rank 2k+1 finally sends the whole vector
 * to rank 2k.
 */
int orc_allgather_algo(const void *const *in, void *const *out, int R, size_t count, int dtype, int algo,
                       orc_opts *opts);

/* Closed form of orc_allreduce_algo at sampled elements (as orc_fold_gathered). */
int orc_fold_gathered_algo(const void *const *vals, const uint64_t *idx, size_t n, int R, size_t count,
                           int dtype, int wire, int algo, void *out);

/*
 * Closed form of the AllReduce result, one element at a time, for sampled
 * checks: vals[r][k] is rank r's input at global element index idx[k] (of a
 * `count`-element vector); out[k] receives the AllReduce result there.
 */
int orc_fold_gathered(const void *const *vals, const uint64_t *idx, size_t n, int R, size_t count,
                      int dtype, int wire, int group_size, void *out);

#ifdef __cplusplus
}
#endif
#endif
