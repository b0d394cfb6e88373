/*
 * ring_oracle.c -- CPU oracle for the ring AllReduce / ReduceScatter / AllGather.
 *
 * TEST INFRASTRUCTURE ONLY: see ring_oracle.h for who may use it, the sources
 * it follows and the readings it takes.  Single-threaded, plain C11, compiled
 * without fast-math and with FP contraction off, so every `+` below is one
 * IEEE binary32 addition.
 *
 * The collectives are simulated literally: every rank owns a work buffer in
 * the wire format and a one-message mailbox; each step first performs every
 * rank's send (a copy of one chunk into the next rank's mailbox), then every
 * rank's receive (the received chunk is added into, or copied over, the same
 * chunk of its own buffer).  orc_fold_gathered is an independent closed form
 * of the same result, used to pin the simulation and for sampled checks of
 * large runs.
 */
#include "ring_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 and bfloat16, from the format definitions.              */
/* ------------------------------------------------------------------------ */

typedef struct {
  int p;     /* significand bits including the hidden bit */
  int emin;  /* exponent of the smallest normal */
  int emax;  /* exponent of the largest finite (= the bias) */
  int mbits; /* stored fraction bits */
  int ebits; /* exponent field bits */
} narrow_fmt;

static const narrow_fmt FMT_F16 = {11, -14, 15, 10, 5};
static const narrow_fmt FMT_BF16 = {8, -126, 127, 7, 8};

static uint32_t f32_bits(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  return u;
}

static float bits_f32(uint32_t u) {
  float x;
  memcpy(&x, &u, 4);
  return x;
}

/* Round the binary32 value x to the nearest value of the narrow format, ties
 * to even, and return that value's encoding. */
static uint16_t round_to_narrow(float x, const narrow_fmt *f) {
  uint32_t u = f32_bits(x);
  uint32_t sign = (u >> 31) << 15;
  uint32_t E = (u >> 23) & 0xffu;
  uint32_t frac = u & 0x7fffffu;
  uint32_t exp_all_ones = ((1u << f->ebits) - 1u) << f->mbits;

  if (E == 0xffu) {
    if (frac == 0) return (uint16_t)(sign | exp_all_ones); /* infinity */
    /* NaN: stays a quiet NaN, keeping the top payload bits */
    return (uint16_t)(sign | exp_all_ones | (1u << (f->mbits - 1)) | (frac >> (23 - f->mbits)));
  }
  if (E == 0 && frac == 0) return (uint16_t)sign; /* signed zero */

  /* |x| = m * 2^q exactly, with m an integer */
  uint32_t m;
  int q;
  if (E == 0) {
    m = frac;
    q = -149;
  } else {
    m = frac | 0x800000u;
    q = (int)E - 150;
  }
  int msb = 0; /* 2^msb <= m < 2^(msb+1) */
  while ((m >> (msb + 1)) != 0) msb++;
  int e = q + msb;                                      /* floor(log2 |x|) */
  int Q = (e > f->emin ? e : f->emin) - (f->p - 1);     /* exponent of one unit in the last place */

  uint64_t M; /* |x| / 2^Q rounded to an integer, ties to even */
  if (q >= Q) {
    M = (uint64_t)m << (q - Q);
  } else {
    int d = Q - q;
    if (d > 40) {
      M = 0;
    } else {
      uint64_t mm = m;
      uint64_t rem = mm & ((1ull << d) - 1ull);
      uint64_t half = 1ull << (d - 1);
      M = mm >> d;
      if (rem > half || (rem == half && (M & 1ull))) M += 1;
    }
  }
  if (M == (1ull << f->p)) { /* rounding carried into the next binade */
    M >>= 1;
    Q += 1;
  }
  if (M < (1ull << (f->p - 1))) /* subnormal or zero: exponent field 0 */
    return (uint16_t)(sign | (uint32_t)M);
  int biased = Q + (f->p - 1) + f->emax;
  if (biased >= (1 << f->ebits) - 1) return (uint16_t)(sign | exp_all_ones); /* overflow */
  return (uint16_t)(sign | ((uint32_t)biased << f->mbits) | (uint32_t)(M - (1ull << (f->p - 1))));
}

/* The binary32 value of a narrow encoding (always exact). */
static float narrow_to_f32(uint16_t h, const narrow_fmt *f) {
  uint32_t sign = (uint32_t)h >> 15;
  uint32_t E = ((uint32_t)h >> f->mbits) & ((1u << f->ebits) - 1u);
  uint32_t frac = (uint32_t)h & ((1u << f->mbits) - 1u);
  float v;
  if (E == (1u << f->ebits) - 1u) {
    if (frac == 0) {
      v = INFINITY;
    } else { /* NaN with the payload moved to the top of the binary32 fraction */
      return bits_f32((sign << 31) | 0x7f800000u | 0x400000u | (frac << (23 - f->mbits)));
    }
  } else if (E == 0) {
    v = ldexpf((float)frac, f->emin - f->mbits);
  } else {
    v = ldexpf((float)(frac + (1u << f->mbits)), (int)E - f->emax - f->mbits);
  }
  return sign ? -v : v;
}

uint16_t orc_f32_to_f16(float x) { return round_to_narrow(x, &FMT_F16); }
uint16_t orc_f32_to_bf16(float x) { return round_to_narrow(x, &FMT_BF16); }
float orc_f16_to_f32(uint16_t h) { return narrow_to_f32(h, &FMT_F16); }
float orc_bf16_to_f32(uint16_t b) { return narrow_to_f32(b, &FMT_BF16); }

/* ------------------------------------------------------------------------ */
/* Element access in the storage and wire formats.                           */
/* ------------------------------------------------------------------------ */

static size_t elem_size(int t) { return t == ORC_F32 ? 4 : 2; }

static int valid_type(int t) { return t == ORC_F32 || t == ORC_F16 || t == ORC_BF16; }

/* Supported (storage, wire) pairs: the same type; binary32 storage carried on
 * a 16-bit wire; or 16-bit storage accumulated in binary32 (exact widening on
 * ingress, binary32 hops, one rounding to the storage format at the end). */
static int supported_pair(int dtype, int wire) {
  if (!valid_type(dtype) || !valid_type(wire)) return 0;
  return dtype == wire || dtype == ORC_F32 || wire == ORC_F32;
}

/* Encoding at j (binary32 bits for ORC_F32). */
static uint32_t get_bits(const void *buf, int t, size_t j) {
  if (t == ORC_F32) {
    uint32_t u;
    memcpy(&u, (const unsigned char *)buf + 4 * j, 4);
    return u;
  }
  uint16_t h;
  memcpy(&h, (const unsigned char *)buf + 2 * j, 2);
  return h;
}

static void put_bits(void *buf, int t, size_t j, uint32_t v) {
  if (t == ORC_F32) {
    memcpy((unsigned char *)buf + 4 * j, &v, 4);
  } else {
    uint16_t h = (uint16_t)v;
    memcpy((unsigned char *)buf + 2 * j, &h, 2);
  }
}

static float bits_to_value(int t, uint32_t v) {
  if (t == ORC_F32) return bits_f32(v);
  if (t == ORC_F16) return orc_f16_to_f32((uint16_t)v);
  return orc_bf16_to_f32((uint16_t)v);
}

static uint32_t value_to_bits(int t, float x) {
  if (t == ORC_F32) return f32_bits(x);
  if (t == ORC_F16) return orc_f32_to_f16(x);
  return orc_f32_to_bf16(x);
}

uint32_t orc_wire_add(int wire, uint32_t a, uint32_t b) {
  float s = bits_to_value(wire, a) + bits_to_value(wire, b); /* one binary32 addition */
  return value_to_bits(wire, s);                             /* identity for binary32 */
}

/* Storage element -> wire encoding (ingress cast: round to nearest even, or
 * exact when the wire is wider). */
static uint32_t ingress(int dtype, int wire, uint32_t v) {
  if (dtype == wire) return v;
  return value_to_bits(wire, bits_to_value(dtype, v));
}

/* Wire encoding -> storage element (egress: exact widening, or one rounding to
 * nearest even when the storage is narrower). */
static uint32_t egress(int dtype, int wire, uint32_t v) {
  if (dtype == wire) return v;
  return value_to_bits(dtype, bits_to_value(wire, v));
}

void orc_f32_to_wire_batch(int wire, const float *x, uint16_t *out, size_t n) {
  for (size_t j = 0; j < n; j++) out[j] = (uint16_t)value_to_bits(wire, x[j]);
}

void orc_wire_add_batch(int wire, const uint16_t *a, const uint16_t *b, uint16_t *out, size_t n) {
  for (size_t j = 0; j < n; j++) out[j] = (uint16_t)orc_wire_add(wire, a[j], b[j]);
}

/* ------------------------------------------------------------------------ */
/* Chunk partition: floor(count / R) per chunk, the last chunk takes the rest. */
/* ------------------------------------------------------------------------ */

size_t orc_chunk_len(size_t count, int R, int c) {
  if (R < 1 || c < 0 || c >= R) return 0;
  size_t base = count / (size_t)R;
  if (c < R - 1) return base;
  return count - (size_t)(R - 1) * base;
}

size_t orc_chunk_off(size_t count, int R, int c) {
  if (R < 1 || c < 0 || c >= R) return 0;
  return (size_t)c * (count / (size_t)R);
}

static int mod(int a, int n) { return ((a % n) + n) % n; }

/* ------------------------------------------------------------------------ */
/* The simulated ring: work buffers, mailboxes, message log, faults.         */
/* ------------------------------------------------------------------------ */

typedef struct {
  unsigned char *data;
  int full;
  int src, chunk;
  size_t len;
} mailbox;

typedef struct {
  int R;
  int wire;
  size_t ew;        /* wire element bytes */
  unsigned char **W; /* work buffer of each rank, in the wire format */
  mailbox *mail;    /* one per rank */
  orc_opts *opts;
  int status;
} ring_sim;

static void sim_free(ring_sim *s) {
  if (s->W) {
    for (int r = 0; r < s->R; r++) free(s->W[r]);
    free(s->W);
  }
  if (s->mail) {
    for (int r = 0; r < s->R; r++) free(s->mail[r].data);
    free(s->mail);
  }
}

static int sim_init(ring_sim *s, int R, int wire, size_t count, size_t mail_cap, orc_opts *opts) {
  memset(s, 0, sizeof(*s));
  s->R = R;
  s->wire = wire;
  s->ew = elem_size(wire);
  s->opts = opts;
  s->W = (unsigned char **)calloc((size_t)R, sizeof(unsigned char *));
  s->mail = (mailbox *)calloc((size_t)R, sizeof(mailbox));
  if (!s->W || !s->mail) return ORC_ENOMEM;
  for (int r = 0; r < R; r++) {
    s->W[r] = (unsigned char *)malloc(count * s->ew + 1);
    s->mail[r].data = (unsigned char *)malloc(mail_cap * s->ew + 1);
    if (!s->W[r] || !s->mail[r].data) return ORC_ENOMEM;
  }
  if (opts) {
    opts->trace_len = 0;
    if (opts->sent_bytes)
      for (int r = 0; r < R; r++) opts->sent_bytes[r] = 0;
  }
  return ORC_OK;
}

static int fault_hits(const orc_opts *o, int kind, int src, int phase, int step) {
  if (!o || o->fault.kind != kind || o->fault.rank != src) return 0;
  if (kind == ORC_FAULT_SILENT)
    return phase > o->fault.phase || (phase == o->fault.phase && step >= o->fault.step);
  return phase == o->fault.phase && step == o->fault.step;
}

static void deliver(ring_sim *s, int src, int dst, int chunk, const unsigned char *data, size_t len) {
  mailbox *mb = &s->mail[dst];
  if (mb->full) { /* a second message before the first was consumed */
    if (s->status == ORC_OK) s->status = ORC_EPROTO;
    return;
  }
  memcpy(mb->data, data, len * s->ew);
  mb->full = 1;
  mb->src = src;
  mb->chunk = chunk;
  mb->len = len;
}

/* Rank src sends `len` wire elements starting at element `off` of its buffer. */
static void sim_send(ring_sim *s, int phase, int step, int src, int dst, int chunk, size_t off,
                     size_t len) {
  orc_opts *o = s->opts;
  if (fault_hits(o, ORC_FAULT_SILENT, src, phase, step)) return; /* rank stopped sending */
  uint64_t bytes = (uint64_t)len * s->ew;
  if (o) {
    if (o->sent_bytes) o->sent_bytes[src] += bytes;
    if (o->trace && o->trace_len < o->trace_cap) {
      orc_msg *m = &o->trace[o->trace_len];
      m->phase = phase;
      m->step = step;
      m->src = src;
      m->dst = dst;
      m->chunk = chunk;
      m->pad = 0;
      m->bytes = bytes;
    }
    o->trace_len++;
  }
  if (fault_hits(o, ORC_FAULT_DROP, src, phase, step)) return; /* lost on the link */
  deliver(s, src, dst, chunk, s->W[src] + off * s->ew, len);
  if (fault_hits(o, ORC_FAULT_DUP, src, phase, step)) deliver(s, src, dst, chunk, s->W[src] + off * s->ew, len);
}

/* Rank dst waits (bounded) for the message of `chunk` from `src`. */
static mailbox *sim_recv(ring_sim *s, int dst, int src, int chunk) {
  mailbox *mb = &s->mail[dst];
  int limit = (s->opts && s->opts->poll_limit > 0) ? s->opts->poll_limit : 16;
  int polls = 0;
  while (!mb->full) {
    if (++polls >= limit) {
      if (s->status == ORC_OK) s->status = ORC_ETIMEOUT;
      return NULL;
    }
  }
  if (mb->src != src || mb->chunk != chunk) {
    if (s->status == ORC_OK) s->status = ORC_EPROTO;
    return NULL;
  }
  return mb;
}

/* Received chunk added into the same chunk of dst's buffer: one rounded add per element. */
static void recv_add(ring_sim *s, int dst, int src, int chunk, size_t off, size_t len) {
  mailbox *mb = sim_recv(s, dst, src, chunk);
  if (!mb) return;
  for (size_t j = 0; j < len; j++) {
    uint32_t mine = get_bits(s->W[dst], s->wire, off + j);
    uint32_t got = get_bits(mb->data, s->wire, j);
    put_bits(s->W[dst], s->wire, off + j, orc_wire_add(s->wire, mine, got));
  }
  mb->full = 0;
}

/* Received chunk copied over the same chunk of dst's buffer. */
static void recv_copy(ring_sim *s, int dst, int src, int chunk, size_t off, size_t len) {
  mailbox *mb = sim_recv(s, dst, src, chunk);
  if (!mb) return;
  memcpy(s->W[dst] + off * s->ew, mb->data, len * s->ew);
  mb->full = 0;
}

/*
 * Ring reduce-scatter among the L ranks first, first+1, ..., first+L-1, with
 * the chunk table of (count, L).  At step t, local rank l sends chunk (l - t)
 * to l+1 and adds chunk (l - t - 1) received from l-1.  Afterwards local rank
 * l holds chunk (l + 1) mod L summed over the group, folded in the order
 * w_c, w_{c+1}, ..., w_{c+L-1}.
 */
static void ring_rs(ring_sim *s, int first, int L, size_t count) {
  for (int t = 0; t < L - 1 && s->status == ORC_OK; t++) {
    for (int l = 0; l < L; l++) {
      int cs = mod(l - t, L);
      sim_send(s, ORC_PHASE_RS, t, first + l, first + mod(l + 1, L), cs, orc_chunk_off(count, L, cs),
               orc_chunk_len(count, L, cs));
    }
    for (int l = 0; l < L && s->status == ORC_OK; l++) {
      int cr = mod(l - t - 1, L);
      recv_add(s, first + l, first + mod(l - 1, L), cr, orc_chunk_off(count, L, cr),
               orc_chunk_len(count, L, cr));
    }
  }
}

/*
 * Ring allgather among the L ranks first..first+L-1 when local rank l starts
 * with the finished chunk (l + shift) mod L: at step t, rank l sends chunk
 * (l + shift - t) to l+1 and stores chunk (l + shift - t - 1) from l-1.
 */
static void ring_ag(ring_sim *s, int first, int L, size_t count, int shift) {
  for (int t = 0; t < L - 1 && s->status == ORC_OK; t++) {
    for (int l = 0; l < L; l++) {
      int cs = mod(l + shift - t, L);
      sim_send(s, ORC_PHASE_AG, t, first + l, first + mod(l + 1, L), cs, orc_chunk_off(count, L, cs),
               orc_chunk_len(count, L, cs));
    }
    for (int l = 0; l < L && s->status == ORC_OK; l++) {
      int cr = mod(l + shift - t - 1, L);
      recv_copy(s, first + l, first + mod(l - 1, L), cr, orc_chunk_off(count, L, cr),
                orc_chunk_len(count, L, cr));
    }
  }
}

/*
 * Inter-group exchange of the two-level ring.  Chunk c is owned, in every
 * group g, by local rank (c - 1) mod L.  Chain step k (k = 0..G-2): the owner
 * in group k sends its partial sum to the owner in group k+1, which adds it,
 * so the total is folded in group order 0, 1, ..., G-1.  Then the owner in
 * group G-1 sends the total to the owners in groups 0..G-2.
 */
static void group_exchange(ring_sim *s, int G, int L, size_t count) {
  for (int k = 0; k < G - 1 && s->status == ORC_OK; k++) {
    for (int c = 0; c < L; c++) {
      int own = mod(c - 1, L);
      sim_send(s, ORC_PHASE_XCHG, k, k * L + own, (k + 1) * L + own, c, orc_chunk_off(count, L, c),
               orc_chunk_len(count, L, c));
    }
    for (int c = 0; c < L && s->status == ORC_OK; c++) {
      int own = mod(c - 1, L);
      recv_add(s, (k + 1) * L + own, k * L + own, c, orc_chunk_off(count, L, c), orc_chunk_len(count, L, c));
    }
  }
  for (int g = 0; g < G - 1 && s->status == ORC_OK; g++) {
    for (int c = 0; c < L; c++) {
      int own = mod(c - 1, L);
      sim_send(s, ORC_PHASE_XBCAST, g, (G - 1) * L + own, g * L + own, c, orc_chunk_off(count, L, c),
               orc_chunk_len(count, L, c));
    }
    for (int c = 0; c < L && s->status == ORC_OK; c++) {
      int own = mod(c - 1, L);
      recv_copy(s, g * L + own, (G - 1) * L + own, c, orc_chunk_off(count, L, c), orc_chunk_len(count, L, c));
    }
  }
}

static size_t max_chunk_len(size_t count, int L) {
  size_t m = 0;
  for (int c = 0; c < L; c++) {
    size_t n = orc_chunk_len(count, L, c);
    if (n > m) m = n;
  }
  return m;
}

/* ------------------------------------------------------------------------ */
/* The collectives.                                                          */
/* ------------------------------------------------------------------------ */

int orc_allreduce(const void *const *in, void *const *out, int R, size_t count, int dtype,
                  int wire, int group_size, orc_opts *opts) {
  if (R < 1 || !in || !out) return ORC_EINVAL;
  if (!supported_pair(dtype, wire)) return ORC_EUNSUPPORTED;
  int L = group_size == 0 ? R : group_size;
  if (L < 1 || R % L != 0) return ORC_EINVAL;
  int G = R / L;
  for (int r = 0; r < R; r++)
    if (count > 0 && (!in[r] || !out[r])) return ORC_EINVAL;

  ring_sim s;
  int st = sim_init(&s, R, wire, count, max_chunk_len(count, L), opts);
  if (st != ORC_OK) {
    sim_free(&s);
    return st;
  }
  for (int r = 0; r < R; r++) /* ingress: storage -> wire */
    for (size_t j = 0; j < count; j++) put_bits(s.W[r], wire, j, ingress(dtype, wire, get_bits(in[r], dtype, j)));

  for (int g = 0; g < G; g++) ring_rs(&s, g * L, L, count); /* reduce-scatter inside each group */
  if (G > 1) group_exchange(&s, G, L, count);              /* one exchange between groups */
  for (int g = 0; g < G; g++) ring_ag(&s, g * L, L, count, 1); /* allgather inside each group */

  if (s.status == ORC_OK)
    for (int r = 0; r < R; r++) /* egress: wire -> storage */
      for (size_t j = 0; j < count; j++) put_bits(out[r], dtype, j, egress(dtype, wire, get_bits(s.W[r], wire, j)));
  st = s.status;
  sim_free(&s);
  return st;
}

int orc_reduce_scatter(const void *const *in, void *const *out, int R, size_t count, int dtype,
                       int wire, orc_opts *opts) {
  if (R < 1 || !in || !out) return ORC_EINVAL;
  if (!supported_pair(dtype, wire)) return ORC_EUNSUPPORTED;
  for (int r = 0; r < R; r++) {
    if (count > 0 && !in[r]) return ORC_EINVAL;
    if (orc_chunk_len(count, R, r) > 0 && !out[r]) return ORC_EINVAL;
  }
  ring_sim s;
  int st = sim_init(&s, R, wire, count, max_chunk_len(count, R), opts);
  if (st != ORC_OK) {
    sim_free(&s);
    return st;
  }
  for (int r = 0; r < R; r++)
    for (size_t j = 0; j < count; j++) put_bits(s.W[r], wire, j, ingress(dtype, wire, get_bits(in[r], dtype, j)));
  ring_rs(&s, 0, R, count);
  if (s.status == ORC_OK) {
    /* rank (c - 1) mod R holds the finished chunk c; output c receives it */
    for (int c = 0; c < R; c++) {
      int holder = mod(c - 1, R);
      size_t off = orc_chunk_off(count, R, c), len = orc_chunk_len(count, R, c);
      for (size_t j = 0; j < len; j++)
        put_bits(out[c], dtype, j, egress(dtype, wire, get_bits(s.W[holder], wire, off + j)));
    }
  }
  st = s.status;
  sim_free(&s);
  return st;
}

int orc_allgather(const void *const *in, void *const *out, int R, size_t count, int dtype,
                  orc_opts *opts) {
  if (R < 1 || !in || !out) return ORC_EINVAL;
  if (!valid_type(dtype)) return ORC_EUNSUPPORTED;
  for (int r = 0; r < R; r++) {
    if (count > 0 && !out[r]) return ORC_EINVAL;
    if (orc_chunk_len(count, R, r) > 0 && !in[r]) return ORC_EINVAL;
  }
  ring_sim s;
  int st = sim_init(&s, R, dtype, count, max_chunk_len(count, R), opts);
  if (st != ORC_OK) {
    sim_free(&s);
    return st;
  }
  /* rank r starts with chunk r */
  for (int r = 0; r < R; r++) {
    size_t off = orc_chunk_off(count, R, r), len = orc_chunk_len(count, R, r);
    if (len) memcpy(s.W[r] + off * s.ew, in[r], len * s.ew);
  }
  ring_ag(&s, 0, R, count, 0);
  if (s.status == ORC_OK)
    for (int r = 0; r < R; r++)
      if (count) memcpy(out[r], s.W[r], count * s.ew);
  st = s.status;
  sim_free(&s);
  return st;
}

/* ------------------------------------------------------------------------ */
/* Closed form: chunk c(i) of element i, then                               */
/*   S_g = x_{gL+c} (+) x_{gL+c+1} (+) ... (+) x_{gL+c+L-1}   (local ranks mod L) */
/*   out = S_0 (+) S_1 (+) ... (+) S_{G-1}                                    */
/* where (+) is one hop on the wire.                                         */
/* ------------------------------------------------------------------------ */

int orc_fold_gathered(const void *const *vals, const uint64_t *idx, size_t n, int R, size_t count,
                      int dtype, int wire, int group_size, void *out) {
  if (R < 1 || !vals || (n > 0 && (!idx || !out))) return ORC_EINVAL;
  if (!supported_pair(dtype, wire)) return ORC_EUNSUPPORTED;
  int L = group_size == 0 ? R : group_size;
  if (L < 1 || R % L != 0) return ORC_EINVAL;
  int G = R / L;
  for (size_t k = 0; k < n; k++) {
    size_t i = (size_t)idx[k];
    if (i >= count) return ORC_EINVAL;
    int c = -1; /* the chunk whose range holds i */
    for (int cc = 0; cc < L; cc++) {
      size_t off = orc_chunk_off(count, L, cc), len = orc_chunk_len(count, L, cc);
      if (i >= off && i < off + len) {
        c = cc;
        break;
      }
    }
    if (c < 0) return ORC_EINVAL;
    uint32_t total = 0;
    for (int g = 0; g < G; g++) {
      uint32_t acc = ingress(dtype, wire, get_bits(vals[g * L + c], dtype, k));
      for (int step = 1; step < L; step++) {
        int r = g * L + (c + step) % L;
        acc = orc_wire_add(wire, acc, ingress(dtype, wire, get_bits(vals[r], dtype, k)));
      }
      total = (g == 0) ? acc : orc_wire_add(wire, total, acc);
    }
    put_bits(out, dtype, k, egress(dtype, wire, total));
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Halving-doubling and naive AllReduce.                                     */
/* ------------------------------------------------------------------------ */

static int floor_pow2(int R) {
  int P = 1;
  while (P * 2 <= R) P *= 2;
  return P;
}

static int log2_exact(int P) {
  int l = 0;
  while ((1 << l) < P) l++;
  return l;
}

/* rank of virtual rank v in halving-doubling (E extra ranks folded in pairs) */
static int hd_rank(int v, int E) { return v < E ? 2 * v + 1 : v + E; }

/* element offset of block b of the (count, P) table; block P is the end */
static size_t block_start(size_t count, int P, int b) {
  return b >= P ? count : orc_chunk_off(count, P, b);
}

static void halving_doubling(ring_sim *s, int R, size_t count) {
  const int P = floor_pow2(R), E = R - P, steps = log2_exact(P);
  /* fold the extra ranks into their odd neighbours */
  for (int k = 0; k < E; k++) sim_send(s, ORC_PHASE_PRE, 0, 2 * k, 2 * k + 1, -1, 0, count);
  for (int k = 0; k < E && s->status == ORC_OK; k++) recv_add(s, 2 * k + 1, 2 * k, -1, 0, count);
  /* recursive halving: every virtual rank owns the block range [lo[v], hi[v]) */
  int lo[64], hi[64];
  for (int v = 0; v < P; v++) {
    lo[v] = 0;
    hi[v] = P;
  }
  for (int t = 0; t < steps && s->status == ORC_OK; t++) {
    const int d = P >> (t + 1);
    int keep_lo[64], keep_hi[64];
    for (int v = 0; v < P; v++) { /* send the half the partner keeps */
      const int mid = (lo[v] + hi[v]) / 2, u = v ^ d;
      const int give_lo = (v & d) ? lo[v] : mid, give_hi = (v & d) ? mid : hi[v];
      keep_lo[v] = (v & d) ? mid : lo[v];
      keep_hi[v] = (v & d) ? hi[v] : mid;
      const size_t a = block_start(count, P, give_lo), b = block_start(count, P, give_hi);
      sim_send(s, ORC_PHASE_RS, t, hd_rank(v, E), hd_rank(u, E), give_lo, a, b - a);
    }
    for (int v = 0; v < P && s->status == ORC_OK; v++) { /* add the partner's copy of the half I keep */
      const size_t a = block_start(count, P, keep_lo[v]), b = block_start(count, P, keep_hi[v]);
      recv_add(s, hd_rank(v, E), hd_rank(v ^ d, E), keep_lo[v], a, b - a);
    }
    for (int v = 0; v < P; v++) {
      lo[v] = keep_lo[v];
      hi[v] = keep_hi[v];
    }
  }
  /* recursive doubling: swap ranges with the partner, nearest partner first */
  for (int t = steps - 1; t >= 0 && s->status == ORC_OK; t--) {
    const int d = P >> (t + 1);
    for (int v = 0; v < P; v++) {
      const size_t a = block_start(count, P, lo[v]), b = block_start(count, P, hi[v]);
      sim_send(s, ORC_PHASE_AG, steps - 1 - t, hd_rank(v, E), hd_rank(v ^ d, E), lo[v], a, b - a);
    }
    int new_lo[64], new_hi[64];
    for (int v = 0; v < P && s->status == ORC_OK; v++) {
      const int u = v ^ d;
      const size_t a = block_start(count, P, lo[u]), b = block_start(count, P, hi[u]);
      recv_copy(s, hd_rank(v, E), hd_rank(u, E), lo[u], a, b - a);
      new_lo[v] = lo[v] < lo[u] ? lo[v] : lo[u];
      new_hi[v] = hi[v] > hi[u] ? hi[v] : hi[u];
    }
    for (int v = 0; v < P; v++) {
      lo[v] = new_lo[v];
      hi[v] = new_hi[v];
    }
  }
  /* hand the result back to the folded ranks */
  for (int k = 0; k < E && s->status == ORC_OK; k++) sim_send(s, ORC_PHASE_POST, 0, 2 * k + 1, 2 * k, -1, 0, count);
  for (int k = 0; k < E && s->status == ORC_OK; k++) recv_copy(s, 2 * k, 2 * k + 1, -1, 0, count);
}

static void naive_reduce_broadcast(ring_sim *s, int R, size_t count) {
  for (int k = 1; k < R && s->status == ORC_OK; k++) { /* the collector adds rank k's vector */
    sim_send(s, ORC_PHASE_RS, k - 1, k, 0, -1, 0, count);
    recv_add(s, 0, k, -1, 0, count);
  }
  for (int k = 1; k < R && s->status == ORC_OK; k++) { /* and sends the sum back */
    sim_send(s, ORC_PHASE_AG, k - 1, 0, k, -1, 0, count);
    recv_copy(s, k, 0, -1, 0, count);
  }
}

/* first chunk held by virtual rank v of the tree AllGather (v = P: the end) */
static int tree_first_chunk(int v, int E) { return v < E ? 2 * v : v + E; }

static void tree_allgather(ring_sim *s, int R, size_t count) {
  const int P = floor_pow2(R), E = R - P, steps = log2_exact(P);
  for (int k = 0; k < E; k++) /* the extra ranks hand their chunks to their odd neighbours */
    sim_send(s, ORC_PHASE_PRE, 0, 2 * k, 2 * k + 1, 2 * k, orc_chunk_off(count, R, 2 * k),
             orc_chunk_len(count, R, 2 * k));
  for (int k = 0; k < E && s->status == ORC_OK; k++)
    recv_copy(s, 2 * k + 1, 2 * k, 2 * k, orc_chunk_off(count, R, 2 * k), orc_chunk_len(count, R, 2 * k));
  /* virtual rank v holds the chunks of virtual ranks [lo[v], hi[v]) */
  int lo[64], hi[64];
  for (int v = 0; v < P; v++) {
    lo[v] = v;
    hi[v] = v + 1;
  }
  for (int t = 0; t < steps && s->status == ORC_OK; t++) {
    const int d = 1 << t;
    for (int v = 0; v < P; v++) {
      const int c0 = tree_first_chunk(lo[v], E), c1 = tree_first_chunk(hi[v], E);
      const size_t a = orc_chunk_off(count, R, c0), b = c1 >= R ? count : orc_chunk_off(count, R, c1);
      sim_send(s, ORC_PHASE_AG, t, hd_rank(v, E), hd_rank(v ^ d, E), c0, a, b - a);
    }
    int new_lo[64], new_hi[64];
    for (int v = 0; v < P && s->status == ORC_OK; v++) {
      const int u = v ^ d;
      const int c0 = tree_first_chunk(lo[u], E), c1 = tree_first_chunk(hi[u], E);
      const size_t a = orc_chunk_off(count, R, c0), b = c1 >= R ? count : orc_chunk_off(count, R, c1);
      recv_copy(s, hd_rank(v, E), hd_rank(u, E), c0, a, b - a);
      new_lo[v] = lo[v] < lo[u] ? lo[v] : lo[u];
      new_hi[v] = hi[v] > hi[u] ? hi[v] : hi[u];
    }
    for (int v = 0; v < P; v++) {
      lo[v] = new_lo[v];
      hi[v] = new_hi[v];
    }
  }
  for (int k = 0; k < E && s->status == ORC_OK; k++) sim_send(s, ORC_PHASE_POST, 0, 2 * k + 1, 2 * k, -1, 0, count);
  for (int k = 0; k < E && s->status == ORC_OK; k++) recv_copy(s, 2 * k, 2 * k + 1, -1, 0, count);
}

static void naive_gather_broadcast(ring_sim *s, int R, size_t count) {
  for (int k = 1; k < R && s->status == ORC_OK; k++) { /* rank 0 collects chunk k */
    const size_t off = orc_chunk_off(count, R, k), len = orc_chunk_len(count, R, k);
    sim_send(s, ORC_PHASE_RS, k - 1, k, 0, k, off, len);
    recv_copy(s, 0, k, k, off, len);
  }
  for (int k = 1; k < R && s->status == ORC_OK; k++) { /* and sends the whole vector out */
    sim_send(s, ORC_PHASE_AG, k - 1, 0, k, -1, 0, count);
    recv_copy(s, k, 0, -1, 0, count);
  }
}

int orc_allgather_algo(const void *const *in, void *const *out, int R, size_t count, int dtype, int algo,
                       orc_opts *opts) {
  if (algo == ORC_ALGO_RING) return orc_allgather(in, out, R, count, dtype, opts);
  if (algo != ORC_ALGO_HALVING_DOUBLING && algo != ORC_ALGO_NAIVE) return ORC_EINVAL;
  if (R < 1 || R > 64 || !in || !out) return ORC_EINVAL;
  if (!valid_type(dtype)) return ORC_EUNSUPPORTED;
  for (int r = 0; r < R; r++) {
    if (count > 0 && !out[r]) return ORC_EINVAL;
    if (orc_chunk_len(count, R, r) > 0 && !in[r]) return ORC_EINVAL;
  }
  ring_sim s;
  int st = sim_init(&s, R, dtype, count, count, opts);
  if (st != ORC_OK) {
    sim_free(&s);
    return st;
  }
  for (int r = 0; r < R; r++) { /* rank r starts with chunk r */
    size_t off = orc_chunk_off(count, R, r), len = orc_chunk_len(count, R, r);
    if (len) memcpy(s.W[r] + off * s.ew, in[r], len * s.ew);
  }
  if (algo == ORC_ALGO_NAIVE)
    naive_gather_broadcast(&s, R, count);
  else
    tree_allgather(&s, R, count);
  if (s.status == ORC_OK)
    for (int r = 0; r < R; r++)
      if (count) memcpy(out[r], s.W[r], count * s.ew);
  st = s.status;
  sim_free(&s);
  return st;
}

int orc_allreduce_algo(const void *const *in, void *const *out, int R, size_t count, int dtype, int wire,
                       int algo, orc_opts *opts) {
  if (algo == ORC_ALGO_RING) return orc_allreduce(in, out, R, count, dtype, wire, 0, opts);
  if (algo != ORC_ALGO_HALVING_DOUBLING && algo != ORC_ALGO_NAIVE) return ORC_EINVAL;
  if (R < 1 || R > 64 || !in || !out) return ORC_EINVAL;
  if (!supported_pair(dtype, wire)) return ORC_EUNSUPPORTED;
  for (int r = 0; r < R; r++)
    if (count > 0 && (!in[r] || !out[r])) return ORC_EINVAL;
  ring_sim s;
  int st = sim_init(&s, R, wire, count, count, opts);
  if (st != ORC_OK) {
    sim_free(&s);
    return st;
  }
  for (int r = 0; r < R; r++)
    for (size_t j = 0; j < count; j++) put_bits(s.W[r], wire, j, ingress(dtype, wire, get_bits(in[r], dtype, j)));
  if (algo == ORC_ALGO_NAIVE)
    naive_reduce_broadcast(&s, R, count);
  else
    halving_doubling(&s, R, count);
  if (s.status == ORC_OK)
    for (int r = 0; r < R; r++)
      for (size_t j = 0; j < count; j++) put_bits(out[r], dtype, j, egress(dtype, wire, get_bits(s.W[r], wire, j)));
  st = s.status;
  sim_free(&s);
  return st;
}

/* Closed forms.  Naive: x_0 (+) x_1 (+) ... (+) x_{R-1}.  Halving-doubling:
 * leaves L_v = x_{2v} (+) x_{2v+1} for v < E, x_{v+E} otherwise; then for
 * d = P/2, P/4, ..., 1: L_v = L_v (+) L_{v+d} for v < d; the result is L_0. */
int orc_fold_gathered_algo(const void *const *vals, const uint64_t *idx, size_t n, int R, size_t count,
                           int dtype, int wire, int algo, void *out) {
  if (algo == ORC_ALGO_RING) return orc_fold_gathered(vals, idx, n, R, count, dtype, wire, 0, out);
  if (algo != ORC_ALGO_HALVING_DOUBLING && algo != ORC_ALGO_NAIVE) return ORC_EINVAL;
  if (R < 1 || R > 64 || !vals || (n > 0 && (!idx || !out))) return ORC_EINVAL;
  if (!supported_pair(dtype, wire)) return ORC_EUNSUPPORTED;
  for (size_t k = 0; k < n; k++) {
    if ((size_t)idx[k] >= count) return ORC_EINVAL;
    uint32_t x[64];
    for (int r = 0; r < R; r++) x[r] = ingress(dtype, wire, get_bits(vals[r], dtype, k));
    uint32_t y;
    if (algo == ORC_ALGO_NAIVE) {
      y = x[0];
      for (int r = 1; r < R; r++) y = orc_wire_add(wire, y, x[r]);
    } else {
      const int P = floor_pow2(R), E = R - P;
      uint32_t leaf[64];
      for (int v = 0; v < P; v++) leaf[v] = v < E ? orc_wire_add(wire, x[2 * v], x[2 * v + 1]) : x[v + E];
      for (int d = P / 2; d >= 1; d /= 2)
        for (int v = 0; v < d; v++) leaf[v] = orc_wire_add(wire, leaf[v], leaf[v + d]);
      y = leaf[0];
    }
    put_bits(out, dtype, k, egress(dtype, wire, y));
  }
  return ORC_OK;
}
