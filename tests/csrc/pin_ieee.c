/*
 * pin_ieee.c -- pins the oracle's IEEE arithmetic to the C compiler's own.
 *
 * Test helper, built and run by tests/test_oracle_ieee.py.  It links the
 * oracle's C source and compares, over whole input spaces:
 *   - binary32 -> binary16 / bfloat16 rounding against the compiler's
 *     (_Float16) and (__bf16) casts (round to nearest, ties to even);
 *   - binary16 / bfloat16 -> binary32 widening against the same types;
 *   - one ring hop on a 16-bit wire (binary32 sum, one rounding) against the
 *     exact sum in binary64 rounded once to the narrow type by the compiler.
 *     binary64 holds the exact sum of two binary16 values, and for bfloat16
 *     a binary64 sum rounded once more is still the correctly rounded result
 *     because 53 >= 2*8 + 2.
 * NaNs compare equal to NaNs (payloads are not pinned).
 *
 * Usage: pin_ieee <test> [lo hi [stride]]: checks inputs lo, lo+stride, ... below hi
 * and prints "<test> <checked> <mismatches> <first bad input>".
 */
#include <inttypes.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "ring_oracle.h"

static uint32_t f2u(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }
static float u2f(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }
static uint16_t h2u(_Float16 h) { uint16_t u; memcpy(&u, &h, 2); return u; }
static _Float16 u2h(uint16_t u) { _Float16 h; memcpy(&h, &u, 2); return h; }
static uint16_t b2u(__bf16 b) { uint16_t u; memcpy(&u, &b, 2); return u; }
static __bf16 u2b(uint16_t u) { __bf16 b; memcpy(&b, &u, 2); return b; }

static int is_nan16(uint16_t v, int ebits) {
  int mbits = 15 - ebits;
  uint32_t e = (v >> mbits) & ((1u << ebits) - 1u);
  return e == (1u << ebits) - 1u && (v & ((1u << mbits) - 1u)) != 0;
}

static int same16(uint16_t a, uint16_t b, int ebits) {
  if (is_nan16(a, ebits) || is_nan16(b, ebits)) return is_nan16(a, ebits) && is_nan16(b, ebits);
  return a == b;
}

static int same32(float a, float b) {
  if (a != a || b != b) return a != a && b != b;
  return f2u(a) == f2u(b);
}

int main(int argc, char **argv) {
  if (argc < 2) return 2;
  const char *t = argv[1];
  uint64_t lo = argc > 2 ? strtoull(argv[2], NULL, 0) : 0;
  uint64_t hi = argc > 3 ? strtoull(argv[3], NULL, 0) : 0;
  int64_t stride = argc > 4 ? (int64_t)strtoull(argv[4], NULL, 0) : 1;
  if (stride < 1) stride = 1;
  uint64_t checked = 0, bad = 0, first = UINT64_MAX;

  if (!strcmp(t, "f32_to_f16") || !strcmp(t, "f32_to_bf16")) {
    int bf = !strcmp(t, "f32_to_bf16");
    if (hi == 0) hi = 1ull << 32;
#pragma omp parallel for reduction(+ : checked, bad) schedule(static)
    for (int64_t k = (int64_t)lo; k < (int64_t)hi; k += stride) {
      float x = u2f((uint32_t)k);
      uint16_t mine = bf ? orc_f32_to_bf16(x) : orc_f32_to_f16(x);
      uint16_t ref = bf ? b2u((__bf16)x) : h2u((_Float16)x);
      checked++;
      if (!same16(mine, ref, bf ? 8 : 5)) {
        bad++;
#pragma omp critical
        if ((uint64_t)k < first) first = (uint64_t)k;
      }
    }
  } else if (!strcmp(t, "f16_to_f32") || !strcmp(t, "bf16_to_f32")) {
    int bf = !strcmp(t, "bf16_to_f32");
    for (uint32_t k = 0; k < 65536; k++) {
      float mine = bf ? orc_bf16_to_f32((uint16_t)k) : orc_f16_to_f32((uint16_t)k);
      float ref = bf ? (float)u2b((uint16_t)k) : (float)u2h((uint16_t)k);
      checked++;
      if (!same32(mine, ref)) {
        bad++;
        if (k < first) first = k;
      }
    }
  } else if (!strcmp(t, "add_f16") || !strcmp(t, "add_bf16")) {
    /* pairs (a, b) = (k >> 16, k & 0xffff) for k in [lo, hi) */
    int bf = !strcmp(t, "add_bf16");
    int wire = bf ? ORC_BF16 : ORC_F16;
    if (hi == 0) hi = 1ull << 32;
#pragma omp parallel for reduction(+ : checked, bad) schedule(static)
    for (int64_t k = (int64_t)lo; k < (int64_t)hi; k += stride) {
      uint16_t a = (uint16_t)((uint64_t)k >> 16), b = (uint16_t)((uint64_t)k & 0xffffu);
      uint16_t mine = (uint16_t)orc_wire_add(wire, a, b);
      uint16_t ref;
      if (bf) {
        double s = (double)(float)u2b(a) + (double)(float)u2b(b);
        ref = b2u((__bf16)s);
      } else {
        double s = (double)(float)u2h(a) + (double)(float)u2h(b);
        ref = h2u((_Float16)s);
      }
      checked++;
      if (!same16(mine, ref, bf ? 8 : 5)) {
        bad++;
#pragma omp critical
        if ((uint64_t)k < first) first = (uint64_t)k;
      }
    }
  } else if (!strcmp(t, "add_f32")) {
    /* binary32 hop: must be the plain IEEE binary32 addition, checked on a
       deterministic pseudo-random sample of [lo, hi) pair indices */
    if (hi == 0) hi = 1ull << 26;
#pragma omp parallel for reduction(+ : checked, bad) schedule(static)
    for (int64_t k = (int64_t)lo; k < (int64_t)hi; k += stride) {
      uint64_t z = (uint64_t)k * 0x9E3779B97F4A7C15ull;
      z ^= z >> 29;
      z *= 0xBF58476D1CE4E5B9ull;
      z ^= z >> 32;
      uint32_t a = (uint32_t)z, b = (uint32_t)(z >> 32);
      /* the binary64 sum of two binary32 values rounded once to binary32 is
         the correctly rounded binary32 sum (53 >= 2*24 + 2) */
      float ref = (float)((double)u2f(a) + (double)u2f(b));
      float mine = u2f(orc_wire_add(ORC_F32, a, b));
      checked++;
      if (!same32(mine, ref)) {
        bad++;
#pragma omp critical
        if ((uint64_t)k < first) first = (uint64_t)k;
      }
    }
  } else {
    return 2;
  }
  printf("%s %" PRIu64 " %" PRIu64 " %" PRIu64 "\n", t, checked, bad, first == UINT64_MAX ? 0 : first);
  return 0;
}
