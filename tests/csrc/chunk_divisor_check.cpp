// Checks the library's division of element indices by the chunk length (a
// multiply and shifts, rr_params.h) against the exact quotient: every
// divisor class (1, powers of two and their neighbours, small odd numbers,
// large and random 64-bit values) and, for each, dividends at 0, around every
// multiple near the low end, around 2^32, 2^63 and 2^64 - 1, and at random.
// Built with a host C++ compiler and run by tests/test_abi_cpu.py; prints
// "checked <n> bad <m>" and the first mismatch.
#include <cinttypes>
#include <cstdio>
#include <vector>

#include "rr_params.h"

static uint64_t next(uint64_t &s) {  // splitmix64
  uint64_t z = (s += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

int main() {
  std::vector<uint64_t> divisors;
  for (uint64_t d = 1; d <= 4096; ++d) divisors.push_back(d);
  for (int k = 12; k < 64; ++k)
    for (int64_t j = -3; j <= 3; ++j) divisors.push_back((1ull << k) + (uint64_t)j);
  divisors.push_back(~0ull);
  divisors.push_back(6250002ull);   // chunks of 50,000,017 over eight ranks
  divisors.push_back(33554432ull);
  uint64_t seed = 12345;
  for (int k = 0; k < 2000; ++k) divisors.push_back(next(seed) >> (next(seed) % 64) | 1ull);
  uint64_t checked = 0, bad = 0;
  for (uint64_t d : divisors) {
    const rr::ChunkDivisor dv = rr::make_chunk_divisor(d);
    std::vector<uint64_t> ns = {0, 1, 2, d - 1, d, d + 1, 2 * d - 1, 2 * d, 3 * d + 1, (1ull << 32) - 1,
                                1ull << 32, (1ull << 32) + 1, (1ull << 63) - 1, 1ull << 63, ~0ull - 1, ~0ull};
    for (uint64_t k = 1; k < 64; ++k) {
      const uint64_t m = k * d;
      if (d != 0 && m / d == k) {
        ns.push_back(m - 1);
        ns.push_back(m);
        ns.push_back(m + 1);
      }
    }
    for (int k = 0; k < 200; ++k) ns.push_back(next(seed) >> (next(seed) % 64));
    for (uint64_t n : ns) {
      const uint64_t q = rr::divide_by_chunk(n, dv.magic, dv.shift1, dv.shift2);
      ++checked;
      if (q != n / d) {
        if (bad++ == 0) std::printf("first mismatch: n=%" PRIu64 " d=%" PRIu64 " got %" PRIu64 "\n", n, d, q);
      }
    }
  }
  std::printf("checked %" PRIu64 " bad %" PRIu64 "\n", checked, bad);
  return bad != 0;
}
