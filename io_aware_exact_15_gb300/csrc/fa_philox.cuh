// Dropout keep decisions from a counter-based generator: Philox4x32 with ten
// rounds (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
// 1, 2, 3", SC 2011).  Element (i, j) of (batch, head) slice bhc uses
//   counter = (j / 16, i, bhc, offset),  key = (seed low word, seed high word)
// and byte j mod 16 of the 128-bit output (word (j / 4) mod 4, byte j mod 4,
// little-endian); it is kept iff that byte >= t, t = rint(256 p).  One call
// covers 16 consecutive keys of one query row.
#pragma once

#include <stdint.h>

#include "fa_ptx.cuh"

namespace fa {

struct PhiloxOut {
  uint32_t w[4];
};

// Ten rounds on the counter; rk[2 r], rk[2 r + 1] are the key of round r,
// i.e. (k0 + r * 0x9E3779B9, k1 + r * 0xBB67AE85) (the Weyl sequence that
// bumps the key between rounds), formed once on the host.
FA_DEV PhiloxOut philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                               const uint32_t (&rk)[20]) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    // the two 32 x 32 -> 64-bit products of the round
    const uint64_t a = static_cast<uint64_t>(0xD2511F53u) * c0;
    const uint64_t b = static_cast<uint64_t>(0xCD9E8D57u) * c2;
    const uint32_t a_hi = static_cast<uint32_t>(a >> 32), a_lo = static_cast<uint32_t>(a);
    const uint32_t b_hi = static_cast<uint32_t>(b >> 32), b_lo = static_cast<uint32_t>(b);
    c0 = b_hi ^ c1 ^ rk[2 * round];
    c1 = b_lo;
    c2 = a_hi ^ c3 ^ rk[2 * round + 1];
    c3 = a_lo;
  }
  PhiloxOut r;
  r.w[0] = c0;
  r.w[1] = c1;
  r.w[2] = c2;
  r.w[3] = c3;
  return r;
}

// Dropout stream of one call: round keys, offset and threshold.
struct DropoutRng {
  const uint32_t (&rk)[20];
  uint32_t offset, t4;  // t4: the threshold t in every byte

  // 0xFF in byte k of the result iff key 4 * w + k of the 16-key group is kept
  FA_DEV static uint32_t keep_bytes(uint32_t word, uint32_t t4) { return __vcmpgeu4(word, t4); }

  // the four words of the 16-key group starting at key 16 * grp of row i
  FA_DEV PhiloxOut group(uint32_t grp, uint32_t i, uint32_t bhc) const {
    return philox4x32_10(grp, i, bhc, offset, rk);
  }
};

// 4 keep bits (bit k = byte k is 0xFF) of a keep_bytes word: the 0/1 bits at
// positions 0, 8, 16, 24 are moved to 28..31 by one multiply (the partial
// products of different bytes land on distinct lower positions, no carries)
FA_DEV uint32_t keep_nibble(uint32_t m) { return ((m & 0x01010101u) * 0x10204080u) >> 28; }

// bf16-pair mask of keys 2 k and 2 k + 1 (k = 0, 1) of a keep_bytes word
FA_DEV uint32_t pair_mask(uint32_t m, int k) {
  return __byte_perm(m, 0u, k == 0 ? 0x1100u : 0x3322u);
}

}  // namespace fa
