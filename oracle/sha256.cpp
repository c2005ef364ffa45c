// Oracle: SHA-256 written from FIPS 180-4 (Secure Hash Standard), sections
// 4.1.2 (functions), 4.2.2 (constants), 5.1.1 (padding), 5.3.3 (initial hash
// value) and 6.2.2 (hash computation).  TEST INFRASTRUCTURE ONLY.
//
// "How the block pool manages KV memory", section "Finding a prefix again":
// since vLLM 0.11 the chained block hash is SHA-256 by default.

#include "oracle.h"

#include <cstring>
#include <vector>

namespace {

// First 32 bits of the fractional parts of the cube roots of the first 64
// primes (FIPS 180-4 section 4.2.2).
const uint32_t K256[64] = {
    0x428a2f98, 0x71374491, 0xb5c0fbcf, 0xe9b5dba5, 0x3956c25b, 0x59f111f1, 0x923f82a4,
    0xab1c5ed5, 0xd807aa98, 0x12835b01, 0x243185be, 0x550c7dc3, 0x72be5d74, 0x80deb1fe,
    0x9bdc06a7, 0xc19bf174, 0xe49b69c1, 0xefbe4786, 0x0fc19dc6, 0x240ca1cc, 0x2de92c6f,
    0x4a7484aa, 0x5cb0a9dc, 0x76f988da, 0x983e5152, 0xa831c66d, 0xb00327c8, 0xbf597fc7,
    0xc6e00bf3, 0xd5a79147, 0x06ca6351, 0x14292967, 0x27b70a85, 0x2e1b2138, 0x4d2c6dfc,
    0x53380d13, 0x650a7354, 0x766a0abb, 0x81c2c92e, 0x92722c85, 0xa2bfe8a1, 0xa81a664b,
    0xc24b8b70, 0xc76c51a3, 0xd192e819, 0xd6990624, 0xf40e3585, 0x106aa070, 0x19a4c116,
    0x1e376c08, 0x2748774c, 0x34b0bcb5, 0x391c0cb3, 0x4ed8aa4a, 0x5b9cca4f, 0x682e6ff3,
    0x748f82ee, 0x78a5636f, 0x84c87814, 0x8cc70208, 0x90befffa, 0xa4506ceb, 0xbef9a3f7,
    0xc67178f2};

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }
inline uint32_t ch(uint32_t x, uint32_t y, uint32_t z) { return (x & y) ^ (~x & z); }
inline uint32_t maj(uint32_t x, uint32_t y, uint32_t z) { return (x & y) ^ (x & z) ^ (y & z); }
inline uint32_t big_sigma0(uint32_t x) { return rotr(x, 2) ^ rotr(x, 13) ^ rotr(x, 22); }
inline uint32_t big_sigma1(uint32_t x) { return rotr(x, 6) ^ rotr(x, 11) ^ rotr(x, 25); }
inline uint32_t small_sigma0(uint32_t x) { return rotr(x, 7) ^ rotr(x, 18) ^ (x >> 3); }
inline uint32_t small_sigma1(uint32_t x) { return rotr(x, 17) ^ rotr(x, 19) ^ (x >> 10); }

void compress(uint32_t H[8], const uint8_t* block) {
  uint32_t W[64];
  for (int t = 0; t < 16; ++t) {
    W[t] = (uint32_t(block[4 * t]) << 24) | (uint32_t(block[4 * t + 1]) << 16) |
           (uint32_t(block[4 * t + 2]) << 8) | uint32_t(block[4 * t + 3]);
  }
  for (int t = 16; t < 64; ++t)
    W[t] = small_sigma1(W[t - 2]) + W[t - 7] + small_sigma0(W[t - 15]) + W[t - 16];
  uint32_t a = H[0], b = H[1], c = H[2], d = H[3], e = H[4], f = H[5], g = H[6], h = H[7];
  for (int t = 0; t < 64; ++t) {
    uint32_t T1 = h + big_sigma1(e) + ch(e, f, g) + K256[t] + W[t];
    uint32_t T2 = big_sigma0(a) + maj(a, b, c);
    h = g;
    g = f;
    f = e;
    e = d + T1;
    d = c;
    c = b;
    b = a;
    a = T1 + T2;
  }
  H[0] += a; H[1] += b; H[2] += c; H[3] += d;
  H[4] += e; H[5] += f; H[6] += g; H[7] += h;
}

}  // namespace

extern "C" void oracle_sha256(const uint8_t* msg, uint64_t len, uint8_t digest[32]) {
  // Initial hash value: first 32 bits of the fractional parts of the square
  // roots of the first 8 primes (FIPS 180-4 section 5.3.3).
  uint32_t H[8] = {0x6a09e667, 0xbb67ae85, 0x3c6ef372, 0xa54ff53a,
                   0x510e527f, 0x9b05688c, 0x1f83d9ab, 0x5be0cd19};
  uint64_t full = len / 64;
  for (uint64_t i = 0; i < full; ++i) compress(H, msg + 64 * i);
  // Padding: a 1 bit, zeros to 56 mod 64 bytes, then the bit length big-endian.
  uint8_t tail[128];
  std::memset(tail, 0, sizeof tail);
  uint64_t rem = len - 64 * full;
  if (rem) std::memcpy(tail, msg + 64 * full, rem);
  tail[rem] = 0x80;
  uint64_t tail_len = (rem < 56) ? 64 : 128;
  uint64_t bits = len * 8;
  for (int i = 0; i < 8; ++i) tail[tail_len - 1 - i] = uint8_t(bits >> (8 * i));
  compress(H, tail);
  if (tail_len == 128) compress(H, tail + 64);
  for (int i = 0; i < 8; ++i) {
    digest[4 * i] = uint8_t(H[i] >> 24);
    digest[4 * i + 1] = uint8_t(H[i] >> 16);
    digest[4 * i + 2] = uint8_t(H[i] >> 8);
    digest[4 * i + 3] = uint8_t(H[i]);
  }
}
