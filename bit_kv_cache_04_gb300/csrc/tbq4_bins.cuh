// TBQ4 index by table lookup.  The index of a normalized value u is the
// number of the 15 ascending midpoints of the 16-entry Lloyd-Max table that lie
// strictly below u (trefon.com, "Matematyka cache KV": 4-bit indices into a
// 16-entry codebook).  Binning u by the float bits of its magnitude >> 20
// (eight bins per octave) puts at most one midpoint in a bin when the nonzero
// midpoints' magnitudes lie more than 2^(1/8) apart (the table's neighbouring
// ratios are 1.28 and more; the host checks it).  Two tables of kTbqBins bins,
// one for u >= +0 and one for u <= -0, hold per bin the count of midpoints
// below every value of the bin and the midpoint inside it (+inf when none), so
// index(u) = base + (u > thr) exactly.  Bin 0 takes every magnitude below key
// k0 + 1 (it holds the zero midpoint), the last bin every magnitude from key
// k0 + kTbqBins - 1 up (infinity included).
#pragma once
#include <cmath>
#include <cstdint>
#include <cstring>

namespace kvq {

constexpr int kTbqBins = 32;

__host__ __device__ inline uint32_t tbq_bits(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  return u;
}

__host__ __device__ inline float tbq_float(uint32_t u) {
  float x;
  memcpy(&x, &u, 4);
  return x;
}

// One below the smallest bin key of a nonzero midpoint's magnitude.
__host__ __device__ inline int tbq4_bin_k0(const float* t) {
  int k = 2047;
  for (int j = 0; j < 15; ++j) {
    const uint32_t m = tbq_bits(t[j]) & 0x7FFFFFFFu;
    const int key = (int)(m >> 20);
    if (m != 0 && key < k) k = key;
  }
  return k - 1;
}

// Entry e of the tables (e < kTbqBins: u >= +0, else u <= -0; bin e mod
// kTbqBins): *thr, *base as above; returns how many midpoints the bin holds.
__host__ __device__ inline int tbq4_bin_entry(const float* t, int k0, int e, float* thr, int* base) {
  const bool neg = e >= kTbqBins;
  const int b = e % kTbqBins;
  const bool last = b == kTbqBins - 1;
  // the bin's magnitudes: [A, B), with A = +0 for bin 0 and no B for the last
  const float A = b == 0 ? 0.f : tbq_float((uint32_t)(k0 + b) << 20);
  const float B = tbq_float((uint32_t)(k0 + b + 1) << 20);
  int below = 0, in = 0;
  float th = INFINITY;
  for (int j = 0; j < 15; ++j) {
    const float x = t[j];
    bool lt, inside;
    if (!neg) {  // u in [A, B)
      lt = x < A;
      inside = !lt && (last || x < B);
    } else {  // u in (-B, -A]; -0 <= +0 holds, so bin 0 holds the zero midpoint
      lt = !last && x <= -B;
      inside = x <= -A && (last || x > -B);
    }
    below += lt ? 1 : 0;
    if (inside) {
      ++in;
      th = x;
    }
  }
  *thr = th;
  *base = below;
  return in;
}

}  // namespace kvq
