// cbq_pack.cpp -- host quantiser behind cbq_pack(): fp32 weights -> codes,
// E8M0 group scales and one E4M3 codebook per row.
//
// "Hibana: Fast Agentic Inference on Unified-Memory Devices", section "Model
// surgery / Three-bit weights": every weight of a 32-weight group is stored
// as a 3-bit index into an 8-entry FP8 codebook, with one 8-bit scale per
// group.  The pages give no rule for choosing the codebook; the one fixed here
// (and in include/cbq.h)
// is: power-of-two group scale from the group maximum, 8-centroid 1-D Lloyd
// per row over the scaled values, centroids rounded to E4M3 and sorted,
// nearest-centroid codes.  The result is deterministic and independent of the
// host (compiled without floating-point contraction).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include "cbq_internal.h"

namespace cbq {

namespace {

// The 127 non-negative finite E4M3 values, ascending; index == byte.
struct E4M3Table {
  double v[127];
  E4M3Table() {
    for (int b = 0; b < 127; ++b) {
      const int e = b >> 3, m = b & 7;
      v[b] = e ? std::ldexp(1.0 + m / 8.0, e - 7) : std::ldexp(m / 8.0, -6);
    }
  }
};
const E4M3Table& table() {
  static const E4M3Table t;
  return t;
}

double e4m3_to_double(uint8_t b) {
  const double mag = table().v[b & 0x7F];
  return (b & 0x80) ? -mag : mag;
}

// Nearest E4M3 byte (ties: even mantissa, i.e. even byte), saturating at 448.
uint8_t double_to_e4m3(double x) {
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  const double ax = std::fabs(x);
  const double* v = table().v;
  if (ax >= v[126]) return sign | 126;
  // first value >= ax
  const int hi = static_cast<int>(std::lower_bound(v, v + 127, ax) - v);
  if (v[hi] == ax) return sign | static_cast<uint8_t>(hi);
  const int lo = hi - 1;
  const double dlo = ax - v[lo], dhi = v[hi] - ax;
  int pick;
  if (dlo < dhi) pick = lo;
  else if (dhi < dlo) pick = hi;
  else pick = (lo % 2 == 0) ? lo : hi;
  return sign | static_cast<uint8_t>(pick);
}

// s = clamp(127 + ceil(log2(amax)), 0, 254); 127 for an all-zero group.
uint8_t scale_byte(const float* w) {
  double amax = 0.0;
  for (int j = 0; j < 32; ++j) amax = std::max(amax, std::fabs(static_cast<double>(w[j])));
  if (amax == 0.0) return 127;
  const int fl = std::ilogb(amax);                       // floor(log2)
  const int cl = (std::ldexp(1.0, fl) == amax) ? fl : fl + 1;
  return static_cast<uint8_t>(std::min(254, std::max(0, 127 + cl)));
}

void put_group(uint8_t* dst, const uint8_t* c32) {
  uint64_t lo = 0;   // bits 0..63  (codes 0..20 and bit 0 of code 21)
  uint32_t hi = 0;   // bits 64..95
  for (int j = 0; j < 32; ++j) {
    const int bit = 3 * j;
    const uint64_t c = c32[j] & 7u;
    if (bit + 3 <= 64) {
      lo |= c << bit;
    } else if (bit >= 64) {
      hi |= static_cast<uint32_t>(c) << (bit - 64);
    } else {  // straddles bit 64
      lo |= c << bit;
      hi |= static_cast<uint32_t>(c >> (64 - bit));
    }
  }
  for (int i = 0; i < 8; ++i) dst[i] = static_cast<uint8_t>(lo >> (8 * i));
  for (int i = 0; i < 4; ++i) dst[8 + i] = static_cast<uint8_t>(hi >> (8 * i));
}

int nearest(double u, const double* c) {
  int best = 0;
  double bd = std::fabs(u - c[0]);
  for (int i = 1; i < 8; ++i) {
    const double d = std::fabs(u - c[i]);
    if (d < bd) {
      bd = d;
      best = i;
    }
  }
  return best;
}

}  // namespace

int pack_host(const float* W, int N, int K, uint8_t* codes, uint8_t* scales,
              uint8_t* codebooks) {
  const int G = K / 32;
  for (long long i = 0; i < static_cast<long long>(N) * K; ++i)
    if (!std::isfinite(W[i])) return CBQ_EINVAL;
  std::vector<double> u(K), sorted(K);
  std::vector<uint8_t> idx(K);
  for (int n = 0; n < N; ++n) {
    const float* wr = W + static_cast<size_t>(n) * K;
    uint8_t* sr = scales + static_cast<size_t>(n) * G;
    for (int g = 0; g < G; ++g) {
      sr[g] = scale_byte(wr + 32 * g);
      const double inv = std::ldexp(1.0, 127 - sr[g]);
      for (int j = 0; j < 32; ++j) u[32 * g + j] = static_cast<double>(wr[32 * g + j]) * inv;
    }
    // Lloyd, 8 centroids, quantile start, 16 rounds
    std::copy(u.begin(), u.end(), sorted.begin());
    std::sort(sorted.begin(), sorted.end());
    double cen[8];
    for (int i = 0; i < 8; ++i) cen[i] = sorted[static_cast<size_t>((2 * i + 1) * K / 16)];
    for (int round = 0; round < 16; ++round) {
      double sum[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      long long cnt[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      for (int k = 0; k < K; ++k) {
        const int c = nearest(u[k], cen);
        sum[c] += u[k];
        ++cnt[c];
      }
      for (int i = 0; i < 8; ++i)
        if (cnt[i]) cen[i] = sum[i] / static_cast<double>(cnt[i]);
    }
    uint8_t cb[8];
    for (int i = 0; i < 8; ++i) cb[i] = double_to_e4m3(cen[i]);
    std::stable_sort(cb, cb + 8, [](uint8_t x, uint8_t y) { return e4m3_to_double(x) < e4m3_to_double(y); });
    std::memcpy(codebooks + static_cast<size_t>(n) * 8, cb, 8);
    double cbv[8];
    for (int i = 0; i < 8; ++i) cbv[i] = e4m3_to_double(cb[i]);
    for (int k = 0; k < K; ++k) idx[k] = static_cast<uint8_t>(nearest(u[k], cbv));
    // tile order: 128-row tile, then k-tile block of the tile's rows x 48 B
    const int t = n / 128, rows_t = std::min(128, N - 128 * t), i = n % 128;
    uint8_t* tile = codes + static_cast<size_t>(t) * 128 * (3 * static_cast<size_t>(K) / 8);
    for (int g = 0; g < G; ++g)
      put_group(tile + static_cast<size_t>(g / 4) * rows_t * 48 + i * 48 + (g % 4) * 12, idx.data() + 32 * g);
  }
  return CBQ_OK;
}

}  // namespace cbq
