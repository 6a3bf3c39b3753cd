// Seeded GPT-2 parameter initialisation on the host.
//
// Generator: SplitMix64 (Steele, Lea, Flood, OOPSLA 2014) used counter-style:
// output j is the finaliser applied to seed + (j+1) * 0x9E3779B97F4A7C15, so
// element i of the canonical parameter vector can be drawn independently from
// outputs 2i and 2i+1.  Gaussian values come from the Box-Muller transform in
// double precision with the C library's log and cos, then one rounding to
// float.  Scales: the GPT-2 init of N(0, 0.02) for the embedding and weight
// matrices, with the matrices that project into the residual stream scaled by
// 1/sqrt(2L); LayerNorm gains 1, biases 0, and wte rows at or past V (the
// padding rows of the classifier) 0.
#include <cmath>
#include <cstdint>
#include <thread>
#include <vector>

#include "model_layout.h"

namespace {

inline uint64_t sm64_output(uint64_t seed, uint64_t j) {
  uint64_t z = seed + (j + 1) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

inline double gaussian(uint64_t seed, uint64_t i) {
  uint64_t x = sm64_output(seed, 2 * i);
  uint64_t y = sm64_output(seed, 2 * i + 1);
  double u1 = ((double)(x >> 11) + 1.0) * 0x1p-53;  // (0, 1]
  double u2 = (double)(y >> 11) * 0x1p-53;          // [0, 1)
  const double two_pi = 2.0 * M_PI;
  double angle = two_pi * u2;
  return std::sqrt(-2.0 * std::log(u1)) * std::cos(angle);
}

void fill_gaussian(float* out, uint64_t first_index, size_t n, double stdev, uint64_t seed) {
  unsigned nt = std::thread::hardware_concurrency();
  if (nt == 0) nt = 1;
  if (nt > 32) nt = 32;
  if (n < (size_t)1 << 16) nt = 1;
  std::vector<std::thread> th;
  size_t per = (n + nt - 1) / nt;
  for (unsigned k = 0; k < nt; k++) {
    size_t a = k * per, b = a + per < n ? a + per : n;
    if (a >= b) break;
    th.emplace_back([=] {
      for (size_t e = a; e < b; e++) out[e] = (float)(gaussian(seed, first_index + e) * stdev);
    });
  }
  for (auto& t : th) t.join();
}

}  // namespace

void init_params_host(const gpt2_config& c, uint64_t seed, float* out) {
  ParamLayout pl = param_layout(c);
  const double sd = 0.02, sd_proj = 0.02 / std::sqrt(2.0 * c.L);
  for (int t = 0; t < GPT2_NUM_TENSORS; t++) {
    float* dst = out + pl.off[t];
    size_t n = pl.numel[t];
    switch (t) {
      case GPT2_WTE: {
        size_t nd = (size_t)c.V * c.C;
        fill_gaussian(dst, pl.off[t], nd, sd, seed);
        for (size_t e = nd; e < n; e++) dst[e] = 0.f;
        break;
      }
      case GPT2_WPE: case GPT2_QKVW: case GPT2_FCW:
        fill_gaussian(dst, pl.off[t], n, sd, seed);
        break;
      case GPT2_ATTPROJW: case GPT2_FCPROJW:
        fill_gaussian(dst, pl.off[t], n, sd_proj, seed);
        break;
      case GPT2_LN1W: case GPT2_LN2W: case GPT2_LNFW:
        for (size_t e = 0; e < n; e++) dst[e] = 1.f;
        break;
      default:
        for (size_t e = 0; e < n; e++) dst[e] = 0.f;
    }
  }
}
