// wp_nf4_host.cpp -- the 16 NormalFloat levels, derived on the host at load time.
//
// QLoRA (Dettmers et al., 2023), 4-bit NormalFloat: quantiles of the standard normal
// at evenly spaced probabilities between 1/2 and an upper probability delta -- 9
// points (8 positive levels and 0) on the positive side, 8 points (7 negative levels
// and 0) on the negative side -- merged with a single zero and divided by the largest
// so the levels span [-1, 1].  delta is the mean of 1 - 1/(2*15) and 1 - 1/(2*16).
// The 4-bit base weights used by the Unsloth fast_lora walkthrough (section 3,
// matmul_lora) and the InvokeAI quantised layer (section 五) are dequantised through
// this table.
//
// The inverse normal CDF is found by bisection on Phi(x) = erfc(-x / sqrt 2) / 2 in
// double precision, and each level is rounded once to float.
#include <algorithm>
#include <cmath>
#include <mutex>

namespace wp {

namespace {

double phi(double x) { return 0.5 * std::erfc(-x / std::sqrt(2.0)); }

double inv_phi(double p) {
  double lo = -40.0, hi = 40.0;
  for (int i = 0; i < 200; ++i) {
    const double mid = 0.5 * (lo + hi);
    if (mid == lo || mid == hi) break;
    if (phi(mid) < p) lo = mid; else hi = mid;
  }
  return 0.5 * (lo + hi);
}

float g_table[16];
std::once_flag g_once;

void build() {
  const double delta = 0.5 * ((1.0 - 1.0 / 30.0) + (1.0 - 1.0 / 32.0));
  const double top = inv_phi(delta);
  double v[16];
  int n = 0;
  for (int j = 0; j < 8; ++j) v[n++] = inv_phi(delta - j * (delta - 0.5) / 8.0) / top;
  for (int j = 0; j < 7; ++j) v[n++] = -inv_phi(delta - j * (delta - 0.5) / 7.0) / top;
  v[n++] = 0.0;
  std::sort(v, v + 16);
  for (int i = 0; i < 16; ++i) g_table[i] = static_cast<float>(v[i]);
}

}  // namespace

void nf4_codebook_host(float out[16]) {
  std::call_once(g_once, build);
  for (int i = 0; i < 16; ++i) out[i] = g_table[i];
}

}  // namespace wp
