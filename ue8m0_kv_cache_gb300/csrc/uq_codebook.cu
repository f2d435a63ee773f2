// uq_codebook.cu -- host computation of the TQ4 codebook ("TurboQuant 완전 정리",
// juhoplayground.github.io, sections "랜덤 회전과 Beta 분포" and "Lloyd-Max 스칼라
// 양자화 (Q_mse)").
//
// After a random rotation, one coordinate of a unit vector in R^d has the
// density f(x) = C_d (1 - x^2)^k on [-1, 1], k = (d-3)/2,
// C_d = Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2)).  The Q_mse codebook is the
// Lloyd-Max quantiser of f: boundaries at the midpoints of neighbouring
// centroids, centroids at the conditional means of their cells.  f is
// symmetric and log-concave, so the fixed point is unique and symmetric; it is
// found on the half-line [0, 1] by alternating the two conditions in double
// precision.  Cell masses are integrated with composite Gauss-Legendre rules
// (nodes from Newton's iteration on the Legendre recurrence); first moments
// use the antiderivative -(1 - x^2)^(k+1) / (2(k+1)) * C_d.
#include <cuda_fp16.h>

#include <cmath>
#include <cstring>
#include <map>
#include <mutex>

#include "uq_internal.h"

namespace uqh {

namespace {

constexpr int kGaussN = 24;    // nodes per panel
constexpr int kPanels = 16;    // panels per cell

struct Gauss {
  double x[kGaussN], w[kGaussN];  // nodes and weights on [-1, 1]
  Gauss() {
    const double pi = std::acos(-1.0);
    for (int i = 0; i < kGaussN; ++i) {
      double z = std::cos(pi * (i + 0.75) / (kGaussN + 0.5));  // initial guess of root i
      double dp = 1.0;
      for (int it = 0; it < 100; ++it) {
        // P_n(z) and P_n'(z) by the three-term recurrence
        double p0 = 1.0, p1 = z;
        for (int n = 2; n <= kGaussN; ++n) {
          const double p2 = ((2.0 * n - 1.0) * z * p1 - (n - 1.0) * p0) / n;
          p0 = p1;
          p1 = p2;
        }
        dp = kGaussN * (z * p1 - p0) / (z * z - 1.0);
        const double dz = p1 / dp;
        z -= dz;
        if (std::fabs(dz) < 1e-16) break;
      }
      x[i] = z;
      w[i] = 2.0 / ((1.0 - z * z) * dp * dp);
    }
  }
};

const Gauss& gauss() {
  static const Gauss g;
  return g;
}

struct Density {
  double k, c;  // exponent (d-3)/2 and normalising constant C_d
  explicit Density(int d)
      : k((d - 3) / 2.0),
        c(std::exp(std::lgamma(d / 2.0) - std::lgamma((d - 1) / 2.0)) / std::sqrt(std::acos(-1.0))) {}
  double f(double x) const {
    const double u = 1.0 - x * x;
    return u <= 0.0 ? 0.0 : c * std::pow(u, k);
  }
  // int_a^b f, 0 <= a <= b <= 1
  double mass(double a, double b) const {
    const Gauss& g = gauss();
    double s = 0.0;
    const double hw = (b - a) / kPanels;
    for (int p = 0; p < kPanels; ++p) {
      const double lo = a + p * hw, mid = lo + 0.5 * hw;
      double t = 0.0;
      for (int i = 0; i < kGaussN; ++i) t += g.w[i] * f(mid + 0.5 * hw * g.x[i]);
      s += 0.5 * hw * t;
    }
    return s;
  }
  // int_a^b x f(x) dx, closed form
  double moment(double a, double b) const {
    const double k1 = k + 1.0;
    return c * (std::pow(1.0 - a * a, k1) - std::pow(1.0 - b * b, k1)) / (2.0 * k1);
  }
};

// Non-negative half of the symmetric Lloyd-Max codebook, ascending.
void lloyd_max_half(int d, int bits, double* c) {
  const int h = 1 << (bits - 1);
  const double sigma = 1.0 / std::sqrt(static_cast<double>(d));
  const Density den(d);
  for (int i = 0; i < h; ++i) c[i] = (i + 0.5) * 3.0 * sigma / h;
  double edges[16 + 1], next[16];
  for (int it = 0; it < 200000; ++it) {
    edges[0] = 0.0;
    for (int i = 1; i < h; ++i) edges[i] = 0.5 * (c[i - 1] + c[i]);
    edges[h] = 1.0;
    double moved = 0.0;
    for (int i = 0; i < h; ++i) {
      next[i] = den.moment(edges[i], edges[i + 1]) / den.mass(edges[i], edges[i + 1]);
      moved = std::fmax(moved, std::fabs(next[i] - c[i]));
    }
    std::memcpy(c, next, sizeof(double) * h);
    if (moved <= 1e-14 * sigma) break;
  }
}

// Nearest f16 value of a non-negative double (ties to even), as a float.
float f16_nearest(double x) {
  if (x >= 65520.0) return INFINITY;
  double quantum;
  if (x < std::ldexp(1.0, -14)) {
    quantum = std::ldexp(1.0, -24);
  } else {
    int e;
    std::frexp(x, &e);  // x in [2^(e-1), 2^e)
    quantum = std::ldexp(1.0, e - 11);
  }
  return static_cast<float>(std::nearbyint(x / quantum) * quantum);
}

std::mutex g_tq_mu;
std::map<int, TqTables> g_tq;

}  // namespace

uq_status tq_codebook_host(int d, int bits, float* mags, float* thresholds) {
  if (bits < 1 || bits > 4 || d < 16 || d > 1024) return UQ_ERR_INVALID_ARG;
  double c[8];
  lloyd_max_half(d, bits, c);
  const int h = 1 << (bits - 1);
  for (int i = 0; i < h; ++i) mags[i] = f16_nearest(c[i]);
  // thresholds between the 2h centroids -c[h-1] < ... < -c[0] < c[0] < ... < c[h-1]
  thresholds[h - 1] = 0.0f;
  for (int i = 0; i + 1 < h; ++i) {
    const float t = static_cast<float>(0.5 * (c[i] + c[i + 1]));
    thresholds[h + i] = t;
    thresholds[h - 2 - i] = -t;
  }
  return UQ_OK;
}

uq_status tq_tables(int d, TqTables* out) {
  std::lock_guard<std::mutex> lk(g_tq_mu);
  auto it = g_tq.find(d);
  if (it == g_tq.end()) {
    TqTables t;
    float mags[8], thr[15];
    const uq_status st = tq_codebook_host(d, 4, mags, thr);
    if (st != UQ_OK) return st;
    uint8_t hi[8], lo[8];
    for (int m = 0; m < 8; ++m) {
      const __half hv = __float2half_rn(mags[m]);  // exact: mags[m] is an f16 value
      uint16_t b;
      std::memcpy(&b, &hv, 2);
      hi[m] = static_cast<uint8_t>(b >> 8);
      lo[m] = static_cast<uint8_t>(b & 0xFF);
    }
    for (int j = 0; j < 7; ++j) t.tpos[j] = thr[8 + j];
    for (int q = 0; q < 2; ++q) {
      t.lut[q] = hi[4 * q] | (hi[4 * q + 1] << 8) | (hi[4 * q + 2] << 16) | (uint32_t(hi[4 * q + 3]) << 24);
      t.lut[2 + q] = lo[4 * q] | (lo[4 * q + 1] << 8) | (lo[4 * q + 2] << 16) | (uint32_t(lo[4 * q + 3]) << 24);
    }
    it = g_tq.emplace(d, t).first;
  }
  *out = it->second;
  return UQ_OK;
}

}  // namespace uqh

extern "C" uq_status uq_tq_codebook(int32_t head_dim, int32_t bits, float* magnitudes, float* thresholds) {
  if (!magnitudes || !thresholds) return UQ_ERR_INVALID_ARG;
  return uqh::tq_codebook_host(head_dim, bits, magnitudes, thresholds);
}
