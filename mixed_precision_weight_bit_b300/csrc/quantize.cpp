// vbq_quantize_rtn: dense weights to the VBQ grid by round-to-nearest, per
// group of 64 weights along the input dimension, at a given bit map (host).
//
// VBQ abstract: every run of 64 consecutive weights has its own bit-width from
// {1,2,4,8}, and the allocation is stored as packed low-bit codes. The pages
// learn the allocation and the weights; given an allocation, the plainest
// encoding of a dense group onto the grid w = s (q - c_b), c_b = (2^b - 1)/2,
// is absmax round-to-nearest: s = max|w| / c_b (rounded to fp16), q the code
// nearest w / s + c_b, clipped to [0, 2^b - 1]. This serves the measurement
// of how far a quantized model's logits move from the dense ones.
#include <cmath>
#include <cstdint>

#include "internal.h"

namespace {

// Nearest fp16 (ties to even) of a finite v >= 0, as bits.
uint16_t f64_to_f16_bits(double v) {
  if (!(v > 0.0)) return 0;
  if (v >= 65520.0) return 0x7C00;  // at or above the midpoint between 65504 and 2^16: infinity
  if (v < std::ldexp(1.0, -14)) return static_cast<uint16_t>(std::nearbyint(std::ldexp(v, 24)));  // subnormal
  int e = 0;
  (void)std::frexp(v, &e);                                // v in [2^(e-1), 2^e)
  double r = std::nearbyint(std::ldexp(v, 11 - e));       // 11 significant bits, in [1024, 2048]
  if (r == 2048.0) {
    r = 1024.0;
    ++e;
  }
  const int biased = e - 1 + 15;
  if (biased >= 31) return 0x7C00;
  return static_cast<uint16_t>((biased << 10) | (static_cast<int>(r) - 1024));
}

double f16_bits_to_f64(uint16_t h) {
  const int ex = (h >> 10) & 31, fr = h & 1023;
  if (ex == 0) return std::ldexp(static_cast<double>(fr), -24);
  return std::ldexp(1024.0 + fr, ex - 25);
}

}  // namespace

using namespace vbq;

extern "C" vbq_status vbq_quantize_rtn(const float* W, int64_t N, int64_t K, const uint8_t* bits, uint8_t* codes,
                                       uint16_t* scales_f16) {
  if (N < 0 || K < 0 || K % GROUP) return fail(VBQ_ERR_SHAPE, "vbq_quantize_rtn: need N, K >= 0 and K % 64 == 0");
  if (N * K > 0 && (!W || !bits || !codes || !scales_f16))
    return fail(VBQ_ERR_INVALID_ARG, "vbq_quantize_rtn: NULL array");
  const int64_t G = K / GROUP;
  for (int64_t r = 0; r < N; ++r)
    for (int64_t g = 0; g < G; ++g) {
      const uint8_t b = bits[r * G + g];
      if (b != 1 && b != 2 && b != 4 && b != 8)
        return fail(VBQ_ERR_BITS, "vbq_quantize_rtn: bits must be 1, 2, 4 or 8 (row " + std::to_string(r) +
                                      ", group " + std::to_string(g) + ")");
      const float* w = W + r * K + g * GROUP;
      double mx = 0.0;
      for (int i = 0; i < GROUP; ++i) {
        if (!std::isfinite(w[i])) return fail(VBQ_ERR_INVALID_ARG, "vbq_quantize_rtn: non-finite weight");
        mx = std::fmax(mx, std::fabs(static_cast<double>(w[i])));
      }
      const double c = (std::ldexp(1.0, b) - 1.0) / 2.0, qmax = std::ldexp(1.0, b) - 1.0;
      const uint16_t sb = f64_to_f16_bits(mx / c);
      if (sb == 0x7C00) return fail(VBQ_ERR_INVALID_ARG, "vbq_quantize_rtn: a group's scale overflows fp16");
      scales_f16[r * G + g] = sb;
      const double s = f16_bits_to_f64(sb);
      uint8_t* q = codes + r * K + g * GROUP;
      for (int i = 0; i < GROUP; ++i) {
        double v = s > 0.0 ? std::nearbyint(static_cast<double>(w[i]) / s + c) : 0.0;
        v = v < 0.0 ? 0.0 : (v > qmax ? qmax : v);
        q[i] = static_cast<uint8_t>(v);
      }
    }
  return VBQ_OK;
}
