// CPU oracle for the VBQ decode path in plain C++: single-threaded, no BLAS,
// written to be checked by eye against the definitions.
//
// TEST INFRASTRUCTURE ONLY. Only the tests, __graft_entry__.smoke() and the
// bench's CPU-baseline leg may load this library. The CUDA path never calls it
// and the two share no code; it restates the definitions of oracle/vbq_oracle.py:
//
// * "Variable Bit-width Quantization: Learning Per-Group Precision for
//   'Bigger-but-Smaller' Language Models", abstract: every run of 64
//   consecutive weights of a row has its own bit-width b in {1,2,4,8}, stored as
//   packed low-bit codes. The abstract gives no code grid; this project's grid
//   is w = s * (q - (2^b - 1)/2), s an fp16 scale, q an unsigned b-bit code.
//   Group g of row r covers columns [64g, 64g + 63].
// * The decode step (same abstract: token-by-token decode) with this
//   project's glue: unit-gain RMSNorm (eps given), attention at position 0 (each
//   query head returns its kv group's v), SwiGLU, fp64 residual, and bf16 (round
//   to nearest, ties to even) at every projection input.
//
// Precision: the dequantized weight is computed in fp32, where it is exact (an
// fp16 scale has 11 significant bits, q - c at most 9). Dot products are summed
// in fp64, one term at a time in column order. Build with -ffp-contract=off so
// that no multiply-add is fused.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

constexpr int64_t kGroup = 64;

// IEEE binary16 bit pattern -> exact value (sign, 5-bit exponent with bias 15, 10-bit fraction).
double half_value(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int exp = (h >> 10) & 0x1F;
  const int frac = h & 0x3FF;
  double v;
  if (exp == 0) {
    v = std::ldexp(static_cast<double>(frac), -24);  // subnormal: frac * 2^-24
  } else if (exp == 31) {
    v = frac ? NAN : INFINITY;
  } else {
    v = std::ldexp(static_cast<double>(frac + 1024), exp - 25);  // (1 + frac/1024) * 2^(exp-15)
  }
  return sign ? -v : v;
}

// bfloat16 bit pattern -> exact value: the upper half of a binary32.
double bf16_value(uint16_t b) {
  const uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

// Round a finite real to the nearest bf16 value, ties to even: 8 significant
// bits, the quantum 2^(e-8) for |v| in [2^(e-1), 2^e), never below 2^-133.
uint16_t bf16_bits(double v) {
  double r = 0.0;
  if (v != 0.0) {
    int e = 0;
    (void)std::frexp(v, &e);
    if (e < -125) e = -125;
    const double quantum = std::ldexp(1.0, e - 8);
    r = std::nearbyint(v / quantum) * quantum;  // the default rounding mode: to nearest, ties to even
  } else {
    r = v;
  }
  const float f = static_cast<float>(r);  // exact: a bf16 value is a binary32 value
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return static_cast<uint16_t>(u >> 16);
}

bool valid_width(uint8_t b) { return b == 1 || b == 2 || b == 4 || b == 8; }

// Checks bit-widths and code ranges; false on any violation.
bool check(const uint8_t* codes, const uint8_t* bits, int64_t N, int64_t K) {
  if (N < 0 || K < 0 || K % kGroup) return false;
  const int64_t G = K / kGroup;
  for (int64_t r = 0; r < N; ++r)
    for (int64_t g = 0; g < G; ++g) {
      const uint8_t b = bits[r * G + g];
      if (!valid_width(b)) return false;
      for (int64_t m = 0; m < kGroup; ++m)
        if (codes[r * K + g * kGroup + m] >= (1u << b)) return false;
    }
  return true;
}

// w = s * (q - c_b) in fp32, c_b = (2^b - 1) / 2.
float weight(uint8_t q, uint8_t b, uint16_t s_bits) {
  const float s = static_cast<float>(half_value(s_bits));
  const float c = static_cast<float>((1u << b) - 1u) / 2.0f;
  return s * (static_cast<float>(q) - c);
}

// y_r = sum_k w_rk x_k in fp64, column order. The scale and the offset of a
// group are decoded once for its 64 weights; each weight is still s * (q - c)
// in fp32, as in weight().
void gemv_rows(const uint8_t* codes, const uint8_t* bits, const uint16_t* scales, int64_t N, int64_t K,
               const double* x, double* y) {
  const int64_t G = K / kGroup;
  for (int64_t r = 0; r < N; ++r) {
    double acc = 0.0;
    for (int64_t g = 0; g < G; ++g) {
      const float s = static_cast<float>(half_value(scales[r * G + g]));
      const float c = static_cast<float>((1u << bits[r * G + g]) - 1u) / 2.0f;
      const uint8_t* q = codes + r * K + g * kGroup;
      const double* xg = x + g * kGroup;
      for (int64_t m = 0; m < kGroup; ++m) acc += static_cast<double>(s * (static_cast<float>(q[m]) - c)) * xg[m];
    }
    y[r] = acc;
  }
}

}  // namespace

extern "C" {

// Shapes of a decode-step stack: per layer q, k, v, o, gate, up, down, then the head.
struct VbqOracleModel {
  int32_t n_layers, d, n_heads, n_kv_heads, head_dim, d_ff, vocab;
  double rms_eps;
};

// W [N][K] fp32. Returns 0, or 1 for invalid inputs.
int vbq_oracle_dequant(const uint8_t* codes, const uint8_t* bits, const uint16_t* scales, int64_t N, int64_t K,
                       float* W) {
  if (!check(codes, bits, N, K)) return 1;
  const int64_t G = K / kGroup;
  for (int64_t r = 0; r < N; ++r)
    for (int64_t k = 0; k < K; ++k) W[r * K + k] = weight(codes[r * K + k], bits[r * G + k / kGroup], scales[r * G + k / kGroup]);
  return 0;
}

// y [N] fp64 = W x for bf16 x [K]. Returns 0, or 1 for invalid inputs.
int vbq_oracle_gemv(const uint8_t* codes, const uint8_t* bits, const uint16_t* scales, int64_t N, int64_t K,
                    const uint16_t* x_bf16, double* y) {
  if (!check(codes, bits, N, K)) return 1;
  std::vector<double> x(static_cast<size_t>(K));
  for (int64_t k = 0; k < K; ++k) x[k] = bf16_value(x_bf16[k]);
  gemv_rows(codes, bits, scales, N, K, x.data(), y);
  return 0;
}

// out [N] = ||W_r||_2 (fp64 sum of squares in column order, then the square root).
int vbq_oracle_row_norms(const uint8_t* codes, const uint8_t* bits, const uint16_t* scales, int64_t N, int64_t K,
                         double* out) {
  if (!check(codes, bits, N, K)) return 1;
  const int64_t G = K / kGroup;
  for (int64_t r = 0; r < N; ++r) {
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double w = weight(codes[r * K + k], bits[r * G + k / kGroup], scales[r * G + k / kGroup]);
      acc += w * w;
    }
    out[r] = std::sqrt(acc);
  }
  return 0;
}

// bf16 bit patterns of n real values (round to nearest, ties to even).
void vbq_oracle_to_bf16(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_bits(v[i]);
}

// One decode step. codes/bits/scales hold n_layers * 7 + 1 matrices in the
// order of each layer's q, k, v, o, gate, up, down, then the head; x is the bf16
// input [d] and logits [vocab] receives the result in fp64.
//   h <- x
//   per layer: u = bf16(rmsnorm(h)); q, k, v = Wq u, Wk u, Wv u
//              a = bf16(attention at position 0 of v); h <- h + Wo a
//              u = bf16(rmsnorm(h)); m = bf16(silu(Wgate u) * (Wup u)); h <- h + Wdown m
//   logits = Whead bf16(rmsnorm(h))
// Returns 0, or 1 for invalid shapes or matrices.
int vbq_oracle_decode_step(const VbqOracleModel* m, const uint8_t* const* codes, const uint8_t* const* bits,
                           const uint16_t* const* scales, const uint16_t* x, double* logits) {
  const int64_t d = m->d, nq = int64_t(m->n_heads) * m->head_dim, nkv = int64_t(m->n_kv_heads) * m->head_dim;
  const int64_t ff = m->d_ff;
  if (m->n_layers < 0 || d <= 0 || m->n_kv_heads <= 0 || m->n_heads % m->n_kv_heads) return 1;
  const int64_t shapes[7][2] = {{nq, d}, {nkv, d}, {nkv, d}, {d, nq}, {ff, d}, {ff, d}, {d, ff}};
  for (int l = 0; l <= m->n_layers; ++l)
    for (int p = 0; p < (l < m->n_layers ? 7 : 1); ++p) {
      const size_t i = static_cast<size_t>(l) * 7 + p;
      const int64_t N = l < m->n_layers ? shapes[p][0] : m->vocab, K = l < m->n_layers ? shapes[p][1] : d;
      if (!check(codes[i], bits[i], N, K)) return 1;
    }
  auto rmsnorm_bf16 = [&](const std::vector<double>& h, std::vector<double>* u) {
    double ss = 0.0;
    for (double v : h) ss += v * v;
    const double inv = std::sqrt(ss / static_cast<double>(h.size()) + m->rms_eps);
    u->resize(h.size());
    for (size_t i = 0; i < h.size(); ++i) (*u)[i] = bf16_value(bf16_bits(h[i] / inv));
  };
  auto proj = [&](size_t i, int64_t N, int64_t K, const std::vector<double>& in, std::vector<double>* out) {
    out->assign(static_cast<size_t>(N), 0.0);
    gemv_rows(codes[i], bits[i], scales[i], N, K, in.data(), out->data());
  };
  std::vector<double> h(static_cast<size_t>(d)), u, q, k, v, a(static_cast<size_t>(nq)), y, g, up, mm;
  for (int64_t i = 0; i < d; ++i) h[i] = bf16_value(x[i]);
  const int64_t group = m->n_heads / m->n_kv_heads;
  for (int l = 0; l < m->n_layers; ++l) {
    const size_t b = static_cast<size_t>(l) * 7;
    rmsnorm_bf16(h, &u);
    proj(b + 0, nq, d, u, &q);
    proj(b + 1, nkv, d, u, &k);
    proj(b + 2, nkv, d, u, &v);
    // A softmax over one key is 1: query head i returns the v of its kv head i / group.
    for (int64_t hd = 0; hd < m->n_heads; ++hd)
      for (int64_t j = 0; j < m->head_dim; ++j)
        a[hd * m->head_dim + j] = bf16_value(bf16_bits(v[(hd / group) * m->head_dim + j]));
    proj(b + 3, d, nq, a, &y);
    for (int64_t i = 0; i < d; ++i) h[i] += y[i];
    rmsnorm_bf16(h, &u);
    proj(b + 4, ff, d, u, &g);
    proj(b + 5, ff, d, u, &up);
    mm.resize(static_cast<size_t>(ff));
    for (int64_t i = 0; i < ff; ++i) mm[i] = bf16_value(bf16_bits(g[i] / (1.0 + std::exp(-g[i])) * up[i]));
    proj(b + 6, d, ff, mm, &y);
    for (int64_t i = 0; i < d; ++i) h[i] += y[i];
  }
  rmsnorm_bf16(h, &u);
  std::vector<double> lg;
  proj(static_cast<size_t>(m->n_layers) * 7, m->vocab, d, u, &lg);
  for (int64_t i = 0; i < m->vocab; ++i) logits[i] = lg[i];
  return 0;
}

}  // extern "C"
