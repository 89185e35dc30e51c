// vbq_pack: logical codes + bit map + scales -> the packed device layout of layout.h.
//
// VBQ abstract ("Variable Bit-width Quantization ..."): once the per-group bit
// allocation is fixed, the weights can be stored as packed low-bit codes. The
// record format, tile order and class ordering are this library's own design.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

#include "internal.h"

namespace {

using namespace vbq;

inline int bits_to_cls(uint8_t b) { return b == 1 ? 0 : b == 2 ? 1 : b == 4 ? 2 : 3; }

// Packs the 64 codes q of one group of class cls as entry j of a step record
// with e entries (layout.h); the record's code bytes start zeroed.
inline void pack_entry(const uint8_t* q, uint32_t cls, uint8_t* rec, uint32_t e, uint32_t j) {
  const uint32_t b = 1u << cls, per_word = 32u / b;
  for (uint32_t m = 0; m < GROUP; ++m) {
    const uint32_t w = m / per_word, r = m % per_word;
    uint32_t* word = reinterpret_cast<uint32_t*>(rec + code_word_off(cls, e, j, w));
    const uint32_t bit = b == 1 ? r : code_bit(b, r);
    *word |= static_cast<uint32_t>(q[m]) << bit;
  }
}

// Entry counts of one super-tile, per group column and class.
void count_super(const uint8_t* bits, int32_t G, int64_t r0, int64_t r1, std::vector<uint32_t>* cnt) {
  cnt->assign(static_cast<size_t>(G) * 4, 0);
  for (int64_t r = r0; r < r1; ++r) {
    const uint8_t* br = bits + r * G;
    for (int32_t g = 0; g < G; ++g) (*cnt)[static_cast<size_t>(g) * 4 + bits_to_cls(br[g])] += 1;
  }
}

// |s| of an fp16 bit pattern, exactly.
double f16_abs(uint16_t h) {
  const uint32_t e = (h >> 10) & 31u, f = h & 1023u;
  if (e == 31) return 1e300;
  return e == 0 ? std::ldexp(static_cast<double>(f), -24) : std::ldexp(static_cast<double>(f | 1024u), static_cast<int>(e) - 25);
}

template <class F>
void parallel_for(int64_t n, F&& f) {
  const int64_t hw = std::max(1u, std::thread::hardware_concurrency());
  const int64_t nt = std::min<int64_t>(hw, std::max<int64_t>(1, n));
  if (nt <= 1) {
    for (int64_t i = 0; i < n; ++i) f(i);
    return;
  }
  std::atomic<int64_t> next{0};
  std::vector<std::thread> th;
  for (int64_t t = 0; t < nt; ++t)
    th.emplace_back([&]() {
      for (int64_t i = next.fetch_add(1); i < n; i = next.fetch_add(1)) f(i);
    });
  for (auto& t : th) t.join();
}

inline uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

}  // namespace

namespace vbq {

// The GEMV plan of a matrix alone (also used after a device change of sms).
vbq_status build_gemv_plan(vbq_matrix* m, cudaStream_t st);
void free_gemv_plan(vbq_matrix* m);

}  // namespace vbq

extern "C" vbq_status vbq_pack(const uint8_t* codes, const uint8_t* bits, const uint16_t* scales_f16, int64_t N,
                               int64_t K, void* stream, vbq_matrix** out) {
  if (!out) return fail(VBQ_ERR_INVALID_ARG, "vbq_pack: out is NULL");
  *out = nullptr;
  if (N < 0 || K < 0) return fail(VBQ_ERR_SHAPE, "vbq_pack: negative N or K");
  if (K % GROUP) return fail(VBQ_ERR_SHAPE, "vbq_pack: K must be a multiple of 64");
  if (K / GROUP > MAX_G) return fail(VBQ_ERR_SHAPE, "vbq_pack: K/64 must be <= 65535");
  if (N >= (int64_t(1) << 31)) return fail(VBQ_ERR_SHAPE, "vbq_pack: N must be < 2^31");
  const int32_t G = static_cast<int32_t>(K / GROUP);
  if (N * G > 0 && (!codes || !bits || !scales_f16)) return fail(VBQ_ERR_INVALID_ARG, "vbq_pack: NULL input array");

  // Validate bit-widths and code ranges before allocating anything.
  std::atomic<int> bad_bits{0}, bad_code{0};
  std::atomic<int64_t> bad_where{-1};
  parallel_for(N, [&](int64_t r) {
    for (int32_t g = 0; g < G; ++g) {
      const uint8_t b = bits[r * G + g];
      if (b != 1 && b != 2 && b != 4 && b != 8) {
        bad_bits = 1;
        bad_where = r * G + g;
        return;
      }
      const uint8_t lim = static_cast<uint8_t>((1u << b) - 1u);
      const uint8_t* q = codes + r * K + static_cast<int64_t>(g) * GROUP;
      uint8_t over = 0;
      for (int m = 0; m < GROUP; ++m) over |= static_cast<uint8_t>(q[m] > lim);
      if (over) {
        bad_code = 1;
        bad_where = r * G + g;
        return;
      }
    }
  });
  if (bad_bits) return fail(VBQ_ERR_BITS, "vbq_pack: bit-width not in {1,2,4,8} at group index " +
                                              std::to_string(bad_where.load()));
  if (bad_code) return fail(VBQ_ERR_CODE_RANGE, "vbq_pack: code >= 2^b in group index " +
                                                    std::to_string(bad_where.load()));

  auto* m = new (std::nothrow) vbq_matrix();
  if (!m) return fail(VBQ_ERR_OOM, "vbq_pack: host allocation");
  m->N = N;
  m->K = K;
  m->G = G;
  if (cudaGetDevice(&m->device) != cudaSuccess) {
    delete m;
    return fail(VBQ_ERR_CUDA, "vbq_pack: no CUDA device");
  }
  const int32_t nt = static_cast<int32_t>((N + TILE - 1) / TILE);
  const int32_t ns = static_cast<int32_t>((N + SROWS - 1) / SROWS);
  m->n_tiles = nt;
  m->n_super = ns;

  // Pass 1: per super-tile, runs and bytes.
  std::vector<std::vector<uint32_t>> counts(ns);
  std::vector<uint64_t> st_bytes(ns, 0), st_runs(ns, 0), st_steps(ns, 0);
  parallel_for(ns, [&](int64_t t) {
    count_super(bits, G, t * SROWS, std::min<int64_t>(N, (t + 1) * SROWS), &counts[t]);
    uint64_t b = 0, runs = 0, steps = 0;
    for (int32_t g = 0; g < G; ++g)
      for (int c = 0; c < 4; ++c) {
        const uint32_t n = counts[t][static_cast<size_t>(g) * 4 + c];
        if (!n) continue;
        b += run_bytes(c, n);
        runs += 1;
        steps += run_steps(c, n);
      }
    st_bytes[t] = b;
    st_runs[t] = runs;
    st_steps[t] = steps;
  });
  std::vector<uint64_t> byte0(ns + 1, 0), run0(ns + 1, 0);
  int64_t n_steps = 0;
  for (int32_t t = 0; t < ns; ++t) {
    byte0[t + 1] = byte0[t] + st_bytes[t];
    run0[t + 1] = run0[t] + st_runs[t];
    n_steps += static_cast<int64_t>(st_steps[t]);
  }
  const uint64_t data_bytes = byte0[ns];
  const uint64_t o_tiles = align256(std::max<uint64_t>(data_bytes, 16));
  const uint64_t total = align256(o_tiles + 8ull * (ns + 1));

  std::vector<uint8_t> host;
  try {
    host.assign(total, 0);
    m->runs.assign(run0[ns], RunInfo{});
  } catch (...) {
    delete m;
    return fail(VBQ_ERR_OOM, "vbq_pack: host staging buffer");
  }

  // Pass 2: write the records.
  parallel_for(ns, [&](int64_t t) {
    const int64_t r0 = t * SROWS, r1 = std::min<int64_t>(N, (t + 1) * SROWS);
    const uint32_t ntl = static_cast<uint32_t>((r1 - r0 + TILE - 1) / TILE);
    uint64_t o = byte0[t];
    uint64_t ri = run0[t];
    std::vector<uint32_t> rows[4];
    for (int32_t g = 0; g < G; ++g) {
      for (int c = 0; c < 4; ++c) rows[c].clear();
      for (int64_t r = r0; r < r1; ++r) rows[bits_to_cls(bits[r * G + g])].push_back(static_cast<uint32_t>(r));
      for (int c = 0; c < 4; ++c) {
        const uint32_t n = static_cast<uint32_t>(rows[c].size());
        if (!n) continue;
        RunInfo& info = m->runs[ri++];
        info.off = o;
        RunHeader h{};
        h.row0 = static_cast<uint32_t>(r0);
        h.g = static_cast<uint16_t>(g);
        h.cls = static_cast<uint8_t>(c);
        h.ntl = static_cast<uint8_t>(ntl);
        h.n = static_cast<uint16_t>(n);
        uint16_t pc[3];
        for (int q = 0; q < 3; ++q) {
          const int64_t lim = r0 + int64_t(q + 1) * TILE;
          pc[q] = static_cast<uint16_t>(std::lower_bound(rows[c].begin(), rows[c].end(), static_cast<uint32_t>(
                                                             std::min<int64_t>(lim, int64_t(UINT32_MAX)))) -
                                        rows[c].begin());
        }
        h.c1 = pc[0];
        h.c2 = pc[1];
        h.c3 = pc[2];
        info.h = h;
        std::memcpy(host.data() + o, &h, sizeof(h));
        o += HEADER_BYTES;
        const uint32_t eps = entries_per_step(c);
        const int b = cls_bits(c);
        for (uint32_t done = 0; done < n; done += eps) {
          const uint32_t e = std::min(eps, n - done);
          uint8_t* rec = host.data() + o;
          uint16_t* sc = reinterpret_cast<uint16_t*>(rec + rec_scale_off(c, e));
          uint8_t* rw = rec + rec_row_off(c, e);
          std::memset(rec, 0, rec_code_bytes(c, e));
          for (uint32_t j = 0; j < e; ++j) {
            const int64_t r = rows[c][done + j];
            pack_entry(codes + r * K + static_cast<int64_t>(g) * GROUP, c, rec, e, j);
            sc[j] = scales_f16[r * G + g];
            rw[j] = static_cast<uint8_t>((r - r0) % TILE);
          }
          o += rec_bytes(c, e);
        }
      }
    }
  });
  std::memcpy(host.data() + o_tiles, byte0.data(), 8ull * (ns + 1));

  // Largest row L1 norm sum_k |w_rk| (exact in double, rounded up to float):
  // every partial sum of a row's products is at most this times max|x|.
  std::vector<double> l1(N, 0.0);
  parallel_for(N, [&](int64_t r) {
    double acc = 0.0;
    for (int32_t g = 0; g < G; ++g) {
      const int b = bits[r * G + g];
      const double c = ((1 << b) - 1) * 0.5;
      double sq = 0.0;
      const uint8_t* q = codes + r * K + static_cast<int64_t>(g) * GROUP;
      for (int mm = 0; mm < GROUP; ++mm) sq += std::fabs(q[mm] - c);
      acc += f16_abs(scales_f16[r * G + g]) * sq;
    }
    l1[r] = acc;
  });
  double l1max = 0.0;
  for (double v : l1) l1max = std::max(l1max, v);
  m->max_row_l1 = l1max >= 3.0e38 ? 3.0e38f : std::nextafter(static_cast<float>(l1max), 3.0e38f);

  int64_t cnt[4] = {0, 0, 0, 0};
  int64_t code_bytes = 0;
  uint16_t max_mag = 0;  // largest |s| as fp16 magnitude bits (monotone in the value for finite fp16)
  for (int64_t i = 0; i < N * G; ++i) {
    const int c = bits_to_cls(bits[i]);
    ++cnt[c];
    code_bytes += 8 * cls_bits(c);
    const uint16_t mag = scales_f16[i] & 0x7FFFu;
    if (mag > max_mag) max_mag = mag;
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = dev_alloc(reinterpret_cast<void**>(&m->dev_base), total);
  if (e != cudaSuccess) {
    delete m;
    cudaGetLastError();
    return fail(e == cudaErrorMemoryAllocation ? VBQ_ERR_OOM : VBQ_ERR_CUDA,
                std::string("vbq_pack: cudaMalloc: ") + cudaGetErrorString(e));
  }
  e = cudaMemcpyAsync(m->dev_base, host.data(), total, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    cudaFree(m->dev_base);
    delete m;
    return cuda_fail(e, "vbq_pack: upload");
  }
  m->data = m->dev_base;
  m->st_byte0 = reinterpret_cast<const uint64_t*>(m->dev_base + o_tiles);
  m->n_runs = static_cast<int64_t>(run0[ns]);
  m->n_steps = n_steps;
  m->data_bytes = static_cast<int64_t>(data_bytes);
  m->code_bytes = code_bytes;
  for (int c = 0; c < 4; ++c) m->groups_by_bits[c] = cnt[c];
  m->max_scale_bits = max_mag;
  {  // fp16 magnitude bits to float (exact)
    const uint32_t ex = (max_mag >> 10) & 31u, f = max_mag & 1023u;
    m->max_scale = ex == 31 ? 1e30f
                   : ex == 0 ? std::ldexp(static_cast<float>(f), -24)
                             : std::ldexp(static_cast<float>(f | 1024u), static_cast<int>(ex) - 25);
  }
  // First run of each (super-tile, group column) block, for the tensor-core path.
  m->block_run.assign(static_cast<size_t>(ns) * G + 1, static_cast<uint32_t>(m->n_runs));
  for (int64_t r = static_cast<int64_t>(m->runs.size()) - 1; r >= 0; --r) {
    const RunInfo& ri = m->runs[r];
    m->block_run[static_cast<size_t>(ri.st()) * G + ri.h.g] = static_cast<uint32_t>(r);
  }

  vbq_status s = build_gemv_plan(m, st);
  if (s != VBQ_OK) {
    cudaFree(m->dev_base);
    delete m;
    return s;
  }
  m->total_bytes = static_cast<int64_t>(total);
  m->meta_bytes = m->total_bytes - code_bytes;
  *out = m;
  return VBQ_OK;
}

extern "C" void vbq_matrix_free(vbq_matrix* m) {
  if (!m) return;
  if (m->dev_base) {
    int cur = 0;
    cudaGetDevice(&cur);
    cudaSetDevice(m->device);
    cudaDeviceSynchronize();
    cudaFree(m->dev_base);
    free_gemv_plan(m);
    tc_forget(m);
    cudaSetDevice(cur);
  }
  delete m;
}

extern "C" vbq_status vbq_matrix_info(const vbq_matrix* m, vbq_info* info) {
  if (!m || !info) return fail(VBQ_ERR_INVALID_ARG, "vbq_matrix_info: NULL argument");
  info->N = m->N;
  info->K = m->K;
  info->code_bytes = m->code_bytes;
  info->meta_bytes = m->meta_bytes;
  info->total_bytes = m->total_bytes;
  info->mean_bits = (m->N * m->K) ? 8.0 * static_cast<double>(m->code_bytes) / static_cast<double>(m->N * m->K) : 0.0;
  info->n_tiles = m->n_tiles;
  info->n_steps = static_cast<int32_t>(std::min<int64_t>(m->n_steps, INT32_MAX));
  for (int c = 0; c < 4; ++c) info->groups_by_bits[c] = m->groups_by_bits[c];
  return VBQ_OK;
}
