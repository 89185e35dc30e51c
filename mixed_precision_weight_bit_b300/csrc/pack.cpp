// vbq_pack: logical codes + bit map + scales -> the packed device layout of layout.h.
//
// VBQ abstract ("Variable Bit-width Quantization ..."): once the per-group bit
// allocation is fixed, the weights can be stored as packed low-bit codes. The
// record format, tile plan and class ordering are this library's own design.
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

// Packs the 64 codes of one group into 8*b bytes.
//  b = 1, 2, 4: bit-planes. Plane p (bit p of every code) fills bytes [8p, 8p+8),
//               with code m's bit at bit m of the plane (little-endian).
//  b = 8:       one byte per code, code m in byte m.
inline void pack_entry(const uint8_t* q, int b, uint8_t* dst) {
  const int nbytes = 8 * b;
  std::memset(dst, 0, nbytes);
  if (b == 8) {
    std::memcpy(dst, q, GROUP);
    return;
  }
  for (int p = 0; p < b; ++p)
    for (int m = 0; m < GROUP; ++m) dst[8 * p + (m >> 3)] |= static_cast<uint8_t>(((q[m] >> p) & 1u) << (m & 7));
}

struct TilePlan {
  std::vector<uint32_t> row0;  // n_tiles + 1
};

// Equal-byte tiles of at most TILE_MAX rows. A row's weight is the bytes its
// groups take in the stream (codes plus scale plus row index).
TilePlan plan_tiles(const uint8_t* bits, int64_t N, int32_t G) {
  TilePlan p;
  std::vector<double> pre(static_cast<size_t>(N) + 1, 0.0);
  for (int64_t r = 0; r < N; ++r) {
    double rb = 0.0;
    const uint8_t* br = bits + r * G;
    for (int32_t g = 0; g < G; ++g) rb += 8.0 * br[g] + 3.0;
    pre[r + 1] = pre[r] + rb;
  }
  p.row0.push_back(0);
  if (N == 0) return p;
  const int64_t nominal = (N + TILE_MAX - 1) / TILE_MAX;
  const double target = pre[N] / static_cast<double>(nominal);
  int64_t start = 0;
  while (start < N) {
    const double thr = pre[start] + target;
    int64_t end = start + 1;
    while (end < N && end - start < TILE_MAX && pre[end] < thr) ++end;
    p.row0.push_back(static_cast<uint32_t>(end));
    start = end;
  }
  return p;
}

struct TileCount {
  uint32_t runs = 0, steps = 0;
  uint64_t bytes = 0;
};

// Run, step and record-byte counts of one tile.
TileCount count_tile(const uint8_t* bits, int32_t G, uint32_t r0, uint32_t r1) {
  TileCount tc;
  for (int32_t g = 0; g < G; ++g) {
    uint32_t n[4] = {0, 0, 0, 0};
    for (uint32_t r = r0; r < r1; ++r) ++n[bits_to_cls(bits[static_cast<int64_t>(r) * G + g])];
    for (int c = 0; c < 4; ++c) {
      if (!n[c]) continue;
      const uint32_t eps = entries_per_step(c);
      tc.runs += 1;
      for (uint32_t done = 0; done < n[c]; done += eps) {
        const uint32_t e = std::min(eps, n[c] - done);
        tc.steps += 1;
        tc.bytes += rec_bytes(c, e);
      }
    }
  }
  return tc;
}

// Writes the runs of one tile: records into data, descriptors and offsets into desc/off.
void fill_tile(const uint8_t* codes, const uint8_t* bits, const uint16_t* scales, int64_t K, int32_t G,
               uint32_t r0, uint32_t r1, uint32_t run0, uint64_t byte0, uint8_t* data, uint32_t* desc,
               uint32_t* off) {
  uint32_t ri = run0;
  uint64_t o = byte0;
  std::vector<uint32_t> rows[4];
  for (int c = 0; c < 4; ++c) rows[c].reserve(r1 - r0);
  for (int32_t g = 0; g < G; ++g) {
    for (int c = 0; c < 4; ++c) rows[c].clear();
    for (uint32_t r = r0; r < r1; ++r) rows[bits_to_cls(bits[static_cast<int64_t>(r) * G + g])].push_back(r);
    for (int c = 0; c < 4; ++c) {
      const uint32_t n = static_cast<uint32_t>(rows[c].size());
      if (!n) continue;
      desc[ri] = make_run(static_cast<uint32_t>(g), static_cast<uint32_t>(c), n);
      off[ri] = static_cast<uint32_t>(o >> 4);
      ++ri;
      const uint32_t eps = entries_per_step(c);
      const int b = cls_bits(c);
      for (uint32_t done = 0; done < n; done += eps) {
        const uint32_t e = std::min(eps, n - done);
        uint8_t* rec = data + o;
        const uint32_t rb = rec_bytes(c, e);
        std::memset(rec, 0, rb);
        uint16_t* sc = reinterpret_cast<uint16_t*>(rec + rec_scale_off(c, e));
        uint8_t* rw = rec + rec_row_off(c, e);
        for (uint32_t j = 0; j < e; ++j) {
          const uint32_t r = rows[c][done + j];
          pack_entry(codes + static_cast<int64_t>(r) * K + static_cast<int64_t>(g) * GROUP, b, rec + j * 8u * b);
          sc[j] = scales[static_cast<int64_t>(r) * G + g];
          rw[j] = static_cast<uint8_t>(r - r0);
        }
        o += rb;
      }
    }
  }
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

  TilePlan plan = plan_tiles(bits, N, G);
  const int32_t nt = static_cast<int32_t>(plan.row0.size()) - 1;
  std::vector<TileCount> tcs(nt);
  parallel_for(nt, [&](int64_t t) { tcs[t] = count_tile(bits, G, plan.row0[t], plan.row0[t + 1]); });
  std::vector<uint32_t> run0(nt + 1, 0);
  std::vector<uint64_t> byte0(nt + 1, 0);
  int64_t n_steps = 0;
  for (int32_t t = 0; t < nt; ++t) {
    run0[t + 1] = run0[t] + tcs[t].runs;
    byte0[t + 1] = byte0[t] + tcs[t].bytes;
    n_steps += tcs[t].steps;
  }
  const uint32_t R = run0[nt];
  const uint64_t data_bytes = byte0[nt];
  if ((data_bytes >> 4) >= (uint64_t(1) << 32)) {
    delete m;
    return fail(VBQ_ERR_SHAPE, "vbq_pack: packed matrix exceeds 64 GiB");
  }

  // One host staging buffer laid out exactly like the device allocation.
  const uint64_t o_desc = align256(std::max<uint64_t>(data_bytes, 16));
  const uint64_t o_off = align256(o_desc + 4ull * std::max<uint32_t>(R, 1));
  const uint64_t o_row0 = align256(o_off + 4ull * (R + 1));
  const uint64_t o_run0 = align256(o_row0 + 4ull * (nt + 1));
  const uint64_t total = align256(o_run0 + 4ull * (nt + 1));
  std::vector<uint8_t> host;
  try {
    host.assign(total, 0);
    m->h_run_desc.assign(R, 0);
    m->h_run_off.assign(R + 1, 0);
  } catch (...) {
    delete m;
    return fail(VBQ_ERR_OOM, "vbq_pack: host staging buffer");
  }
  parallel_for(nt, [&](int64_t t) {
    fill_tile(codes, bits, scales_f16, K, G, plan.row0[t], plan.row0[t + 1], run0[t], byte0[t], host.data(),
              m->h_run_desc.data(), m->h_run_off.data());
  });
  m->h_run_off[R] = static_cast<uint32_t>(data_bytes >> 4);
  std::memcpy(host.data() + o_desc, m->h_run_desc.data(), 4ull * R);
  std::memcpy(host.data() + o_off, m->h_run_off.data(), 4ull * (R + 1));
  std::memcpy(host.data() + o_row0, plan.row0.data(), 4ull * (nt + 1));
  std::memcpy(host.data() + o_run0, run0.data(), 4ull * (nt + 1));

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
  cudaError_t e = cudaMalloc(&m->dev_base, total);
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
  m->run_desc = reinterpret_cast<const uint32_t*>(m->dev_base + o_desc);
  m->run_off = reinterpret_cast<const uint32_t*>(m->dev_base + o_off);
  m->tile_row0 = reinterpret_cast<const uint32_t*>(m->dev_base + o_row0);
  m->tile_run0 = reinterpret_cast<const uint32_t*>(m->dev_base + o_run0);
  m->h_tile_row0 = plan.row0;
  m->h_tile_run0 = run0;
  m->n_tiles = nt;
  m->n_runs = static_cast<int32_t>(R);
  m->n_steps = n_steps;
  m->data_bytes = static_cast<int64_t>(data_bytes);
  m->code_bytes = code_bytes;
  for (int c = 0; c < 4; ++c) m->groups_by_bits[c] = cnt[c];
  {  // the largest (tile, column) record span
    int64_t best = 0;
    for (int32_t t = 0; t < nt; ++t) {
      uint32_t r = run0[t];
      while (r < run0[t + 1]) {
        uint32_t e = r + 1;
        while (e < run0[t + 1] && run_g(m->h_run_desc[e]) == run_g(m->h_run_desc[r])) ++e;
        best = std::max<int64_t>(best, 16ll * (m->h_run_off[e] - m->h_run_off[r]));
        r = e;
      }
    }
    m->max_col_bytes = best;
  }
  {  // fp16 magnitude bits to float (exact)
    const uint32_t e = (max_mag >> 10) & 31u, f = max_mag & 1023u;
    m->tc_max_scale = e == 31 ? 1e30f
                      : e == 0 ? std::ldexp(static_cast<float>(f), -24)
                               : std::ldexp(static_cast<float>(f | 1024u), static_cast<int>(e) - 25);
  }

  // The plan of a GEMV over this matrix alone.
  Plan pl = make_plan({seg_tables(m)}, plan_ctas(data_bytes, gpu_info().sms), MAX_UNITS_PER_CTA);
  e = upload_plan(pl, MAX_NB, {m->data}, st, &m->plan);
  if (e != cudaSuccess) {
    cudaFree(m->dev_base);
    delete m;
    return cuda_fail(e, "vbq_pack: plan upload");
  }
  m->total_bytes = static_cast<int64_t>(total) + m->plan.bytes;
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
    free_plan(&m->plan);
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
