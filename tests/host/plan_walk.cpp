// Host check of the packed layout and the batch-1 work plans (CPU only, no GPU).
//
// Builds pack.cpp, plan.cpp and gemv_plan.cpp against a stub CUDA runtime
// whose "device" memory is host memory. It packs seeded random matrices and
// checks that
//   * walking the stream tile by tile (run header, then steps) decodes every
//     (row, group) exactly once, back to its logical codes and fp16 scale,
//     with runs in (tile, group column, class) order and rows increasing;
//   * replaying every warp of every CTA of a plan exactly as the batch-1
//     kernel does (its byte pieces concatenated into its stream, the first
//     run header from the plan, later headers from the stream) visits every
//     step once, consumes exactly the bytes the warp copies, and keeps each
//     CTA inside its window of SLOTS_MAX super-tiles and CCAP staged columns;
//     per-super-tile arrival counts match;
//   * the same holds for plans over several matrices (as for [q; k; v]) and
//     for several CTA counts.
// Exit status 0 on success; the first failed checks are printed.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <random>
#include <string>
#include <vector>

#include "../../mixed_precision_weight_bit_b300/csrc/internal.h"

// ---------------------------------------------------------------- stub runtime

extern "C" {
cudaError_t cudaGetDevice(int* d) { *d = 0; return cudaSuccess; }
cudaError_t cudaSetDevice(int) { return cudaSuccess; }
cudaError_t cudaDeviceSynchronize(void) { return cudaSuccess; }
cudaError_t cudaMalloc(void** p, size_t n) { *p = std::malloc(n ? n : 1); return *p ? cudaSuccess : cudaErrorMemoryAllocation; }
cudaError_t cudaFree(void* p) { std::free(p); return cudaSuccess; }
cudaError_t cudaMemcpyAsync(void* d, const void* s, size_t n, cudaMemcpyKind, cudaStream_t) { std::memcpy(d, s, n); return cudaSuccess; }
cudaError_t cudaMemsetAsync(void* d, int v, size_t n, cudaStream_t) { std::memset(d, v, n); return cudaSuccess; }
cudaError_t cudaStreamSynchronize(cudaStream_t) { return cudaSuccess; }
cudaError_t cudaGetLastError(void) { return cudaSuccess; }
const char* cudaGetErrorString(cudaError_t) { return "stub"; }
}

namespace vbq {
static std::string g_err;
vbq_status fail(vbq_status s, const std::string& d) { g_err = d; return s; }
vbq_status cuda_fail(cudaError_t, const char* w) { g_err = w; return VBQ_ERR_CUDA; }
void note_launches(int64_t) {}
void tc_forget(const vbq_matrix*) {}
cudaError_t dev_alloc(void** p, size_t n) { return cudaMalloc(p, n); }
static int g_sms = 148;
const GpuInfo& gpu_info() {
  static GpuInfo gi;
  gi.device = 0;
  gi.sms = g_sms;
  gi.max_smem_optin = 232448;
  return gi;
}
}  // namespace vbq

using namespace vbq;

static int g_failures = 0;
#define CHECK(cond, ...)                                        \
  do {                                                          \
    if (!(cond)) {                                              \
      std::fprintf(stderr, "FAIL %s:%d: ", __FILE__, __LINE__); \
      std::fprintf(stderr, __VA_ARGS__);                        \
      std::fprintf(stderr, "\n");                               \
      if (++g_failures > 10) std::exit(1);                      \
    }                                                           \
  } while (0)

struct Logical {
  int64_t N, K;
  std::vector<uint8_t> codes, bits;
  std::vector<uint16_t> scales;
};

static Logical make_matrix(int64_t N, int64_t K, const double p[4], uint32_t seed, int mode) {
  Logical L{N, K, {}, {}, {}};
  const int64_t G = K / 64;
  std::mt19937_64 rng(seed);
  std::uniform_real_distribution<double> U(0.0, 1.0);
  L.bits.resize(N * G);
  L.codes.resize(N * K);
  L.scales.resize(N * G);
  for (int64_t r = 0; r < N; ++r)
    for (int64_t g = 0; g < G; ++g) {
      int b;
      if (mode == 1) {          // row-clustered: first half mean 6 bits, second half 1 bit
        b = r < N / 2 ? (U(rng) < 0.5 ? 4 : 8) : 1;
      } else if (mode == 2) {   // column-banded: first quarter of groups 8-bit
        b = g < G / 4 ? 8 : 1;
      } else {
        const double u = U(rng);
        b = u < p[0] ? 1 : u < p[0] + p[1] ? 2 : u < p[0] + p[1] + p[2] ? 4 : 8;
      }
      L.bits[r * G + g] = static_cast<uint8_t>(b);
      L.scales[r * G + g] = static_cast<uint16_t>(0x2000 + (rng() & 0x0FFF));
      for (int m = 0; m < 64; ++m) L.codes[r * K + g * 64 + m] = static_cast<uint8_t>(rng() & ((1u << b) - 1u));
    }
  return L;
}

// Code m of entry j of a step record of class cls with e entries (layout.h).
static uint32_t decode_code(const uint8_t* rec, uint32_t cls, uint32_t e, uint32_t j, uint32_t m) {
  const uint32_t b = 1u << cls, per_word = 32u / b, r = m % per_word;
  uint32_t w;
  std::memcpy(&w, rec + code_word_off(cls, e, j, m / per_word), 4);
  return (w >> (b == 1 ? r : code_bit(b, r))) & ((1u << b) - 1u);
}

// Checks the entries of one step (entries i0 .. i0+e-1 of its run) against the
// logical matrix and marks them seen.
static void check_step(const Logical& L, const RunHeader& h, const uint8_t* rec, uint32_t e, uint32_t i0,
                       std::vector<uint8_t>* seen, int64_t* last_row) {
  const int64_t G = L.K / 64;
  const uint32_t cls = h.cls;
  for (uint32_t j = 0; j < e; ++j) {
    const uint16_t sc = *reinterpret_cast<const uint16_t*>(rec + rec_scale_off(cls, e) + 2 * j);
    const uint32_t row_in = rec[rec_row_off(cls, e) + j];
    const uint32_t tile = entry_tile(h, i0 + j);
    CHECK(tile < h.ntl, "entry tile inside the super-tile");
    const int64_t r = int64_t(h.row0) + int64_t(tile) * TILE + row_in;
    CHECK(r < L.N, "row %lld beyond N", (long long)r);
    if (r >= L.N) continue;
    CHECK(r > *last_row, "rows of a run must increase");
    *last_row = r;
    const int64_t gi = r * G + h.g;
    CHECK(L.bits[gi] == (1 << cls), "class of (%lld, %u)", (long long)r, h.g);
    CHECK(L.scales[gi] == sc, "scale of (%lld, %u)", (long long)r, h.g);
    for (uint32_t m = 0; m < 64; ++m)
      CHECK(decode_code(rec, cls, e, j, m) == L.codes[r * L.K + int64_t(h.g) * 64 + m], "code %u of (%lld, %u)", m,
            (long long)r, h.g);
    (*seen)[gi] += 1;
  }
}

// Walks the whole stream super-tile by super-tile, as the dequant kernel does.
static void check_stream(const vbq_matrix* M, const Logical& L) {
  const int64_t G = L.K / 64;
  std::vector<uint8_t> seen(L.N * G, 0);
  std::vector<uint64_t> tb(M->n_super + 1);
  std::memcpy(tb.data(), M->st_byte0, 8 * tb.size());
  size_t run_index = 0;
  for (int32_t t = 0; t < M->n_super; ++t) {
    uint64_t o = tb[t];
    int last_key = -1;
    const int64_t rows = std::min<int64_t>(L.N - int64_t(t) * SROWS, SROWS);
    while (o < tb[t + 1]) {
      RunHeader h;
      std::memcpy(&h, M->data + o, sizeof(h));
      CHECK(run_index < M->runs.size() && M->runs[run_index].off == o &&
                std::memcmp(&M->runs[run_index].h, &h, sizeof(h)) == 0, "run list entry");
      CHECK(h.row0 == static_cast<uint32_t>(t) * SROWS, "header super-tile");
      CHECK(h.ntl == (rows + TILE - 1) / TILE, "header tile count");
      CHECK(h.c1 <= h.c2 && h.c2 <= h.c3 && h.c3 <= h.n, "prefix counts");
      const int key = h.g * 4 + h.cls;
      CHECK(key > last_key, "runs in (g, class) order");
      last_key = key;
      ++run_index;
      o += HEADER_BYTES;
      int64_t last_row = -1;
      const uint32_t eps = entries_per_step(h.cls);
      for (uint32_t done = 0; done < h.n; done += eps) {
        const uint32_t e = std::min<uint32_t>(eps, h.n - done);
        check_step(L, h, M->data + o, e, done, &seen, &last_row);
        o += rec_bytes(h.cls, e);
      }
    }
    CHECK(o == tb[t + 1], "super-tile %d ends at its table offset", t);
  }
  CHECK(run_index == M->runs.size(), "every run walked");
  for (size_t i = 0; i < seen.size(); ++i) CHECK(seen[i] == 1, "group %zu seen %d times", i, seen[i]);
  // Byte accounting.
  int64_t cb = 0;
  for (uint8_t b : L.bits) cb += 8 * b;
  CHECK(cb == M->code_bytes, "code bytes");
  CHECK(M->total_bytes == M->code_bytes + M->meta_bytes, "total = code + meta");
}

// Replays an item plan: every warp's stream (its pieces), walked like the kernel.
static void check_plan(const std::vector<const vbq_matrix*>& mats, const std::vector<const Logical*>& logi,
                       const ItemPlan& P, const std::vector<std::vector<uint64_t>>& pieces_per_warp) {
  std::vector<std::vector<uint8_t>> seen(mats.size());
  for (size_t s = 0; s < mats.size(); ++s) seen[s].assign(logi[s]->N * (logi[s]->K / 64), 0);
  std::vector<uint32_t> arrivals(P.n_item_super, 0);
  for (int32_t c = 0; c < P.n_ctas; ++c) {
    const CtaPlan& cp = P.ctas[c];
    CHECK(cp.n_slots <= static_cast<uint32_t>(SLOTS_MAX), "CTA %d touches %u super-tiles", c, cp.n_slots);
    const uint32_t ncols = (cp.a1 - cp.a0) + (cp.b1 - cp.b0);
    CHECK(ncols <= static_cast<uint32_t>(CCAP), "CTA %d stages %u columns", c, ncols);
    for (uint32_t t = 0; t < cp.n_slots; ++t) arrivals[cp.st_base + t] += 1;
    for (int w = 0; w < KW; ++w) {
      const size_t wi = static_cast<size_t>(c) * KW + w;
      // The warp's stream: its pieces concatenated.
      std::vector<uint8_t> st;
      for (uint64_t pc : pieces_per_warp[wi]) {
        const uint8_t* a = reinterpret_cast<const uint8_t*>((pc >> 20) << 4);
        const uint64_t n = (pc & 0xFFFFFu) << 4;
        st.insert(st.end(), a, a + n);
      }
      const WarpPlan& wp = P.warps[wi];
      uint64_t o = 0;
      for (uint32_t si = 0; si < wp.nsub; ++si) {
        const SubRange& sr = wp.sub[si];
        CHECK(sr.seg < mats.size(), "sub-range segment");
        const Logical& L = *logi[sr.seg];
        RunHeader h = sr.first;
        uint32_t k = sr.k0, left = sr.nsteps;
        if (left == 0) continue;
        if (k == 0) {
          CHECK(o + HEADER_BYTES <= st.size(), "header inside the stream");
          RunHeader sh;
          std::memcpy(&sh, st.data() + o, sizeof(sh));
          CHECK(std::memcmp(&sh, &h, sizeof(h)) == 0, "plan header equals the stream header");
          o += HEADER_BYTES;
        }
        while (true) {
          const uint32_t nrs = run_steps(h.cls, h.n);
          CHECK(k < nrs, "start step inside the run");
          const uint32_t kend = std::min(nrs, k + left);
          const uint32_t item_st = P.st_off[sr.seg] + h.row0 / SROWS;
          CHECK(item_st >= cp.st_base && item_st < cp.st_base + cp.n_slots, "super-tile inside the CTA window");
          CHECK((h.g >= cp.a0 && h.g < cp.a1) || (h.g >= cp.b0 && h.g < cp.b1), "column %u staged by CTA %d", h.g, c);
          CHECK(col_slot(cp, h.g) < ncols, "column slot");
          const uint32_t eps = entries_per_step(h.cls), nfull = h.n / eps, e_last = h.n - nfull * eps;
          int64_t last_row = -1;
          const uint32_t k_start = k;
          for (; k < kend; ++k) {
            const uint32_t e = k < nfull ? eps : e_last;
            CHECK(o + rec_bytes(h.cls, e) <= st.size(), "step inside the stream");
            if (o + rec_bytes(h.cls, e) > st.size()) return;
            check_step(L, h, st.data() + o, e, k * eps, &seen[sr.seg], &last_row);
            o += rec_bytes(h.cls, e);
          }
          left -= kend - k_start;
          if (left == 0) break;
          CHECK(o + HEADER_BYTES <= st.size(), "next header inside the stream");
          if (o + HEADER_BYTES > st.size()) return;
          std::memcpy(&h, st.data() + o, sizeof(h));
          o += HEADER_BYTES;
          k = 0;
        }
      }
      CHECK(o == st.size(), "CTA %d warp %d consumes %llu of %zu streamed bytes", c, w, (unsigned long long)o,
            st.size());
    }
  }
  for (size_t s = 0; s < mats.size(); ++s)
    for (size_t i = 0; i < seen[s].size(); ++i) CHECK(seen[s][i] == 1, "seg %zu group %zu seen %d times", s, i, seen[s][i]);
  for (uint32_t t = 0; t < P.n_item_super; ++t) CHECK(arrivals[t] == P.arrivals[t], "arrivals of super-tile %u", t);
}

static vbq_matrix* pack(const Logical& L) {
  vbq_matrix* m = nullptr;
  const vbq_status s = vbq_pack(L.codes.data(), L.bits.data(), L.scales.data(), L.N, L.K, nullptr, &m);
  CHECK(s == VBQ_OK, "vbq_pack failed: %s", g_err.c_str());
  return m;
}

static void plan_and_check(const std::vector<const vbq_matrix*>& mats, const std::vector<const Logical*>& logi,
                           int32_t n_ctas) {
  std::vector<SegPlanInput> segs;
  for (const vbq_matrix* m : mats) {
    SegPlanInput s;
    s.runs = &m->runs;
    s.data = m->data;
    s.n_super = static_cast<uint32_t>(m->n_super);
    s.G = static_cast<uint32_t>(m->G);
    segs.push_back(s);
  }
  ItemPlan ip;
  const char* why = "";
  int32_t n = n_ctas;
  while (!make_item_plan(segs, n, &ip, &why)) n *= 2;
  std::vector<std::vector<uint64_t>> per_warp;
  CHECK(append_pieces(ip, segs, &per_warp), "pieces");
  per_warp.resize(static_cast<size_t>(ip.n_ctas) * KW);
  check_plan(mats, logi, ip, per_warp);
}

int main() {
  const double p0[4] = {0.69, 0.15, 0.11, 0.05};
  const double one[4][4] = {{1, 0, 0, 0}, {0, 1, 0, 0}, {0, 0, 1, 0}, {0, 0, 0, 1}};
  struct Case { int64_t N, K; const double* p; int mode; };
  std::vector<Case> cases = {
      {1, 64, p0, 0},      {3, 128, p0, 0},     {257, 640, p0, 0},   {511, 192, p0, 0},   {768, 768, p0, 0},
      {4099, 128, p0, 0},  {300, 1024, p0, 0},  {1024, 1024, p0, 1}, {1024, 1024, p0, 2}, {200, 512, one[0], 0},
      {200, 512, one[1], 0}, {200, 512, one[2], 0}, {200, 512, one[3], 0}, {2048, 4096, p0, 0}, {20000, 128, p0, 0},
      {5000, 8192, p0, 0}, {3000, 640, p0, 1},
  };
  uint32_t seed = 1;
  for (const Case& cs : cases) {
    const Logical L = make_matrix(cs.N, cs.K, cs.p, seed++, cs.mode);
    vbq_matrix* m = pack(L);
    if (!m) continue;
    check_stream(m, L);
    for (int32_t ctas : {1, 7, 148}) plan_and_check({m}, {&L}, ctas);
    vbq_matrix_free(m);
  }
  {  // three matrices in one item, as [q; k; v]
    const Logical q = make_matrix(600, 512, p0, 101, 0), k = make_matrix(130, 512, p0, 102, 0),
                  v = make_matrix(257, 512, p0, 103, 0);
    vbq_matrix *mq = pack(q), *mk = pack(k), *mv = pack(v);
    for (int32_t ctas : {1, 5, 148}) plan_and_check({mq, mk, mv}, {&q, &k, &v}, ctas);
    vbq_matrix_free(mq);
    vbq_matrix_free(mk);
    vbq_matrix_free(mv);
  }
  {  // invalid inputs are rejected before anything is allocated
    Logical L = make_matrix(4, 128, p0, 7, 0);
    vbq_matrix* m = nullptr;
    L.bits[3] = 3;
    CHECK(vbq_pack(L.codes.data(), L.bits.data(), L.scales.data(), 4, 128, nullptr, &m) == VBQ_ERR_BITS && !m,
          "bad bit-width");
    L = make_matrix(4, 128, p0, 7, 0);
    L.bits[0] = 1;
    L.codes[5] = 2;
    CHECK(vbq_pack(L.codes.data(), L.bits.data(), L.scales.data(), 4, 128, nullptr, &m) == VBQ_ERR_CODE_RANGE && !m,
          "code out of range");
    CHECK(vbq_pack(L.codes.data(), L.bits.data(), L.scales.data(), 4, 100, nullptr, &m) == VBQ_ERR_SHAPE, "K % 64");
  }
  if (g_failures) return 1;
  std::printf("plan walk ok\n");
  return 0;
}
