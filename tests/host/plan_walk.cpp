// Host check of the packed layout and the GEMV work plans (CPU only, no GPU).
//
// Builds pack.cpp and plan.cpp against a stub CUDA runtime whose "device"
// memory is host memory. It packs seeded random matrices, then replays what
// each warp of the GEMV kernel walks: the units of its CTA, its slice of each
// unit, run by run and step by step. It checks that
//   * every warp's slices add up to the bytes it copies, and that the records it
//     walks sit exactly at the offsets the copies put them;
//   * every step of every tile is walked exactly once per launch;
//   * decoding every walked record (codes, fp16 scale, row) gives back the
//     logical codes and scales;
//   * split tiles have consistent split/nsplit/pbase/counter numbers, no CTA has
//     more than 32 units, and the CTA ranges have about equal bytes.
// Exit status 0 on success; the first failed check is printed.
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
#define CHECK(cond, ...)                                   \
  do {                                                     \
    if (!(cond)) {                                         \
      std::fprintf(stderr, "FAIL %s:%d: ", __FILE__, __LINE__); \
      std::fprintf(stderr, __VA_ARGS__);                   \
      std::fprintf(stderr, "\n");                          \
      if (++g_failures > 10) std::exit(1);                 \
    }                                                      \
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

// Replays the kernel's walk over one launch's plan. segs[i] is the packed matrix i.
static void check_plan(const std::vector<const vbq_matrix*>& mats, const std::vector<const Logical*>& logi,
                       const Plan& pl, const DevicePlan& dp, int W, bool balance = true) {
  const int SPW = SLICES / W;
  // Every step of every run of every matrix: visit count.
  std::vector<std::vector<std::vector<uint8_t>>> seen(mats.size());
  uint64_t total = 0;
  for (size_t s = 0; s < mats.size(); ++s) {
    seen[s].resize(mats[s]->n_runs);
    for (int32_t r = 0; r < mats[s]->n_runs; ++r) seen[s][r].assign(run_steps(mats[s]->h_run_desc[r]), 0);
    total += mats[s]->data_bytes;
  }
  CHECK(pl.units.size() == static_cast<size_t>(pl.n_ctas) * pl.umax, "unit slots");
  CHECK(dp.n_ctas == pl.n_ctas && dp.umax == pl.umax, "device plan shape");
  std::vector<uint64_t> cta_bytes(pl.n_ctas, 0);
  std::vector<uint64_t> cta_cost(pl.n_ctas, 0);  // the planner's work model over what each CTA walks
  std::vector<uint32_t> cnt_units(pl.n_counters, 0);
  std::vector<uint32_t> cta_units(pl.n_ctas, 0);
  for (int32_t c = 0; c < pl.n_ctas; ++c) {
    // The kernel counts a CTA's units as the non-empty slots, which come first.
    uint32_t nu = 0;
    bool gap = false;
    for (int32_t i = 0; i < pl.umax; ++i) {
      const bool used = dp.units[static_cast<size_t>(c) * pl.umax + i].nsplit > 0;
      if (used && gap) CHECK(false, "CTA %d: used slot after an empty one", c);
      if (used) ++nu; else gap = true;
    }
    cta_units[c] = nu;
    CHECK(pl.umax <= MAX_UNITS_PER_CTA, "umax %d", pl.umax);
    const uint32_t u0 = static_cast<uint32_t>(c) * pl.umax, u1 = u0 + nu;
    for (int w = 0; w < W; ++w) {
      uint64_t stream = 0;  // bytes this warp copies, in order
      // The warp's piece list: one piece per unit with a non-empty slice, in unit order.
      const uint64_t* pieces = W == 16 ? dp.pieces16 : dp.pieces8;
      const uint32_t* pstart = W == 16 ? dp.start16 : dp.start8;
      const uint32_t* pbytes = W == 16 ? dp.bytes16 : dp.bytes8;
      uint32_t pi = pstart[c * W + w];
      for (uint32_t u = u0; u < u1; ++u) {
        const UnitRec ur = dp.units[u];
        CHECK(ur.seg < mats.size(), "unit seg");
        const vbq_matrix* M = mats[ur.seg];
        const Logical& LG = *logi[ur.seg];
        CHECK(ur.tile < static_cast<uint32_t>(M->n_tiles), "unit tile");
        CHECK(ur.split < ur.nsplit, "split index");
        const uint32_t r0 = M->h_tile_row0[ur.tile], rows = M->h_tile_row0[ur.tile + 1] - r0;
        CHECK(ur.r0 == r0 && ur.rows == rows, "unit rows");
        if (ur.nsplit > 1) {
          CHECK(ur.cnt < pl.n_counters, "counter index");
          CHECK(static_cast<uint64_t>(ur.pbase) + static_cast<uint64_t>(ur.nsplit) * rows <= pl.partial_rows,
                "partial range");
          if (w == 0) cnt_units[ur.cnt] += 1;
        }
        const SliceRec f = dp.slices[static_cast<size_t>(u) * SLICES + w * SPW];
        const SliceRec l = dp.slices[static_cast<size_t>(u) * SLICES + w * SPW + SPW - 1];
        if (SPW == 2) {
          const SliceRec mid = dp.slices[static_cast<size_t>(u) * SLICES + w * SPW];
          CHECK(mid.b1 == l.b0, "slices of a warp are contiguous");
        }
        const uint64_t b0 = uint64_t(f.b0) * 16, b1 = uint64_t(l.b1) * 16;
        CHECK(b1 >= b0, "slice bytes");
        if (b1 > b0) {
          CHECK(pi < pstart[c * W + w + 1], "CTA %d warp %d: too few pieces", c, w);
          const uint64_t q = pieces[pi++];
          CHECK(((q >> 20) << 4) == reinterpret_cast<uint64_t>(M->data + b0), "piece address");
          CHECK(((q & 0xFFFFFu) << 4) == b1 - b0, "piece length");
        }
        {  // the first group column the kernel prefetches
          const uint32_t g0 = (SPW > 1 && f.b1 == f.b0) ? l.g0 : f.g0;
          if (b1 > b0) {
            const uint32_t r = (SPW > 1 && f.b1 == f.b0) ? l.run0 : f.run0;
            CHECK(g0 == run_g(M->h_run_desc[r]), "slice g0");
          }
        }
        cta_bytes[c] += b1 - b0;
        // Walk runs and steps exactly as the kernel does.
        uint64_t o = b0;
        const uint32_t run_end = l.run1 + (l.k1 > 0 ? 1u : 0u);
        uint32_t k = f.k0;
        for (uint32_t run = f.run0; run < run_end; ++run, k = 0) {
          CHECK(run < static_cast<uint32_t>(M->n_runs), "run index %u of %d", run, M->n_runs);
          CHECK(run >= M->h_tile_run0[ur.tile] && run < M->h_tile_run0[ur.tile + 1], "run outside the unit's tile");
          const uint32_t d = M->h_run_desc[run];
          const uint32_t cls = run_cls(d), n = run_n(d), eps = entries_per_step(cls);
          const uint32_t kend = (run == l.run1) ? l.k1 : (n + eps - 1) / eps;
          if (k == 0 && kend > 0) CHECK(o == uint64_t(M->h_run_off[run]) * 16, "run start offset");
          if (k == 0 && kend > 0) {
            const bool col = run == 0 || run_g(M->h_run_desc[run - 1]) != run_g(d) ||
                             std::binary_search(M->h_tile_run0.begin(), M->h_tile_run0.end(), run);
            cta_cost[c] += kCostRun + (col ? kCostColumn : 0u);
          }
          if (kend > k) cta_cost[c] += uint64_t(kend - k) * kCostStep[cls];
          for (; k < kend; ++k) {
            CHECK(k < seen[ur.seg][run].size(), "step index");
            seen[ur.seg][run][k] += 1;
            const uint32_t e = std::min(eps, n - k * eps);
            const uint8_t* rec = M->data + o;
            const int b = 1 << cls;
            const uint32_t g = run_g(d);
            for (uint32_t j = 0; j < e; ++j) {
              const uint32_t row = rec[rec_row_off(cls, e) + j];
              CHECK(row < rows, "row in tile");
              uint16_t sc;
              std::memcpy(&sc, rec + rec_scale_off(cls, e) + 2 * j, 2);
              const int64_t R = r0 + row;
              CHECK(LG.bits[R * (LG.K / 64) + g] == b, "class of (row, g)");
              CHECK(LG.scales[R * (LG.K / 64) + g] == sc, "scale of (row, g)");
              const uint8_t* ent = rec + j * 8u * b;
              for (int m = 0; m < 64; ++m) {
                uint32_t q = 0;  // bit-planes for 1, 2 and 4 bits, bytes for 8 bits
                if (b == 8) {
                  q = ent[m];
                } else {
                  for (int p = 0; p < b; ++p) q |= ((ent[8 * p + (m >> 3)] >> (m & 7)) & 1u) << p;
                }
                if (q != LG.codes[R * LG.K + g * 64 + m]) {
                  CHECK(false, "code mismatch row %lld g %u m %d", static_cast<long long>(R), g, m);
                  break;
                }
              }
            }
            o += rec_bytes(cls, e);
          }
        }
        CHECK(o == b1, "walked bytes %llu != slice end %llu", static_cast<unsigned long long>(o),
              static_cast<unsigned long long>(b1));
        stream += b1 - b0;
      }
      CHECK(pi == pstart[c * W + w + 1], "CTA %d warp %d: extra pieces", c, w);
      CHECK(pbytes[c * W + w] == stream, "CTA %d warp %d: piece bytes", c, w);
    }
  }
  for (size_t s = 0; s < mats.size(); ++s)
    for (int32_t r = 0; r < mats[s]->n_runs; ++r)
      for (size_t k = 0; k < seen[s][r].size(); ++k)
        CHECK(seen[s][r][k] == 1, "seg %zu run %d step %zu walked %d times", s, r, k, seen[s][r][k]);
  for (uint32_t i = 0; i < pl.n_counters; ++i) CHECK(cnt_units[i] >= 2, "split tile with <2 units");
  // Balance: no CTA far above the mean of the work model (one step and one
  // column of slack per unit, since cuts fall on step borders).
  if (balance && pl.n_ctas > 1 && W == 16) {
    uint64_t tot = 0;
    for (uint64_t v : cta_cost) tot += v;
    const double mean = static_cast<double>(tot) / pl.n_ctas;
    for (int32_t c = 0; c < pl.n_ctas; ++c)
      CHECK(cta_cost[c] <= mean * 1.02 + 200.0 + 250.0 * cta_units[c], "CTA %d carries cost %llu, mean %.0f", c,
            static_cast<unsigned long long>(cta_cost[c]), mean);
  }
}

int main() {
  const double cfg0[4] = {0.69, 0.15, 0.11, 0.05};
  const double all8[4] = {0, 0, 0, 1};
  const double all1[4] = {1, 0, 0, 0};
  struct Case { int64_t N, K; const double* p; int mode; };
  const Case cases[] = {
      {768, 768, cfg0, 0},   {1, 64, cfg0, 0},     {3, 128, cfg0, 0},     {300, 1024, cfg0, 0},
      {257, 640, cfg0, 0},   {4099, 128, cfg0, 0}, {200, 512, all8, 0},   {200, 512, all1, 0},
      {1024, 1024, cfg0, 1}, {1024, 1024, cfg0, 2}, {2048, 4096, cfg0, 0}, {5000, 64, cfg0, 0},
      {40000, 64, all1, 0},
  };
  std::vector<Logical> keep;
  keep.reserve(32);
  std::vector<vbq_matrix*> packed;
  uint32_t seed = 1;
  for (const Case& cs : cases) {
    keep.push_back(make_matrix(cs.N, cs.K, cs.p, seed++, cs.mode));
    const Logical& L = keep.back();
    vbq_matrix* m = nullptr;
    const vbq_status st = vbq_pack(L.codes.data(), L.bits.data(), L.scales.data(), L.N, L.K, nullptr, &m);
    CHECK(st == VBQ_OK, "pack %lldx%lld: %s", static_cast<long long>(cs.N), static_cast<long long>(cs.K),
          g_err.c_str());
    packed.push_back(m);
    // The matrix's own plan, as the 1- and 2-column kernels (16 warps) and the 4-column kernel (8 warps) read it.
    Plan pl = make_plan({seg_tables(m)}, m->plan.n_ctas, MAX_UNITS_PER_CTA);
    check_plan({m}, {&L}, pl, m->plan, 16);
    check_plan({m}, {&L}, pl, m->plan, 8);
    // Whole-column plans (the tensor-core path): every unit starts and ends at a column start.
    for (int P : {1, 148}) {
      Plan pc = make_plan({seg_tables(m)}, P, MAX_UNITS_PER_CTA, true);
      DevicePlan dc;
      CHECK(upload_plan(pc, 64, {m->data}, nullptr, &dc) == cudaSuccess, "upload");
      check_plan({m}, {&L}, pc, dc, 16, /*balance=*/false);  // cuts fall only on column starts
      for (size_t u = 0; u < pc.units.size(); ++u) {
        if (pc.units[u].nsplit == 0) continue;
        const SliceRec& a0 = pc.slices[u * SLICES];
        const SliceRec& a1 = pc.slices[u * SLICES + SLICES - 1];
        auto col_start = [&](uint32_t r) {
          return r == 0 || r >= static_cast<uint32_t>(m->n_runs) ||
                 run_g(m->h_run_desc[r - 1]) != run_g(m->h_run_desc[r]) ||
                 std::binary_search(m->h_tile_run0.begin(), m->h_tile_run0.end(), r);
        };
        CHECK(a0.k0 == 0 && a1.k1 == 0 && col_start(a0.run0) && col_start(a1.run1), "unit %zu not on columns", u);
      }
      CHECK(m->max_col_bytes <= 17408, "column span %lld", static_cast<long long>(m->max_col_bytes));
      free_plan(&dc);
    }
    // Other CTA counts, including more CTAs than tiles and a single CTA.
    for (int P : {1, 7, 148, 600}) {
      Plan p2 = make_plan({seg_tables(m)}, P, MAX_UNITS_PER_CTA);
      DevicePlan d2;
      CHECK(upload_plan(p2, 4, {m->data}, nullptr, &d2) == cudaSuccess, "upload");
      check_plan({m}, {&L}, p2, d2, 16);
      free_plan(&d2);
    }
  }
  // Fused launches of several matrices (as the decode step's [q;k;v] and [gate;up]).
  {
    const std::vector<const vbq_matrix*> ms = {packed[3], packed[4], packed[6]};
    const std::vector<const Logical*> ls = {&keep[3], &keep[4], &keep[6]};
    std::vector<SegTables> segs;
    for (const vbq_matrix* m : ms) segs.push_back(seg_tables(m));
    for (int P : {1, 5, 148}) {
      Plan p = make_plan(segs, P, MAX_UNITS_PER_CTA);
      DevicePlan d;
      CHECK(upload_plan(p, 1, {ms[0]->data, ms[1]->data, ms[2]->data}, nullptr, &d) == cudaSuccess, "upload");
      check_plan(ms, ls, p, d, 16);
      free_plan(&d);
    }
  }
  for (vbq_matrix* m : packed) vbq_matrix_free(m);
  if (g_failures) {
    std::fprintf(stderr, "%d check(s) failed\n", g_failures);
    return 1;
  }
  std::printf("plan walk ok\n");
  return 0;
}
