// Work plans for the GEMV kernels (plan.h). Host code only.
#include "plan.h"

#include <algorithm>
#include <cstring>

namespace vbq {

namespace {

constexpr uint64_t kMinCtaBytes = 32 * 1024;

// A step border in the stream of a launch: step k of run `run` of segment `seg`.
// The end of a segment is (seg, n_runs, 0).
struct Pos {
  int seg = 0;
  uint32_t run = 0, k = 0;
  uint64_t gbyte = 0;  // offset in the launch's stream
};

struct Stream {
  const std::vector<SegTables>& segs;
  std::vector<uint64_t> base;  // stream offset of each segment, plus the total

  explicit Stream(const std::vector<SegTables>& s) : segs(s) {
    base.assign(s.size() + 1, 0);
    for (size_t i = 0; i < s.size(); ++i)
      base[i + 1] = base[i] + (s[i].n_runs ? uint64_t(s[i].run_off[s[i].n_runs]) * 16u : 0u);
  }
  uint64_t total() const { return base.back(); }

  uint64_t run_start(int seg, uint32_t run) const { return uint64_t(segs[seg].run_off[run]) * 16u; }

  // Nearest step border to local byte t of segment seg.
  Pos snap_local(int seg, uint64_t t) const {
    const SegTables& S = segs[seg];
    Pos p;
    p.seg = seg;
    if (t >= run_start(seg, S.n_runs)) {
      p.run = S.n_runs;
      p.gbyte = base[seg] + run_start(seg, S.n_runs);
      return p;
    }
    // last run whose start <= t
    uint32_t lo = 0, hi = S.n_runs;  // invariant: start(lo) <= t < start(hi)
    while (hi - lo > 1) {
      const uint32_t mid = (lo + hi) / 2;
      if (run_start(seg, mid) <= t) lo = mid; else hi = mid;
    }
    const uint32_t d = S.run_desc[lo];
    const uint64_t full = full_step_bytes(run_cls(d));
    const uint32_t nst = run_steps(d);
    uint64_t k = (t - run_start(seg, lo) + full / 2) / full;
    if (k >= nst) {
      p.run = lo + 1;
      p.k = 0;
      p.gbyte = base[seg] + run_start(seg, lo + 1);
    } else {
      p.run = lo;
      p.k = static_cast<uint32_t>(k);
      p.gbyte = base[seg] + run_start(seg, lo) + k * full;
    }
    return p;
  }

  // Nearest step border to stream byte t.
  Pos snap(uint64_t t) const {
    for (size_t s = 0; s < segs.size(); ++s)
      if (t < base[s + 1]) return snap_local(static_cast<int>(s), t - base[s]);
    return end();
  }

  Pos end() const {
    Pos p;
    p.seg = static_cast<int>(segs.size()) - 1;
    p.run = segs.empty() ? 0 : segs.back().n_runs;
    p.gbyte = total();
    return p;
  }

  // Moves a position at the end of a segment to the start of the next non-empty one.
  Pos normalize(Pos p) const {
    while (p.seg + 1 < static_cast<int>(segs.size()) && p.run >= static_cast<uint32_t>(segs[p.seg].n_runs)) {
      ++p.seg;
      p.run = 0;
      p.k = 0;
    }
    return p;
  }

  uint32_t tile_of(int seg, uint32_t run) const {
    const SegTables& S = segs[seg];
    const uint32_t* b = S.tile_run0;
    // last tile whose first run <= run
    const uint32_t* it = std::upper_bound(b, b + S.n_tiles + 1, run);
    return static_cast<uint32_t>((it - b) - 1);
  }
};

SliceRec slice_of(const Stream& st, const Pos& a, const Pos& b) {
  SliceRec r{};
  r.run0 = a.run;
  r.k0 = a.k;
  r.run1 = b.run;
  r.k1 = b.k;
  r.b0 = static_cast<uint32_t>((a.gbyte - st.base[a.seg]) >> 4);
  r.b1 = static_cast<uint32_t>((b.gbyte - st.base[a.seg]) >> 4);
  r.g0 = (b.gbyte > a.gbyte) ? run_g(st.segs[a.seg].run_desc[a.run]) : 0u;
  return r;
}

bool build(const Stream& st, int32_t P, int max_units, Plan* out) {
  const uint64_t total = st.total();
  std::vector<Pos> cut(P + 1);
  cut[0] = st.normalize(st.snap(0));
  cut[P] = st.end();
  for (int32_t c = 1; c < P; ++c) {
    cut[c] = st.normalize(st.snap(total * static_cast<uint64_t>(c) / static_cast<uint64_t>(P)));
    if (cut[c].gbyte < cut[c - 1].gbyte) cut[c] = cut[c - 1];
  }
  // Units in stream order, with their CTA and slices.
  std::vector<UnitRec> units;
  std::vector<SliceRec> slices;
  std::vector<int32_t> owner;
  int umax = 1;
  for (int32_t c = 0; c < P; ++c) {
    Pos pos = cut[c];
    int nunits = 0;
    while (pos.gbyte < cut[c + 1].gbyte) {
      pos = st.normalize(pos);
      const SegTables& S = st.segs[pos.seg];
      const uint32_t t = st.tile_of(pos.seg, pos.run);
      Pos tend;
      tend.seg = pos.seg;
      tend.run = S.tile_run0[t + 1];
      tend.gbyte = st.base[pos.seg] + st.run_start(pos.seg, tend.run);
      const Pos uend = cut[c + 1].gbyte < tend.gbyte ? cut[c + 1] : tend;
      UnitRec u{};
      u.seg = static_cast<uint32_t>(pos.seg);
      u.tile = t;
      u.r0 = S.tile_row0[t];
      u.rows = S.tile_row0[t + 1] - S.tile_row0[t];
      units.push_back(u);
      owner.push_back(c);
      // Warp slices: equal bytes, snapped to step borders inside the unit.
      Pos prev = pos;
      for (int j = 1; j <= SLICES; ++j) {
        Pos nx;
        if (j == SLICES) {
          nx = uend;
        } else {
          const uint64_t tgt = pos.gbyte + (uend.gbyte - pos.gbyte) * static_cast<uint64_t>(j) / SLICES;
          nx = st.snap_local(pos.seg, tgt - st.base[pos.seg]);
          if (nx.gbyte < prev.gbyte) nx = prev;
          if (nx.gbyte > uend.gbyte) nx = uend;
        }
        SliceRec sr = slice_of(st, prev, nx);
        if (nx.gbyte == prev.gbyte) {  // empty slice: start = end
          sr.run1 = sr.run0;
          sr.k1 = sr.k0;
        }
        slices.push_back(sr);
        prev = nx;
      }
      ++nunits;
      pos = uend;
    }
    if (nunits > max_units) return false;
    umax = std::max(umax, nunits);
  }

  // Split tiles. Units of one tile are consecutive in stream order.
  Plan pl;
  pl.n_ctas = P;
  pl.umax = umax;
  size_t i = 0;
  while (i < units.size()) {
    size_t j = i + 1;
    while (j < units.size() && units[j].seg == units[i].seg && units[j].tile == units[i].tile) ++j;
    const uint32_t ns = static_cast<uint32_t>(j - i);
    for (size_t q = i; q < j; ++q) {
      units[q].split = static_cast<uint32_t>(q - i);
      units[q].nsplit = ns;
      units[q].pbase = ns > 1 ? static_cast<uint32_t>(pl.partial_rows) : 0u;
      units[q].cnt = ns > 1 ? pl.n_counters : 0u;
    }
    if (ns > 1) {
      pl.partial_rows += static_cast<uint64_t>(ns) * units[i].rows;
      pl.n_counters += 1;
    }
    i = j;
  }
  // Slots: CTA c owns [c*umax, (c+1)*umax).
  pl.units.assign(static_cast<size_t>(P) * umax, UnitRec{});
  pl.slices.assign(static_cast<size_t>(P) * umax * SLICES, SliceRec{});
  std::vector<int> fill(P, 0);
  for (size_t u = 0; u < units.size(); ++u) {
    const int32_t c = owner[u];
    const size_t slot = static_cast<size_t>(c) * umax + fill[c]++;
    pl.units[slot] = units[u];
    for (int j = 0; j < SLICES; ++j) pl.slices[slot * SLICES + j] = slices[u * SLICES + j];
  }
  *out = std::move(pl);
  return true;
}

}  // namespace

int32_t plan_ctas(uint64_t total_bytes, int sms) {
  const uint64_t by_bytes = (total_bytes + kMinCtaBytes - 1) / kMinCtaBytes;
  return static_cast<int32_t>(std::max<uint64_t>(1, std::min<uint64_t>(static_cast<uint64_t>(sms), by_bytes)));
}

Plan make_plan(const std::vector<SegTables>& segs, int32_t n_ctas, int max_units) {
  Stream st(segs);
  Plan p;
  int32_t P = std::max<int32_t>(1, n_ctas);
  if (st.total() == 0) {
    p.n_ctas = 0;
    p.umax = 0;
    return p;
  }
  while (!build(st, P, max_units, &p)) P = P + P / 2 + 1;
  return p;
}

cudaError_t upload_plan(const Plan& p, int max_nb, cudaStream_t stream, DevicePlan* out) {
  auto al = [](uint64_t b) { return (b + 255) & ~uint64_t(255); };
  const uint64_t o_units = 0;
  const uint64_t o_slices = al(o_units + sizeof(UnitRec) * std::max<size_t>(1, p.units.size()));
  const uint64_t o_cnt = al(o_slices + sizeof(SliceRec) * std::max<size_t>(1, p.slices.size()));
  const uint64_t o_part = al(o_cnt + 4ull * std::max<uint32_t>(1, p.n_counters));
  const uint64_t total = al(o_part + 4ull * std::max<uint64_t>(1, p.partial_rows * max_nb));
  std::vector<uint8_t> host(o_cnt, 0);
  if (!p.units.empty()) std::memcpy(host.data() + o_units, p.units.data(), sizeof(UnitRec) * p.units.size());
  if (!p.slices.empty()) std::memcpy(host.data() + o_slices, p.slices.data(), sizeof(SliceRec) * p.slices.size());
  uint8_t* d = nullptr;
  cudaError_t e = cudaMalloc(&d, total);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyAsync(d, host.data(), o_cnt, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(d + o_cnt, 0, total - o_cnt, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) {
    cudaFree(d);
    return e;
  }
  out->base = d;
  out->units = reinterpret_cast<const UnitRec*>(d + o_units);
  out->slices = reinterpret_cast<const SliceRec*>(d + o_slices);
  out->counters = reinterpret_cast<uint32_t*>(d + o_cnt);
  out->partial = reinterpret_cast<float*>(d + o_part);
  out->n_ctas = p.n_ctas;
  out->umax = p.umax;
  out->bytes = static_cast<int64_t>(total);
  return cudaSuccess;
}

void free_plan(DevicePlan* p) {
  if (p->base) cudaFree(p->base);
  *p = DevicePlan{};
}

}  // namespace vbq
