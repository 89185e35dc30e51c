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
  uint64_t gcost = 0;  // estimated work before this position
};

struct Stream {
  const std::vector<SegTables>& segs;
  std::vector<uint64_t> base;   // stream byte offset of each segment, plus the total
  std::vector<uint64_t> cbase;  // stream cost offset of each segment, plus the total
  std::vector<std::vector<uint64_t>> cpre;  // per segment: cost before each run (n_runs + 1)
  std::vector<std::vector<uint32_t>> cols;  // per segment: first run of every (tile, column), then n_runs
  bool whole_columns = false;

  explicit Stream(const std::vector<SegTables>& s, bool by_columns = false) : segs(s), whole_columns(by_columns) {
    base.assign(s.size() + 1, 0);
    cbase.assign(s.size() + 1, 0);
    cpre.resize(s.size());
    for (size_t i = 0; i < s.size(); ++i) {
      base[i + 1] = base[i] + (s[i].n_runs ? uint64_t(s[i].run_off[s[i].n_runs]) * 16u : 0u);
      std::vector<uint64_t>& c = cpre[i];
      c.assign(static_cast<size_t>(s[i].n_runs) + 1, 0);
      for (int32_t r = 0; r < s[i].n_runs; ++r) {
        const uint32_t d = s[i].run_desc[r];
        const bool col_start = r == 0 || run_g(s[i].run_desc[r - 1]) != run_g(d) || is_tile_start(i, r);
        c[r + 1] = c[r] + head_cost(d, col_start) + uint64_t(run_steps(d)) * kCostStep[run_cls(d)];
      }
      cbase[i + 1] = cbase[i] + c.back();
    }
    cols.resize(s.size());
    for (size_t i = 0; i < s.size(); ++i) {
      for (int32_t r = 0; r < s[i].n_runs; ++r)
        if (r == 0 || run_g(s[i].run_desc[r - 1]) != run_g(s[i].run_desc[r]) || is_tile_start(i, r))
          cols[i].push_back(static_cast<uint32_t>(r));
      cols[i].push_back(static_cast<uint32_t>(s[i].n_runs));
    }
  }
  static uint64_t head_cost(uint32_t, bool col_start) { return kCostRun + (col_start ? kCostColumn : 0u); }
  bool is_tile_start(size_t seg, int32_t r) const {
    const SegTables& S = segs[seg];
    return std::binary_search(S.tile_run0, S.tile_run0 + S.n_tiles + 1, static_cast<uint32_t>(r));
  }
  uint64_t total() const { return base.back(); }
  uint64_t total_cost() const { return cbase.back(); }

  uint64_t run_start(int seg, uint32_t run) const { return uint64_t(segs[seg].run_off[run]) * 16u; }

  Pos at(int seg, uint32_t run, uint32_t k) const {
    const SegTables& S = segs[seg];
    Pos p;
    p.seg = seg;
    if (run >= static_cast<uint32_t>(S.n_runs)) {
      p.run = S.n_runs;
      p.gbyte = base[seg] + run_start(seg, S.n_runs);
      p.gcost = cbase[seg] + cpre[seg].back();
      return p;
    }
    const uint32_t d = S.run_desc[run];
    if (k >= run_steps(d)) return at(seg, run + 1, 0);
    p.run = run;
    p.k = k;
    p.gbyte = base[seg] + run_start(seg, run) + uint64_t(k) * full_step_bytes(run_cls(d));
    p.gcost = cbase[seg] + cpre[seg][run] + (k ? (cpre[seg][run + 1] - cpre[seg][run] -
                                                  uint64_t(run_steps(d)) * kCostStep[run_cls(d)]) +
                                                     uint64_t(k) * kCostStep[run_cls(d)]
                                               : 0u);
    return p;
  }

  // Nearest step border (or column start, in whole-column mode) to local cost t of segment seg.
  Pos snap_local(int seg, uint64_t t) const {
    const SegTables& S = segs[seg];
    const std::vector<uint64_t>& c = cpre[seg];
    if (t >= c.back()) return at(seg, S.n_runs, 0);
    if (whole_columns) {
      const std::vector<uint32_t>& cs = cols[seg];
      // last column start whose cost <= t, and the next one
      size_t lo = 0, hi = cs.size() - 1;
      while (hi - lo > 1) {
        const size_t mid = (lo + hi) / 2;
        if (c[cs[mid]] <= t) lo = mid; else hi = mid;
      }
      const uint64_t a = c[cs[lo]], b = c[cs[hi]];
      return at(seg, (t - a <= b - t) ? cs[lo] : cs[hi], 0);
    }
    // last run whose cost start <= t
    const uint32_t r = static_cast<uint32_t>(std::upper_bound(c.begin(), c.end(), t) - c.begin()) - 1u;
    const uint32_t d = S.run_desc[r];
    const uint64_t head = c[r + 1] - c[r] - uint64_t(run_steps(d)) * kCostStep[run_cls(d)];
    const uint64_t step = kCostStep[run_cls(d)];
    const uint64_t into = t - c[r];
    const uint64_t k = into <= head ? 0u : (into - head + step / 2) / step;
    return at(seg, r, static_cast<uint32_t>(std::min<uint64_t>(k, run_steps(d))));
  }

  // Nearest step border to stream cost t.
  Pos snap(uint64_t t) const {
    for (size_t s = 0; s < segs.size(); ++s)
      if (t < cbase[s + 1]) return snap_local(static_cast<int>(s), t - cbase[s]);
    return end();
  }

  Pos end() const {
    Pos p;
    p.seg = static_cast<int>(segs.size()) - 1;
    p.run = segs.empty() ? 0 : segs.back().n_runs;
    p.gbyte = total();
    p.gcost = total_cost();
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
  const uint64_t total = st.total_cost();
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
      const Pos tend = st.at(pos.seg, S.tile_run0[t + 1], 0);
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
          const uint64_t tgt = pos.gcost + (uend.gcost - pos.gcost) * static_cast<uint64_t>(j) / SLICES;
          nx = st.snap_local(pos.seg, tgt - st.cbase[pos.seg]);
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

Plan make_plan(const std::vector<SegTables>& segs, int32_t n_ctas, int max_units, bool whole_columns) {
  Stream st(segs, whole_columns);
  Plan p;
  int32_t P = std::max<int32_t>(1, n_ctas);
  if (st.total() == 0 || st.total_cost() == 0) {
    p.n_ctas = 0;
    p.umax = 0;
    return p;
  }
  while (!build(st, P, max_units, &p)) P = P + P / 2 + 1;
  return p;
}

bool append_pieces(const Plan& p, const std::vector<const uint8_t*>& seg_data, int W,
                   std::vector<std::vector<uint64_t>>* per_warp) {
  const int spw = SLICES / W;
  bool ok = true;
  per_warp->resize(static_cast<size_t>(p.n_ctas) * W);
  for (int32_t c = 0; c < p.n_ctas; ++c)
    for (int32_t i = 0; i < p.umax; ++i) {
      const size_t slot = static_cast<size_t>(c) * p.umax + i;
      const UnitRec& u = p.units[slot];
      if (u.nsplit == 0) break;
      for (int w = 0; w < W; ++w) {
        const SliceRec& f = p.slices[slot * SLICES + w * spw];
        const SliceRec& l = p.slices[slot * SLICES + w * spw + spw - 1];
        if (l.b1 > f.b0) {
          const uint8_t* a = seg_data[u.seg] + uint64_t(f.b0) * 16u;
          const uint64_t n = uint64_t(l.b1 - f.b0) * 16u;
          ok = ok && piece_fits(a, n);
          (*per_warp)[static_cast<size_t>(c) * W + w].push_back(make_piece(a, n));
        }
      }
    }
  return ok;
}

PieceSet finish_pieces(const std::vector<std::vector<uint64_t>>& per_warp) {
  PieceSet ps;
  ps.start.assign(per_warp.size() + 1, 0);
  ps.bytes.assign(per_warp.size(), 0);
  for (size_t i = 0; i < per_warp.size(); ++i) {
    ps.start[i + 1] = ps.start[i] + static_cast<uint32_t>(per_warp[i].size());
    uint64_t b = 0;
    for (uint64_t q : per_warp[i]) {
      ps.pieces.push_back(q);
      b += (q & 0xFFFFFu) << 4;
    }
    ps.bytes[i] = static_cast<uint32_t>(b);
  }
  return ps;
}

cudaError_t upload_plan(const Plan& p, int max_nb, const std::vector<const uint8_t*>& seg_data,
                        cudaStream_t stream, DevicePlan* out) {
  auto al = [](uint64_t b) { return (b + 255) & ~uint64_t(255); };
  std::vector<std::vector<uint64_t>> w16, w8;
  if (!append_pieces(p, seg_data, 16, &w16) || !append_pieces(p, seg_data, 8, &w8)) return cudaErrorInvalidValue;
  const PieceSet p16 = finish_pieces(w16), p8 = finish_pieces(w8);
  const uint64_t o_units = 0;
  const uint64_t o_slices = al(o_units + sizeof(UnitRec) * std::max<size_t>(1, p.units.size()));
  const uint64_t o_p16 = al(o_slices + sizeof(SliceRec) * std::max<size_t>(1, p.slices.size()));
  const uint64_t o_s16 = al(o_p16 + 8ull * std::max<size_t>(1, p16.pieces.size()));
  const uint64_t o_b16 = al(o_s16 + 4ull * p16.start.size());
  const uint64_t o_p8 = al(o_b16 + 4ull * std::max<size_t>(1, p16.bytes.size()));
  const uint64_t o_s8 = al(o_p8 + 8ull * std::max<size_t>(1, p8.pieces.size()));
  const uint64_t o_b8 = al(o_s8 + 4ull * p8.start.size());
  const uint64_t o_cnt = al(o_b8 + 4ull * std::max<size_t>(1, p8.bytes.size()));
  const uint64_t o_part = al(o_cnt + 4ull * std::max<uint32_t>(1, p.n_counters));
  const uint64_t total = al(o_part + 4ull * std::max<uint64_t>(1, p.partial_rows * max_nb));
  std::vector<uint8_t> host(o_cnt, 0);
  auto put = [&](uint64_t off, const void* src, size_t n) {
    if (n) std::memcpy(host.data() + off, src, n);
  };
  put(o_units, p.units.data(), sizeof(UnitRec) * p.units.size());
  put(o_slices, p.slices.data(), sizeof(SliceRec) * p.slices.size());
  put(o_p16, p16.pieces.data(), 8 * p16.pieces.size());
  put(o_s16, p16.start.data(), 4 * p16.start.size());
  put(o_b16, p16.bytes.data(), 4 * p16.bytes.size());
  put(o_p8, p8.pieces.data(), 8 * p8.pieces.size());
  put(o_s8, p8.start.data(), 4 * p8.start.size());
  put(o_b8, p8.bytes.data(), 4 * p8.bytes.size());
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
  out->pieces16 = reinterpret_cast<const uint64_t*>(d + o_p16);
  out->start16 = reinterpret_cast<const uint32_t*>(d + o_s16);
  out->bytes16 = reinterpret_cast<const uint32_t*>(d + o_b16);
  out->pieces8 = reinterpret_cast<const uint64_t*>(d + o_p8);
  out->start8 = reinterpret_cast<const uint32_t*>(d + o_s8);
  out->bytes8 = reinterpret_cast<const uint32_t*>(d + o_b8);
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
