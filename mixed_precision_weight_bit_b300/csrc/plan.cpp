// Work plans for the batch-1 kernels (plan.h).
#include "plan.h"

#include <algorithm>
#include <cmath>

namespace vbq {

namespace {

struct Flat {
  int seg;
  uint32_t run;        // run index in its segment
  uint32_t item_st;    // item super-tile
  uint32_t g;
  uint64_t step0;      // item step index of the run's first step
  uint32_t steps;
  double cost0;        // cost of all steps before the run
  double head;         // extra cost of the run's first step (run set-up, column preparation)
  double step_cost;
};

struct Flattened {
  std::vector<Flat> runs;
  uint64_t total_steps = 0;
  double total_cost = 0.0;
  uint32_t G = 0;

  // Index of the run holding item step pos (pos < total_steps).
  size_t run_of(uint64_t pos) const {
    size_t lo = 0, hi = runs.size();
    while (hi - lo > 1) {
      const size_t mid = (lo + hi) / 2;
      if (runs[mid].step0 <= pos) lo = mid; else hi = mid;
    }
    return lo;
  }
  double cost(uint64_t pos) const {
    if (pos >= total_steps) return total_cost;
    const Flat& f = runs[run_of(pos)];
    const uint64_t k = pos - f.step0;
    return f.cost0 + (k > 0 ? f.head + static_cast<double>(k) * f.step_cost : 0.0);
  }
  // The step border whose cost is nearest to c.
  uint64_t pos_for(double c) const {
    if (runs.empty() || c <= 0.0) return 0;
    if (c >= total_cost) return total_steps;
    size_t lo = 0, hi = runs.size();
    while (hi - lo > 1) {
      const size_t mid = (lo + hi) / 2;
      if (runs[mid].cost0 <= c) lo = mid; else hi = mid;
    }
    const Flat& f = runs[lo];
    const double within = c - f.cost0 - f.head;
    double k = within / f.step_cost;
    if (within < 0.0) k = (c - f.cost0) < 0.5 * (f.head + f.step_cost) ? 0.0 : 1.0;
    uint64_t ki = static_cast<uint64_t>(std::llround(std::max(0.0, k)));
    ki = std::min<uint64_t>(ki, f.steps);
    return f.step0 + ki;
  }
  // Super-tiles and group columns touched by steps [p0, p1) (p1 > p0).
  void window(uint64_t p0, uint64_t p1, uint32_t* st0, uint32_t* nslots, uint32_t* ncols, uint32_t cols[4]) const {
    const Flat& a = runs[run_of(p0)];
    const Flat& b = runs[run_of(p1 - 1)];
    *st0 = a.item_st;
    *nslots = b.item_st - a.item_st + 1;
    if (a.item_st == b.item_st) {
      cols[0] = a.g; cols[1] = b.g + 1; cols[2] = 0; cols[3] = 0;
    } else if (b.item_st == a.item_st + 1 && b.g + 1 < a.g) {
      cols[0] = 0; cols[1] = b.g + 1; cols[2] = a.g; cols[3] = G;
    } else {
      cols[0] = 0; cols[1] = G; cols[2] = 0; cols[3] = 0;
    }
    *ncols = (cols[1] - cols[0]) + (cols[3] - cols[2]);
  }
  bool fits(uint64_t p0, uint64_t p1) const {
    uint32_t st0, ns, nc, cols[4];
    window(p0, p1, &st0, &ns, &nc, cols);
    return ns <= static_cast<uint32_t>(SLOTS_MAX) && nc <= static_cast<uint32_t>(CCAP);
  }
};

Flattened flatten(const std::vector<SegPlanInput>& segs, std::vector<uint32_t>* st_off, uint32_t* n_item_super) {
  Flattened F;
  uint32_t off = 0;
  st_off->clear();
  for (const SegPlanInput& s : segs) {
    st_off->push_back(off);
    off += s.n_super;
    F.G = std::max(F.G, s.G);
  }
  *n_item_super = off;
  double cost = 0.0;
  uint64_t step = 0;
  for (size_t si = 0; si < segs.size(); ++si) {
    const std::vector<RunInfo>& rr = *segs[si].runs;
    uint32_t last_st = UINT32_MAX, last_g = UINT32_MAX;
    for (size_t r = 0; r < rr.size(); ++r) {
      const RunInfo& ri = rr[r];
      Flat f;
      f.seg = static_cast<int>(si);
      f.run = static_cast<uint32_t>(r);
      f.item_st = (*st_off)[si] + ri.st();
      f.g = ri.h.g;
      f.step0 = step;
      f.steps = run_steps(ri.h.cls, ri.h.n);
      f.cost0 = cost;
      f.step_cost = kCostStep[ri.h.cls];
      f.head = kCostRun + ((ri.st() != last_st || ri.h.g != last_g) ? kCostColumn : 0.0);
      last_st = ri.st();
      last_g = ri.h.g;
      F.runs.push_back(f);
      step += f.steps;
      cost += f.head + f.steps * f.step_cost;
    }
  }
  F.total_steps = step;
  F.total_cost = cost;
  return F;
}

}  // namespace

bool make_item_plan(const std::vector<SegPlanInput>& segs, int32_t n_ctas, ItemPlan* out, const char** why) {
  ItemPlan& P = *out;
  P = ItemPlan{};
  P.n_ctas = n_ctas;
  Flattened F = flatten(segs, &P.st_off, &P.n_item_super);
  P.total_cost = F.total_cost;
  P.arrivals.assign(P.n_item_super, 0);
  P.ctas.assign(n_ctas, CtaPlan{});
  P.warps.assign(static_cast<size_t>(n_ctas) * KW, WarpPlan{});
  P.sub_b0.assign(static_cast<size_t>(n_ctas) * KW * MAX_SEG, 0);
  if (F.total_steps == 0) return true;

  // CTA ranges: equal shares of the remaining cost, each kept inside the
  // super-tile and column limits (the largest end that fits, found by bisection).
  std::vector<uint64_t> cut(n_ctas + 1, 0);
  uint64_t pos = 0;
  for (int32_t c = 0; c < n_ctas; ++c) {
    cut[c] = pos;
    if (pos >= F.total_steps) continue;
    const double c0 = F.cost(pos);
    const double target = c0 + (F.total_cost - c0) / static_cast<double>(n_ctas - c);
    uint64_t end = (c == n_ctas - 1) ? F.total_steps : std::max<uint64_t>(F.pos_for(target), pos + 1);
    end = std::min<uint64_t>(end, F.total_steps);
    if (!F.fits(pos, end)) {
      uint64_t lo = pos + 1, hi = end;  // fits(pos, lo) holds: one step touches one super-tile and column
      while (hi - lo > 1) {
        const uint64_t mid = lo + (hi - lo) / 2;
        if (F.fits(pos, mid)) lo = mid; else hi = mid;
      }
      end = lo;
    }
    pos = end;
  }
  cut[n_ctas] = pos;
  if (pos < F.total_steps) {
    *why = "the item needs more CTAs than given (each CTA may touch 2 super-tiles and 64 group columns)";
    return false;
  }

  for (int32_t c = 0; c < n_ctas; ++c) {
    const uint64_t p0 = cut[c], p1 = cut[c + 1];
    CtaPlan& cp = P.ctas[c];
    if (p1 <= p0) continue;
    uint32_t st0, ns, nc, cols[4];
    F.window(p0, p1, &st0, &ns, &nc, cols);
    cp.st_base = st0;
    cp.n_slots = ns;
    cp.a0 = cols[0];
    cp.a1 = cols[1];
    cp.b0 = cols[2];
    cp.b1 = cols[3];
    for (uint32_t t = 0; t < ns; ++t) P.arrivals[st0 + t] += 1;
    // Warp ranges: equal cost shares of the CTA range.
    const double ca = F.cost(p0), cb = F.cost(p1);
    uint64_t wa = p0;
    for (int w = 0; w < KW; ++w) {
      uint64_t wb = (w == KW - 1) ? p1 : F.pos_for(ca + (cb - ca) * (w + 1) / KW);
      wb = std::min(std::max(wb, wa), p1);
      WarpPlan& wp = P.warps[static_cast<size_t>(c) * KW + w];
      // Sub-ranges: one per segment the range crosses.
      uint64_t q = wa;
      while (q < wb) {
        const size_t fi = F.run_of(q);
        const Flat& f = F.runs[fi];
        const SegPlanInput& S = segs[f.seg];
        const RunInfo& ri = (*S.runs)[f.run];
        size_t fj = fi;
        while (fj + 1 < F.runs.size() && F.runs[fj + 1].seg == f.seg && F.runs[fj + 1].step0 < wb) ++fj;
        const uint64_t seg_end = std::min<uint64_t>(wb, F.runs[fj].step0 + F.runs[fj].steps);
        if (wp.nsub >= MAX_SEG) {
          *why = "a warp range crosses more segments than supported";
          return false;
        }
        SubRange& sr = wp.sub[wp.nsub++];
        sr.first = ri.h;
        sr.seg = static_cast<uint32_t>(f.seg);
        sr.k0 = static_cast<uint32_t>(q - f.step0);
        sr.nsteps = static_cast<uint32_t>(seg_end - q);
        const uint64_t b0 = sr.k0 == 0 ? ri.off : ri.off + HEADER_BYTES + uint64_t(sr.k0) * full_step_bytes(ri.h.cls);
        const size_t fe = F.run_of(seg_end - 1);
        const Flat& fl = F.runs[fe];
        const RunInfo& re = (*S.runs)[fl.run];
        const uint64_t ke = seg_end - fl.step0;  // steps of the last run inside the range (>= 1)
        const uint64_t b1 = ke == fl.steps ? re.off + run_bytes(re.h.cls, re.h.n)
                                           : re.off + HEADER_BYTES + ke * full_step_bytes(re.h.cls);
        sr.bytes = static_cast<uint32_t>(b1 - b0);
        P.sub_b0[(static_cast<size_t>(c) * KW + w) * MAX_SEG + (wp.nsub - 1)] = b0;
        q = seg_end;
      }
      wa = wb;
    }
  }
  for (CtaPlan& cp : P.ctas)
    for (uint32_t t = 0; t < cp.n_slots; ++t) cp.expect[t] = P.arrivals[cp.st_base + t];
  return true;
}

bool append_pieces(const ItemPlan& p, const std::vector<SegPlanInput>& segs,
                   std::vector<std::vector<uint64_t>>* per_warp) {
  const size_t nw = static_cast<size_t>(p.n_ctas) * KW;
  if (per_warp->size() < nw) per_warp->resize(nw);
  for (size_t w = 0; w < nw; ++w) {
    const WarpPlan& wp = p.warps[w];
    for (uint32_t s = 0; s < wp.nsub; ++s) {
      const SubRange& sr = wp.sub[s];
      if (sr.nsteps == 0) continue;
      const SegPlanInput& S = segs[sr.seg];
      const uint64_t b0 = p.sub_b0[w * MAX_SEG + s];
      const uint8_t* a = S.data + b0;
      uint64_t left = sr.bytes;
      while (left > 0) {  // pieces below 16 MiB each
        const uint64_t take = std::min<uint64_t>(left, uint64_t(1) << 23);
        if (!piece_fits(a, take)) return false;
        (*per_warp)[w].push_back(make_piece(a, take));
        a += take;
        left -= take;
      }
    }
  }
  return true;
}

PieceSet finish_pieces(const std::vector<std::vector<uint64_t>>& per_warp) {
  PieceSet ps;
  ps.start.push_back(0);
  for (const auto& v : per_warp) {
    uint64_t b = 0;
    for (uint64_t pc : v) {
      ps.pieces.push_back(pc);
      b += (pc & 0xFFFFFu) << 4;
    }
    ps.start.push_back(static_cast<uint32_t>(ps.pieces.size()));
    ps.bytes.push_back(static_cast<uint32_t>(b));
  }
  return ps;
}

}  // namespace vbq
