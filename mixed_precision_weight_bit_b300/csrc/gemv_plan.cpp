// The batch-1 GEMV plan of one packed matrix: built once by vbq_pack (host code).
#include <cstring>
#include <vector>

#include "internal.h"

namespace vbq {


vbq_status build_gemv_plan(vbq_matrix* m, cudaStream_t st) {
  GemvPlanDev& P = m->gemv;
  P = GemvPlanDev{};
  if (m->N == 0 || m->K == 0) return VBQ_OK;
  const int sms = gpu_info().sms;
  std::vector<SegPlanInput> segs(1);
  segs[0].runs = &m->runs;
  segs[0].data = m->data;
  segs[0].n_super = static_cast<uint32_t>(m->n_super);
  segs[0].G = static_cast<uint32_t>(m->G);
  ItemPlan ip;
  const char* why = "";
  int32_t n_ctas = sms > 0 ? sms : 1;
  // Grow the grid until every CTA range fits in TS_MAX tiles.
  while (!make_item_plan(segs, n_ctas, &ip, &why)) {
    if (n_ctas > (1 << 20)) return fail(VBQ_ERR_UNSUPPORTED, std::string("vbq_pack: ") + why);
    n_ctas *= 2;
  }
  std::vector<std::vector<uint64_t>> per_warp;
  if (!append_pieces(ip, segs, &per_warp))
    return fail(VBQ_ERR_UNSUPPORTED, "vbq_pack: weight address beyond 2^48");
  const PieceSet ps = finish_pieces(per_warp);
  auto al = [](size_t b) { return (b + 255) & ~size_t(255); };
  const size_t nt = static_cast<size_t>(m->n_super);
  const size_t o_w = 0;
  const size_t o_c = o_w + al(sizeof(WarpPlan) * ip.warps.size());
  const size_t o_arr = o_c + al(sizeof(CtaPlan) * ip.ctas.size());
  const size_t o_cnt = o_arr + al(4 * nt);
  const size_t o_acc = o_cnt + al(4 * nt);
  const size_t o_p = o_acc + al(8 * nt * SROWS);
  const size_t o_ps = o_p + al(8 * std::max<size_t>(1, ps.pieces.size()));
  const size_t o_pb = o_ps + al(4 * ps.start.size());
  const size_t total = o_pb + al(4 * std::max<size_t>(1, ps.bytes.size()));
  std::vector<uint8_t> host(total, 0);
  std::memcpy(host.data() + o_w, ip.warps.data(), sizeof(WarpPlan) * ip.warps.size());
  std::memcpy(host.data() + o_c, ip.ctas.data(), sizeof(CtaPlan) * ip.ctas.size());
  std::memcpy(host.data() + o_arr, ip.arrivals.data(), 4 * nt);
  if (!ps.pieces.empty()) std::memcpy(host.data() + o_p, ps.pieces.data(), 8 * ps.pieces.size());
  std::memcpy(host.data() + o_ps, ps.start.data(), 4 * ps.start.size());
  if (!ps.bytes.empty()) std::memcpy(host.data() + o_pb, ps.bytes.data(), 4 * ps.bytes.size());
  void* base = nullptr;
  cudaError_t e = dev_alloc(reinterpret_cast<void**>(&base), total);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "vbq_pack: plan allocation");
  }
  e = cudaMemcpyAsync(base, host.data(), total, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    cudaFree(base);
    return cuda_fail(e, "vbq_pack: plan upload");
  }
  uint8_t* b = static_cast<uint8_t*>(base);
  P.base = base;
  P.warps = reinterpret_cast<const WarpPlan*>(b + o_w);
  P.ctas = reinterpret_cast<const CtaPlan*>(b + o_c);
  P.arrivals = reinterpret_cast<const uint32_t*>(b + o_arr);
  P.counters = reinterpret_cast<uint32_t*>(b + o_cnt);
  P.acc = reinterpret_cast<unsigned long long*>(b + o_acc);
  P.pieces = reinterpret_cast<const uint64_t*>(b + o_p);
  P.pstart = reinterpret_cast<const uint32_t*>(b + o_ps);
  P.pbytes = reinterpret_cast<const uint32_t*>(b + o_pb);
  P.n_ctas = ip.n_ctas;
  P.bytes = static_cast<int64_t>(total);
  return VBQ_OK;
}

void free_gemv_plan(vbq_matrix* m) {
  if (m->gemv.base) cudaFree(m->gemv.base);
  m->gemv = GemvPlanDev{};
}

}  // namespace vbq
