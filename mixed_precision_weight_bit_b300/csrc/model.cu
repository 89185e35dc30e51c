// vbq_decode_step: one batch-1 decode step through a stack of VBQ projections.
//
// VBQ abstract ("Variable Bit-width Quantization ..."): packed per-group codes
// speed up token-by-token decode, whose speed memory bandwidth sets. The pages
// give no architecture, so the glue is this library's reading (decode.cuh):
// unit-gain RMSNorm, attention at position 0 (each query head returns its kv
// group's v), SwiGLU, fp32 residual, and bf16 at every projection input.
//
// A step is one persistent cooperative launch (vbq_decode_kernel): per layer
// the items [q;k;v], o, [gate;up], down, then the head, linked by per-super-tile
// flags instead of grid barriers. Each warp streams its share of every item's
// packed weights back to back, so the next item's weights arrive while a CTA
// waits for its inputs. Items, work plans and per-warp piece lists are built
// once, here.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "decode.cuh"
#include "internal.h"

using namespace vbq;

namespace {

enum { P_Q = 0, P_K, P_V, P_O, P_GATE, P_UP, P_DOWN, P_PER_LAYER };
enum { L_QKV = 0, L_O, L_GU, L_DOWN, L_PER_LAYER };

int64_t proj_n(const vbq_model_desc& d, int p) {
  switch (p) {
    case P_Q: return int64_t(d.n_heads) * d.head_dim;
    case P_K:
    case P_V: return int64_t(d.n_kv_heads) * d.head_dim;
    case P_O:
    case P_DOWN: return d.d;
    default: return d.d_ff;
  }
}
int64_t proj_k(const vbq_model_desc& d, int p) {
  switch (p) {
    case P_O: return int64_t(d.n_heads) * d.head_dim;
    case P_DOWN: return d.d_ff;
    default: return d.d;
  }
}

int64_t n_super_of(int64_t n) { return (n + SROWS - 1) / SROWS; }
uint32_t decode_smem_bytes() { return smem_layout(kRingSlots).total + 2 * kItemSmem; }
static_assert(smem_layout(kRingSlots).total + 2 * kItemSmem <= 232448, "shared memory of the decode kernel");


// Scratch of one item, in 8-byte words from the scratch base: 64-bit sums,
// float outputs (none for the head, which writes the logits), and the
// per-super-tile arrival counters, flags and statistics.
struct ItemBuf {
  int64_t acc = 0, out = -1, cnt = 0, flag = 0, stats = 0;
  int64_t n_super = 0;
};

// The step scratch. Sums and counters must be zero before the first step and
// every step leaves them so; flags hold the epoch of the launch that set them.
struct Layout {
  int64_t h0 = 0, h0_flag = 0, h0_stats = 0, n_super_in = 0;
  std::vector<ItemBuf> items;
  int64_t total = 0;
};

// n_super per item, in step order.
Layout layout_of(const vbq_model_desc& d, const std::vector<int64_t>& item_super) {
  Layout L;
  int64_t w = 0;
  auto take = [&](int64_t words) {  // 128-byte aligned, so counters, flags and statistics share no cache line
    const int64_t o = w;
    w += (words + 15) & ~int64_t(15);
    return o;
  };
  L.n_super_in = n_super_of(d.d);
  L.h0 = take(L.n_super_in * SROWS / 2);
  L.h0_flag = take((L.n_super_in + 1) / 2);
  L.h0_stats = take(L.n_super_in);
  const size_t n = item_super.size();
  for (size_t i = 0; i < n; ++i) {
    ItemBuf b;
    b.n_super = item_super[i];
    b.acc = take(b.n_super * SROWS);
    if (i + 1 < n) b.out = take(b.n_super * SROWS / 2);
    b.cnt = take((b.n_super + 1) / 2);
    b.flag = take((b.n_super + 1) / 2);
    b.stats = take(b.n_super);
    L.items.push_back(b);
  }
  L.total = w;
  return L;
}

}  // namespace

struct vbq_model {
  vbq_model_desc desc{};
  std::vector<const vbq_matrix*> mats;
  int device = 0;
  int sms = 0;
  int32_t n_items = 0;
  Layout lay;
  uint64_t* ws = nullptr;            // step scratch (Layout), then the host-step staging
  uint16_t* x_stage = nullptr;
  float* logits_stage = nullptr;
  bool trace = false;
  uint16_t* tr_in = nullptr;
  float* tr_out = nullptr;
  std::vector<int64_t> in_off, out_off;
  int64_t in_total = 0, out_total = 0;
  std::vector<std::vector<uint32_t>> item_st_off;
  std::vector<int64_t> item_super;
  void* prog_mem = nullptr;          // plans, piece lists and the item arrays
  const CtaPlan* ctas = nullptr;     // [n_items][sms]
  const WarpPlan* warps = nullptr;   // [n_items][sms][KW]
  const uint64_t* pieces = nullptr;
  const uint32_t* pstart = nullptr;
  const uint32_t* pbytes = nullptr;
  DItem* items_ws = nullptr;         // items over ws
  DItem* items_static = nullptr;     // items over the static scratch (null if the model does not fit it)
  uint64_t* static_base = nullptr;
  int* err = nullptr;
  // Host copies kept for the context step: each warp's pieces of every item in
  // step order, and per item each warp's piece count once that item is in.
  std::vector<std::vector<uint64_t>> per_warp;
  std::vector<std::vector<uint32_t>> marks;
  // Context steps (vbq_model_set_context): the KV caches, the rotated query,
  // the attention output, and the programs of the segmented launches.
  int32_t max_ctx = 0;
  double rope_theta = 10000.0;
  uint16_t* kv = nullptr;            // bf16 [n_layers][2][n_kv_heads][max_ctx][head_dim]
  uint16_t* q_rot = nullptr;         // bf16 [n_heads * head_dim]
  float* attn_out = nullptr;         // [n_heads * head_dim]
  void* ctx_mem = nullptr;
  DItem* items_ctx = nullptr;        // items over ws, the o items reading attn_out
  const uint64_t* seg_pieces = nullptr;
  const uint32_t* seg_start = nullptr;  // [n_seg][n_warps + 1]
  const uint32_t* seg_bytes = nullptr;  // [n_seg][n_warps]
  std::vector<int32_t> seg_item0;    // first item of each segment, then n_items
};

namespace {

// The static scratch of vbq_decode_step_noalloc (defined at the bottom of this file).
vbq_status step_scratch_address(int dev, uint64_t** out);
constexpr int64_t kStepScratchWords = int64_t(4) << 20;  // 32 MiB

float l1_of(std::initializer_list<const vbq_matrix*> ms) {
  float v = 0.0f;
  for (const vbq_matrix* m : ms) v = std::max(v, m->max_row_l1);
  return v;
}

// Flag values: one per launch, unique across models and devices (0 is never used).
uint32_t next_epoch() {
  static std::atomic<uint32_t> counter{0};
  uint32_t e;
  do {
    e = counter.fetch_add(1u) + 1u;
  } while (e == 0u);
  return e;
}

// The items of one step over the scratch at base.
std::vector<DItem> make_items(const vbq_model* m, uint64_t* base, bool trace, bool ctx = false) {
  const vbq_model_desc& d = m->desc;
  const Layout& L = m->lay;
  auto words = [&](int64_t off) { return base + off; };
  auto tin = [&](int p) -> uint16_t* { return trace ? m->tr_in + m->in_off[p] : nullptr; };
  auto tout = [&](int p) -> float* { return trace ? m->tr_out + m->out_off[p] : nullptr; };
  const int64_t nq = proj_n(d, P_Q);
  // The residual read by the next RMSNorm: its vector and statistics.
  const float* res_vec = reinterpret_cast<const float*>(words(L.h0));
  ResStats res{reinterpret_cast<const float2*>(words(L.h0_stats)), reinterpret_cast<const uint32_t*>(words(L.h0_flag)),
               static_cast<int32_t>(L.n_super_in), d.d};
  std::vector<DItem> items;
  auto base_item = [&](int idx, int mode, int K, float l1) {
    const ItemBuf& b = L.items[idx];
    DItem it{};
    for (size_t s = 0; s < m->item_st_off[idx].size() && s < static_cast<size_t>(MAX_SEG); ++s)
      it.seg_st_off[s] = m->item_st_off[idx][s];
    it.mode = mode;
    it.K = K;
    it.l1 = l1;
    it.eps = d.rms_eps;
    it.n_super = static_cast<int32_t>(b.n_super);
    it.acc = reinterpret_cast<unsigned long long*>(words(b.acc));
    it.cnt = reinterpret_cast<uint32_t*>(words(b.cnt));
    it.flag = reinterpret_cast<uint32_t*>(words(b.flag));
    it.out = b.out >= 0 ? reinterpret_cast<float*>(words(b.out)) : nullptr;
    it.out_n = b.n_super * SROWS;
    return it;
  };
  auto rms_input = [&](DItem& it) {
    it.src = res_vec;
    it.src_flag = res.flag;
    it.src_nsuper = res.n_super;
    it.rs = res;
  };
  auto residual_output = [&](DItem& it, int idx) {  // out = res_vec + y; the next RMSNorm reads it
    it.res = res_vec;
    it.out_n = d.d;
    it.stats = reinterpret_cast<float2*>(words(L.items[idx].stats));
    res_vec = it.out;
    res = ResStats{it.stats, it.flag, it.n_super, d.d};
  };
  for (int l = 0; l < d.n_layers; ++l) {
    const vbq_matrix* const* W = &m->mats[static_cast<size_t>(l) * P_PER_LAYER];
    const int p0 = l * P_PER_LAYER, i0 = l * L_PER_LAYER;
    const float l1_qkv = l1_of({W[P_Q], W[P_K], W[P_V]});
    const ResStats rs_qkv = res;
    DItem qkv = base_item(i0 + L_QKV, X_RMS, d.d, l1_qkv);  // [q; k; v] = W bf16(rmsnorm(h))
    rms_input(qkv);
    qkv.trace_x = tin(p0 + P_Q);
    for (int s = 0; s < 3; ++s) {
      qkv.trace_y[s] = tout(p0 + P_Q + s);
      qkv.trace_n[s] = proj_n(d, P_Q + s);
    }
    items.push_back(qkv);
    const std::vector<uint32_t>& so = m->item_st_off[i0 + L_QKV];
    {  // h += W_o bf16(v of each head's kv group)
      DItem it = base_item(i0 + L_O, X_GQA, static_cast<int>(nq), l1_of({W[P_O]}));
      it.src = qkv.out;
      it.src_flag = qkv.flag;
      it.src_nsuper = qkv.n_super;
      it.rs = rs_qkv;
      it.l1_src = l1_qkv;
      it.v_off = int64_t(so[2]) * SROWS;
      it.v_st0 = static_cast<int32_t>(so[2]);
      it.v_st1 = static_cast<int32_t>(so[2] + n_super_of(proj_n(d, P_V)));
      it.head_dim = d.head_dim;
      it.group = d.n_heads / d.n_kv_heads;
      if (ctx) {
        // The context step: o reads the attention output, [n_heads][head_dim] in
        // order, which a launch before this one completed (no flags to wait on).
        // Each element is a convex combination of v's, so the bound through v
        // (rs, l1_src) still holds.
        it.src = m->attn_out;
        it.v_off = 0;
        it.v_st0 = it.v_st1 = 0;
        it.group = 1;
      }
      it.trace_x = tin(p0 + P_O);
      it.trace_y[0] = tout(p0 + P_O);
      it.trace_n[0] = d.d;
      residual_output(it, i0 + L_O);
      items.push_back(it);
    }
    const ResStats rs_gu = res;
    DItem gu = base_item(i0 + L_GU, X_RMS, d.d, l1_of({W[P_GATE], W[P_UP]}));  // [gate; up] = W bf16(rmsnorm(h))
    rms_input(gu);
    gu.trace_x = tin(p0 + P_GATE);
    for (int s = 0; s < 2; ++s) {
      gu.trace_y[s] = tout(p0 + P_GATE + s);
      gu.trace_n[s] = d.d_ff;
    }
    items.push_back(gu);
    const std::vector<uint32_t>& sg = m->item_st_off[i0 + L_GU];
    {  // h += W_down bf16(silu(gate) * up)
      DItem it = base_item(i0 + L_DOWN, X_SWIGLU, d.d_ff, l1_of({W[P_DOWN]}));
      it.src = gu.out;
      it.src_flag = gu.flag;
      it.src_nsuper = gu.n_super;
      it.rs = rs_gu;
      it.up_off = int64_t(sg[1]) * SROWS;
      it.l1_gate = W[P_GATE]->max_row_l1;
      it.l1_up = W[P_UP]->max_row_l1;
      it.trace_x = tin(p0 + P_DOWN);
      it.trace_y[0] = tout(p0 + P_DOWN);
      it.trace_n[0] = d.d;
      residual_output(it, i0 + L_DOWN);
      items.push_back(it);
    }
  }
  {  // logits = W_head bf16(rmsnorm(h)), written by the conversions into the launch's buffer
    const int ih = d.n_layers * L_PER_LAYER, ph = d.n_layers * P_PER_LAYER;
    DItem it = base_item(ih, X_RMS, d.d, l1_of({m->mats[ph]}));
    rms_input(it);
    it.out = nullptr;
    it.out_n = d.vocab;
    it.trace_x = tin(ph);
    items.push_back(it);
  }
  return items;
}

cudaError_t upload_items(const std::vector<DItem>& items, DItem* dst) {
  return cudaMemcpy(dst, items.data(), sizeof(DItem) * items.size(), cudaMemcpyHostToDevice);
}

// Test hooks (vbq_debug_set): the cycles a flag wait may take before the
// kernel records a timeout (default about a second), whether waits look for a
// flag value that no launch writes, and how many words of the static scratch
// vbq_decode_step_noalloc may use.
std::atomic<long long> g_spin_limit{kSpinCycles};
std::atomic<int> g_never_ready{0};
std::atomic<int64_t> g_noalloc_words{0};

// Items [i0, i1) of a step in one launch. pieces/pstart/pbytes: the warps'
// piece lists of exactly those items; the step input is converted only by the
// launch that starts at item 0; every launch of a step shares its epoch.
cudaError_t launch_decode_range(const vbq_model* m, const DItem* items, int32_t i0, int32_t i1, const uint64_t* pieces,
                                const uint32_t* pstart, const uint32_t* pbytes, uint32_t epoch, uint64_t* base,
                                const uint16_t* x, float* out, cudaStream_t st, int* err) {
  const Layout& L = m->lay;
  DecodeArgs a{};
  a.items = items + i0;
  a.ctas = m->ctas + static_cast<size_t>(i0) * m->sms;
  a.warps = m->warps + static_cast<size_t>(i0) * m->sms * KW;
  a.n_items = i1 - i0;
  a.pieces = pieces;
  a.pstart = pstart;
  a.pbytes = pbytes;
  a.x = x;
  a.d = i0 == 0 ? m->desc.d : 0;
  a.h0 = reinterpret_cast<float*>(base + L.h0);
  a.h0_stats = reinterpret_cast<float2*>(base + L.h0_stats);
  a.h0_flag = reinterpret_cast<uint32_t*>(base + L.h0_flag);
  a.logits = out;
  a.epoch = epoch;
  a.wait_epoch = g_never_ready.load() ? (a.epoch | 0x80000000u) : a.epoch;
  a.spin_limit = g_spin_limit.load();
  a.ns = kRingSlots;
  a.err = err;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(m->sms), 1, 1);
  cfg.blockDim = dim3(KW * 32, 1, 1);
  cfg.dynamicSmemBytes = decode_smem_bytes();
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA is resident: the flag waits need it
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  note_launches(1);
  return cudaLaunchKernelEx(&cfg, vbq_decode_kernel, a);
}

cudaError_t launch_decode(const vbq_model* m, const DItem* items, uint64_t* base, const uint16_t* x, float* out,
                          cudaStream_t st, int* err) {
  return launch_decode_range(m, items, 0, m->n_items, m->pieces, m->pstart, m->pbytes, next_epoch(), base, x, out, st,
                             err);
}

void prepare_decode_kernel() {
  static std::mutex mu;
  static std::map<int, bool> done;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return;
  cudaFuncSetAttribute(vbq_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, decode_smem_bytes());
  done[dev] = true;
}

}  // namespace

extern "C" void vbq_model_free(vbq_model* m);

extern "C" vbq_status vbq_model_create(const vbq_model_desc* desc, const vbq_matrix* const* mats, vbq_model** out) {
  if (!out) return fail(VBQ_ERR_INVALID_ARG, "vbq_model_create: out is NULL");
  *out = nullptr;
  if (!desc || !mats) return fail(VBQ_ERR_INVALID_ARG, "vbq_model_create: NULL desc or mats");
  const vbq_model_desc d = *desc;
  if (d.n_layers < 0 || d.d <= 0 || d.n_heads <= 0 || d.n_kv_heads <= 0 || d.head_dim <= 0 || d.d_ff <= 0 ||
      d.vocab <= 0 || d.n_heads % d.n_kv_heads || !(d.rms_eps >= 0.0f))
    return fail(VBQ_ERR_SHAPE, "vbq_model_create: invalid shapes");
  if (d.d % GROUP || d.d_ff % GROUP || (int64_t(d.n_heads) * d.head_dim) % GROUP)
    return fail(VBQ_ERR_SHAPE, "vbq_model_create: d, d_ff and n_heads*head_dim must be multiples of 64");
  if (d.d > XT_MAX || int64_t(d.n_heads) * d.head_dim > XT_MAX || d.d_ff > XCAP)
    return fail(VBQ_ERR_UNSUPPORTED, "vbq_model_create: d and n_heads*head_dim must be at most " +
                                         std::to_string(XT_MAX) + " and d_ff at most " + std::to_string(XCAP));
  const int nm = d.n_layers * P_PER_LAYER + 1;
  int dev = 0;
  VBQ_CUDA_TRY(cudaGetDevice(&dev));
  for (int i = 0; i < nm; ++i) {
    const vbq_matrix* w = mats[i];
    if (!w) return fail(VBQ_ERR_INVALID_ARG, "vbq_model_create: NULL matrix " + std::to_string(i));
    const int p = i < nm - 1 ? i % P_PER_LAYER : -1;
    const int64_t n = p >= 0 ? proj_n(d, p) : d.vocab;
    const int64_t k = p >= 0 ? proj_k(d, p) : d.d;
    if (w->N != n || w->K != k)
      return fail(VBQ_ERR_SHAPE, "vbq_model_create: matrix " + std::to_string(i) + " is " + std::to_string(w->N) +
                                     "x" + std::to_string(w->K) + ", expected " + std::to_string(n) + "x" +
                                     std::to_string(k));
    if (w->device != dev) return fail(VBQ_ERR_INVALID_ARG, "vbq_model_create: matrices on another device");
  }
  auto* m = new (std::nothrow) vbq_model();
  if (!m) return fail(VBQ_ERR_OOM, "vbq_model_create");
  m->desc = d;
  m->device = dev;
  m->sms = gpu_info().sms;
  m->err = device_check_word();
  if (!m->err) {
    delete m;
    return fail(VBQ_ERR_CUDA, "vbq_model_create: no device check word");
  }
  m->mats.assign(mats, mats + nm);
  // Trace offsets: inputs shared by q/k/v and by gate/up.
  m->in_off.assign(nm, 0);
  m->out_off.assign(nm, 0);
  int64_t io = 0, oo = 0;
  for (int i = 0; i < nm; ++i) {
    const int pp = i < nm - 1 ? i % P_PER_LAYER : -1;
    if (pp == P_K || pp == P_V) {
      m->in_off[i] = m->in_off[i - (pp - P_Q)];
    } else if (pp == P_UP) {
      m->in_off[i] = m->in_off[i - 1];
    } else {
      m->in_off[i] = io;
      io += pp >= 0 ? proj_k(d, pp) : d.d;
    }
    m->out_off[i] = oo;
    oo += pp >= 0 ? proj_n(d, pp) : d.vocab;
  }
  m->in_total = io;
  m->out_total = oo;

  // One plan per item, each over exactly one CTA per SM; the piece lists of all items in turn.
  std::vector<std::vector<uint64_t>> per_warp;
  std::vector<WarpPlan> all_warps;
  std::vector<CtaPlan> all_ctas;
  auto add_plan = [&](std::initializer_list<const vbq_matrix*> ms) -> vbq_status {
    std::vector<SegPlanInput> segs;
    for (const vbq_matrix* w : ms) {
      SegPlanInput s;
      s.runs = &w->runs;
      s.data = w->data;
      s.n_super = static_cast<uint32_t>(w->n_super);
      s.G = static_cast<uint32_t>(w->G);
      segs.push_back(s);
    }
    ItemPlan pl;
    const char* why = "";
    if (!make_item_plan(segs, m->sms, &pl, &why))
      return fail(VBQ_ERR_UNSUPPORTED, std::string("vbq_model_create: ") + why);
    if (!append_pieces(pl, segs, &per_warp))
      return fail(VBQ_ERR_UNSUPPORTED, "vbq_model_create: weight address beyond 2^48");
    per_warp.resize(static_cast<size_t>(m->sms) * KW);
    std::vector<uint32_t> mk(per_warp.size());
    for (size_t w = 0; w < per_warp.size(); ++w) mk[w] = static_cast<uint32_t>(per_warp[w].size());
    m->marks.push_back(std::move(mk));
    all_warps.insert(all_warps.end(), pl.warps.begin(), pl.warps.end());
    all_ctas.insert(all_ctas.end(), pl.ctas.begin(), pl.ctas.end());
    m->item_st_off.push_back(pl.st_off);
    m->item_super.push_back(pl.n_item_super);
    return VBQ_OK;
  };
  vbq_status s = VBQ_OK;
  for (int l = 0; l <= d.n_layers && s == VBQ_OK; ++l) {
    const vbq_matrix* const* W = &m->mats[static_cast<size_t>(l) * P_PER_LAYER];
    if (l == d.n_layers) {
      s = add_plan({W[0]});
    } else if ((s = add_plan({W[P_Q], W[P_K], W[P_V]})) == VBQ_OK && (s = add_plan({W[P_O]})) == VBQ_OK &&
               (s = add_plan({W[P_GATE], W[P_UP]})) == VBQ_OK) {
      s = add_plan({W[P_DOWN]});
    }
  }
  if (s != VBQ_OK) {
    vbq_model_free(m);
    return s;
  }
  m->n_items = static_cast<int32_t>(m->item_super.size());
  m->lay = layout_of(d, m->item_super);

  // Device memory: the step scratch, the host-step staging, then the plans, the piece lists and both item arrays.
  const PieceSet ps = finish_pieces(per_warp);
  auto al = [](int64_t b) { return (b + 255) & ~int64_t(255); };
  const int64_t b_ws = al(8 * m->lay.total), b_x = al(2 * int64_t(d.d)), b_lg = al(4 * int64_t(d.vocab));
  cudaError_t e = dev_alloc(reinterpret_cast<void**>(&m->ws), b_ws + b_x + b_lg);
  if (e == cudaSuccess) e = cudaMemset(m->ws, 0, b_ws);
  if (e != cudaSuccess) {
    vbq_model_free(m);
    return cuda_fail(e, "vbq_model_create: workspace");
  }
  m->x_stage = reinterpret_cast<uint16_t*>(reinterpret_cast<char*>(m->ws) + b_ws);
  m->logits_stage = reinterpret_cast<float*>(reinterpret_cast<char*>(m->ws) + b_ws + b_x);
  const int64_t o_c = 0, o_w = al(int64_t(sizeof(CtaPlan) * all_ctas.size()));
  const int64_t o_p = o_w + al(int64_t(sizeof(WarpPlan) * all_warps.size()));
  const int64_t o_s = o_p + al(8 * int64_t(std::max<size_t>(1, ps.pieces.size())));
  const int64_t o_b = o_s + al(4 * int64_t(ps.start.size()));
  const int64_t o_i1 = o_b + al(4 * int64_t(std::max<size_t>(1, ps.bytes.size())));
  const int64_t o_i2 = o_i1 + al(int64_t(sizeof(DItem)) * m->n_items);
  const int64_t total = o_i2 + al(int64_t(sizeof(DItem)) * m->n_items);
  e = dev_alloc(&m->prog_mem, total);
  char* pm = static_cast<char*>(m->prog_mem);
  if (e == cudaSuccess) e = cudaMemcpy(pm + o_c, all_ctas.data(), sizeof(CtaPlan) * all_ctas.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(pm + o_w, all_warps.data(), sizeof(WarpPlan) * all_warps.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess && !ps.pieces.empty())
    e = cudaMemcpy(pm + o_p, ps.pieces.data(), 8 * ps.pieces.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(pm + o_s, ps.start.data(), 4 * ps.start.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess && !ps.bytes.empty())
    e = cudaMemcpy(pm + o_b, ps.bytes.data(), 4 * ps.bytes.size(), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    vbq_model_free(m);
    return cuda_fail(e, "vbq_model_create: programs");
  }
  m->ctas = reinterpret_cast<const CtaPlan*>(pm + o_c);
  m->warps = reinterpret_cast<const WarpPlan*>(pm + o_w);
  m->pieces = reinterpret_cast<const uint64_t*>(pm + o_p);
  m->pstart = reinterpret_cast<const uint32_t*>(pm + o_s);
  m->pbytes = reinterpret_cast<const uint32_t*>(pm + o_b);
  m->items_ws = reinterpret_cast<DItem*>(pm + o_i1);
  e = upload_items(make_items(m, m->ws, false), m->items_ws);
  // The program over the static scratch of vbq_decode_step_noalloc, when the model fits it. That entry
  // point's set-up happens here, with the model's device current, so that its calls allocate nothing.
  if (e == cudaSuccess && m->lay.total <= kStepScratchWords) {
    uint64_t* sb = nullptr;
    vbq_status ss = step_scratch_address(dev, &sb);
    if (ss != VBQ_OK) {
      vbq_model_free(m);
      return ss;
    }
    m->static_base = sb;
    m->items_static = reinterpret_cast<DItem*>(pm + o_i2);
    e = upload_items(make_items(m, sb, false), m->items_static);
  }
  if (e != cudaSuccess) {
    vbq_model_free(m);
    return cuda_fail(e, "vbq_model_create: items");
  }
  prepare_decode_kernel();
  m->per_warp = std::move(per_warp);
  *out = m;
  return VBQ_OK;
}

extern "C" void vbq_model_free(vbq_model* m) {
  if (!m) return;
  int cur = 0;
  cudaGetDevice(&cur);
  cudaSetDevice(m->device);
  cudaDeviceSynchronize();
  cudaFree(m->ws);
  cudaFree(m->prog_mem);
  cudaFree(m->tr_in);
  cudaFree(m->tr_out);
  cudaFree(m->kv);
  cudaFree(m->ctx_mem);
  cudaSetDevice(cur);
  delete m;
}

extern "C" vbq_status vbq_decode_step(vbq_model* m, const uint16_t* x_dev, float* logits_dev, void* stream) {
  if (!m || !x_dev || !logits_dev) return fail(VBQ_ERR_INVALID_ARG, "vbq_decode_step: NULL argument");
  if (reinterpret_cast<uintptr_t>(logits_dev) % 4 || reinterpret_cast<uintptr_t>(x_dev) % 4)
    return fail(VBQ_ERR_INVALID_ARG, "vbq_decode_step: misaligned buffer (x and logits need 4-byte alignment)");
  int dev = 0;
  VBQ_CUDA_TRY(cudaGetDevice(&dev));
  if (dev != m->device) return fail(VBQ_ERR_INVALID_ARG, "vbq_decode_step: model is on another device");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  VBQ_CUDA_TRY(launch_decode(m, m->items_ws, m->ws, x_dev, logits_dev, st, m->err));
  if (m->trace) {
    const int64_t ph = int64_t(m->desc.n_layers) * P_PER_LAYER;
    VBQ_CUDA_TRY(cudaMemcpyAsync(m->tr_out + m->out_off[ph], logits_dev, 4 * static_cast<size_t>(m->desc.vocab),
                                 cudaMemcpyDeviceToDevice, st));
  }
  return VBQ_OK;
}

extern "C" vbq_status vbq_decode_step_host(vbq_model* m, const uint16_t* x_host, float* logits_host, void* stream) {
  if (!m || !x_host || !logits_host) return fail(VBQ_ERR_INVALID_ARG, "vbq_decode_step_host: NULL argument");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  VBQ_CUDA_TRY(cudaMemcpyAsync(m->x_stage, x_host, 2 * static_cast<size_t>(m->desc.d), cudaMemcpyHostToDevice, st));
  vbq_status s = vbq_decode_step(m, m->x_stage, m->logits_stage, stream);
  if (s != VBQ_OK) return s;
  VBQ_CUDA_TRY(cudaMemcpyAsync(logits_host, m->logits_stage, 4 * static_cast<size_t>(m->desc.vocab),
                               cudaMemcpyDeviceToHost, st));
  VBQ_CUDA_TRY(cudaStreamSynchronize(st));
  return VBQ_OK;
}

extern "C" vbq_status vbq_model_set_trace(vbq_model* m, int32_t enable) {
  if (!m) return fail(VBQ_ERR_INVALID_ARG, "vbq_model_set_trace: NULL model");
  if (enable && !m->tr_in) {
    VBQ_CUDA_TRY(cudaMalloc(&m->tr_in, 2 * static_cast<size_t>(m->in_total)));
    VBQ_CUDA_TRY(cudaMalloc(&m->tr_out, 4 * static_cast<size_t>(m->out_total)));
  }
  m->trace = enable != 0;
  VBQ_CUDA_TRY(cudaDeviceSynchronize());  // no step may be reading the items
  VBQ_CUDA_TRY(upload_items(make_items(m, m->ws, m->trace), m->items_ws));
  if (m->items_ctx) VBQ_CUDA_TRY(upload_items(make_items(m, m->ws, m->trace, true), m->items_ctx));
  return VBQ_OK;
}

extern "C" vbq_status vbq_model_trace_info(const vbq_model* m, int64_t* in_off, int64_t* out_off, int64_t* in_total,
                                           int64_t* out_total) {
  if (!m) return fail(VBQ_ERR_INVALID_ARG, "vbq_model_trace_info: NULL model");
  const size_t nm = m->in_off.size();
  if (in_off)
    for (size_t i = 0; i < nm; ++i) in_off[i] = m->in_off[i];
  if (out_off)
    for (size_t i = 0; i < nm; ++i) out_off[i] = m->out_off[i];
  if (in_total) *in_total = m->in_total;
  if (out_total) *out_total = m->out_total;
  return VBQ_OK;
}

extern "C" vbq_status vbq_model_read_trace(const vbq_model* m, uint16_t* in_host, float* out_host) {
  if (!m || !in_host || !out_host) return fail(VBQ_ERR_INVALID_ARG, "vbq_model_read_trace: NULL argument");
  if (!m->tr_in) return fail(VBQ_ERR_INVALID_ARG, "vbq_model_read_trace: trace was never enabled");
  VBQ_CUDA_TRY(cudaDeviceSynchronize());
  VBQ_CUDA_TRY(cudaMemcpy(in_host, m->tr_in, 2 * static_cast<size_t>(m->in_total), cudaMemcpyDeviceToHost));
  VBQ_CUDA_TRY(cudaMemcpy(out_host, m->tr_out, 4 * static_cast<size_t>(m->out_total), cudaMemcpyDeviceToHost));
  return VBQ_OK;
}

// ---------------------------------------------------------------- allocation-free decode step
//
// ---- context steps -----------------------------------------------------------
//
// vbq_decode_step_at runs the same items as vbq_decode_step, cut after each
// layer's [q;k;v] item into n_layers + 1 launches; between them, one layer's
// attention: its q and new k turned by the rotary embedding at pos and k, v
// appended to the layer's cache (vbq_attn_prep_kernel), then attention of the
// query heads over positions 0 .. pos (vbq_attention_decode) into attn_out,
// which the layer's o item reads. Every launch of a step shares its epoch; a
// launch's flags are all set when the next launch starts.

extern "C" vbq_status vbq_model_set_context(vbq_model* m, int32_t max_context, double rope_theta) {
  if (!m) return fail(VBQ_ERR_INVALID_ARG, "vbq_model_set_context: NULL model");
  const vbq_model_desc& d = m->desc;
  if (max_context < 0 || max_context > 65536)
    return fail(VBQ_ERR_SHAPE, "vbq_model_set_context: max_context must be in [0, 65536]");
  if (max_context > 0 && (d.head_dim != 64 && d.head_dim != 128))
    return fail(VBQ_ERR_UNSUPPORTED, "vbq_model_set_context: head_dim must be 64 or 128");
  if (max_context > 0 && d.n_heads / d.n_kv_heads > 8)
    return fail(VBQ_ERR_UNSUPPORTED, "vbq_model_set_context: at most 8 query heads per kv head");
  if (max_context > 0 && !(rope_theta > 1.0)) return fail(VBQ_ERR_INVALID_ARG, "vbq_model_set_context: theta must be > 1");
  int cur = 0;
  VBQ_CUDA_TRY(cudaGetDevice(&cur));
  if (cur != m->device) return fail(VBQ_ERR_INVALID_ARG, "vbq_model_set_context: model is on another device");
  VBQ_CUDA_TRY(cudaDeviceSynchronize());  // no step may be using what is freed
  cudaFree(m->kv);
  cudaFree(m->ctx_mem);
  m->kv = nullptr;
  m->ctx_mem = nullptr;
  m->q_rot = nullptr;
  m->attn_out = nullptr;
  m->items_ctx = nullptr;
  m->max_ctx = 0;
  m->seg_item0.clear();
  if (max_context == 0) return VBQ_OK;

  // Segments: items [seg_item0[s], seg_item0[s + 1]), cut after every [q;k;v] item.
  std::vector<int32_t> b{0};
  for (int l = 0; l < d.n_layers; ++l) b.push_back(l * L_PER_LAYER + L_QKV + 1);
  b.push_back(m->n_items);
  const size_t n_seg = b.size() - 1, nw = m->per_warp.size();
  // Each segment's piece lists, warp after warp.
  std::vector<uint64_t> pieces;
  std::vector<uint32_t> start, bytes;
  for (size_t sg = 0; sg < n_seg; ++sg) {
    for (size_t w = 0; w < nw; ++w) {
      const uint32_t p0 = b[sg] == 0 ? 0u : m->marks[b[sg] - 1][w];
      const uint32_t p1 = m->marks[b[sg + 1] - 1][w];
      start.push_back(static_cast<uint32_t>(pieces.size()));
      uint64_t by = 0;
      for (uint32_t p = p0; p < p1; ++p) {
        pieces.push_back(m->per_warp[w][p]);
        by += (m->per_warp[w][p] & 0xFFFFFu) << 4;
      }
      bytes.push_back(static_cast<uint32_t>(by));
    }
    start.push_back(static_cast<uint32_t>(pieces.size()));
  }
  const int64_t hd = int64_t(d.n_heads) * d.head_dim;
  const size_t kv_elems = size_t(d.n_layers) * 2 * d.n_kv_heads * size_t(max_context) * d.head_dim;
  auto al = [](size_t v) { return (v + 255) & ~size_t(255); };
  const size_t o_q = 0, o_a = o_q + al(2 * hd), o_i = o_a + al(4 * hd);
  const size_t o_p = o_i + al(sizeof(DItem) * m->n_items);
  const size_t o_s = o_p + al(8 * std::max<size_t>(1, pieces.size()));
  const size_t o_b = o_s + al(4 * start.size());
  const size_t total = o_b + al(4 * bytes.size());
  cudaError_t e = dev_alloc(reinterpret_cast<void**>(&m->kv), std::max<size_t>(2, 2 * kv_elems));
  if (e == cudaSuccess) e = cudaMemset(m->kv, 0, std::max<size_t>(2, 2 * kv_elems));
  if (e == cudaSuccess) e = dev_alloc(&m->ctx_mem, total);
  char* cm = static_cast<char*>(m->ctx_mem);
  if (e == cudaSuccess && !pieces.empty()) e = cudaMemcpy(cm + o_p, pieces.data(), 8 * pieces.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(cm + o_s, start.data(), 4 * start.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess && !bytes.empty()) e = cudaMemcpy(cm + o_b, bytes.data(), 4 * bytes.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) {
    m->q_rot = reinterpret_cast<uint16_t*>(cm + o_q);
    m->attn_out = reinterpret_cast<float*>(cm + o_a);
    m->items_ctx = reinterpret_cast<DItem*>(cm + o_i);
    m->seg_pieces = reinterpret_cast<const uint64_t*>(cm + o_p);
    m->seg_start = reinterpret_cast<const uint32_t*>(cm + o_s);
    m->seg_bytes = reinterpret_cast<const uint32_t*>(cm + o_b);
    e = upload_items(make_items(m, m->ws, m->trace, true), m->items_ctx);
  }
  if (e != cudaSuccess) {
    cudaFree(m->kv);
    cudaFree(m->ctx_mem);
    m->kv = nullptr;
    m->ctx_mem = nullptr;
    m->items_ctx = nullptr;
    return cuda_fail(e, "vbq_model_set_context");
  }
  m->max_ctx = max_context;
  m->rope_theta = rope_theta;
  m->seg_item0 = b;
  return VBQ_OK;
}

extern "C" vbq_status vbq_model_kv_cache(const vbq_model* m, int32_t layer, uint16_t** k, uint16_t** v,
                                         int64_t* stride) {
  if (!m || !k || !v || !stride) return fail(VBQ_ERR_INVALID_ARG, "vbq_model_kv_cache: NULL argument");
  if (!m->kv) return fail(VBQ_ERR_INVALID_ARG, "vbq_model_kv_cache: no context set (vbq_model_set_context)");
  if (layer < 0 || layer >= m->desc.n_layers) return fail(VBQ_ERR_SHAPE, "vbq_model_kv_cache: layer out of range");
  const size_t per = size_t(m->desc.n_kv_heads) * size_t(m->max_ctx) * m->desc.head_dim;
  *k = m->kv + size_t(layer) * 2 * per;
  *v = *k + per;
  *stride = m->max_ctx;
  return VBQ_OK;
}

extern "C" vbq_status vbq_decode_step_at(vbq_model* m, const uint16_t* x_dev, int32_t pos, float* logits_dev,
                                         void* stream) {
  if (!m || !x_dev || !logits_dev) return fail(VBQ_ERR_INVALID_ARG, "vbq_decode_step_at: NULL argument");
  if (reinterpret_cast<uintptr_t>(logits_dev) % 4 || reinterpret_cast<uintptr_t>(x_dev) % 4)
    return fail(VBQ_ERR_INVALID_ARG, "vbq_decode_step_at: misaligned buffer (x and logits need 4-byte alignment)");
  if (!m->items_ctx) return fail(VBQ_ERR_INVALID_ARG, "vbq_decode_step_at: no context set (vbq_model_set_context)");
  if (pos < 0 || pos >= m->max_ctx) return fail(VBQ_ERR_SHAPE, "vbq_decode_step_at: need 0 <= pos < max_context");
  int dev = 0;
  VBQ_CUDA_TRY(cudaGetDevice(&dev));
  if (dev != m->device) return fail(VBQ_ERR_INVALID_ARG, "vbq_decode_step_at: model is on another device");
  const vbq_model_desc& d = m->desc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const uint32_t epoch = next_epoch();
  const size_t nw = m->per_warp.size(), n_seg = m->seg_item0.size() - 1;
  for (size_t sg = 0; sg < n_seg; ++sg) {
    VBQ_CUDA_TRY(launch_decode_range(m, m->items_ctx, m->seg_item0[sg], m->seg_item0[sg + 1], m->seg_pieces,
                                     m->seg_start + sg * (nw + 1), m->seg_bytes + sg * nw, epoch, m->ws, x_dev,
                                     logits_dev, st, m->err));
    if (sg + 1 == n_seg) break;
    const int l = static_cast<int>(sg);  // the segment ended with layer l's [q;k;v]
    const Layout& L = m->lay;
    const int iq = l * L_PER_LAYER + L_QKV;
    const float* qkv = reinterpret_cast<const float*>(m->ws + L.items[iq].out);
    const std::vector<uint32_t>& so = m->item_st_off[iq];
    uint16_t *kc = nullptr, *vc = nullptr;
    int64_t stride = 0;
    vbq_status s = vbq_model_kv_cache(m, l, &kc, &vc, &stride);
    if (s != VBQ_OK) return s;
    s = launch_attn_prep(qkv, int64_t(so[0]) * SROWS, int64_t(so[1]) * SROWS, int64_t(so[2]) * SROWS, m->q_rot, kc,
                         vc, d.n_heads, d.n_kv_heads, d.head_dim, stride, pos, m->rope_theta, st);
    if (s != VBQ_OK) return s;
    s = vbq_attention_decode(m->q_rot, kc, vc, d.n_heads, d.n_kv_heads, d.head_dim, stride, pos + 1, m->attn_out,
                             stream);
    if (s != VBQ_OK) return s;
  }
  if (m->trace) {
    const int64_t ph = int64_t(d.n_layers) * P_PER_LAYER;
    VBQ_CUDA_TRY(cudaMemcpyAsync(m->tr_out + m->out_off[ph], logits_dev, 4 * static_cast<size_t>(d.vocab),
                                 cudaMemcpyDeviceToDevice, st));
  }
  return VBQ_OK;
}

// vbq_decode_step keeps its step scratch (each item's fixed-point sums,
// float outputs, arrival counters, flags and statistics) in memory that
// vbq_model_create allocated for the model. Some callers cannot tie device
// memory to a model they step: real-time loops whose device memory is fixed
// before the loop starts, or hosts that hand out device memory only from their
// own pool. vbq_decode_step_noalloc serves them: it launches the same kernel
// with the step's scratch in the file-scope array below, and allocates nothing.

namespace {

// Step scratch of vbq_decode_step_noalloc, in the Layout of the model:
// 4,194,304 8-byte words = 32 MiB on every device that loads this library,
// held until the process exits.
static __device__ __align__(256) uint64_t g_step_scratch[kStepScratchWords];

std::mutex g_step_scratch_mu;
std::map<int, uint64_t*> g_step_scratch_addr;  // device ordinal -> device address of g_step_scratch

// Device address of g_step_scratch on device dev, which must be current. The
// first call on a device looks it up and clears the array; later calls only
// read the cached value.
vbq_status step_scratch_address(int dev, uint64_t** out) {
  std::lock_guard<std::mutex> lock(g_step_scratch_mu);
  auto it = g_step_scratch_addr.find(dev);
  if (it != g_step_scratch_addr.end()) {
    *out = it->second;
    return VBQ_OK;
  }
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_step_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(g_step_scratch)");
  // Steps need the sums and counters at zero; they leave them so.
  e = cudaMemset(p, 0, sizeof(uint64_t) * kStepScratchWords);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "clearing g_step_scratch");
  g_step_scratch_addr[dev] = static_cast<uint64_t*>(p);
  *out = static_cast<uint64_t*>(p);
  return VBQ_OK;
}

}  // namespace

extern "C" vbq_status vbq_decode_step_noalloc(vbq_model* m, const uint16_t* x_dev, float* logits_dev, void* stream) {
  if (!m || !x_dev || !logits_dev) return fail(VBQ_ERR_INVALID_ARG, "vbq_decode_step_noalloc: NULL argument");
  if (reinterpret_cast<uintptr_t>(logits_dev) % 4 || reinterpret_cast<uintptr_t>(x_dev) % 4)
    return fail(VBQ_ERR_INVALID_ARG,
                "vbq_decode_step_noalloc: misaligned buffer (x and logits need 4-byte alignment)");
  const int64_t limit = g_noalloc_words.load() > 0 ? std::min(g_noalloc_words.load(), kStepScratchWords)
                                                    : kStepScratchWords;
  if (m->lay.total > limit)
    return fail(VBQ_ERR_SHAPE, "vbq_decode_step_noalloc: the step needs " + std::to_string(m->lay.total) +
                                   " scratch words of 8 bytes (per item: fixed-point sums, outputs, counters and "
                                   "flags); the static scratch holds " +
                                   std::to_string(limit));
  int dev = 0;
  VBQ_CUDA_TRY(cudaGetDevice(&dev));
  if (dev != m->device) return fail(VBQ_ERR_INVALID_ARG, "vbq_decode_step_noalloc: model is on another device");
  if (!m->items_static) return fail(VBQ_ERR_CUDA, "vbq_decode_step_noalloc: the static scratch was not set up");
  cudaError_t e = launch_decode(m, m->items_static, m->static_base, x_dev, logits_dev,
                                static_cast<cudaStream_t>(stream), m->err);
  if (e != cudaSuccess) return cuda_fail(e, "vbq_decode_step_noalloc: launch");
  return VBQ_OK;
}

extern "C" vbq_status vbq_debug_set(int32_t key, int64_t value) {
  switch (key) {
    case VBQ_DEBUG_WAIT_LIMIT:
      if (value < 0) return fail(VBQ_ERR_INVALID_ARG, "vbq_debug_set: negative wait limit");
      g_spin_limit.store(value == 0 ? kSpinCycles : value);
      return VBQ_OK;
    case VBQ_DEBUG_NEVER_READY:
      g_never_ready.store(value != 0);
      return VBQ_OK;
    case VBQ_DEBUG_ALLOC_CAP:
      if (value < 0) return fail(VBQ_ERR_INVALID_ARG, "vbq_debug_set: negative byte count");
      set_alloc_cap(value);
      return VBQ_OK;
    case VBQ_DEBUG_NOALLOC_WORDS:
      if (value < 0) return fail(VBQ_ERR_INVALID_ARG, "vbq_debug_set: negative word count");
      g_noalloc_words.store(value);
      return VBQ_OK;
    default:
      return fail(VBQ_ERR_INVALID_ARG, "vbq_debug_set: unknown key " + std::to_string(key));
  }
}
