// vbq_decode_step: one batch-1 decode step through a stack of VBQ projections.
//
// VBQ abstract ("Variable Bit-width Quantization ..."): packed per-group codes
// speed up token-by-token decode, whose speed memory bandwidth sets. The pages give no
// architecture, so the glue below is this library's reading: unit-gamma
// RMSNorm, attention at position 0 (a softmax over one key is 1, so each query
// head returns its kv group's v), SwiGLU, fp32 residual, and bf16 at every
// projection input.
//
// A step is one persistent kernel (vbq_decode_kernel in gemv.cuh): one CTA per
// SM runs h = x, then per layer four GEMV items, then the head:
//   [q;k;v] (RMSNorm in its prologue), o (GQA gather in its prologue, residual
//   in its epilogue), [gate;up] (RMSNorm prologue), down (SwiGLU prologue,
//   residual epilogue),
// with a grid barrier between items. Each warp streams its share of every
// item's packed weights back to back, so the next item's weights are already
// arriving while the CTAs wait at a barrier. The items, their work plans and
// the per-warp piece lists are built once, when the model is created.
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"
#include "launch.h"

using namespace vbq;

namespace {

enum { P_Q = 0, P_K, P_V, P_O, P_GATE, P_UP, P_DOWN, P_PER_LAYER };
enum { L_QKV = 0, L_O, L_GU, L_DOWN, L_PER_LAYER };

constexpr int DEC_W = 16;     // warps per CTA of the decode kernel
constexpr int DEC_NSLOT = 2;  // ring slots per warp

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

int64_t round64(int64_t n) { return (n + 63) & ~int64_t(63); }

// Float offsets of one step's activations inside a region: the grid-barrier
// counters, h, [q;k;v] and [gate;up]. The counters must be zero before a step;
// each step leaves them so. (Split-tile partial rows and arrival counters live
// in each item's work plan, which the model owns.)
struct Layout {
  int64_t bar = 0, h = 0, qkv = 0, gu = 0, total = 0;
};

Layout layout_of(const vbq_model_desc& d) {
  Layout L;
  L.bar = 0;
  L.h = 64;
  L.qkv = L.h + round64(d.d);
  L.gu = L.qkv + round64(proj_n(d, P_Q) + 2 * proj_n(d, P_K));
  L.total = L.gu + round64(2 * int64_t(d.d_ff));
  return L;
}

}  // namespace

struct vbq_model {
  vbq_model_desc desc{};
  std::vector<const vbq_matrix*> mats;
  int device = 0;
  int sms = 0;
  Layout lay;
  float* ws = nullptr;              // this model's step scratch (Layout), then the host-step staging
  uint16_t* x_stage = nullptr;
  float* logits_stage = nullptr;
  bool trace = false;
  uint16_t* tr_in = nullptr;
  float* tr_out = nullptr;
  std::vector<int64_t> in_off, out_off;
  int64_t in_total = 0, out_total = 0;
  std::vector<DevicePlan> plans;    // per item
  void* prog_mem = nullptr;         // piece lists and the items of both programs
  const uint64_t* pieces = nullptr;
  const uint32_t* pstart = nullptr;
  const uint32_t* pbytes = nullptr;
  Item* items_ws = nullptr;         // items over ws
  Item* items_static = nullptr;     // items over the static scratch (null if the model does not fit it)
  ZeroSpec pre_ws[2] = {}, pre_static[2] = {};  // what each program clears before its first barrier
  float* static_base = nullptr;
  int32_t n_items = 0;
  int* err = nullptr;               // the device check word of the model's device
};

namespace {

// The static scratch of vbq_decode_step_noalloc (defined at the bottom of this file).
vbq_status step_scratch_address(int dev, float** out);
constexpr int64_t kStepScratchFloats = 65536;

// The items of one step over the scratch at `base`. Each item clears the
// output of the item two after it (the outputs that split tiles add into);
// pre receives the outputs of the first two items, cleared before the first
// grid barrier.
std::vector<Item> make_items(const vbq_model* m, float* base, bool trace, ZeroSpec pre[2]) {
  const vbq_model_desc& d = m->desc;
  const Layout& L = m->lay;
  float* h = base + L.h;
  float* qkv = base + L.qkv;
  float* gu = base + L.gu;
  const int64_t nq = proj_n(d, P_Q), nkv = proj_n(d, P_K);
  auto tin = [&](int p) -> uint16_t* { return trace ? m->tr_in + m->in_off[p] : nullptr; };
  auto tout = [&](int p) -> float* { return trace ? m->tr_out + m->out_off[p] : nullptr; };
  std::vector<Item> items;
  std::vector<ZeroSpec> outputs;  // per item: what its split tiles add into (n = 0: adds onto h)
  std::vector<CopySpec> traces;   // per item: its traced output, copied by the next item
  auto item_for = [&](int li) {
    Item it{};
    it.plan = plan_view(m->plans[li]);
    it.ep = EP_STORE;
    return it;
  };
  auto add_seg = [&](Item& it, const vbq_matrix* w, float* y, float* ty) {
    it.seg[it.nseg] = view_of(w, y, static_cast<int32_t>(w->N), ty);
    it.nseg += 1;
  };
  for (int l = 0; l < d.n_layers; ++l) {
    const vbq_matrix* const* W = &m->mats[static_cast<size_t>(l) * P_PER_LAYER];
    const int p0 = l * P_PER_LAYER, l0 = l * L_PER_LAYER;
    {  // [q; k; v] = W u, u = bf16(rmsnorm(h))
      Item it = item_for(l0 + L_QKV);
      add_seg(it, W[P_Q], qkv, nullptr);
      add_seg(it, W[P_K], qkv + nq, nullptr);
      add_seg(it, W[P_V], qkv + nq + nkv, nullptr);
      it.xs.mode = X_RMSNORM;
      it.xs.K = d.d;
      it.xs.h = h;
      it.xs.eps = d.rms_eps;
      it.xs.trace_x = tin(p0 + P_Q);
      items.push_back(it);
      outputs.push_back(ZeroSpec{qkv, 0, static_cast<int32_t>(nq + 2 * nkv)});
      traces.push_back(CopySpec{qkv, tout(p0 + P_Q), trace ? static_cast<int32_t>(nq + 2 * nkv) : 0});
    }
    {  // h += Wo a, a = bf16(v of each head's kv group)
      Item it = item_for(l0 + L_O);
      add_seg(it, W[P_O], h, tout(p0 + P_O));
      it.xs.mode = X_GQA;
      it.xs.K = static_cast<int32_t>(nq);
      it.xs.v = qkv + nq + nkv;
      it.xs.head_dim = d.head_dim;
      it.xs.group = d.n_heads / d.n_kv_heads;
      it.xs.trace_x = tin(p0 + P_O);
      it.ep = EP_RESID;
      it.resid = h;
      items.push_back(it);
      outputs.push_back(ZeroSpec{nullptr, 0, 0});
      traces.push_back(CopySpec{});
    }
    {  // [gate; up] = W u, u = bf16(rmsnorm(h))
      Item it = item_for(l0 + L_GU);
      add_seg(it, W[P_GATE], gu, nullptr);
      add_seg(it, W[P_UP], gu + d.d_ff, nullptr);
      it.xs.mode = X_RMSNORM;
      it.xs.K = d.d;
      it.xs.h = h;
      it.xs.eps = d.rms_eps;
      it.xs.trace_x = tin(p0 + P_GATE);
      items.push_back(it);
      outputs.push_back(ZeroSpec{gu, 0, 2 * d.d_ff});
      traces.push_back(CopySpec{gu, tout(p0 + P_GATE), trace ? 2 * d.d_ff : 0});
    }
    {  // h += Wdown bf16(silu(gate) * up)
      Item it = item_for(l0 + L_DOWN);
      add_seg(it, W[P_DOWN], h, tout(p0 + P_DOWN));
      it.xs.mode = X_SWIGLU;
      it.xs.K = d.d_ff;
      it.xs.gate = gu;
      it.xs.up = gu + d.d_ff;
      it.xs.trace_x = tin(p0 + P_DOWN);
      it.ep = EP_RESID;
      it.resid = h;
      items.push_back(it);
      outputs.push_back(ZeroSpec{nullptr, 0, 0});
      traces.push_back(CopySpec{});
    }
  }
  {  // logits = Whead bf16(rmsnorm(h)), into the launch's output
    const int lh = d.n_layers * L_PER_LAYER, ph = d.n_layers * P_PER_LAYER;
    Item it = item_for(lh);
    add_seg(it, m->mats[ph], nullptr, nullptr);  // traced by a copy after the launch
    it.xs.mode = X_RMSNORM;
    it.xs.K = d.d;
    it.xs.h = h;
    it.xs.eps = d.rms_eps;
    it.xs.trace_x = tin(ph);
    items.push_back(it);
    outputs.push_back(ZeroSpec{nullptr, 0, d.vocab});  // the launch's logits
    traces.push_back(CopySpec{});
  }
  for (size_t i = 1; i < items.size(); ++i) items[i].tcopy = traces[i - 1];
  for (size_t i = 0; i < items.size(); ++i) items[i].zero = i + 2 < items.size() ? outputs[i + 2] : ZeroSpec{};
  for (int i = 0; i < 2; ++i) pre[i] = static_cast<size_t>(i) < outputs.size() ? outputs[i] : ZeroSpec{};
  return items;
}

cudaError_t upload_items(const std::vector<Item>& items, Item* dst) {
  return cudaMemcpy(dst, items.data(), sizeof(Item) * items.size(), cudaMemcpyHostToDevice);
}

cudaError_t launch_decode(const vbq_model* m, const Item* items, const ZeroSpec* pre, float* base,
                          const uint16_t* x, float* out, cudaStream_t st, int* err) {
  DecodeArgs a{};
  a.prog.items = items;
  a.prog.n_items = m->n_items;
  a.prog.pieces = m->pieces;
  a.prog.pstart = m->pstart;
  a.prog.pbytes = m->pbytes;
  a.prog.h = base + m->lay.h;
  a.prog.d = m->desc.d;
  a.prog.grid_bar = reinterpret_cast<uint32_t*>(base + m->lay.bar);
  a.prog.err = err;
  a.prog.pre[0] = pre[0];
  a.prog.pre[1] = pre[1];
  a.x = x;
  a.out = out;
  // The grid-barrier and split-tile counters are zero here: the scratch starts
  // zeroed, and every launch leaves them at zero when it ends.
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(m->sms), 1, 1);
  cfg.blockDim = dim3(DEC_W * 32, 1, 1);
  cfg.dynamicSmemBytes = GemvSmem<1, DEC_W, DEC_NSLOT>::kBytesStaged;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA is resident: the grid barriers need it
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  note_launches(1);
  return cudaLaunchKernelEx(&cfg, vbq_decode_kernel<DEC_W, DEC_NSLOT>, a);
}

void prepare_decode_kernel() {
  static std::mutex mu;
  static std::map<int, bool> done;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return;
  cudaFuncSetAttribute(vbq_decode_kernel<DEC_W, DEC_NSLOT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       GemvSmem<1, DEC_W, DEC_NSLOT>::kBytesStaged);
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
      d.vocab <= 0 || d.n_heads % d.n_kv_heads || d.head_dim % 2 || !(d.rms_eps >= 0.0f))
    return fail(VBQ_ERR_SHAPE, "vbq_model_create: invalid shapes");
  if (d.d > XCAP || d.d_ff > XCAP || int64_t(d.n_heads) * d.head_dim > XCAP)
    return fail(VBQ_ERR_UNSUPPORTED, "vbq_model_create: d, d_ff and n_heads*head_dim must be at most " +
                                         std::to_string(XCAP) + " (the decode kernel stages x in shared memory)");
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

  // One plan per item, every one over exactly one CTA per SM; the piece lists of all items in turn.
  std::vector<std::vector<uint64_t>> per_warp;
  auto add_plan = [&](std::initializer_list<const vbq_matrix*> ms) -> vbq_status {
    std::vector<SegTables> segs;
    std::vector<const uint8_t*> data;
    for (const vbq_matrix* w : ms) {
      segs.push_back(seg_tables(w));
      data.push_back(w->data);
    }
    Plan pl = make_plan(segs, m->sms, MAX_UNITS_PER_CTA);
    if (pl.n_ctas != m->sms && pl.n_ctas != 0)
      return fail(VBQ_ERR_UNSUPPORTED, "vbq_model_create: a projection needs more than one CTA per SM");
    if (pl.n_ctas == 0) {  // an empty projection: one empty slot per CTA
      pl.n_ctas = m->sms;
      pl.umax = 1;
      pl.units.assign(m->sms, UnitRec{});
      pl.slices.assign(static_cast<size_t>(m->sms) * SLICES, SliceRec{});
    }
    if (!append_pieces(pl, data, DEC_W, &per_warp))
      return fail(VBQ_ERR_UNSUPPORTED, "vbq_model_create: weight address beyond 2^48 or a warp piece of 16 MiB or more");
    DevicePlan dp;
    cudaError_t err = upload_plan(pl, 1, data, nullptr, &dp);
    if (err != cudaSuccess) return cuda_fail(err, "vbq_model_create: plan upload");
    m->plans.push_back(dp);
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
  m->n_items = static_cast<int32_t>(m->plans.size());
  m->lay = layout_of(d);

  // Device memory: the step scratch, the host-step staging, the piece lists and both item arrays.
  const PieceSet ps = finish_pieces(per_warp);
  auto al = [](int64_t b) { return (b + 255) & ~int64_t(255); };
  const int64_t b_ws = al(4 * m->lay.total), b_x = al(2 * int64_t(d.d)), b_lg = al(4 * int64_t(d.vocab));
  cudaError_t e = cudaMalloc(&m->ws, b_ws + b_x + b_lg);
  if (e == cudaSuccess) e = cudaMemset(m->ws, 0, b_ws);
  if (e != cudaSuccess) {
    vbq_model_free(m);
    return cuda_fail(e, "vbq_model_create: workspace");
  }
  m->x_stage = reinterpret_cast<uint16_t*>(reinterpret_cast<char*>(m->ws) + b_ws);
  m->logits_stage = reinterpret_cast<float*>(reinterpret_cast<char*>(m->ws) + b_ws + b_x);
  const int64_t o_p = 0, o_s = al(8 * int64_t(std::max<size_t>(1, ps.pieces.size())));
  const int64_t o_b = o_s + al(4 * int64_t(ps.start.size()));
  const int64_t o_i1 = o_b + al(4 * int64_t(std::max<size_t>(1, ps.bytes.size())));
  const int64_t o_i2 = o_i1 + al(int64_t(sizeof(Item)) * m->n_items);
  const int64_t total = o_i2 + al(int64_t(sizeof(Item)) * m->n_items);
  e = cudaMalloc(&m->prog_mem, total);
  char* pm = static_cast<char*>(m->prog_mem);
  if (e == cudaSuccess && !ps.pieces.empty())
    e = cudaMemcpy(pm + o_p, ps.pieces.data(), 8 * ps.pieces.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(pm + o_s, ps.start.data(), 4 * ps.start.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess && !ps.bytes.empty())
    e = cudaMemcpy(pm + o_b, ps.bytes.data(), 4 * ps.bytes.size(), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    vbq_model_free(m);
    return cuda_fail(e, "vbq_model_create: programs");
  }
  m->pieces = reinterpret_cast<const uint64_t*>(pm + o_p);
  m->pstart = reinterpret_cast<const uint32_t*>(pm + o_s);
  m->pbytes = reinterpret_cast<const uint32_t*>(pm + o_b);
  m->items_ws = reinterpret_cast<Item*>(pm + o_i1);
  e = upload_items(make_items(m, m->ws, false, m->pre_ws), m->items_ws);
  // The program over the static scratch of vbq_decode_step_noalloc, when the model fits it. That entry
  // point's set-up happens here, with the model's device current, so that its calls allocate nothing.
  if (e == cudaSuccess && m->lay.total <= kStepScratchFloats) {
    float* sb = nullptr;
    vbq_status ss = step_scratch_address(dev, &sb);
    if (ss != VBQ_OK) {
      vbq_model_free(m);
      return ss;
    }
    m->static_base = sb;
    m->items_static = reinterpret_cast<Item*>(pm + o_i2);
    e = upload_items(make_items(m, sb, false, m->pre_static), m->items_static);
  }
  if (e != cudaSuccess) {
    vbq_model_free(m);
    return cuda_fail(e, "vbq_model_create: items");
  }
  prepare_decode_kernel();
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
  for (DevicePlan& p : m->plans) free_plan(&p);
  cudaSetDevice(cur);
  delete m;
}

extern "C" vbq_status vbq_decode_step(vbq_model* m, const uint16_t* x_dev, float* logits_dev, void* stream) {
  if (!m || !x_dev || !logits_dev) return fail(VBQ_ERR_INVALID_ARG, "vbq_decode_step: NULL argument");
  if (reinterpret_cast<uintptr_t>(logits_dev) % 4 || reinterpret_cast<uintptr_t>(x_dev) % 4)
    return fail(VBQ_ERR_INVALID_ARG, "vbq_decode_step: misaligned buffer (x and logits need 4-byte alignment)");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (m->trace)  // traced outputs that add onto the residual are sums of adds
    VBQ_CUDA_TRY(cudaMemsetAsync(m->tr_out, 0, 4 * static_cast<size_t>(m->out_total), st));
  VBQ_CUDA_TRY(launch_decode(m, m->items_ws, m->pre_ws, m->ws, x_dev, logits_dev, st, m->err));
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
  VBQ_CUDA_TRY(upload_items(make_items(m, m->ws, m->trace, m->pre_ws), m->items_ws));
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
// vbq_decode_step keeps its step scratch (activations and the grid-barrier
// counters) in memory that vbq_model_create allocated for the model. Some callers cannot tie device memory to a model
// they step: code that runs while another component is capturing the stream
// into its own graph, real-time loops whose device memory is fixed before the
// loop starts, or hosts that hand out device memory only from their own pool.
// vbq_decode_step_noalloc serves them: it launches the same kernel with the
// step's scratch in the file-scope array below, and allocates nothing.

namespace {

// Step scratch of vbq_decode_step_noalloc, in the Layout of the model: 65,536
// floats = 256 KiB on every device that loads this library, held until the
// process exits.
static __device__ __align__(256) float g_step_scratch[kStepScratchFloats];

std::mutex g_step_scratch_mu;
std::map<int, float*> g_step_scratch_addr;  // device ordinal -> device address of g_step_scratch

// Device address of g_step_scratch on device dev, which must be current. The
// first call on a device looks it up; later calls only read the cached value.
vbq_status step_scratch_address(int dev, float** out) {
  std::lock_guard<std::mutex> lock(g_step_scratch_mu);
  auto it = g_step_scratch_addr.find(dev);
  if (it != g_step_scratch_addr.end()) {
    *out = it->second;
    return VBQ_OK;
  }
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_step_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(g_step_scratch)");
  // Steps need the counters at zero; they leave them so.
  e = cudaMemset(p, 0, sizeof(float) * kStepScratchFloats);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "clearing g_step_scratch");
  g_step_scratch_addr[dev] = static_cast<float*>(p);
  *out = static_cast<float*>(p);
  return VBQ_OK;
}

}  // namespace

extern "C" vbq_status vbq_decode_step_noalloc(vbq_model* m, const uint16_t* x_dev, float* logits_dev, void* stream) {
  if (!m || !x_dev || !logits_dev) return fail(VBQ_ERR_INVALID_ARG, "vbq_decode_step_noalloc: NULL argument");
  if (reinterpret_cast<uintptr_t>(logits_dev) % 4 || reinterpret_cast<uintptr_t>(x_dev) % 4)
    return fail(VBQ_ERR_INVALID_ARG,
                "vbq_decode_step_noalloc: misaligned buffer (x and logits need 4-byte alignment)");
  if (m->lay.total > kStepScratchFloats)
    return fail(VBQ_ERR_SHAPE, "vbq_decode_step_noalloc: the step needs " + std::to_string(m->lay.total) +
                                   " scratch floats (barrier block, h, q/k/v and gate/up, each rounded up to 64); the "
                                   "static scratch holds " +
                                   std::to_string(kStepScratchFloats));
  int dev = 0;
  VBQ_CUDA_TRY(cudaGetDevice(&dev));
  if (dev != m->device) return fail(VBQ_ERR_INVALID_ARG, "vbq_decode_step_noalloc: model is on another device");
  if (!m->items_static) return fail(VBQ_ERR_CUDA, "vbq_decode_step_noalloc: the static scratch was not set up");
  cudaError_t e = launch_decode(m, m->items_static, m->pre_static, m->static_base, x_dev, logits_dev,
                                static_cast<cudaStream_t>(stream), m->err);
  if (e != cudaSuccess) return cuda_fail(e, "vbq_decode_step_noalloc: launch");
  return VBQ_OK;
}
