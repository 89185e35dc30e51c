// vbq_decode_step: one batch-1 decode step through a stack of VBQ projections.
//
// VBQ abstract ("Variable Bit-width Quantization ..."): the packed recipe makes
// memory-bandwidth-bound autoregressive decode faster. The pages give no
// architecture, so the glue below is this library's reading: unit-gamma
// RMSNorm, attention at position 0 (a softmax over one key is 1, so each query
// head returns its kv group's v), SwiGLU, fp32 residual, and bf16 at every
// projection input.
//
// Each step is 1 + 4*n_layers + 1 kernels: h = x; per layer the fused
// [q;k;v] GEMV (RMSNorm in its prologue), the o GEMV (GQA gather in its
// prologue, residual add in its epilogue), the fused [gate;up] GEMV (RMSNorm
// prologue), and the down GEMV (SwiGLU prologue, residual epilogue); then the
// head GEMV. Each of these launches has its own work plan over its matrices,
// made when the model is created. The sequence is captured once into a CUDA
// graph. Its edges are programmatic: each GEMV starts streaming its weights
// while the previous one finishes, and waits (griddepcontrol.wait) only before
// touching activations.
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

__global__ void init_h_kernel(const uint16_t* __restrict__ x, float* __restrict__ h, int32_t d) {
  grid_dep_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < d; i += gridDim.x * blockDim.x)
    h[i] = __uint_as_float(static_cast<uint32_t>(x[i]) << 16);
}

}  // namespace

struct vbq_model {
  vbq_model_desc desc{};
  std::vector<const vbq_matrix*> mats;
  int device = 0;
  void* ws = nullptr;
  float* h = nullptr;
  float* qkv = nullptr;
  float* gu = nullptr;
  uint16_t* x_stage = nullptr;
  float* logits_stage = nullptr;
  bool trace = false;
  uint16_t* tr_in = nullptr;
  float* tr_out = nullptr;
  std::vector<int64_t> in_off, out_off;
  int64_t in_total = 0, out_total = 0;
  cudaStream_t cap_stream = nullptr;
  cudaGraphExec_t exec = nullptr;
  const uint16_t* g_x = nullptr;
  float* g_logits = nullptr;
  int64_t kernels_per_step = 0;
  std::vector<DevicePlan> plans;  // per layer: [q;k;v], o, [gate;up], down; then the head
  uint64_t max_partial_rows = 0;
  uint32_t max_counters = 0;
};

namespace {

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

void free_graph(vbq_model* m) {
  if (m->exec) cudaGraphExecDestroy(m->exec);
  m->exec = nullptr;
}


void add_seg(GemvArgs& a, const vbq_matrix* m, float* y, float* trace_y) {
  a.seg[a.nseg] = view_of(m, y, static_cast<int32_t>(m->N), trace_y);
  a.nseg += 1;
}

enum { L_QKV = 0, L_O, L_GU, L_DOWN, L_PER_LAYER };

// Where one step's activations live.
struct StepBuffers {
  float* h;
  float* qkv;
  float* gu;
  // Split-tile scratch shared by every launch of the step (the launches run in
  // stream order, and each touches it only after griddepcontrol.wait). When
  // null, each launch uses its plan's own storage.
  float* partial;
  uint32_t* counters;
};

GemvArgs proj_args(const vbq_model* m, int launch, const StepBuffers& b, int* err) {
  GemvArgs a{};
  a.err = err;
  a.ep = EP_STORE;
  a.plan = plan_view(m->plans[launch]);
  if (b.partial) {
    a.plan.partial = b.partial;
    a.plan.counters = b.counters;
  }
  return a;
}

// Enqueues one step; every kernel after the first may launch programmatically.
// skip_init: the caller has already enqueued h = x.
cudaError_t enqueue_step(const vbq_model* m, const uint16_t* x, float* logits, const StepBuffers& b, bool trace,
                         cudaStream_t st, int* err, bool skip_init = false) {
  const vbq_model_desc& d = m->desc;
  const int L = d.n_layers;
  const int64_t nq = proj_n(d, P_Q), nkv = proj_n(d, P_K);
  float* q_out = b.qkv;
  float* k_out = b.qkv + nq;
  float* v_out = b.qkv + nq + nkv;
  auto tin = [&](int p) -> uint16_t* { return trace ? m->tr_in + m->in_off[p] : nullptr; };
  auto tout = [&](int p) -> float* { return trace ? m->tr_out + m->out_off[p] : nullptr; };
  auto n_ctas = [&](int launch) { return m->plans[launch].n_ctas; };

  cudaError_t e = cudaSuccess;
  if (!skip_init) {
    note_launches(1);
    init_h_kernel<<<(d.d + 255) / 256, 256, 0, st>>>(x, b.h, d.d);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }

  for (int l = 0; l < L; ++l) {
    const vbq_matrix* const* W = &m->mats[static_cast<size_t>(l) * P_PER_LAYER];
    const int p0 = l * P_PER_LAYER;
    const int l0 = l * L_PER_LAYER;
    {  // [q; k; v] = W u, u = bf16(rmsnorm(h))
      GemvArgs a = proj_args(m, l0 + L_QKV, b, err);
      add_seg(a, W[P_Q], q_out, tout(p0 + P_Q));
      add_seg(a, W[P_K], k_out, tout(p0 + P_K));
      add_seg(a, W[P_V], v_out, tout(p0 + P_V));
      a.xs.mode = X_RMSNORM;
      a.xs.K = d.d;
      a.xs.h = b.h;
      a.xs.eps = d.rms_eps;
      a.xs.trace_x = tin(p0 + P_Q);
      if ((e = launch_gemv(1, a, n_ctas(l0 + L_QKV), st, true)) != cudaSuccess) return e;
    }
    {  // h += Wo a, a = bf16(v of each head's kv group)
      GemvArgs a = proj_args(m, l0 + L_O, b, err);
      add_seg(a, W[P_O], b.h, tout(p0 + P_O));
      a.xs.mode = X_GQA;
      a.xs.K = static_cast<int32_t>(nq);
      a.xs.v = v_out;
      a.xs.head_dim = d.head_dim;
      a.xs.group = d.n_heads / d.n_kv_heads;
      a.xs.trace_x = tin(p0 + P_O);
      a.ep = EP_RESID;
      a.resid = b.h;
      if ((e = launch_gemv(1, a, n_ctas(l0 + L_O), st, true)) != cudaSuccess) return e;
    }
    {  // [gate; up] = W u, u = bf16(rmsnorm(h))
      GemvArgs a = proj_args(m, l0 + L_GU, b, err);
      add_seg(a, W[P_GATE], b.gu, tout(p0 + P_GATE));
      add_seg(a, W[P_UP], b.gu + d.d_ff, tout(p0 + P_UP));
      a.xs.mode = X_RMSNORM;
      a.xs.K = d.d;
      a.xs.h = b.h;
      a.xs.eps = d.rms_eps;
      a.xs.trace_x = tin(p0 + P_GATE);
      if ((e = launch_gemv(1, a, n_ctas(l0 + L_GU), st, true)) != cudaSuccess) return e;
    }
    {  // h += Wdown bf16(silu(gate) * up)
      GemvArgs a = proj_args(m, l0 + L_DOWN, b, err);
      add_seg(a, W[P_DOWN], b.h, tout(p0 + P_DOWN));
      a.xs.mode = X_SWIGLU;
      a.xs.K = d.d_ff;
      a.xs.gate = b.gu;
      a.xs.up = b.gu + d.d_ff;
      a.xs.trace_x = tin(p0 + P_DOWN);
      a.ep = EP_RESID;
      a.resid = b.h;
      if ((e = launch_gemv(1, a, n_ctas(l0 + L_DOWN), st, true)) != cudaSuccess) return e;
    }
  }
  {  // logits = Whead bf16(rmsnorm(h))
    const int lh = L * L_PER_LAYER;
    GemvArgs a = proj_args(m, lh, b, err);
    const int ph = L * P_PER_LAYER;
    add_seg(a, m->mats[ph], logits, tout(ph));
    a.xs.mode = X_RMSNORM;
    a.xs.K = d.d;
    a.xs.h = b.h;
    a.xs.eps = d.rms_eps;
    a.xs.trace_x = tin(ph);
    if ((e = launch_gemv(1, a, n_ctas(lh), st, true)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

vbq_status build_graph(vbq_model* m, const uint16_t* x, float* logits) {
  free_graph(m);
  int* err = device_check_word();
  if (!err) return fail(VBQ_ERR_CUDA, "device check word");
  warm_gemv(1);
  const int64_t before = vbq_launch_count(0);
  VBQ_CUDA_TRY(cudaStreamBeginCapture(m->cap_stream, cudaStreamCaptureModeThreadLocal));
  const StepBuffers b{m->h, m->qkv, m->gu, nullptr, nullptr};
  cudaError_t e = enqueue_step(m, x, logits, b, m->trace, m->cap_stream, err);
  cudaGraph_t graph = nullptr;
  cudaError_t e2 = cudaStreamEndCapture(m->cap_stream, &graph);
  // Capturing enqueues nothing: the counter tracks launches that actually run.
  m->kernels_per_step = vbq_launch_count(0) - before;
  note_launches(-m->kernels_per_step);
  if (e != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    return cuda_fail(e, "decode step capture");
  }
  if (e2 != cudaSuccess) return cuda_fail(e2, "cudaStreamEndCapture");
  e = cudaGraphInstantiate(&m->exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) {
    m->exec = nullptr;
    return cuda_fail(e, "cudaGraphInstantiate");
  }
  m->g_x = x;
  m->g_logits = logits;
  return VBQ_OK;
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
  m->mats.assign(mats, mats + nm);
  const int64_t nqkv = proj_n(d, P_Q) + 2 * proj_n(d, P_K);
  auto al = [](int64_t b) { return (b + 255) & ~int64_t(255); };
  const int64_t b_h = al(4 * d.d), b_qkv = al(4 * nqkv), b_gu = al(8 * int64_t(d.d_ff));
  const int64_t b_x = al(2 * d.d), b_lg = al(4 * int64_t(d.vocab));
  cudaError_t e = cudaMalloc(&m->ws, b_h + b_qkv + b_gu + b_x + b_lg);
  if (e != cudaSuccess) {
    delete m;
    return cuda_fail(e, "vbq_model_create: workspace");
  }
  char* p = static_cast<char*>(m->ws);
  m->h = reinterpret_cast<float*>(p);
  m->qkv = reinterpret_cast<float*>(p + b_h);
  m->gu = reinterpret_cast<float*>(p + b_h + b_qkv);
  m->x_stage = reinterpret_cast<uint16_t*>(p + b_h + b_qkv + b_gu);
  m->logits_stage = reinterpret_cast<float*>(p + b_h + b_qkv + b_gu + b_x);
  e = cudaStreamCreateWithFlags(&m->cap_stream, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    cudaFree(m->ws);
    delete m;
    return cuda_fail(e, "vbq_model_create: stream");
  }
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
  // One plan per launch of the step, each over the launch's matrices.
  const int sms = gpu_info().sms;
  auto add_plan = [&](std::initializer_list<const vbq_matrix*> ms) -> cudaError_t {
    std::vector<SegTables> segs;
    uint64_t bytes = 0;
    for (const vbq_matrix* w : ms) {
      segs.push_back(seg_tables(w));
      bytes += static_cast<uint64_t>(w->data_bytes);
    }
    Plan pl = make_plan(segs, plan_ctas(bytes, sms), MAX_UNITS_PER_CTA);
    m->max_partial_rows = std::max<uint64_t>(m->max_partial_rows, pl.partial_rows);
    m->max_counters = std::max<uint32_t>(m->max_counters, pl.n_counters);
    DevicePlan dp;
    cudaError_t err = upload_plan(pl, 1, nullptr, &dp);
    if (err == cudaSuccess) m->plans.push_back(dp);
    return err;
  };
  for (int l = 0; l <= d.n_layers; ++l) {
    const vbq_matrix* const* W = &m->mats[static_cast<size_t>(l) * P_PER_LAYER];
    cudaError_t err;
    if (l == d.n_layers) {
      err = add_plan({W[0]});
    } else if ((err = add_plan({W[P_Q], W[P_K], W[P_V]})) == cudaSuccess && (err = add_plan({W[P_O]})) == cudaSuccess &&
               (err = add_plan({W[P_GATE], W[P_UP]})) == cudaSuccess) {
      err = add_plan({W[P_DOWN]});
    }
    if (err != cudaSuccess) {
      vbq_model_free(m);
      return cuda_fail(err, "vbq_model_create: plan upload");
    }
  }
  *out = m;
  return VBQ_OK;
}

extern "C" void vbq_model_free(vbq_model* m) {
  if (!m) return;
  int cur = 0;
  cudaGetDevice(&cur);
  cudaSetDevice(m->device);
  cudaDeviceSynchronize();
  free_graph(m);
  if (m->cap_stream) cudaStreamDestroy(m->cap_stream);
  cudaFree(m->ws);
  cudaFree(m->tr_in);
  cudaFree(m->tr_out);
  for (DevicePlan& p : m->plans) free_plan(&p);
  cudaSetDevice(cur);
  delete m;
}

extern "C" vbq_status vbq_decode_step(vbq_model* m, const uint16_t* x_dev, float* logits_dev, void* stream) {
  if (!m || !x_dev || !logits_dev) return fail(VBQ_ERR_INVALID_ARG, "vbq_decode_step: NULL argument");
  if (reinterpret_cast<uintptr_t>(logits_dev) % 4 || reinterpret_cast<uintptr_t>(x_dev) % 2)
    return fail(VBQ_ERR_INVALID_ARG, "vbq_decode_step: misaligned buffer");
  if (!m->exec || m->g_x != x_dev || m->g_logits != logits_dev) {
    vbq_status s = build_graph(m, x_dev, logits_dev);
    if (s != VBQ_OK) return s;
  }
  VBQ_CUDA_TRY(cudaGraphLaunch(m->exec, static_cast<cudaStream_t>(stream)));
  note_launches(m->kernels_per_step);
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
  free_graph(m);
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
// vbq_decode_step keeps its activations in a workspace that vbq_model_create
// allocates, and it builds a CUDA graph on its first call and whenever the x or
// logits pointers change; instantiating that graph allocates too. Some callers
// cannot allow any allocation at step time: code that runs while another
// component is capturing the stream into its own graph (cudaMalloc is illegal
// during capture), real-time loops whose device memory is fixed before the loop
// starts, or hosts that hand out device memory only from their own pool.
// vbq_decode_step_noalloc serves them. It launches the same kernels in the same
// order, directly on the caller's stream, and keeps the activations in the
// file-scope array below.

namespace {

// g_step_scratch holds, in 64-float blocks: a status block, the split-tile
// arrival counters, h [d], [q;k;v], [gate;up], and the split-tile partial rows.
// 262,144 floats = 1 MiB on every device that loads this library, held until
// the process exits.
constexpr int64_t kStepScratchFloats = 262144;
static __device__ __align__(256) float g_step_scratch[kStepScratchFloats];

std::mutex g_step_scratch_mu;
std::map<int, float*> g_step_scratch_addr;  // device ordinal -> device address of g_step_scratch

// Device address of g_step_scratch on the current device. The first call on a
// device looks it up (and sets the GEMV kernel attributes); later calls only
// read the cached address.
vbq_status step_scratch_address(int dev, float** out) {
  std::lock_guard<std::mutex> lock(g_step_scratch_mu);
  auto it = g_step_scratch_addr.find(dev);
  if (it != g_step_scratch_addr.end()) {
    *out = it->second;
    return VBQ_OK;
  }
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_step_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "vbq_decode_step_noalloc: cudaGetSymbolAddress(g_step_scratch)");
  warm_gemv(1);
  g_step_scratch_addr[dev] = static_cast<float*>(p);
  *out = static_cast<float*>(p);
  return VBQ_OK;
}

// h = x, after clearing the status word and the arrival counters (`nclear` words at `clear`).
__global__ void init_h_clear_kernel(const uint16_t* __restrict__ x, float* __restrict__ h, int32_t d,
                                    uint32_t* __restrict__ clear, int32_t nclear) {
  grid_dep_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nclear; i += gridDim.x * blockDim.x) clear[i] = 0u;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < d; i += gridDim.x * blockDim.x)
    h[i] = __uint_as_float(static_cast<uint32_t>(x[i]) << 16);
}

int64_t round64(int64_t n) { return (n + 63) & ~int64_t(63); }

}  // namespace

extern "C" vbq_status vbq_decode_step_noalloc(vbq_model* m, const uint16_t* x_dev, float* logits_dev, void* stream) {
  if (!m || !x_dev || !logits_dev) return fail(VBQ_ERR_INVALID_ARG, "vbq_decode_step_noalloc: NULL argument");
  if (reinterpret_cast<uintptr_t>(logits_dev) % 4 || reinterpret_cast<uintptr_t>(x_dev) % 2)
    return fail(VBQ_ERR_INVALID_ARG, "vbq_decode_step_noalloc: misaligned buffer");
  const vbq_model_desc& d = m->desc;
  const int64_t n_cnt = round64(m->max_counters);
  const int64_t n_h = round64(d.d);
  const int64_t n_qkv = round64(proj_n(d, P_Q) + 2 * proj_n(d, P_K));
  const int64_t n_gu = round64(2 * int64_t(d.d_ff));
  const int64_t n_part = round64(static_cast<int64_t>(m->max_partial_rows));
  const int64_t need = 64 + n_cnt + n_h + n_qkv + n_gu + n_part;
  if (need > kStepScratchFloats)
    return fail(VBQ_ERR_SHAPE, "vbq_decode_step_noalloc: the step needs " + std::to_string(need) +
                                   " scratch floats (status, counters, h, q/k/v, gate/up and split-tile partials, "
                                   "each rounded up to 64); the static scratch holds " +
                                   std::to_string(kStepScratchFloats));
  int dev = 0;
  VBQ_CUDA_TRY(cudaGetDevice(&dev));
  if (dev != m->device) return fail(VBQ_ERR_INVALID_ARG, "vbq_decode_step_noalloc: model is on another device");
  float* base = nullptr;
  vbq_status s = step_scratch_address(dev, &base);
  if (s != VBQ_OK) return s;
  StepBuffers b{};
  uint32_t* counters = reinterpret_cast<uint32_t*>(base + 64);
  b.counters = counters;
  b.h = base + 64 + n_cnt;
  b.qkv = b.h + n_h;
  b.gu = b.qkv + n_qkv;
  b.partial = b.gu + n_gu;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The status word and the counters must start at zero; the first kernel clears them.
  note_launches(1);
  init_h_clear_kernel<<<(d.d + 255) / 256, 256, 0, st>>>(x_dev, b.h, d.d, reinterpret_cast<uint32_t*>(base),
                                                         static_cast<int32_t>(64 + n_cnt));
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = enqueue_step(m, x_dev, logits_dev, b, false, st, reinterpret_cast<int*>(base), true);
  if (e != cudaSuccess) return cuda_fail(e, "vbq_decode_step_noalloc: launch");
  return VBQ_OK;
}
