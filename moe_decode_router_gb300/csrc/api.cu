// C ABI of the Flint MoE library: argument validation, per-device set-up, the
// CUDA-graph cache of the BF16 decode stack, and the built-in scratch of the
// no-allocation decode call.  See include/flint_moe.h.
#include <atomic>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <vector>

#include "flint_common.cuh"
#include "flint_internal.h"
#include "flint_moe.h"

namespace flint {

// Device error word: kernels OR an error bit into it when a bounded wait
// gives up.  Kernels get its address as a parameter.
__device__ unsigned int g_flint_error;

namespace {

constexpr size_t MAX_GRAPHS = 32;

// Cycle limit of the persistent decode kernel's waits on data of other thread
// blocks (flint_moe_set_wait_limit).
std::atomic<long long> g_wait_limit{WAIT_LIMIT_CYCLES};

// Decode kernels used for NVFP4 weights (flint_moe_set_decode_kernel).
std::atomic<int> g_decode_kernel{FLINT_MOE_DECODE_CHAINED};
bool use_persistent(const flint_moe_dims* d) {
  return d->weight_dtype == FLINT_MOE_W_NVFP4 && g_decode_kernel.load() == FLINT_MOE_DECODE_PERSISTENT;
}

struct GraphEntry {
  std::vector<uintptr_t> key;
  cudaGraphExec_t exec;
};

struct DeviceState {
  bool ready = false;
  int sm_count = 0;
  int gu_grid = 0;     // three-kernel path: gate/up CTAs
  int fused_grid = 0;  // persistent kernel: one CTA per SM, at most one per router expert
  unsigned* err = nullptr;
  cudaStream_t capture_stream = nullptr;
  std::vector<GraphEntry> graphs;
};

std::mutex g_mu;
std::map<int, DeviceState> g_devices;

int to_status(cudaError_t e) { return e == cudaSuccess ? FLINT_MOE_OK : FLINT_MOE_ERR_CUDA; }

// Device address of the error word on the current device (looked up once per
// device; creates nothing).  Called with g_mu held.
std::map<int, unsigned*> g_err_words;
int error_word(unsigned** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  auto it = g_err_words.find(dev);
  if (it == g_err_words.end()) {
    unsigned* p = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_flint_error) != cudaSuccess || p == nullptr)
      return FLINT_MOE_ERR_CUDA;
    it = g_err_words.emplace(dev, p).first;
  }
  *out = it->second;
  return FLINT_MOE_OK;
}

int fused_grid_for(int sm_count) { return sm_count < E ? sm_count : E; }

// Called with g_mu held.
int device_state(DeviceState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  DeviceState& s = g_devices[dev];
  if (!s.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FLINT_MOE_ERR_CUDA;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FLINT_MOE_ERR_CUDA;
    if (major != 10) return FLINT_MOE_ERR_UNSUPPORTED;  // built for sm_103a only
    s.gu_grid = s.sm_count < MAX_GU_GRID ? s.sm_count : MAX_GU_GRID;
    s.fused_grid = fused_grid_for(s.sm_count);
    int st = error_word(&s.err);
    if (st != FLINT_MOE_OK) return st;
    if (decode_kernels_init(dev) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
    if (fused_kernels_init(s.sm_count) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
    if (dense_kernels_init() != cudaSuccess) return FLINT_MOE_ERR_CUDA;
    if (medium_kernels_init() != cudaSuccess) return FLINT_MOE_ERR_CUDA;
    if (prefill_kernels_init(dev) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
    if (cudaStreamCreateWithFlags(&s.capture_stream, cudaStreamNonBlocking) != cudaSuccess)
      return FLINT_MOE_ERR_CUDA;
    s.ready = true;
  }
  *out = &s;
  return FLINT_MOE_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_dims(const flint_moe_dims* d) {
  if (d == nullptr) return FLINT_MOE_ERR_INVALID_ARG;
  if (d->hidden != H || d->n_experts != E || d->n_shared != 1 || d->inter != I || d->top_k != TOPK)
    return FLINT_MOE_ERR_UNSUPPORTED;
  if (d->weight_dtype != FLINT_MOE_W_NVFP4 && d->weight_dtype != FLINT_MOE_W_BF16) return FLINT_MOE_ERR_UNSUPPORTED;
  if (!(d->rms_eps >= 0.f) || !std::isfinite(d->rms_eps)) return FLINT_MOE_ERR_INVALID_ARG;
  return FLINT_MOE_OK;
}

int check_layer(const flint_moe_dims* d, const flint_moe_layer* L) {
  if (L == nullptr || L->router_w == nullptr || L->experts == nullptr) return FLINT_MOE_ERR_INVALID_ARG;
  if (!aligned(L->router_w, 16) || !aligned(L->experts, 16)) return FLINT_MOE_ERR_INVALID_ARG;
  if (d->weight_dtype == FLINT_MOE_W_NVFP4 && (L->tensor_scales == nullptr || !aligned(L->tensor_scales, 16)))
    return FLINT_MOE_ERR_INVALID_ARG;
  if (L->norm_w != nullptr && !aligned(L->norm_w, 16)) return FLINT_MOE_ERR_INVALID_ARG;
  return FLINT_MOE_OK;
}

bool opt_aligned(const void* p) { return p == nullptr || aligned(p, 16); }

// A byte range [p, p + n) of one argument; null or empty ranges are skipped.
struct Range {
  const void* p;
  size_t n;
};

// True if the byte ranges [a, a + na) and [b, b + nb) share a byte.
bool overlap(const Range& a, const Range& b) {
  if (a.p == nullptr || b.p == nullptr || a.n == 0 || b.n == 0) return false;
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a.p), pb = reinterpret_cast<uintptr_t>(b.p);
  return pa < pb + b.n && pb < pa + a.n;
}

// True if a buffer the call writes shares a byte with another buffer of the
// call (written or read).  Buffers that are only read may share bytes.
bool outputs_overlap(const std::vector<Range>& outs, const std::vector<Range>& ins) {
  for (size_t i = 0; i < outs.size(); ++i) {
    for (size_t j = i + 1; j < outs.size(); ++j)
      if (overlap(outs[i], outs[j])) return true;
    for (const Range& r : ins)
      if (overlap(outs[i], r)) return true;
  }
  return false;
}

// The read-only buffers of one sublayer.
void add_layer_ranges(const flint_moe_dims* d, const flint_moe_layer& L, std::vector<Range>& ins) {
  const bool f4 = d->weight_dtype == FLINT_MOE_W_NVFP4;
  ins.push_back({L.router_w, (size_t)E * H * 2});
  ins.push_back({L.experts, (size_t)NE * (f4 ? F4_EXPERT : B16_EXPERT)});
  if (f4) ins.push_back({L.tensor_scales, (size_t)NE * 2 * 4});
  ins.push_back({L.norm_w, (size_t)H * 2});
}

LayerArgs layer_args(const flint_moe_layer& L) {
  LayerArgs a;
  a.router_w = L.router_w;
  a.experts = static_cast<const uint8_t*>(L.experts);
  a.tscale = L.tensor_scales;
  a.norm_w = L.norm_w;
  return a;
}

size_t decode_ws_needed() { return decode_path_ws_bytes(); }

// Largest token count of one prefill call (keeps every pair index and
// work-item count far inside int32).
constexpr int PREFILL_MAX_TOKENS = 1 << 20;

// Scratch of flint_moe_decode_layer_noalloc: one fixed array in the device
// image (held by every GPU that loads the library, for the whole process).
// In host code its name is only a stand-in; kernels get the device address
// looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FLINT_MOE_NOALLOC_SCRATCH_BYTES];
static_assert(MT_MAX == FLINT_MOE_MAX_MEDIUM_BATCH && BMAX == FLINT_MOE_MAX_DECODE_BATCH, "batch caps");
static_assert(decode_path_ws_bytes() <= FLINT_MOE_NOALLOC_SCRATCH_BYTES,
              "the built-in scratch must hold the decode workspace of 8 tokens");

struct NoallocState {
  bool ready = false;
  int gu_grid = 0;
  int fused_grid = 0;
  unsigned* err = nullptr;
  void* scratch = nullptr;
};
std::map<int, NoallocState> g_noalloc;

// Once per device, with that device current; creates nothing and allocates
// nothing.  Its first call on a device must not happen during a stream
// capture (symbol look-ups are not capturable): that returns
// FLINT_MOE_ERR_INVALID_ARG.  Called with g_mu held.
int noalloc_state(cudaStream_t stream, NoallocState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  NoallocState& s = g_noalloc[dev];
  if (!s.ready) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
    if (cap != cudaStreamCaptureStatusNone) return FLINT_MOE_ERR_INVALID_ARG;
    int sms = 0, major = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
      return FLINT_MOE_ERR_CUDA;
    if (major != 10) return FLINT_MOE_ERR_UNSUPPORTED;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return FLINT_MOE_ERR_CUDA;
    int st = error_word(&s.err);
    if (st != FLINT_MOE_OK) return st;
    if (decode_kernels_init(dev) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
    if (fused_kernels_init(sms) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
    s.scratch = ptr;
    s.gu_grid = sms < MAX_GU_GRID ? sms : MAX_GU_GRID;
    s.fused_grid = fused_grid_for(sms);
    s.ready = true;
  }
  *out = &s;
  return FLINT_MOE_OK;
}

// One decode sublayer (chained or persistent kernels) over a workspace of
// decode_ws_needed() bytes.
int launch_one_layer(const flint_moe_dims* dims, const flint_moe_layer& layer, const void* x, int B, void* y,
                     int32_t* ids, float* w, void* ws, int gu_grid, int fused_grid, unsigned* err,
                     cudaStream_t stream) {
  const LayerArgs la = layer_args(layer);
  if (use_persistent(dims)) {
    if (fused_grid < DN_TILES) return FLINT_MOE_ERR_UNSUPPORTED;
    return to_status(launch_fused_stack(&la, 1, x, B, dims->rms_eps, y, nullptr, ids, w, carve_fused_ws(ws),
                                        fused_grid, err, g_wait_limit.load(), stream));
  }
  return to_status(launch_decode_chain(dims->weight_dtype == FLINT_MOE_W_NVFP4 ? 0 : 1, la, x, nullptr, B,
                                       dims->rms_eps, y, nullptr, nullptr, ids, w, carve_decode_ws(ws, MAX_GU_GRID),
                                       gu_grid, err, stream, true));
}

}  // namespace
}  // namespace flint

using namespace flint;

extern "C" {

size_t flint_moe_packed_bytes(const flint_moe_dims* dims) {
  if (check_dims(dims) != FLINT_MOE_OK) return 0;
  return (size_t)NE * (dims->weight_dtype == FLINT_MOE_W_NVFP4 ? F4_EXPERT : B16_EXPERT);
}

size_t flint_moe_workspace_bytes(const flint_moe_dims* dims, int max_tokens) {
  if (check_dims(dims) != FLINT_MOE_OK || max_tokens < 1) return 0;
  if (max_tokens > PREFILL_MAX_TOKENS) return 0;
  const size_t dec = decode_ws_needed();
  if (dims->weight_dtype != FLINT_MOE_W_NVFP4) return max_tokens <= BMAX ? dec : 0;  // medium, prefill: NVFP4 only
  size_t n = prefill_ws_bytes(max_tokens);
  if (n < dec) n = dec;
  // Any decode call of 9..64 tokens is a call of at most max_tokens tokens.
  if (max_tokens > BMAX && n < medium_ws_bytes()) n = medium_ws_bytes();
  return n;
}

int flint_moe_pack_weights(const flint_moe_dims* dims, const void* gate_up, const uint8_t* gate_up_scales,
                           const void* down, const uint8_t* down_scales, void* packed, size_t packed_bytes,
                           flint_moe_stream_t stream) {
  int st = check_dims(dims);
  if (st != FLINT_MOE_OK) return st;
  const bool f4 = dims->weight_dtype == FLINT_MOE_W_NVFP4;
  if (gate_up == nullptr || down == nullptr || packed == nullptr) return FLINT_MOE_ERR_INVALID_ARG;
  if (f4 && (gate_up_scales == nullptr || down_scales == nullptr)) return FLINT_MOE_ERR_INVALID_ARG;
  if (!f4 && (gate_up_scales != nullptr || down_scales != nullptr)) return FLINT_MOE_ERR_INVALID_ARG;
  if (!aligned(gate_up, 16) || !aligned(down, 16) || !aligned(packed, 16) || !opt_aligned(gate_up_scales) ||
      !opt_aligned(down_scales))
    return FLINT_MOE_ERR_INVALID_ARG;
  if (packed_bytes < flint_moe_packed_bytes(dims)) return FLINT_MOE_ERR_WORKSPACE;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != FLINT_MOE_OK) return st;
  return to_status(launch_pack(f4 ? 0 : 1, gate_up, gate_up_scales, down, down_scales, packed,
                               reinterpret_cast<cudaStream_t>(stream)));
}

int flint_moe_decode_layer(const flint_moe_dims* dims, const flint_moe_layer* layer, const void* x, int B, void* y,
                           int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes, flint_moe_stream_t stream) {
  int st = check_dims(dims);
  if (st != FLINT_MOE_OK) return st;
  if ((st = check_layer(dims, layer)) != FLINT_MOE_OK) return st;
  if (B < 1) return FLINT_MOE_ERR_INVALID_ARG;
  const bool medium = B > BMAX;
  if (B > MT_MAX || (medium && dims->weight_dtype != FLINT_MOE_W_NVFP4)) return FLINT_MOE_ERR_UNSUPPORTED;
  if (x == nullptr || y == nullptr || ws == nullptr || x == y) return FLINT_MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(ws, 256) || !opt_aligned(topk_ids) || !opt_aligned(topk_w))
    return FLINT_MOE_ERR_INVALID_ARG;
  const size_t ws_need = medium ? medium_ws_bytes() : decode_ws_needed();
  if (ws_bytes < ws_need) return FLINT_MOE_ERR_WORKSPACE;
  const size_t act = (size_t)B * H * 2, sel = (size_t)B * TOPK * 4;
  std::vector<Range> ins{{x, act}};
  add_layer_ranges(dims, *layer, ins);
  if (outputs_overlap({{y, act}, {ws, ws_need}, {topk_ids, sel}, {topk_w, sel}}, ins))
    return FLINT_MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != FLINT_MOE_OK) return st;
  if (medium)
    return to_status(launch_medium_chain(layer_args(*layer), x, nullptr, B, dims->rms_eps, y, topk_ids, topk_w,
                                         carve_medium_ws(ws), ds->gu_grid, ds->err,
                                         reinterpret_cast<cudaStream_t>(stream), true));
  return launch_one_layer(dims, *layer, x, B, y, topk_ids, topk_w, ws, ds->gu_grid, ds->fused_grid, ds->err,
                          reinterpret_cast<cudaStream_t>(stream));
}

int flint_moe_decode_stack(const flint_moe_dims* dims, const flint_moe_layer* layers, int n_layers, const void* x,
                           int B, void* y, int32_t* ids_per_layer, float* w_per_layer, void* ys_per_layer, void* ws,
                           size_t ws_bytes, flint_moe_stream_t stream) {
  int st = check_dims(dims);
  if (st != FLINT_MOE_OK) return st;
  if (layers == nullptr || n_layers < 1 || n_layers > 4096) return FLINT_MOE_ERR_INVALID_ARG;
  for (int i = 0; i < n_layers; ++i)
    if ((st = check_layer(dims, &layers[i])) != FLINT_MOE_OK) return st;
  if (B < 1) return FLINT_MOE_ERR_INVALID_ARG;
  const bool medium = B > BMAX;
  if (B > MT_MAX || (medium && dims->weight_dtype != FLINT_MOE_W_NVFP4)) return FLINT_MOE_ERR_UNSUPPORTED;
  if (x == nullptr || y == nullptr || ws == nullptr || x == y) return FLINT_MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(ws, 256) || !opt_aligned(ids_per_layer) ||
      !opt_aligned(w_per_layer) || !opt_aligned(ys_per_layer))
    return FLINT_MOE_ERR_INVALID_ARG;
  const size_t ws_need = medium ? medium_ws_bytes() : decode_ws_needed();
  if (ws_bytes < ws_need) return FLINT_MOE_ERR_WORKSPACE;
  {
    const size_t act = (size_t)B * H * 2, sel = (size_t)n_layers * B * TOPK * 4;
    std::vector<Range> ins{{x, act}};
    for (int i = 0; i < n_layers; ++i) add_layer_ranges(dims, layers[i], ins);
    if (outputs_overlap({{y, act}, {ws, ws_need}, {ids_per_layer, sel}, {w_per_layer, sel},
                         {ys_per_layer, (size_t)n_layers * act}},
                        ins))
      return FLINT_MOE_ERR_INVALID_ARG;
  }

  if (!medium && use_persistent(dims)) {
    // One cooperative launch per 64 sublayers; nothing to capture or cache.
    std::vector<LayerArgs> la;
    la.reserve((size_t)n_layers);
    for (int i = 0; i < n_layers; ++i) la.push_back(layer_args(layers[i]));
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState* ds = nullptr;
    if ((st = device_state(&ds)) != FLINT_MOE_OK) return st;
    if (ds->fused_grid < DN_TILES) return FLINT_MOE_ERR_UNSUPPORTED;
    return to_status(launch_fused_stack(la.data(), n_layers, x, B, dims->rms_eps, y, ys_per_layer, ids_per_layer,
                                        w_per_layer, carve_fused_ws(ws), ds->fused_grid, ds->err,
                                        g_wait_limit.load(), reinterpret_cast<cudaStream_t>(stream)));
  }

  std::vector<uintptr_t> key;
  key.reserve(16 + 4 * (size_t)n_layers);
  key.push_back((uintptr_t)dims->weight_dtype);
  uint32_t eps_bits;
  std::memcpy(&eps_bits, &dims->rms_eps, 4);
  key.push_back(eps_bits);
  key.push_back((uintptr_t)n_layers);
  key.push_back((uintptr_t)B);
  key.push_back((uintptr_t)x);
  key.push_back((uintptr_t)y);
  key.push_back((uintptr_t)ids_per_layer);
  key.push_back((uintptr_t)w_per_layer);
  key.push_back((uintptr_t)ys_per_layer);
  key.push_back((uintptr_t)ws);
  for (int i = 0; i < n_layers; ++i) {
    key.push_back((uintptr_t)layers[i].router_w);
    key.push_back((uintptr_t)layers[i].experts);
    key.push_back((uintptr_t)layers[i].tensor_scales);
    key.push_back((uintptr_t)layers[i].norm_w);
  }

  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != FLINT_MOE_OK) return st;
  cudaStream_t user = reinterpret_cast<cudaStream_t>(stream);
  for (auto& ge : ds->graphs)
    if (ge.key == key) return to_status(cudaGraphLaunch(ge.exec, user));

  const DecodeWs w = carve_decode_ws(ws, MAX_GU_GRID);
  const MediumWs mw = carve_medium_ws(ws);
  cudaStream_t cs = ds->capture_stream;
  cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  cudaError_t le = cudaSuccess;
  for (int i = 0; i < n_layers && le == cudaSuccess && medium; ++i) {
    // The first sublayer normalises x itself; every other one finds its
    // x_hat in the workspace, left there by the previous sublayer's combine
    // from its output.
    const bool last = i == n_layers - 1;
    void* ys = ys_per_layer ? static_cast<uint8_t*>(ys_per_layer) + (size_t)i * B * H * 2 : nullptr;
    int32_t* ids = ids_per_layer ? ids_per_layer + (size_t)i * B * TOPK : nullptr;
    float* wl = w_per_layer ? w_per_layer + (size_t)i * B * TOPK : nullptr;
    void* yout = last ? y : (ys ? ys : mw.y_mid);
    LayerArgs nxt{};
    if (!last) nxt = layer_args(layers[i + 1]);
    le = launch_medium_chain(layer_args(layers[i]), i == 0 ? x : nullptr, last ? nullptr : &nxt, B, dims->rms_eps,
                             yout, ids, wl, mw, ds->gu_grid, ds->err, cs, true);
    if (le == cudaSuccess && last && ys) le = cudaMemcpyAsync(ys, y, (size_t)B * H * 2, cudaMemcpyDeviceToDevice, cs);
  }
  for (int i = 0; i < n_layers && le == cudaSuccess && !medium; ++i) {
    const bool last = i == n_layers - 1;
    const void* xin = i == 0 ? x : w.y_mid;
    void* yout = last ? y : w.y_mid;
    // The previous sublayer's down kernel leaves the sum of squares of its
    // output for this sublayer's RMSNorm.
    const void* ss_in = (i > 0 && layers[i].norm_w != nullptr) ? w.ss_part : nullptr;
    void* ss_out = (!last && layers[i + 1].norm_w != nullptr) ? w.ss_part : nullptr;
    void* ys = ys_per_layer ? static_cast<uint8_t*>(ys_per_layer) + (size_t)i * B * H * 2 : nullptr;
    int32_t* ids = ids_per_layer ? ids_per_layer + (size_t)i * B * TOPK : nullptr;
    float* wl = w_per_layer ? w_per_layer + (size_t)i * B * TOPK : nullptr;
    le = launch_decode_chain(dims->weight_dtype == FLINT_MOE_W_NVFP4 ? 0 : 1, layer_args(layers[i]), xin, ss_in, B,
                             dims->rms_eps, yout, ys, ss_out, ids, wl, w, ds->gu_grid, ds->err, cs, true);
  }
  cudaGraph_t graph = nullptr;
  e = cudaStreamEndCapture(cs, &graph);
  if (le != cudaSuccess || e != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();
    return FLINT_MOE_ERR_CUDA;
  }
  cudaGraphExec_t exec = nullptr;
  e = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  if (ds->graphs.size() >= MAX_GRAPHS) {
    cudaGraphExecDestroy(ds->graphs.front().exec);
    ds->graphs.erase(ds->graphs.begin());
  }
  ds->graphs.push_back(GraphEntry{std::move(key), exec});
  return to_status(cudaGraphLaunch(exec, user));
}

int flint_moe_decode_layer_noalloc(const flint_moe_dims* dims, const flint_moe_layer* layer, const void* x, int B,
                                   void* y, int32_t* topk_ids, float* topk_w, flint_moe_stream_t stream) {
  int st = check_dims(dims);
  if (st != FLINT_MOE_OK) return st;
  if ((st = check_layer(dims, layer)) != FLINT_MOE_OK) return st;
  if (B < 1) return FLINT_MOE_ERR_INVALID_ARG;
  if (B > FLINT_MOE_NOALLOC_MAX_TOKENS) return FLINT_MOE_ERR_WORKSPACE;  // beyond the built-in scratch
  if (x == nullptr || y == nullptr || x == y) return FLINT_MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16) || !opt_aligned(topk_ids) || !opt_aligned(topk_w))
    return FLINT_MOE_ERR_INVALID_ARG;
  const size_t act = (size_t)B * H * 2, sel = (size_t)B * TOPK * 4;
  std::vector<Range> ins{{x, act}};
  add_layer_ranges(dims, *layer, ins);
  if (outputs_overlap({{y, act}, {topk_ids, sel}, {topk_w, sel}}, ins)) return FLINT_MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  NoallocState* ns = nullptr;
  if ((st = noalloc_state(s, &ns)) != FLINT_MOE_OK) return st;
  return launch_one_layer(dims, *layer, x, B, y, topk_ids, topk_w, ns->scratch, ns->gu_grid, ns->fused_grid, ns->err,
                          s);
}

int flint_moe_prefill_layer(const flint_moe_dims* dims, const flint_moe_layer* layer, const void* x, int T, void* y,
                            int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes, flint_moe_stream_t stream) {
  int st = check_dims(dims);
  if (st != FLINT_MOE_OK) return st;
  if (dims->weight_dtype != FLINT_MOE_W_NVFP4) return FLINT_MOE_ERR_UNSUPPORTED;
  if ((st = check_layer(dims, layer)) != FLINT_MOE_OK) return st;
  if (T < 1) return FLINT_MOE_ERR_INVALID_ARG;
  if (T > PREFILL_MAX_TOKENS) return FLINT_MOE_ERR_UNSUPPORTED;
  if (x == nullptr || y == nullptr || ws == nullptr || x == y) return FLINT_MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(ws, 256) || !opt_aligned(topk_ids) || !opt_aligned(topk_w))
    return FLINT_MOE_ERR_INVALID_ARG;
  if (ws_bytes < prefill_ws_bytes(T)) return FLINT_MOE_ERR_WORKSPACE;
  {
    const size_t act = (size_t)T * H * 2, sel = (size_t)T * TOPK * 4;
    std::vector<Range> ins{{x, act}};
    add_layer_ranges(dims, *layer, ins);
    if (outputs_overlap({{y, act}, {ws, prefill_ws_bytes(T)}, {topk_ids, sel}, {topk_w, sel}}, ins))
      return FLINT_MOE_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != FLINT_MOE_OK) return st;
  return to_status(launch_prefill(layer_args(*layer), x, T, dims->rms_eps, y, topk_ids, topk_w, ws, ds->sm_count,
                                  ds->err, reinterpret_cast<cudaStream_t>(stream)));
}

// Shapes of the dense GEMV: 16 | N, 256 | K, K <= DENSE_MAX_BK, N < 2^24.
bool dense_shape_ok(int N, int K) {
  return N >= 16 && N % 16 == 0 && N < (1 << 24) && K >= 256 && K % 256 == 0 && K <= DENSE_MAX_BK;
}

size_t flint_moe_dense_packed_bytes(int N, int K) { return dense_shape_ok(N, K) ? dense_packed_bytes(N, K) : 0; }

int flint_moe_pack_dense(const uint8_t* codes, const uint8_t* scales, int N, int K, void* packed, size_t packed_bytes,
                         flint_moe_stream_t stream) {
  if (!dense_shape_ok(N, K)) return FLINT_MOE_ERR_UNSUPPORTED;
  if (codes == nullptr || scales == nullptr || packed == nullptr) return FLINT_MOE_ERR_INVALID_ARG;
  if (!aligned(codes, 16) || !aligned(scales, 16) || !aligned(packed, 16)) return FLINT_MOE_ERR_INVALID_ARG;
  if (packed_bytes < dense_packed_bytes(N, K)) return FLINT_MOE_ERR_WORKSPACE;
  if (outputs_overlap({{packed, dense_packed_bytes(N, K)}},
                      {{codes, (size_t)N * K / 2}, {scales, (size_t)N * K / 16}}))
    return FLINT_MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* ds = nullptr;
  int st = device_state(&ds);
  if (st != FLINT_MOE_OK) return st;
  return to_status(launch_pack_dense(codes, scales, N, K, packed, reinterpret_cast<cudaStream_t>(stream)));
}

int flint_moe_dense_gemv(const void* packed, int N, int K, float tensor_scale, const void* x, int B, void* y,
                         flint_moe_stream_t stream) {
  if (!dense_shape_ok(N, K)) return FLINT_MOE_ERR_UNSUPPORTED;
  if (B < 1) return FLINT_MOE_ERR_INVALID_ARG;
  if (B > BMAX || (long long)B * K > DENSE_MAX_BK) return FLINT_MOE_ERR_UNSUPPORTED;
  if (packed == nullptr || x == nullptr || y == nullptr) return FLINT_MOE_ERR_INVALID_ARG;
  if (!aligned(packed, 16) || !aligned(x, 16) || !aligned(y, 16)) return FLINT_MOE_ERR_INVALID_ARG;
  if (!std::isfinite(tensor_scale)) return FLINT_MOE_ERR_INVALID_ARG;
  if (outputs_overlap({{y, (size_t)B * N * 2}}, {{x, (size_t)B * K * 2}, {packed, dense_packed_bytes(N, K)}}))
    return FLINT_MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState* ds = nullptr;
  int st = device_state(&ds);
  if (st != FLINT_MOE_OK) return st;
  return to_status(launch_dense_gemv(packed, N, K, tensor_scale, x, B, y, ds->sm_count, ds->err,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

int flint_moe_release(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  int cur = -1;
  cudaGetDevice(&cur);
  int rc = FLINT_MOE_OK;
  for (auto& kv : g_devices) {
    if (cudaSetDevice(kv.first) != cudaSuccess) {
      rc = FLINT_MOE_ERR_CUDA;
      continue;
    }
    for (auto& ge : kv.second.graphs)
      if (cudaGraphExecDestroy(ge.exec) != cudaSuccess) rc = FLINT_MOE_ERR_CUDA;
    kv.second.graphs.clear();
  }
  if (cur >= 0) cudaSetDevice(cur);
  return rc;
}

int flint_moe_device_error(int reset) {
  std::lock_guard<std::mutex> lk(g_mu);
  unsigned* err = nullptr;
  int st = error_word(&err);
  if (st != FLINT_MOE_OK) return st;
  unsigned v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  if (cudaMemcpy(&v, err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  if (reset && cudaMemset(err, 0, sizeof(unsigned)) != cudaSuccess) return FLINT_MOE_ERR_CUDA;
  return (int)(v & 0x7FFFFFFFu);
}

int flint_moe_device_status(int reset) {
  const int v = flint_moe_device_error(reset);
  if (v < 0) return v;
  if (v & (int)(ERR_WAIT_FULL | ERR_WAIT_EMPTY | ERR_DRAIN | ERR_POLL)) return FLINT_MOE_ERR_TIMEOUT;
  if (v & (int)ERR_LAYOUT) return FLINT_MOE_ERR_CUDA;
  return FLINT_MOE_OK;  // ERR_ROUTER_BOUND alone: the routing was recomputed exactly
}

int flint_moe_set_decode_kernel(int kernel) {
  if (kernel != FLINT_MOE_DECODE_CHAINED && kernel != FLINT_MOE_DECODE_PERSISTENT) return FLINT_MOE_ERR_INVALID_ARG;
  g_decode_kernel.store(kernel);
  return FLINT_MOE_OK;
}

int flint_moe_set_wait_limit(long long cycles) {
  g_wait_limit.store(cycles > 0 ? cycles : WAIT_LIMIT_CYCLES);
  return FLINT_MOE_OK;
}

const char* flint_moe_status_string(int status) {
  switch (status) {
    case FLINT_MOE_OK: return "ok";
    case FLINT_MOE_ERR_INVALID_ARG: return "invalid argument";
    case FLINT_MOE_ERR_UNSUPPORTED: return "unsupported shape, batch or format";
    case FLINT_MOE_ERR_WORKSPACE: return "workspace or output buffer too small";
    case FLINT_MOE_ERR_CUDA: return "CUDA runtime error";
    case FLINT_MOE_ERR_TIMEOUT: return "a bounded device wait gave up";
    default: return "unknown status";
  }
}

}  // extern "C"
