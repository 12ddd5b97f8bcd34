// Host-buffer entry points (declared in include/strata_moe.h): one call copies the activations from
// host memory into the workspace's I/O area, runs the layer (or the stack) exactly as the device-buffer
// call does, copies the result back to host memory and synchronises the stream.
//
// With page-locked host buffers and a non-default stream the three steps are captured once as a CUDA
// graph and replayed by later calls with the same arguments, so a call costs one graph launch and one
// synchronisation on the host instead of a copy, a launch per kernel and a copy.  Page-locked
// activations move through the host buffers' device mappings (a copy kernel in, the layer's own stores
// out): a copy-engine transfer of a few KB costs several microseconds of latency on the call's path,
// and at tens of MB the SMs move the bytes faster than the copy engines.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"

using namespace strata;

namespace {

#define STRATA_TRY_HOST(expr)              \
  do {                                     \
    const strata_status _st = (expr);      \
    if (_st != STRATA_OK) return _st;      \
  } while (0)

// A host-buffer call synchronises its stream, so it cannot be part of a capture.
strata_status not_capturing(cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return STRATA_E_CUDA;
  return cs == cudaStreamCaptureStatusNone ? STRATA_OK : STRATA_E_INVAL;
}

// The device address of page-locked host memory at p, or nullptr when p is pageable (or unmapped).
inline void* mapped(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // an unregistered pointer may leave an error behind on older drivers
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// The device address of the page-locked host buffer [p, p + bytes), or nullptr: its first and last
// bytes must both be page-locked and mapped the same distance apart (the buffer lies in one allocation
// or registration, as the header requires); anything else takes the copy engines.
inline void* mapped_range(const void* p, size_t bytes) {
  void* m0 = mapped(p);
  if (!m0 || bytes == 0) return m0;
  void* m1 = mapped((const char*)p + bytes - 1);
  return m1 == (char*)m0 + (bytes - 1) ? m0 : nullptr;
}

// dst[i] = src[i], 16-byte words; one side is page-locked host memory reached through its device
// mapping, the other the workspace's I/O area.
__global__ void __launch_bounds__(256) host_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                        size_t n) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

// A host buffer's mapping the kernels can use directly: present and 16-byte aligned.
inline bool usable_map(const void* map) { return map && ((uintptr_t)map & 15) == 0; }

// Copy `bytes` (a multiple of 16) from src to dst on s: host_copy_kernel when the mapped side `map`
// (the device address of the host buffer) is usable -- on this system SM loads and stores through
// the mapping beat the copy engines both for a few KB (latency) and for tens of MB (measured at 21 MB
// each way) -- else a copy-engine transfer of the host pointer `host`.
strata_status copy_host(void* dst, const void* src, size_t bytes, const void* map, bool to_device, const void* host,
                        cudaStream_t s) {
  if (usable_map(map)) {
    const size_t n = bytes / 16;
    const int blocks = (int)std::min<size_t>((n + 255) / 256, 8 * 152);
    STRATA_LAUNCH(KID_HOST_COPY, s,
                  host_copy_kernel<<<blocks, 256, 0, s>>>((const uint4*)src, (uint4*)dst, n));
    return cudaGetLastError() == cudaSuccess ? STRATA_OK : STRATA_E_CUDA;
  }
  const cudaError_t e = to_device ? cudaMemcpyAsync(dst, host, bytes, cudaMemcpyHostToDevice, s)
                                  : cudaMemcpyAsync((void*)host, src, bytes, cudaMemcpyDeviceToHost, s);
  return e == cudaSuccess ? STRATA_OK : STRATA_E_CUDA;
}

// Everything a captured graph depends on: the pointers it copies from and to, the sizes, the
// experts' descriptors (by value), the stream and the device.
struct HostKey {
  int kind = 0;  // 0: layer, 1: stack
  int device = 0;
  int32_t T = 0, flags = 0, n_layers = 0;
  const void* w_router = nullptr;
  const void* bias = nullptr;
  const void* x_host = nullptr;
  const void* out_host = nullptr;
  const void* x_map = nullptr;    // their device mappings (a re-registered buffer may map elsewhere)
  const void* out_map = nullptr;
  const void* ids = nullptr;
  const void* weights = nullptr;
  const void* ws = nullptr;
  size_t ws_bytes = 0;
  const void* stream = nullptr;
  std::vector<strata_experts_t> ex;

  bool operator==(const HostKey& o) const {
    if (kind != o.kind || device != o.device || T != o.T || flags != o.flags || n_layers != o.n_layers ||
        w_router != o.w_router || bias != o.bias || x_host != o.x_host || out_host != o.out_host ||
        x_map != o.x_map || out_map != o.out_map || ids != o.ids ||
        weights != o.weights || ws != o.ws || ws_bytes != o.ws_bytes || stream != o.stream || ex.size() != o.ex.size())
      return false;
    for (size_t i = 0; i < ex.size(); ++i)
      if (ex[i].blobs != o.ex[i].blobs || ex[i].blob_stride != o.ex[i].blob_stride ||
          ex[i].n_expert != o.ex[i].n_expert || ex[i].q2_offset != o.ex[i].q2_offset ||
          ex[i].shared_blob != o.ex[i].shared_blob)
        return false;
    return true;
  }
};

struct HostGraph {
  HostKey key;
  cudaGraphExec_t exec = nullptr;
  unsigned long long launches = 0;  // the library's kernels in the graph
  unsigned long long last_use = 0;
};

constexpr size_t kMaxGraphs = 16;
std::mutex g_mu;
std::vector<HostGraph> g_graphs;
unsigned long long g_clock = 0;

// The graph for `key`, captured by `enqueue` on first use; nullptr (and *st set) if capture failed.
template <typename Enqueue>
cudaGraphExec_t graph_for(const HostKey& key, cudaStream_t s, Enqueue enqueue, strata_status* st,
                          unsigned long long* launches) {
  for (HostGraph& g : g_graphs)
    if (g.key == key) {
      g.last_use = ++g_clock;
      *launches = g.launches;
      return g.exec;
    }
  const unsigned long long before = launches_this_thread();
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    *st = STRATA_E_CUDA;
    return nullptr;
  }
  const strata_status est = enqueue();
  cudaGraph_t graph = nullptr;
  const cudaError_t ce = cudaStreamEndCapture(s, &graph);
  if (est != STRATA_OK || ce != cudaSuccess || !graph) {
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();
    *st = est != STRATA_OK ? est : STRATA_E_CUDA;
    return nullptr;
  }
  cudaGraphExec_t exec = nullptr;
  const cudaError_t ie = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (ie != cudaSuccess) {
    *st = STRATA_E_CUDA;
    return nullptr;
  }
  if (g_graphs.size() >= kMaxGraphs) {  // drop the least recently used
    size_t lru = 0;
    for (size_t i = 1; i < g_graphs.size(); ++i)
      if (g_graphs[i].last_use < g_graphs[lru].last_use) lru = i;
    cudaGraphExecDestroy(g_graphs[lru].exec);
    g_graphs.erase(g_graphs.begin() + (long)lru);
  }
  // capture counted the launches it recorded; replays count them again, so take them back out here
  *launches = launches_this_thread() - before;
  count_launches(0ull - *launches);
  g_graphs.push_back(HostGraph{key, exec, *launches, ++g_clock});
  return exec;
}

// Runs `enqueue` (copy in, compute, copy out on s) from a cached graph when it can, else directly,
// then synchronises s.
template <typename Enqueue>
strata_status run_host_call(const HostKey& key, cudaStream_t s, bool page_locked, Enqueue enqueue) {
  const bool graphable = s != nullptr && s != cudaStreamLegacy && page_locked && !profiling_armed();
  if (graphable) {
    std::lock_guard<std::mutex> lock(g_mu);
    strata_status st = STRATA_OK;
    unsigned long long n = 0;
    cudaGraphExec_t exec = graph_for(key, s, enqueue, &st, &n);
    if (!exec) return st;
    if (cudaGraphLaunch(exec, s) != cudaSuccess) return STRATA_E_CUDA;
    count_launches(n);
  } else {
    const strata_status st = enqueue();
    if (st != STRATA_OK) return st;
  }
  return cudaStreamSynchronize(s) == cudaSuccess ? STRATA_OK : STRATA_E_CUDA;
}

}  // namespace

extern "C" {

strata_status strata_moe_layer_host(const strata_experts_t* ex, const uint16_t* w_router, const float* bias,
                                    const float* x_host, int32_t T, int32_t flags, float* out_host, int32_t* ids,
                                    float* weights, void* ws, size_t ws_bytes, void* stream) {
  if (!x_host || !out_host) return STRATA_E_INVAL;
  const strata_status chk = check_layer_args(ex, 1, w_router, bias, flags, T, ws, ws_bytes);
  if (chk != STRATA_OK) return chk;
  if (T == 0) return STRATA_OK;
  const size_t bytes = sizeof(float) * (size_t)T * H;
  const char* xa = (const char*)x_host;
  const char* oa = (const char*)out_host;
  if (xa < oa + bytes && oa < xa + bytes) return STRATA_E_INVAL;  // the host buffers overlap
  const WsLayout L = ws_layout(T);
  float* dx = (float*)((char*)ws + L.io);
  float* dout = dx + (size_t)T * H;
  cudaStream_t s = (cudaStream_t)stream;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return STRATA_E_CUDA;
  STRATA_TRY_HOST(not_capturing(s));
  const void* xm = mapped_range(x_host, bytes);
  const void* om = mapped_range(out_host, bytes);
  HostKey key;
  key.kind = 0;
  key.device = dev;
  key.T = T;
  key.flags = flags;
  key.w_router = w_router;
  key.bias = bias;
  key.x_host = x_host;
  key.out_host = out_host;
  key.x_map = xm;
  key.out_map = om;
  key.ids = ids;
  key.weights = weights;
  key.ws = ws;
  key.ws_bytes = ws_bytes;
  key.stream = stream;
  key.ex.assign(ex, ex + 1);
  // a decode layer (T <= 8) stores each output element once, so it writes straight into out_host's
  // mapping, which saves the copy-out step; a prefill layer first sets its output and then adds every
  // expert's weighted contribution into it (fp32 reductions): those stay in device memory and the
  // result is copied out once
  const bool direct_out = T <= DECODE_T_MAX && usable_map(om);
  auto enqueue = [&]() -> strata_status {
    STRATA_TRY_HOST(copy_host(dx, xm, bytes, xm, true, x_host, s));
    STRATA_TRY_HOST(strata_moe_layer(ex, w_router, bias, dx, T, flags, direct_out ? (float*)om : dout, ids, weights,
                                     ws, ws_bytes, stream));
    return direct_out ? STRATA_OK : copy_host((void*)om, dout, bytes, om, false, out_host, s);
  };
  return run_host_call(key, s, xm && om, enqueue);
}

strata_status strata_moe_stack_host(const strata_experts_t* ex, const uint16_t* w_router, const float* bias,
                                    int32_t n_layers, float* x_host, int32_t T, int32_t* ids, float* weights,
                                    void* ws, size_t ws_bytes, void* stream) {
  if (!x_host || n_layers < 0) return STRATA_E_INVAL;
  const strata_status chk = check_layer_args(ex, n_layers, w_router, bias, 0, T, ws, ws_bytes);
  if (chk != STRATA_OK) return chk;
  if (T == 0 || n_layers == 0) return STRATA_OK;
  const size_t bytes = sizeof(float) * (size_t)T * H;
  const WsLayout L = ws_layout(T);
  float* dx = (float*)((char*)ws + L.io);
  cudaStream_t s = (cudaStream_t)stream;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return STRATA_E_CUDA;
  STRATA_TRY_HOST(not_capturing(s));
  const void* xm = mapped_range(x_host, bytes);
  HostKey key;
  key.kind = 1;
  key.device = dev;
  key.T = T;
  key.n_layers = n_layers;
  key.w_router = w_router;
  key.bias = bias;
  key.x_host = x_host;
  key.out_host = x_host;
  key.x_map = xm;
  key.out_map = xm;
  key.ids = ids;
  key.weights = weights;
  key.ws = ws;
  key.ws_bytes = ws_bytes;
  key.stream = stream;
  key.ex.assign(ex, ex + n_layers);
  auto enqueue = [&]() -> strata_status {
    STRATA_TRY_HOST(copy_host(dx, xm, bytes, xm, true, x_host, s));
    STRATA_TRY_HOST(strata_moe_stack(ex, w_router, bias, n_layers, dx, T, ids, weights, ws, ws_bytes, stream));
    return copy_host((void*)xm, dx, bytes, xm, false, x_host, s);
  };
  return run_host_call(key, s, xm != nullptr, enqueue);
}

}  // extern "C"
