// Host-buffer entry points (declared in include/strata_moe.h): one call copies the activations from
// host memory into the workspace's I/O area, runs the layer (or the stack) exactly as the device-buffer
// call does, copies the result back to host memory and synchronises the stream.
//
// With page-locked host buffers and a non-default stream the three steps are captured once as a CUDA
// graph and replayed by later calls with the same arguments, so a call costs one graph launch and one
// synchronisation on the host instead of a copy, a launch per kernel and a copy.
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"

using namespace strata;

namespace {

inline bool page_locked(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // an unregistered pointer may leave an error behind on older drivers
    return false;
  }
  return a.type == cudaMemoryTypeHost;
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
  const void* ids = nullptr;
  const void* weights = nullptr;
  const void* ws = nullptr;
  size_t ws_bytes = 0;
  const void* stream = nullptr;
  std::vector<strata_experts_t> ex;

  bool operator==(const HostKey& o) const {
    if (kind != o.kind || device != o.device || T != o.T || flags != o.flags || n_layers != o.n_layers ||
        w_router != o.w_router || bias != o.bias || x_host != o.x_host || out_host != o.out_host || ids != o.ids ||
        weights != o.weights || ws != o.ws || ws_bytes != o.ws_bytes || stream != o.stream || ex.size() != o.ex.size())
      return false;
    for (size_t i = 0; i < ex.size(); ++i)
      if (ex[i].blobs != o.ex[i].blobs || ex[i].blob_stride != o.ex[i].blob_stride ||
          ex[i].n_expert != o.ex[i].n_expert || ex[i].q2_offset != o.ex[i].q2_offset)
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
strata_status run_host_call(const HostKey& key, cudaStream_t s, const void* a, const void* b, Enqueue enqueue) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return STRATA_E_CUDA;
  if (cs != cudaStreamCaptureStatusNone) return STRATA_E_INVAL;  // a synchronising call cannot be captured
  const bool graphable = s != nullptr && s != cudaStreamLegacy && page_locked(a) && page_locked(b) &&
                         !profiling_armed();
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
  HostKey key;
  key.kind = 0;
  key.device = dev;
  key.T = T;
  key.flags = flags;
  key.w_router = w_router;
  key.bias = bias;
  key.x_host = x_host;
  key.out_host = out_host;
  key.ids = ids;
  key.weights = weights;
  key.ws = ws;
  key.ws_bytes = ws_bytes;
  key.stream = stream;
  key.ex.assign(ex, ex + 1);
  auto enqueue = [&]() -> strata_status {
    if (cudaMemcpyAsync(dx, x_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return STRATA_E_CUDA;
    const strata_status st = strata_moe_layer(ex, w_router, bias, dx, T, flags, dout, ids, weights, ws, ws_bytes, stream);
    if (st != STRATA_OK) return st;
    return cudaMemcpyAsync(out_host, dout, bytes, cudaMemcpyDeviceToHost, s) == cudaSuccess ? STRATA_OK
                                                                                             : STRATA_E_CUDA;
  };
  return run_host_call(key, s, x_host, out_host, enqueue);
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
  HostKey key;
  key.kind = 1;
  key.device = dev;
  key.T = T;
  key.n_layers = n_layers;
  key.w_router = w_router;
  key.bias = bias;
  key.x_host = x_host;
  key.out_host = x_host;
  key.ids = ids;
  key.weights = weights;
  key.ws = ws;
  key.ws_bytes = ws_bytes;
  key.stream = stream;
  key.ex.assign(ex, ex + n_layers);
  auto enqueue = [&]() -> strata_status {
    if (cudaMemcpyAsync(dx, x_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return STRATA_E_CUDA;
    const strata_status st = strata_moe_stack(ex, w_router, bias, n_layers, dx, T, ids, weights, ws, ws_bytes, stream);
    if (st != STRATA_OK) return st;
    return cudaMemcpyAsync(x_host, dx, bytes, cudaMemcpyDeviceToHost, s) == cudaSuccess ? STRATA_OK
                                                                                         : STRATA_E_CUDA;
  };
  return run_host_call(key, s, x_host, x_host, enqueue);
}

}  // extern "C"
