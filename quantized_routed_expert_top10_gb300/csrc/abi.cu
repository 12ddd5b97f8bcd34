// C ABI of the routed-expert MoE block (declared in include/strata_moe.h): argument checks,
// workspace carving and the launch sequence of each step.
#include <cstdio>

#include "common.cuh"

using namespace strata;

namespace {

inline bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

inline strata_status cuda_status(cudaError_t e) { return e == cudaSuccess ? STRATA_OK : STRATA_E_CUDA; }

strata_status check_T(int32_t T) { return (T < 0 || T > TMAX) ? STRATA_E_INVAL : STRATA_OK; }

strata_status check_E(int32_t E) {
  return (E < 32 || E > EMAX || (E % 32) != 0) ? STRATA_E_INVAL : STRATA_OK;
}

strata_status check_ws(const void* ws, size_t ws_bytes, int32_t T) {
  if (!ws) return STRATA_E_INVAL;
  if (!aligned(ws, 256)) return STRATA_E_ALIGN;
  if (ws_bytes < ws_layout(T).total) return STRATA_E_WORKSPACE;
  return STRATA_OK;
}

strata_status check_experts(const strata_experts_t* ex) {
  if (!ex || !ex->blobs) return STRATA_E_INVAL;
  if (check_E(ex->n_expert) != STRATA_OK) return STRATA_E_INVAL;
  if (ex->q2_offset != 1 && ex->q2_offset != 2) return STRATA_E_INVAL;
  if (ex->blob_stride < BLOB) return STRATA_E_INVAL;
  if (!aligned(ex->blobs, 256) || (ex->blob_stride % 256) != 0) return STRATA_E_ALIGN;
  if (ex->shared_blob && !aligned(ex->shared_blob, 256)) return STRATA_E_ALIGN;
  return STRATA_OK;
}

#define STRATA_TRY(expr)                    \
  do {                                      \
    const strata_status _st = (expr);       \
    if (_st != STRATA_OK) return _st;       \
  } while (0)
#define STRATA_CUDA(expr)                          \
  do {                                             \
    const cudaError_t _e = (expr);                 \
    if (_e != cudaSuccess) return STRATA_E_CUDA;   \
  } while (0)

// Steps 1-3 for T tokens into the workspace (ids/weights to the given pointers). Also leaves the
// quantised expert input in ws.qx.  Reads x (rmsnorm applied first when `norm`).
// For a prefill layer (T > DECODE_T_MAX) the router's prep pass also writes the expert path's fp16 token
// copy and initialises out (x for residual layers, else zeros) for the fused combine.
strata_status route_and_group(const float* x, int T, int norm, const uint16_t* w_router, const float* bias, int E,
                              int q2_offset, int32_t* ids, float* weights, float* logits_user,
                              const WsLayout& L, char* ws, cudaStream_t s, float* out = nullptr) {
  if (T <= DECODE_T_MAX) {
    STRATA_CUDA(launch_route_decode(x, T, norm, w_router, bias, E, q2_offset, ids, weights, logits_user, L, ws, s));
    return STRATA_OK;
  }
  float* lparts = (float*)(ws + L.logits);
  STRATA_CUDA(launch_router_tc(x, norm ? (float*)(ws + L.inv_rms) : nullptr, T, w_router, E, ws + L.xbf, lparts,
                               (int*)(ws + L.status), s, out ? (uint8_t*)(ws + L.x16) : nullptr, out));
  STRATA_CUDA(launch_top_k(lparts, T, E, bias, logits_user, ids, weights, s));
  STRATA_CUDA(launch_group(ids, T, E, (int32_t*)(ws + L.expert_off), (int32_t*)(ws + L.pair),
                           (int32_t*)(ws + L.active), nullptr, L, ws, s));
  return STRATA_OK;
}

strata_status layer_impl(const strata_experts_t* ex, const uint16_t* w_router, const float* bias, const float* x,
                         int32_t T, int32_t flags, float* out, int32_t* ids, float* weights, void* ws,
                         size_t ws_bytes, cudaStream_t s, const DecodeNext* next = nullptr) {
  STRATA_TRY(check_T(T));
  if (!w_router || !x || !out) return STRATA_E_INVAL;
  STRATA_TRY(check_experts(ex));
  if (flags & ~STRATA_MOE_RESIDUAL_RMSNORM) return STRATA_E_INVAL;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(w_router, 16) || (bias && !aligned(bias, 4)))
    return STRATA_E_ALIGN;
  STRATA_TRY(check_ws(ws, ws_bytes, T));
  if (T == 0) return STRATA_OK;
  const WsLayout L = ws_layout(T);
  char* w = (char*)ws;
  int32_t* ids_d = ids ? ids : (int32_t*)(w + L.ids);
  float* wts_d = weights ? weights : (float*)(w + L.weights);
  const int norm = (flags & STRATA_MOE_RESIDUAL_RMSNORM) ? 1 : 0;
  if (T <= DECODE_T_MAX) {
    const int alias = (x < out + (size_t)T * H && out < x + (size_t)T * H) ? 1 : 0;  // in-place call
    STRATA_CUDA(launch_decode_fused(*ex, w_router, bias, x, T, norm, alias, out, ids_d, wts_d, next, L, w, s));
    return STRATA_OK;
  }
  STRATA_TRY(route_and_group(x, T, norm, w_router, bias, ex->n_expert, ex->q2_offset, ids_d, wts_d, nullptr, L, w, s,
                             out));
  STRATA_CUDA(launch_experts_tc(*ex, (const uint8_t*)(w + L.x16), T, (const int32_t*)(w + L.expert_off),
                                (const int32_t*)(w + L.pair), (const int32_t*)(w + L.active),
                                (const int32_t*)(w + L.n_active), nullptr, wts_d, out, (uint8_t*)(w + L.xg),
                                (uint8_t*)(w + L.hg),
                                (uint8_t*)(w + L.tcmeta), (int*)(w + L.status), s, ex->shared_blob));
  return STRATA_OK;
}

}  // namespace

// The checks strata_moe_layer / strata_moe_stack make before enqueueing anything, for the host-buffer
// calls to make before they touch the device (n_ex descriptors, all with the same expert count).
strata_status strata::check_layer_args(const strata_experts_t* ex, int n_ex, const uint16_t* w_router,
                                       const float* bias, int32_t flags, int32_t T, const void* ws,
                                       size_t ws_bytes) {
  STRATA_TRY(check_T(T));
  if (!ex || n_ex < 0 || !w_router) return STRATA_E_INVAL;
  for (int l = 0; l < n_ex; ++l) {
    STRATA_TRY(check_experts(&ex[l]));
    if (ex[l].n_expert != ex[0].n_expert) return STRATA_E_INVAL;
  }
  if (flags & ~STRATA_MOE_RESIDUAL_RMSNORM) return STRATA_E_INVAL;
  if (!aligned(w_router, 16) || (bias && !aligned(bias, 4))) return STRATA_E_ALIGN;
  return check_ws(ws, ws_bytes, T);
}

extern "C" {

size_t strata_moe_workspace_bytes(int32_t T) {
  if (T < 0 || T > TMAX) return 0;
  return ws_layout(T).total;
}

strata_status strata_moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws) return STRATA_E_INVAL;
  if (!aligned(ws, 256)) return STRATA_E_ALIGN;
  if (ws_bytes < WS_HEADER) return STRATA_E_WORKSPACE;
  // the header and, when the workspace holds it, the decode exchange area (tag 0 = no value)
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes < DX_END ? WS_HEADER : DX_END, (cudaStream_t)stream));
}

strata_status strata_moe_route(const float* x, int32_t T, const uint16_t* w_router, const float* bias,
                               int32_t n_expert, int32_t* ids, float* weights, float* logits, void* ws,
                               size_t ws_bytes, void* stream) {
  STRATA_TRY(check_T(T));
  STRATA_TRY(check_E(n_expert));
  if (!x || !w_router || !ids || !weights) return STRATA_E_INVAL;
  if (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(ids, 4) || !aligned(weights, 4) ||
      (bias && !aligned(bias, 4)) || (logits && !aligned(logits, 4)))
    return STRATA_E_ALIGN;
  STRATA_TRY(check_ws(ws, ws_bytes, T));
  if (T == 0) return STRATA_OK;
  const WsLayout L = ws_layout(T);
  char* w = (char*)ws;
  cudaStream_t s = (cudaStream_t)stream;
  if (T <= DECODE_T_MAX) {
    STRATA_CUDA(launch_route_decode(x, T, 0, w_router, bias, n_expert, 1, ids, weights, logits, L, w, s));
    return STRATA_OK;
  }
  float* lparts = (float*)(w + L.logits);
  STRATA_CUDA(launch_router_tc(x, nullptr, T, w_router, n_expert, w + L.xbf, lparts, (int*)(w + L.status), s));
  STRATA_CUDA(launch_top_k(lparts, T, n_expert, bias, logits, ids, weights, s));
  return STRATA_OK;
}

strata_status strata_moe_group(const int32_t* ids, int32_t T, int32_t n_expert, int32_t* expert_off, int32_t* pair,
                               int32_t* active, int32_t* n_active, void* ws, size_t ws_bytes, void* stream) {
  STRATA_TRY(check_T(T));
  STRATA_TRY(check_E(n_expert));
  if (!ids || !expert_off || !pair || !active || !n_active) return STRATA_E_INVAL;
  if (!aligned(ids, 4) || !aligned(expert_off, 4) || !aligned(pair, 4) || !aligned(active, 4) || !aligned(n_active, 4))
    return STRATA_E_ALIGN;
  STRATA_TRY(check_ws(ws, ws_bytes, T));
  if (T == 0) return STRATA_OK;
  const WsLayout L = ws_layout(T);
  STRATA_CUDA(launch_group(ids, T, n_expert, expert_off, pair, active, n_active, L, (char*)ws, (cudaStream_t)stream));
  return STRATA_OK;
}

strata_status strata_moe_experts(const strata_experts_t* ex, const float* x, int32_t T, const int32_t* expert_off,
                                 const int32_t* pair, const int32_t* active, const int32_t* n_active, float* parts,
                                 void* ws, size_t ws_bytes, void* stream) {
  STRATA_TRY(check_T(T));
  STRATA_TRY(check_experts(ex));
  if (!x || !expert_off || !pair || !active || !n_active || !parts) return STRATA_E_INVAL;
  if (!aligned(x, 16) || !aligned(parts, 16) || !aligned(expert_off, 4) || !aligned(pair, 4) || !aligned(active, 4) ||
      !aligned(n_active, 4))
    return STRATA_E_ALIGN;
  STRATA_TRY(check_ws(ws, ws_bytes, T));
  if (T == 0) return STRATA_OK;
  const WsLayout L = ws_layout(T);
  char* w = (char*)ws;
  cudaStream_t s = (cudaStream_t)stream;
  STRATA_CUDA(launch_x16(x, nullptr, T, (uint8_t*)(w + L.x16), s));
  STRATA_CUDA(launch_experts_tc(*ex, (const uint8_t*)(w + L.x16), T, expert_off, pair, active, n_active, parts,
                                nullptr, nullptr, (uint8_t*)(w + L.xg), (uint8_t*)(w + L.hg), (uint8_t*)(w + L.tcmeta),
                                (int*)(w + L.status), s));
  return STRATA_OK;
}

strata_status strata_moe_combine(const float* parts, const float* weights, int32_t T, const float* residual,
                                 float* out, void* stream) {
  STRATA_TRY(check_T(T));
  if (!parts || !weights || !out) return STRATA_E_INVAL;
  if (!aligned(parts, 16) || !aligned(out, 16) || !aligned(weights, 4) || (residual && !aligned(residual, 16)))
    return STRATA_E_ALIGN;
  if (T == 0) return STRATA_OK;
  STRATA_CUDA(launch_combine(parts, weights, T, residual, out, (cudaStream_t)stream));
  return STRATA_OK;
}

strata_status strata_moe_layer(const strata_experts_t* ex, const uint16_t* w_router, const float* bias, const float* x,
                               int32_t T, int32_t flags, float* out, int32_t* ids, float* weights, void* ws,
                               size_t ws_bytes, void* stream) {
  return layer_impl(ex, w_router, bias, x, T, flags, out, ids, weights, ws, ws_bytes, (cudaStream_t)stream);
}

strata_status strata_moe_stack(const strata_experts_t* ex, const uint16_t* w_router, const float* bias,
                               int32_t n_layers, float* x, int32_t T, int32_t* ids, float* weights, void* ws,
                               size_t ws_bytes, void* stream) {
  if (!ex || n_layers < 0) return STRATA_E_INVAL;
  STRATA_TRY(check_T(T));
  for (int l = 0; l < n_layers; ++l) {
    STRATA_TRY(check_experts(&ex[l]));
    if (ex[l].n_expert != ex[0].n_expert) return STRATA_E_INVAL;
  }
  if (n_layers == 0 || T == 0) return STRATA_OK;
  const int E = ex[0].n_expert;
  // decode stacks alternate between x and a workspace buffer, so no layer writes the array it reads
  // (the one-kernel layer then needs no release/acquire pair around its router exchange); an odd
  // stack ends with one copy back into x
  float* bufs[2] = {x, T <= DECODE_T_MAX && ws ? (float*)((char*)ws + ws_layout(T).xpp) : x};
  for (int l = 0; l < n_layers; ++l) {
    // decode layers look one layer ahead: the next router on this layer's input names the experts to
    // prefetch into L2
    DecodeNext next{};
    if (l + 1 < n_layers)
      next = DecodeNext{w_router + (size_t)(l + 1) * E * H, bias ? bias + (size_t)(l + 1) * E : nullptr,
                        (const uint8_t*)ex[l + 1].blobs, ex[l + 1].blob_stride};
    STRATA_TRY(layer_impl(&ex[l], w_router + (size_t)l * E * H, bias ? bias + (size_t)l * E : nullptr, bufs[l & 1], T,
                          STRATA_MOE_RESIDUAL_RMSNORM, bufs[(l + 1) & 1], ids ? ids + (size_t)l * T * K : nullptr,
                          weights ? weights + (size_t)l * T * K : nullptr, ws, ws_bytes, (cudaStream_t)stream,
                          l + 1 < n_layers ? &next : nullptr));
  }
  if (bufs[n_layers & 1] != x)
    STRATA_CUDA(cudaMemcpyAsync(x, bufs[n_layers & 1], sizeof(float) * (size_t)T * H, cudaMemcpyDeviceToDevice,
                                (cudaStream_t)stream));
  return STRATA_OK;
}

strata_status strata_moe_wait_selftest(void* ws, size_t ws_bytes, uint64_t limit_ns, void* stream) {
  STRATA_TRY(check_ws(ws, ws_bytes, 1));
  if (limit_ns < 1000 || limit_ns > 2000000000ull) return STRATA_E_INVAL;
  const WsLayout L = ws_layout(1);
  uint64_t* word = (uint64_t*)((char*)ws + L.logits);
  STRATA_CUDA(cudaMemsetAsync(word, 0, sizeof(uint64_t), (cudaStream_t)stream));
  // tag 0xA5A5A5A5: the word holds tag 0 and nothing writes it during the call
  STRATA_CUDA(launch_wait_selftest(word, 0xA5A5A5A5u, (unsigned long long)limit_ns, (int*)((char*)ws + L.status),
                                   (cudaStream_t)stream));
  return STRATA_OK;
}

strata_status strata_pack_q2_0(const uint8_t* canonical, uint8_t* packed, int64_t n_blobs) {
  if (!canonical || !packed || n_blobs < 0) return STRATA_E_INVAL;
  const uint8_t* c_end = canonical + n_blobs * BLOB;
  const uint8_t* p_end = packed + n_blobs * BLOB;
  if (n_blobs && canonical < p_end && packed < c_end) return STRATA_E_INVAL;
  pack_host(canonical, packed, n_blobs);
  return STRATA_OK;
}

strata_status strata_unpack_q2_0(const uint8_t* packed, uint8_t* canonical, int64_t n_blobs) {
  if (!canonical || !packed || n_blobs < 0) return STRATA_E_INVAL;
  const uint8_t* c_end = canonical + n_blobs * BLOB;
  const uint8_t* p_end = packed + n_blobs * BLOB;
  if (n_blobs && canonical < p_end && packed < c_end) return STRATA_E_INVAL;
  unpack_host(packed, canonical, n_blobs);
  return STRATA_OK;
}

strata_status strata_pack_q2_0_device(const uint8_t* canonical, int64_t src_stride, uint8_t* packed,
                                      int64_t dst_stride, int64_t n_blobs, void* stream) {
  if (!canonical || !packed || n_blobs < 0) return STRATA_E_INVAL;
  if (src_stride < BLOB || dst_stride < BLOB) return STRATA_E_INVAL;
  if (!aligned(canonical, 2) || (src_stride & 1) || !aligned(packed, 256) || (dst_stride % 256)) return STRATA_E_ALIGN;
  if (n_blobs == 0) return STRATA_OK;
  STRATA_CUDA(launch_pack_device(canonical, src_stride, packed, dst_stride, n_blobs, (cudaStream_t)stream));
  return STRATA_OK;
}

strata_status strata_poll_status(const void* ws, void* stream) {
  if (!ws) return STRATA_E_INVAL;
  int v = 0;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return STRATA_E_CUDA;
  if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return STRATA_E_CUDA;
  if (v & ST_TIMEOUT) return STRATA_E_TIMEOUT;
  if (v & ST_CORRUPT) return STRATA_E_CORRUPT;
  return STRATA_OK;
}

strata_status strata_clear_status(void* ws, void* stream) {
  if (!ws) return STRATA_E_INVAL;
  return cuda_status(cudaMemsetAsync(ws, 0, sizeof(int), (cudaStream_t)stream));
}

const char* strata_status_str(strata_status s) {
  switch (s) {
    case STRATA_OK: return "STRATA_OK";
    case STRATA_E_INVAL: return "STRATA_E_INVAL: invalid argument";
    case STRATA_E_ALIGN: return "STRATA_E_ALIGN: misaligned pointer or stride";
    case STRATA_E_UNSUPPORTED: return "STRATA_E_UNSUPPORTED: unsupported shape";
    case STRATA_E_CUDA: return "STRATA_E_CUDA: CUDA runtime error";
    case STRATA_E_TIMEOUT: return "STRATA_E_TIMEOUT: bounded device wait expired";
    case STRATA_E_WORKSPACE: return "STRATA_E_WORKSPACE: workspace too small";
    case STRATA_E_CORRUPT: return "STRATA_E_CORRUPT: invalid data seen on the device";
  }
  return "unknown strata_status";
}

}  // extern "C"
