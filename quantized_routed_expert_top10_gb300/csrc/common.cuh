// Internal definitions shared by the sm_103a kernels of the routed-expert MoE block.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "strata_moe.h"

namespace strata {

// Dimensions fixed by the model ("The byte budget, in code": H = 2560, FF = 640, QK = 64, top-10).
constexpr int H = STRATA_MOE_H;
constexpr int FF = STRATA_MOE_FF;
constexpr int K = STRATA_MOE_K;
constexpr int QK = STRATA_MOE_QK;
constexpr int EMAX = STRATA_MOE_E_MAX;
constexpr int TMAX = STRATA_MOE_T_MAX;
constexpr int KB_GU = H / QK;  // 40 k-blocks along gate/up's contraction
constexpr int KB_D = FF / QK;  // 10 k-blocks along down's contraction
constexpr int RT = 128;        // rows per row tile
constexpr int RT_GU = FF / RT; // 5 gate/up row tiles
constexpr int RT_D = H / RT;   // 20 down row tiles
// Packed gate/up region: slabs of 16 rows; per (slab, kb) a 576-byte piece (gate codes of the 16
// rows, up codes, {gate d, up d} per row); a slab's 40 pieces are contiguous (23,040 bytes).
constexpr int SLAB = 16;                  // rows per gate/up slab
constexpr int N_SLAB = FF / SLAB;         // 40 slabs
constexpr int SLAB_KB = 576;              // bytes per (slab, kb) piece
constexpr int SLAB_BYTES = KB_GU * SLAB_KB;  // 23,040 bytes per slab
constexpr int GU_CHUNK = (RT / SLAB) * SLAB_KB;  // 4,608 bytes: one kb of a 128-row tile (8 pieces)
constexpr int D_CHUNK = 2304;  // bytes per (rt, kb) down chunk
constexpr int64_t D_REGION = 921600;
constexpr int64_t BLOB = STRATA_MOE_BLOB_BYTES;

constexpr int ROUTER_KSPLIT = 2;  // prefill router: splits of the 2,560-term contraction over CTAs
constexpr int DECODE_T_MAX = 8;  // T <= this: fused single-kernel routing (router + top-10 + grouping)

// Device status bits (ws word 0).
constexpr int ST_CORRUPT = 1;
constexpr int ST_TIMEOUT = 2;

// A 64-wide block of an activation vector, quantised to 16-bit integers q ~= v / s and split into
// hi (signed) and lo (unsigned) bytes, laid out for the Q2_0 code masks: word (q4, m) holds the
// values of weights 16*q4 + 4*b + m, b = 0..3 (byte b), matching (codes & (3 << 2m)) of code word q4.
struct __align__(16) QBlock {
  uint32_t hi[16];
  uint32_t lo[16];
  float s64;    // s / 64, s = max|v| / 32767
  int32_t qoff; // 64 * q2_offset * sum(q)
  int32_t pad[2];
};
static_assert(sizeof(QBlock) == 144, "QBlock layout");

// Workspace layout for a call with T tokens (byte offsets, each 256-aligned).  The first
// WS_HEADER bytes (status word and counters) are the same for every T and are zeroed once by
// strata_moe_workspace_init; kernels that use a counter reset it before they finish.
constexpr size_t WS_HEADER = 12288;
constexpr size_t WS_STATUS = 0;     // int32 status word
constexpr size_t WS_CNT_ROUTE = 64; // int32 router last-CTA counter
// Sync words of the one-kernel decode layer (int32 indices from WS_SYNC): the exit counter and the
// call epoch (the tag of the values one call exchanges through the area below).
constexpr size_t WS_SYNC = 4096;
constexpr int WS_SYNC_EXIT = 1;
constexpr int WS_SYNC_EPOCH = 32;  // own 128-byte line
constexpr int WS_SYNC_SMRANK = 64;  // [256] per-SM arrival tickets (which of an SM's CTAs is which)
constexpr int WS_SYNC_WORDS = WS_SYNC_SMRANK + 256;
constexpr int WS_NREP = 16;        // replicas of the router dot products (every CTA reads all of them)
static_assert(WS_SYNC + sizeof(int32_t) * WS_SYNC_WORDS <= WS_HEADER, "decode sync words must fit the header");
// Decode exchange area, right after the header at the same offset for every T >= 1: 64-bit words
// (value bits, call tag), each written once per call and polled by the CTAs that need it, so a
// reader learns that a value is there from the value itself.  strata_moe_workspace_init zeroes it;
// tag 0 never marks a value.
constexpr size_t DX_DOTS = WS_HEADER;                                              // [WS_NREP][8][EMAX]
// pair slots: the routed pairs t*K + k, then one per token for a layer's shared expert (K*T + t)
constexpr int DECODE_PAIRS = DECODE_T_MAX * (K + 1);
constexpr size_t DX_H = DX_DOTS + sizeof(uint64_t) * WS_NREP * DECODE_T_MAX * EMAX;  // [DECODE_PAIRS][FF]
constexpr size_t DX_PARTS = DX_H + sizeof(uint64_t) * DECODE_PAIRS * FF;           // [DECODE_PAIRS][H]
constexpr size_t DX_PRED = DX_PARTS + sizeof(uint64_t) * DECODE_PAIRS * H;         // [8][EMAX] next layer
constexpr size_t DX_PRED_IDS = DX_PRED + sizeof(uint64_t) * DECODE_T_MAX * EMAX;     // [1 + 8 * K]
constexpr size_t DX_END = (DX_PRED_IDS + sizeof(uint64_t) * (1 + DECODE_T_MAX * K) + 255) / 256 * 256;
static_assert(DX_END % 256 == 0 && DX_PRED_IDS % 256 == 0, "exchange area regions stay 256-byte aligned");

struct WsLayout {
  size_t status, cnt_route;
  size_t logits;      // fp32 [ROUTER_KSPLIT][T][EMAX] partial router logits (T > DECODE_T_MAX: one slice per
                      // split of the contraction; the decode path uses slice 0 as [T][EMAX] logits)
  size_t ids;         // int32 [T][K]
  size_t weights;     // fp32 [T][K]
  size_t inv_rms;     // fp32 [T] 1/rms of each token (residual layers, T > DECODE_T_MAX)
  size_t xbf;         // bf16 [2][T][H] router operand: x_hi, x_lo (T > DECODE_T_MAX)
  size_t expert_off;  // int32 [EMAX + 1]
  size_t pair;        // int32 [T*K]
  size_t active;      // int32 [EMAX]
  size_t n_active;    // int32 [4]: n_active
  size_t chunk_cnt;   // int32 [n_chunks][EMAX]
  size_t qx;          // QBlock [T][KB_GU] quantised layer input (T <= DECODE_T_MAX routing kernel)
  size_t xpp;         // fp32 [T][H] (T <= DECODE_T_MAX): the other buffer of a decode stack's ping-pong
  size_t x16;         // tensor-core expert path: fp16 token copy [KB_GU][T][128 B]
  size_t xg;          //                          the same per padded slot, swizzled [KB_GU][rows][128 B]
  size_t hg;          //                          fp16 h per padded slot, swizzled [KB_D][rows][128 B]
  size_t tcmeta;      //                                      expert ranges, tiles, counts
  size_t io;          // fp32 [2][T][H]: device copies of a host-buffer call's input and output
  size_t total;
  int n_chunks;
};

constexpr int GROUP_CHUNK = 2048;  // pairs per grouping chunk

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Sizes of the tensor-core path's buffers (experts_tc.cu).
int64_t tc_rows_cap(int T);
size_t tc_x16_bytes(int T);
size_t tc_xg_bytes(int T);
size_t tc_hg_bytes(int T);
size_t tc_meta_bytes(int T);

inline WsLayout ws_layout(int T) {
  WsLayout L{};
  const int P = T * K;
  L.n_chunks = (P + GROUP_CHUNK - 1) / GROUP_CHUNK;
  if (L.n_chunks < 1) L.n_chunks = 1;
  L.status = WS_STATUS;
  L.cnt_route = WS_CNT_ROUTE;
  size_t o = DX_END;
  auto take = [&](size_t bytes) { size_t at = o; o = align256(o + bytes); return at; };
  L.logits = take(sizeof(float) * (size_t)ROUTER_KSPLIT * T * EMAX);
  L.ids = take(sizeof(int32_t) * (size_t)P);
  L.weights = take(sizeof(float) * (size_t)P);
  L.inv_rms = take(T > DECODE_T_MAX ? sizeof(float) * (size_t)T : 0);
  L.xbf = take(T > DECODE_T_MAX ? sizeof(uint16_t) * 2 * (size_t)T * H : 0);
  L.expert_off = take(sizeof(int32_t) * (EMAX + 1));
  L.pair = take(sizeof(int32_t) * (size_t)P);
  L.active = take(sizeof(int32_t) * EMAX);
  L.n_active = take(sizeof(int32_t) * 4);
  L.chunk_cnt = take(sizeof(int32_t) * (size_t)L.n_chunks * EMAX);
  L.qx = take(sizeof(QBlock) * (size_t)T * KB_GU);
  L.xpp = take(T <= DECODE_T_MAX ? sizeof(float) * (size_t)T * H : 0);
  L.x16 = take(tc_x16_bytes(T));
  L.xg = take(tc_xg_bytes(T));
  L.hg = take(tc_hg_bytes(T));
  L.tcmeta = take(tc_meta_bytes(T));
  L.io = take(sizeof(float) * 2 * (size_t)T * H);
  L.total = T > 0 ? o : WS_HEADER;
  return L;
}
// ---------------------------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ void set_status(int* status, int bit) { atomicOr(status, bit); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Quantise one 64-value block held as two values per lane (lane l: v0 = v[2l], v1 = v[2l+1]) into
// a QBlock.  Must be called by a full warp; `tmp` is 64 int32 of shared memory for this warp.
__device__ __forceinline__ void quantise_block_warp(float v0, float v1, int q2_offset, QBlock* dst,
                                                    int32_t* tmp) {
  const int lane = threadIdx.x & 31;
  const float amax = warp_max(fmaxf(fabsf(v0), fabsf(v1)));
  int q0 = 0, q1 = 0;
  if (amax > 0.f) {
    const float inv = 32767.f / amax;
    q0 = max(-32767, min(32767, __float2int_rn(v0 * inv)));
    q1 = max(-32767, min(32767, __float2int_rn(v1 * inv)));
  }
  tmp[2 * lane] = q0;
  tmp[2 * lane + 1] = q1;
  int qs = q0 + q1;
#pragma unroll
  for (int o = 16; o; o >>= 1) qs += __shfl_xor_sync(0xffffffffu, qs, o);
  __syncwarp();
  // lane -> word: lanes 0..15 hi words, 16..31 lo words; word index w = q4 * 4 + m.
  const int w = lane & 15;
  const int q4 = w >> 2, m = w & 3;
  uint32_t word = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const int v = tmp[16 * q4 + 4 * b + m];
    const uint32_t byte = (lane < 16) ? (uint32_t)((v >> 8) & 0xFF) : (uint32_t)(v & 0xFF);
    word |= byte << (8 * b);
  }
  if (lane < 16) dst->hi[w] = word; else dst->lo[w] = word;
  if (lane == 0) {
    dst->s64 = (amax > 0.f) ? (amax / 32767.f) * (1.f / 64.f) : 0.f;
    dst->qoff = 64 * q2_offset * qs;
  }
  __syncwarp();
}

// Sum over the code masks of one 16-byte Q2_0 code row against one QBlock's words, returning
// 64 * (sum_i c_i * q_i); the caller subtracts qoff and scales by d * s64.
struct Masked { uint32_t m[16]; };

__device__ __forceinline__ Masked mask_codes(uint4 c) {
  Masked r;
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    r.m[4 * q + 0] = w[q] & 0x03030303u;
    r.m[4 * q + 1] = w[q] & 0x0C0C0C0Cu;
    r.m[4 * q + 2] = w[q] & 0x30303030u;
    r.m[4 * q + 3] = w[q] & 0xC0C0C0C0u;
  }
  return r;
}

__device__ __forceinline__ int dot64(const Masked& c, const uint32_t* hi, const uint32_t* lo) {
  int ah[4] = {0, 0, 0, 0}, al[4] = {0, 0, 0, 0};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      ah[m] = dp4a_us(c.m[4 * q + m], hi[4 * q + m], ah[m]);
      al[m] = dp4a_uu(c.m[4 * q + m], lo[4 * q + m], al[m]);
    }
  }
  // ah[m] = 4^m * S_hi,m  ->  64 * S_hi = 64 ah0 + 16 ah1 + 4 ah2 + ah3 (exact in int32).
  const int sh = ((ah[0] * 4 + ah[1]) * 4 + ah[2]) * 4 + ah[3];
  const int sl = ((al[0] * 4 + al[1]) * 4 + al[2]) * 4 + al[3];
  return sh * 256 + sl;
}

}  // namespace strata

// Launchers implemented in the .cu files (all enqueue on `stream`, return cudaGetLastError()).
namespace strata {
// Launch accounting (instrument.cu): every launch is bracketed by kernel_begin / kernel_end, which count
// it and record the caller's armed timing events around it.  Ids equal the ABI's STRATA_KERNEL_*.
enum KernelId : int {
  KID_DECODE_LAYER = 0, KID_ROUTE_DECODE, KID_ROUTER_PREP, KID_ROUTER_TC, KID_TOP_K, KID_GROUP_HIST, KID_GROUP_SCAN,
  KID_GROUP_SCATTER, KID_TC_PREPARE, KID_TC_GATHER, KID_TC_GATEUP, KID_TC_DOWN, KID_COMBINE, KID_PACK, KID_HOST_COPY,
  KID_WAIT_SELFTEST, KID_BLOB_CRC32, KID_COUNT
};
void kernel_begin(int kid, cudaStream_t s);
void kernel_end(int kid, cudaStream_t s);
// Argument checks of a layer / stack call with n_ex expert descriptors (abi.cu).
strata_status check_layer_args(const strata_experts_t* ex, int n_ex, const uint16_t* w_router, const float* bias,
                               int32_t flags, int32_t T, const void* ws, size_t ws_bytes);
// True while the calling thread has event timing armed for some kernel (its launches must then be
// enqueued one by one, not replayed from a graph).
bool profiling_armed();
// Counts n launches made by replaying a graph that holds n of the library's kernels (n may wrap to
// take back launches that a capture counted).
void count_launches(unsigned long long n);
// Launch sites the calling thread has passed so far (captured ones included).
unsigned long long launches_this_thread();
// Launch of a kernel of the prefill chain with programmatic stream serialisation: it may start while
// the kernel before it on the stream finishes (that kernel lets it once every CTA has begun), and it
// reaches past its prologue only through griddep_wait(), which returns once the kernel before it has
// completed and its memory is visible.  Kernels launched this way call griddep_launch_dependents()
// and griddep_wait() (device_common.cuh) before touching memory that other launches write or read.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

#define STRATA_LAUNCH(kid, s, ...) \
  do {                             \
    kernel_begin((kid), (s));      \
    __VA_ARGS__;                   \
    kernel_end((kid), (s));        \
  } while (0)

// CRC-32 of packed blobs (checksum.cu): on the host, and one CTA per blob on the device.
uint32_t blob_crc32_host(const uint8_t* data, int64_t n);
cudaError_t launch_blob_crc32(const uint8_t* blobs, int64_t stride, int64_t n_blobs, uint32_t* crc, cudaStream_t s);
// The decode layer's bounded waits on conditions that never hold, with limit_ns (decode_fused.cu).
cudaError_t launch_wait_selftest(const uint64_t* word, uint32_t tag, unsigned long long limit_ns, int* status,
                                 cudaStream_t s);
cudaError_t launch_route_decode(const float* x, int T, int apply_rmsnorm, const uint16_t* w_router,
                                const float* bias, int E, int q2_offset, int32_t* ids, float* weights,
                                float* logits_out, const WsLayout& L, char* ws, cudaStream_t s);
// Router logits of a prefill chunk: bf16 hi/lo copies of x (times 1/rms, written to inv_rms, when it is
// non-null) in xbf, then the tensor-core GEMM into the partial-logit slices.  A layer call also passes
// x16 (receives the expert path's fp16 token copy, with the same 1/rms) and out (receives x when inv_rms
// is non-null -- the residual -- else zeros, for the down kernel to add the experts' outputs into).
cudaError_t launch_router_tc(const float* x, float* inv_rms, int T, const uint16_t* w_router, int E, void* xbf,
                             float* parts, int* status, cudaStream_t s, uint8_t* x16 = nullptr,
                             float* out = nullptr);
cudaError_t launch_top_k(const float* parts, int T, int E, const float* bias, float* logits_out, int32_t* ids,
                         float* weights, cudaStream_t s);
cudaError_t launch_group(const int32_t* ids, int T, int E, int32_t* expert_off, int32_t* pair,
                         int32_t* active, int32_t* n_active, const WsLayout& L, char* ws, cudaStream_t s);
// A 2-D tensor map (CUtensorMap, 64-byte aligned storage) over a row-major matrix of `rows` rows of
// `inner` elements of CUtensorMapDataType `dtype`, rows row_stride bytes apart; boxes of box_inner x
// box_rows elements, 128-byte swizzle, out-of-range elements read as zeros.  False if encoding fails.
bool make_tensor_map_2d(void* map, int dtype, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride,
                        uint32_t box_inner, uint32_t box_rows);
// fp16 token copy X16 of x (times inv_rms[t] when non-null) for the tensor-core expert path.
cudaError_t launch_x16(const float* x, const float* inv_rms, int T, uint8_t* x16, cudaStream_t s);
// Tile lists, then the gate/up and down kernels over the grouping.  out == null: y of every pair into
// parts [T*K][H]; otherwise out[t] += weights[t][k] * y (out already holds the residual or zeros), and
// a non-null shared_blob adds that expert's output for every token with weight 1.
cudaError_t launch_experts_tc(const strata_experts_t& ex, const uint8_t* x16, int T, const int32_t* expert_off,
                              const int32_t* pair, const int32_t* active, const int32_t* n_active, float* parts,
                              const float* weights, float* out, uint8_t* xg, uint8_t* hg, uint8_t* meta, int* status,
                              cudaStream_t s, const void* shared_blob = nullptr);
cudaError_t launch_combine(const float* parts, const float* weights, int T, const float* residual,
                           float* out, cudaStream_t s);
// The next layer of a decode stack, for the lookahead (its router on this layer's input predicts its
// experts, which are prefetched into L2 while this layer finishes).
struct DecodeNext {
  const uint16_t* wr;  // [E][H] bf16
  const float* bias;   // [E] or null
  const uint8_t* blobs;
  int64_t stride;
};
cudaError_t launch_decode_fused(const strata_experts_t& ex, const uint16_t* w_router, const float* bias,
                                const float* x, int T, int residual, int alias, float* out, int32_t* ids, float* weights,
                                const DecodeNext* next, const WsLayout& L, char* ws, cudaStream_t s);
cudaError_t launch_pack_device(const uint8_t* canonical, int64_t src_stride, uint8_t* packed,
                               int64_t dst_stride, int64_t n_blobs, cudaStream_t s);
}  // namespace strata

namespace strata {
void pack_host(const uint8_t* canonical, uint8_t* packed, int64_t n_blobs);
void unpack_host(const uint8_t* packed, uint8_t* canonical, int64_t n_blobs);
}  // namespace strata
