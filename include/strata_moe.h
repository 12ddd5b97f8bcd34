/* strata_moe.h -- C ABI of the GB300 (sm_103a) routed-expert MoE block.
 *
 * The block (one layer of a 48-layer, 512-expert, top-10 model; H = 2560, FF = 640):
 *   1. router logits   l[t][e] = sum_h x[t][h] * Wr[e][h] (+ bias[e])            (BF16 GEMV/GEMM)
 *   2. top-10           softmax over E, stable descending order, first 10, renormalised
 *   3. grouping         pairs (t, k) counting-sorted by expert
 *   4. expert FFN       y = down(silu(gate x) * (up x)) with Q2_0 weights dequantised in-kernel
 *   5. combine          out[t] = sum_k w[t][k] * y[t][k]   (+ x[t] for residual layers)
 * Sources, by page title and section:
 *   - zwxr.cn news/242664 "MoE 遇上消费级显卡", section "一次路由的完整旅程": moe_route's BF16 GEMV
 *     (project_bf16) to 512 logits, native_router_top10 (softmax over all 512, stable descending
 *     argsort, gather, renormalise with ggml's lower clamp -> ids[10], weights[10]), the grouped
 *     expert kernel, and moe_combine.
 *   - ai.thesatyajit.com "Strata engine", section "The byte budget, in code": H = 2560, FF = 640,
 *     QK = 64, blob = 3 * H*FF*18/64 = 1,382,400 bytes; section "The CPU kernels": Q2_0 codes
 *     {0,1,2,3} mean {-1,0,1,2} x scale, and the in-block bit order of unpack64_q2_0.
 *   - momoyeyu.github.io "ai-infra-strata", section "提示词处理": tokens gathered per expert so one
 *     weight read serves several tokens; the dequantisation is fused into the matrix kernel.
 *   - The SwiGLU form and the rmsnorm residual stack come from the benchmark statement of the block.
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers owned by the caller unless marked "host".  The library never
 *     allocates or frees device memory; scratch lives in the caller's workspace `ws`.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only enqueue work; they
 *     return before it runs and do not synchronise, except strata_poll_status and the two
 *     host-buffer calls (strata_moe_layer_host, strata_moe_stack_host).
 *   - Arguments checkable on the host are checked first; a bad one returns an error and enqueues
 *     nothing.  T == 0 is a valid empty call (returns STRATA_OK, enqueues nothing).
 *   - Conditions only the device can see (an expert id >= E, a bounded wait that expired) set
 *     bits in a status word inside `ws`; read it with strata_poll_status.  Kernels never trap.
 *   - fp32 tensors are row-major and 16-byte aligned; ws must be 256-byte aligned and initialised
 *     once with strata_moe_workspace_init before first use; afterwards every call leaves it
 *     reusable.  Two calls that share a ws must not overlap in time (same stream, or ordered).
 *
 * Packed expert blob ("GPU layout", written by strata_pack_q2_0*; same 1,382,400 bytes as the
 * canonical blob; every piece starts on a 16-byte boundary when the blob is 256-byte aligned):
 *   canonical: gate [640][2560], up [640][2560], down [2560][640], each row-major, as Q2_0 blocks of
 *     64 consecutive weights {fp16 d, 16 code bytes}; weight i of a block in code byte i/4 at bits
 *     2*(i%4); value d * (c - q2_offset).
 *   packed gate/up region, bytes [0, 921600): for slab s = 0..39 (rows 16*s .. 16*s + 15 of gate and
 *     up), for k-block kb = 0..39, a 576-byte piece at (s*40 + kb)*576:
 *        [0, 256)     gate codes of the slab's 16 rows, 16 bytes per row, row order
 *        [256, 512)   up codes, same order
 *        [512, 576)   per row r: {fp16 gate d, fp16 up d} at 512 + 4*r
 *     so one slab (all 40 k-blocks, 23,040 bytes) is contiguous, and the 8 pieces of one k-block of
 *     a 128-row tile sit 23,040 bytes apart.
 *   packed down region, bytes [921600, 1382400): for row tile rt = 0..19, kb = 0..9, a 2304-byte
 *     chunk at 921600 + (rt*10 + kb)*2304: [0, 2048) codes of 128 rows, [2048, 2304) fp16 d per row.
 *   Code bytes keep the canonical in-block order.
 */
#ifndef STRATA_MOE_H_
#define STRATA_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define STRATA_MOE_H 2560
#define STRATA_MOE_FF 640
#define STRATA_MOE_E_MAX 512
#define STRATA_MOE_K 10
#define STRATA_MOE_QK 64
#define STRATA_MOE_BLOB_BYTES 1382400
#define STRATA_MOE_T_MAX 8192 /* the pages' largest prefill chunk (8,192 tokens) */

/* strata_moe_layer flags */
#define STRATA_MOE_RESIDUAL_RMSNORM 1 /* out = x + moe(rmsnorm(x)), rmsnorm(x) = x / sqrt(mean(x^2) + 1e-6) */

typedef enum strata_status {
  STRATA_OK = 0,
  STRATA_E_INVAL = -1,       /* null pointer, size out of range, bad enum value */
  STRATA_E_ALIGN = -2,       /* a pointer or stride breaks the alignment rule of its argument */
  STRATA_E_UNSUPPORTED = -3, /* a shape the library does not implement */
  STRATA_E_CUDA = -4,        /* a CUDA runtime call (launch, copy) failed */
  STRATA_E_TIMEOUT = -5,     /* a bounded device-side wait expired (device status) */
  STRATA_E_WORKSPACE = -6,   /* ws_bytes smaller than strata_moe_workspace_bytes(T) */
  STRATA_E_CORRUPT = -7      /* the device saw invalid data, e.g. an expert id >= E (device status) */
} strata_status;

/* The experts of one layer. */
typedef struct strata_experts {
  const void* blobs;   /* device: expert e's packed blob at blobs + e * blob_stride; 256-byte aligned */
  int64_t blob_stride; /* bytes; multiple of 256 and >= STRATA_MOE_BLOB_BYTES */
  int32_t n_expert;    /* E: experts routed over; multiple of 32 in [32, 512] */
  int32_t q2_offset;   /* 1: codes {0,1,2,3} = {-1,0,1,2} x d (the pages); 2: the c-2 reading */
  /* device, nullable: the layer's shared expert, a packed blob (256-byte aligned) of the same shape and
   * format.  wayneh.tw "strata-local-moe-inference" lists a shared expert that runs on the GPU for every
   * token; the pages give neither its width nor a gate, so it is read as an expert of the routed
   * experts' shape whose output on the same input is added with weight 1 to the routed experts'
   * weighted sum (strata_moe_layer, strata_moe_stack and the host-buffer calls; strata_moe_experts
   * computes the routed pairs only and ignores it).  NULL: no shared expert. */
  const void* shared_blob;
} strata_experts_t;

/* Bytes of workspace a call with T tokens needs (any entry point below). */
size_t strata_moe_workspace_bytes(int32_t T);

/* Zero the workspace's counters, status word and call epoch and, when ws_bytes covers it (any
 * workspace sized for T >= 1), the decode path's exchange area, whose 64-bit words carry the tag of
 * the call that wrote them (enqueued on stream).  Call once after allocating, with the size the calls
 * will pass. */
strata_status strata_moe_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Steps 1-2. x fp32 [T][2560] (the router input, already normalised if the layer normalises);
 * w_router bf16 bit patterns [E][2560]; bias fp32 [E] or NULL; E = n_expert (multiple of 32 in
 * [32, 512]).  Outputs: ids int32 [T][10] in descending probability (equal probabilities: lower
 * id first), weights fp32 [T][10] = p / max(sum of the 10 p, 2^-14); logits fp32 [T][E] or NULL
 * (includes the bias).  Logits accumulate in fp32. */
strata_status strata_moe_route(const float* x, int32_t T, const uint16_t* w_router, const float* bias,
                               int32_t n_expert, int32_t* ids, float* weights, float* logits, void* ws,
                               size_t ws_bytes, void* stream);

/* Step 3. ids int32 [T][10] -> expert_off int32 [E+1] (exclusive prefix of per-expert counts),
 * pair int32 [T*10]: pair numbers p = t*10 + k sorted by expert, ascending p within an expert;
 * active int32 [E]: experts with >= 1 pair in increasing id (entries past n_active undefined);
 * n_active int32 [1].  An id outside [0, E) sets STRATA_E_CORRUPT in the status word and that
 * pair is dropped. */
strata_status strata_moe_group(const int32_t* ids, int32_t T, int32_t n_expert, int32_t* expert_off,
                               int32_t* pair, int32_t* active, int32_t* n_active, void* ws,
                               size_t ws_bytes, void* stream);

/* Step 3 without a caller workspace (this entry point has no counterpart on the pages).
 * Some callers cannot call cudaMalloc at all: code running inside an engine whose device memory
 * belongs to its own pool or to another runtime, or a process that must not grow its device
 * footprint after start-up.  This call takes the same inputs and writes the same outputs as
 * strata_moe_group (bit for bit), but its scratch -- the per-chunk expert histograms -- is a fixed
 * array of STRATA_MOE_GROUP_NOALLOC_SCRATCH_BYTES (256 KiB) in the library's own device memory, so it
 * allocates nothing and takes no ws.
 *   - The array is sized for the largest T the ABI allows; T outside [0, STRATA_MOE_T_MAX] returns
 *     STRATA_E_INVAL.
 *   - Every GPU that loads the library holds the array until the process exits.  The first call on
 *     a device looks up the array's device address (with that device current) and caches it, so
 *     make that first call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents (every word a call reads
 *     it first writes, so nothing has to be cleared): calls whose GPU work overlaps -- other streams,
 *     other host threads -- race on it; order them.
 *   - There is no device status word: an id outside [0, E) drops its pair, which shows as
 *     expert_off[E] < T*10. */
#define STRATA_MOE_GROUP_NOALLOC_SCRATCH_BYTES (256 * 1024)
strata_status strata_moe_group_noalloc(const int32_t* ids, int32_t T, int32_t n_expert, int32_t* expert_off,
                                       int32_t* pair, int32_t* active, int32_t* n_active, void* stream);

/* Step 4. For every pair p = t*10 + k listed by the grouping: parts[p][:] = expert(x[t]) with the
 * expert that owns p.  x fp32 [T][2560]; grouping arrays as strata_moe_group writes them; parts
 * fp32 [T][10][2560].  Weights are the packed blobs of ex (host pointer to the struct).  Computed
 * as grouped tensor-core GEMMs (x rounded to fp16, fp32 accumulation) for every T.  The grouping
 * arrays are checked on the device before any expert work: an active entry naming an expert outside
 * [0, n_expert) or a slot range outside [0, T*10), or active entries that are not strictly increasing
 * or whose slot ranges are out of order or overlap, set STRATA_E_CORRUPT and the call computes nothing
 * (parts keeps its contents); a pair number outside [0, T*10) sets STRATA_E_CORRUPT and that slot is
 * skipped. */
strata_status strata_moe_experts(const strata_experts_t* ex, const float* x, int32_t T,
                                 const int32_t* expert_off, const int32_t* pair, const int32_t* active,
                                 const int32_t* n_active, float* parts, void* ws, size_t ws_bytes,
                                 void* stream);

/* Step 5. out[t][h] = (residual ? residual[t][h] : 0) + (sum over k = 0..9, in order, of
 * weights[t][k] * parts[t][k][h]).  residual may be NULL; out may alias residual. */
strata_status strata_moe_combine(const float* parts, const float* weights, int32_t T,
                                 const float* residual, float* out, void* stream);

/* Steps 1-5 for one layer. flags = 0: out = moe(x); flags = STRATA_MOE_RESIDUAL_RMSNORM: out =
 * x + moe(rmsnorm(x)) with router and experts both reading rmsnorm(x).  out may alias x.  ids /
 * weights (nullable) receive the routing.  Workspace as for any call with T tokens.
 * With ex->shared_blob, the shared expert's output (weight 1) is added to the routed experts' weighted
 * sum before the residual.
 * Summation order: for T <= 8 the ten weighted expert outputs of a token are added in k order (then
 * the shared expert's) and repeated calls give the same bits.  For T > 8 the combine is fused into the down projection: out is
 * first set to x (residual layers) or 0, and each expert's weighted output is added into it with fp32
 * atomic additions as the expert finishes, so the order of a token's ten additions -- and the last
 * bits of out -- can differ from call to call (the routing, computed before, does not). */
strata_status strata_moe_layer(const strata_experts_t* ex, const uint16_t* w_router, const float* bias,
                               const float* x, int32_t T, int32_t flags, float* out, int32_t* ids,
                               float* weights, void* ws, size_t ws_bytes, void* stream);

/* n_layers residual layers in sequence on x (in place): x <- x + moe_l(rmsnorm(x)).
 * ex: host array [n_layers]; w_router: device bf16 [n_layers][E][2560]; bias: device fp32
 * [n_layers][E] or NULL; ids / weights (nullable): device [n_layers][T][10]. */
strata_status strata_moe_stack(const strata_experts_t* ex, const uint16_t* w_router, const float* bias,
                               int32_t n_layers, float* x, int32_t T, int32_t* ids, float* weights,
                               void* ws, size_t ws_bytes, void* stream);

/* strata_moe_layer for activations in HOST memory: x_host (host, fp32 [T][2560]) is copied into the
 * workspace's I/O area, the layer runs there exactly as strata_moe_layer runs it (same kernels, same
 * results bit for bit), the output is copied to out_host (host, fp32 [T][2560]), and the call returns
 * after synchronising `stream`, so out_host holds the result on return.  ids / weights (nullable) are
 * DEVICE arrays as for strata_moe_layer.  x_host and out_host must not overlap (STRATA_E_INVAL).
 *   - Page-locked host buffers (cudaHostAlloc / cudaHostRegister) with a device mapping and 16-byte
 *     alignment are reached through that mapping: x_host is read by a copy kernel, and a decode layer
 *     (T <= 8) stores its output straight into out_host while a prefill layer computes it in the
 *     workspace and a copy kernel writes it out.  Each buffer must lie within one page-locked
 *     allocation or registration (its first and last bytes are checked).  Pageable or unaligned
 *     buffers go through the copy engines.
 *   - When x_host and out_host are page-locked and `stream` is not the legacy default stream, the
 *     first call captures copy-in, layer and copy-out as one CUDA graph and later calls with the same
 *     arguments (every pointer and size, flags, stream, current device and the fields of *ex) replay
 *     it: one graph launch per call.  Up to 16 graphs are kept per process, the least recently used
 *     dropped.  Otherwise (pageable buffers, the default stream, or event timing armed by
 *     strata_moe_profile_arm) the steps are enqueued one by one.
 *   - The host buffers are read and written by the GPU during the call only; their contents may
 *     change freely between calls, as may every device array's contents.
 *   - Must not be called while `stream` is being captured: returns STRATA_E_INVAL.
 *   - Workspace as for strata_moe_layer (strata_moe_workspace_bytes includes the I/O area); calls
 *     sharing a workspace must not overlap in time. */
strata_status strata_moe_layer_host(const strata_experts_t* ex, const uint16_t* w_router, const float* bias,
                                    const float* x_host, int32_t T, int32_t flags, float* out_host, int32_t* ids,
                                    float* weights, void* ws, size_t ws_bytes, void* stream);

/* strata_moe_stack for activations in HOST memory: x_host (host, fp32 [T][2560]) is copied in, the
 * n_layers residual layers run as in strata_moe_stack, the result is copied back into x_host, and the
 * call returns after synchronising `stream`.  Graph capture and replay, workspace and errors as for
 * strata_moe_layer_host (the key includes all n_layers descriptors of ex). */
strata_status strata_moe_stack_host(const strata_experts_t* ex, const uint16_t* w_router, const float* bias,
                                    int32_t n_layers, float* x_host, int32_t T, int32_t* ids, float* weights,
                                    void* ws, size_t ws_bytes, void* stream);

/* Failure-detection self-test (no counterpart on the pages).  Every wait in the library's kernels is
 * bounded: past a limit (2 s) it records STRATA_E_TIMEOUT in the workspace's status word and the
 * kernel returns instead of hanging.  This call runs the decode layer's two kinds of wait -- a poll of
 * an exchange word for a tag, and an mbarrier phase -- in one CTA on conditions that never hold, with
 * the limit limit_ns (in [1000, 2e9]), so both expire: afterwards strata_poll_status returns
 * STRATA_E_TIMEOUT, strata_clear_status clears it, and the context stays usable.  Uses the first 8
 * bytes of the workspace's logits area as the never-written word (set to 0 first); ws as for T = 1.
 * Enqueued on stream; takes about 2 x limit_ns on the device. */
strata_status strata_moe_wait_selftest(void* ws, size_t ws_bytes, uint64_t limit_ns, void* stream);

/* Blob checksums, for verifying an upload or a device pack against the bytes it came from.
 * zwxr.cn news/242664, section "与静态 offload 方案的本质差异": every expert slot is read back and
 * checked after it is filled, and the engine refuses to run when a check fails.  The checksum is the
 * common CRC-32 (IEEE 802.3 polynomial, reflected, preset and final inversion all ones: the value
 * zlib's crc32 gives) of each blob's STRATA_MOE_BLOB_BYTES bytes; blob j starts at blobs + j*stride,
 * stride >= STRATA_MOE_BLOB_BYTES.  Host: blobs and crc [n_blobs] are host memory.  Device: blobs in
 * device memory (256-byte aligned, stride a multiple of 256), crc a device array [n_blobs] written
 * on stream, one CTA per blob.  n_blobs == 0 is an empty call. */
strata_status strata_blob_crc32(const uint8_t* blobs, int64_t stride, int64_t n_blobs, uint32_t* crc);
strata_status strata_blob_crc32_device(const void* blobs, int64_t stride, int64_t n_blobs, uint32_t* crc,
                                       void* stream);

/* Canonical -> packed blob layout, host memory (host pointers), n_blobs consecutive blobs of
 * STRATA_MOE_BLOB_BYTES each.  Pure byte permutation; src and dst must not overlap. */
strata_status strata_pack_q2_0(const uint8_t* canonical, uint8_t* packed, int64_t n_blobs);

/* Packed -> canonical, host memory: the inverse of strata_pack_q2_0. */
strata_status strata_unpack_q2_0(const uint8_t* packed, uint8_t* canonical, int64_t n_blobs);

/* Canonical -> packed on the device: blob j from canonical + j*src_stride to packed +
 * j*dst_stride (dst_stride multiple of 256, dst 256-byte aligned, src 2-byte aligned). */
strata_status strata_pack_q2_0_device(const uint8_t* canonical, int64_t src_stride, uint8_t* packed,
                                      int64_t dst_stride, int64_t n_blobs, void* stream);

/* Synchronise stream, read and return the workspace status word (STRATA_OK if no device-side
 * error was recorded since the last strata_moe_workspace_init or strata_clear_status). */
strata_status strata_poll_status(const void* ws, void* stream);

/* Reset the workspace status word (enqueued on stream). */
strata_status strata_clear_status(void* ws, void* stream);

/* Static string naming a status code. */
const char* strata_status_str(strata_status s);

/* ---- Diagnostics: launch accounting and kernel timing -------------------------------------------
 * Not part of the method: these let a caller measure the library's kernels with its own CUDA events.
 * Kernel ids (every kernel the library launches): */
#define STRATA_KERNEL_DECODE_LAYER 0   /* whole layer for T <= 8, one cooperative launch */
#define STRATA_KERNEL_ROUTE_DECODE 1   /* router GEMV + top-10 + grouping, T <= 8 (strata_moe_route) */
#define STRATA_KERNEL_ROUTER_PREP 2    /* bf16 hi/lo copies of x for the router GEMM (and 1/rms), T > 8; in a layer call
                                          also the experts' fp16 token copy and the output's initial value
                                          (strata_moe_experts: the fp16 token copy alone) */
#define STRATA_KERNEL_ROUTER_TC 3      /* router GEMM on the tensor cores, T > 8 */
#define STRATA_KERNEL_TOP_K 4
#define STRATA_KERNEL_GROUP_HIST 5
#define STRATA_KERNEL_GROUP_SCAN 6
#define STRATA_KERNEL_GROUP_SCATTER 7
#define STRATA_KERNEL_TC_PREPARE 8     /* tile list of the tensor-core expert path */
#define STRATA_KERNEL_TC_GATHER 9      /* fp16 token gather per expert */
#define STRATA_KERNEL_TC_GATEUP 10     /* Q2_0 gate/up + SwiGLU grouped GEMM (tcgen05) */
#define STRATA_KERNEL_TC_DOWN 11       /* Q2_0 down grouped GEMM (tcgen05); in a layer call also the combine */
#define STRATA_KERNEL_COMBINE 12       /* strata_moe_combine */
#define STRATA_KERNEL_PACK 13
#define STRATA_KERNEL_HOST_COPY 14     /* copy between page-locked host memory and the workspace (host-buffer calls) */
#define STRATA_KERNEL_WAIT_SELFTEST 15 /* strata_moe_wait_selftest */
#define STRATA_KERNEL_BLOB_CRC32 16    /* strata_blob_crc32_device */
#define STRATA_KERNEL_COUNT 17

/* Number of kernels this process has launched through the library so far (all threads). */
uint64_t strata_moe_launch_count(void);

/* Arm event timing of one kernel for the calling host thread: of the launches of kernel `kernel` made
 * from this thread after this call, the first `skip` are not recorded and the next n record
 * start_events[i] on the launch's stream just before launch i and stop_events[i] just after it
 * (cudaEventRecord; i = 0 .. n-1), so cudaEventElapsedTime(start_events[i], stop_events[i]) is that
 * launch's duration on the device.  The arrays are host arrays of cudaEvent_t handles owned by the
 * caller; the library keeps the two array pointers (not copies) until it is re-armed or disarmed, so
 * they must stay valid until then.  n == 0 disarms.  Not meant for stream capture (event records in a
 * captured stream are ordering nodes, not timestamps).  Returns STRATA_E_INVAL for a bad kernel id,
 * skip < 0, n < 0, or NULL arrays with n > 0. */
strata_status strata_moe_profile_arm(int32_t kernel, int32_t skip, void* const* start_events, void* const* stop_events,
                                     int32_t n);

/* How many launches of `kernel` were recorded since it was last armed (calling thread); -1 for a bad id. */
int32_t strata_moe_profile_recorded(int32_t kernel);

#ifdef __cplusplus
}
#endif
#endif /* STRATA_MOE_H_ */
