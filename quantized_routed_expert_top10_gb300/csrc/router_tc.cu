// Router logits for prefill chunks on the tensor cores (tcgen05), sm_103a.
//
// zwxr.cn news/242664, section "一次路由的完整旅程": moe_route projects the normalised activation
// with a BF16 projection to 512 expert logits.  For a chunk of T tokens this is the GEMM
//   logits[T][E] = X[T][2560] * Wr[E][2560]^T (+ bias),
// run with the router rows (bf16, exact) as A (M = 128 experts) and the tokens as B (N = 128), so
// the accumulator's TMEM lanes are experts and the epilogue's stores are coalesced along experts.
// A prep pass writes x (times the token's 1/rms for residual layers) as two bf16 matrices,
// x_hi = bf16(x) and x_lo = bf16(x - x_hi); both products accumulate into the same fp32 TMEM
// accumulator, so each term carries x to about 16 significant bits (relative error ~2^-17).
// The x_hi and x_lo tiles of a k-block lie one after the other in shared memory, so together they are
// one 256-row operand: a single MMA (N = 256) takes both products, x_hi's into accumulator columns
// [0, 128) and x_lo's into [128, 256).  A CTA covers 128 tokens and ET 128-row tiles of router rows
// against the one token operand, with one accumulator of 256 columns per expert tile: two tiles when
// that still gives every SM a CTA (each token tile is then read once per 256 experts), else one.
// The contraction is split two ways over CTAs (ROUTER_KSPLIT; 1,280 columns each); a CTA writes
// x_hi's + x_lo's product to its slice of the partial-logit buffer and the top-k kernel adds the
// slices in a fixed order (and the bias), so results do not depend on scheduling.  The tensor core's
// fp32 accumulation over 80 steps keeps the error on a logit (~1e-5) far below the 1e-4 band within
// which tied logits may order either way.
// Pipeline: one thread streams the 2 + ET 128 x 64 operand tiles of each k-block with TMA (tensor
// maps, 128-byte swizzle) into a ring of stages, one thread issues the MMAs, four warps drain TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "tc_common.cuh"

namespace strata {

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
bool make_tensor_map_2d(void* map, int dtype, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride,
                        uint32_t box_inner, uint32_t box_rows) {
  using EncodeTiled = PFN_cuTensorMapEncodeTiled_v12000;
  static EncodeTiled fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<EncodeTiled>(p);
  }
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_stride};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return fn(reinterpret_cast<CUtensorMap*>(map), (CUtensorMapDataType)dtype, 2, const_cast<void*>(base), dims,
            strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

constexpr int RT_T = 128;  // tokens per tile (MMA N)
constexpr int RT_E = 128;  // experts per tile (MMA M)
constexpr int RT_THREADS = 128;
constexpr uint32_t RT_TILE = 128 * 128;  // 128 rows x 64 bf16
template <int ET>
struct RtGeo {  // ET expert tiles per CTA
  static constexpr uint32_t STAGE = (2 + ET) * RT_TILE;  // x_hi, x_lo, then the router rows of each tile
  static constexpr int NS = ET == 1 ? 4 : 3;              // ring stages
  static constexpr size_t SMEM = (size_t)NS * STAGE + 1024;
};
constexpr int RT_KBS = KB_GU / ROUTER_KSPLIT;  // k-blocks per CTA
static_assert(KB_GU % ROUTER_KSPLIT == 0 && RT_KBS % 2 == 0, "even split of the contraction");

__host__ __device__ __forceinline__ uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// 2-D tiled TMA load of box {64 elements, 128 rows} at (k0, row0), completing on bar.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int k0, int row0, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(k0), "r"(row0), "r"(smem_u32(bar))
      : "memory");
}

// x (fp32 [T][H]) -> x_hi, x_lo (bf16 [T][H]), times 1/rms(x[t]) when inv_rms is non-null (which then
// also receives the factors).  For a layer call also x16 (the expert path's fp16 token copy, same
// scaling) and out = x (residual layers, skipped when out is x itself) or 0: the down kernel adds the
// experts' weighted outputs into it.  One warp per token row; every read of the row precedes the
// warp's stores to out, so out may be x.
__global__ void __launch_bounds__(256) router_prep_kernel(const float* x, int T, __nv_bfloat16* __restrict__ xh,
                                                          __nv_bfloat16* __restrict__ xl,
                                                          float* __restrict__ inv_rms, uint8_t* __restrict__ x16,
                                                          float* out) {
  griddep_launch_dependents();
  griddep_wait();
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= T) return;
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)t * H);
  float4* orow = out ? reinterpret_cast<float4*>(out + (size_t)t * H) : nullptr;
  const bool init_out = out && (!inv_rms || out != x);
  constexpr int PER = H / 4 / 32;  // 20 float4 per lane
  float sc = 1.f;
  if (inv_rms) {
    float ss = 0.f;
#pragma unroll 4
    for (int i = 0; i < PER; ++i) {
      const float4 v = xr[lane + 32 * i];
      ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
    ss = warp_sum(ss);
    sc = 1.f / sqrtf(ss / (float)H + 1e-6f);
    if (lane == 0) inv_rms[t] = sc;
  }
#pragma unroll 4
  for (int i = 0; i < PER; ++i) {
    const float4 v = xr[lane + 32 * i];  // read before this lane's store to the same float4 of out
    const float f[4] = {v.x * sc, v.y * sc, v.z * sc, v.w * sc};
    __nv_bfloat16 hi[4], lo[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      hi[q] = __float2bfloat16_rn(f[q]);
      lo[q] = __float2bfloat16_rn(f[q] - __bfloat162float(hi[q]));  // the difference is exact in fp32
    }
    const size_t o = (size_t)t * H + 4 * (lane + 32 * i);
    *reinterpret_cast<uint2*>(xh + o) = *reinterpret_cast<const uint2*>(hi);
    *reinterpret_cast<uint2*>(xl + o) = *reinterpret_cast<const uint2*>(lo);
    if (x16) tc::x16_store_chunk(v, i, sc, t, T, x16);
    if (init_out) orow[lane + 32 * i] = inv_rms ? v : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

template <int ET>
__global__ void __launch_bounds__(RT_THREADS, 1) router_tc_kernel(const __grid_constant__ CUtensorMap map_xh,
                                                                  const __grid_constant__ CUtensorMap map_xl,
                                                                  const __grid_constant__ CUtensorMap map_wr, int T,
                                                                  int E, float* __restrict__ parts, int* status) {
  constexpr int RT_ET = ET, RT_NS = RtGeo<ET>::NS;
  constexpr uint32_t RT_STAGE = RtGeo<ET>::STAGE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[RT_NS], empty[RT_NS], done;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * RT_T, e0 = blockIdx.y * RT_E * RT_ET;
  const int kb0 = blockIdx.z * RT_KBS;
  griddep_launch_dependents();
  if (warp == 2) tc::tmem_alloc(&tmem_base, 512);
  if (tid == 0) {
    for (int s = 0; s < RT_NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
    fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  griddep_wait();  // x_hi / x_lo come from the prep kernel
  const uint32_t tmem = tmem_base;
  bool ok = true;
  if (tid == 0) {
    // ---- producer: three TMA tiles per k-block ----
    int kbl = 0;
    for (; kbl < RT_KBS; ++kbl) {
      const int s = kbl % RT_NS;
      if (kbl >= RT_NS && !mbar_wait(&empty[s], (uint32_t)((kbl / RT_NS - 1) & 1), status)) {
        ok = false;
        break;
      }
      uint8_t* st = smem + (size_t)s * RT_STAGE;
      const int k = (kb0 + kbl) * QK;
      mbar_expect_tx(&full[s], RT_STAGE);
      tma_load_2d(st, &map_xh, k, t0, &full[s]);
      tma_load_2d(st + RT_TILE, &map_xl, k, t0, &full[s]);
#pragma unroll
      for (int j = 0; j < RT_ET; ++j)  // rows past E read as zeros
        tma_load_2d(st + (2 + j) * RT_TILE, &map_wr, k, e0 + j * RT_E, &full[s]);
    }
    for (int back = 1; back <= RT_NS && back <= kbl; ++back)  // copies still in flight after a failure
      mbar_wait(&full[(kbl - back) % RT_NS], (uint32_t)(((kbl - back) / RT_NS) & 1), status);
  } else if (tid == 32) {
    // ---- MMA issuer ----
    const uint32_t idesc = idesc_bf16_f32(RT_E, 2 * RT_T);  // N: the tile's tokens as x_hi, then as x_lo
    for (int kbl = 0; kbl < RT_KBS; ++kbl) {
      const int s = kbl % RT_NS;
      if (!mbar_wait(&full[s], (uint32_t)((kbl / RT_NS) & 1), status)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint8_t* st = smem + (size_t)s * RT_STAGE;
      const uint64_t bx = tc::smem_desc_sw128(smem_u32(st));  // x_hi rows, then x_lo rows
      const uint64_t bd = tc::smem_desc_sw128(smem_u32(st + 2 * RT_TILE));
      // the expert tiles' MMAs alternate, so each accumulator's next MMA never waits on its last
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int j = 0; j < RT_ET; ++j)
          tc::mma_f16(tmem + (uint32_t)(j * 2 * RT_T), bd + (uint64_t)((j * RT_TILE) >> 4) + 2 * kk, bx + 2 * kk, idesc,
                      (kbl > 0 || kk > 0) ? 1u : 0u);
      tc::mma_commit(&empty[s]);
    }
    tc::mma_commit(&done);  // after every MMA this thread issued
  }
  // ---- epilogue: warps 0..3 own TMEM lane quadrants = expert rows; columns are tokens.  Each 4 x 4
  // block of (experts, tokens) is transposed across 4 lanes, so lane 4g + j stores experts 4g .. 4g + 3
  // of token j as one 16-byte store (experts past E land in the row's unused tail: rows hold EMAX) ----
  __syncwarp();
  ok = mbar_wait(&done, 0u, status) && ok;
  tc::fence_after_sync();
  const int j4 = lane & 3;
#pragma unroll 1
  for (int c = 0; c < RT_ET * (RT_T / 16); ++c) {
    const int j = c / (RT_T / 16), ch = c % (RT_T / 16);  // expert tile, 16-token chunk
    const int e4 = e0 + j * RT_E + 32 * warp + 4 * (lane >> 2);
    float hi[16], lo[16];
    const uint32_t acc = tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(j * 2 * RT_T + 16 * ch);
    tc::tmem_ld16(acc, hi);
    tc::tmem_ld16(acc + RT_T, lo);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      uint32_t a[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = __float_as_uint(hi[4 * m + i] + lo[4 * m + i]);
      tc::transpose4_lanes(a, j4);
      const int t = t0 + 16 * ch + 4 * m + j4;
      if (ok && e4 < E && t < T)
        *reinterpret_cast<uint4*>(parts + ((size_t)blockIdx.z * T + t) * EMAX + e4) = make_uint4(a[0], a[1], a[2], a[3]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tc::tmem_dealloc(tmem, 512);
    tc::tmem_relinquish();
  }
}

// Tensor map of a row-major bf16 matrix [rows][H]: boxes of 64 columns x 128 rows, 128-byte swizzle,
// rows past the end read as zeros.
bool make_map(CUtensorMap* m, const void* base, int rows) {
  return make_tensor_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, H, rows, (uint64_t)H * 2, 64, 128);
}

int g_rt_attr[64];  // per device: dynamic shared memory set; multiprocessor count
int g_rt_sms[64];

}  // namespace

cudaError_t launch_router_tc(const float* x, float* inv_rms, int T, const uint16_t* w_router, int E, void* xbf,
                             float* parts, int* status, cudaStream_t s, uint8_t* x16, float* out) {
  __nv_bfloat16* xh = reinterpret_cast<__nv_bfloat16*>(xbf);
  __nv_bfloat16* xl = xh + (size_t)T * H;
  STRATA_LAUNCH(KID_ROUTER_PREP, s,
                launch_pdl(router_prep_kernel, (T + 7) / 8, 256, 0, s, x, T, xh, xl, inv_rms, x16, out));
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  CUtensorMap mh, ml, mw;
  if (!make_map(&mh, xh, T) || !make_map(&ml, xl, T) || !make_map(&mw, w_router, E)) return cudaErrorInvalidValue;
  int dev = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  int sms = (dev >= 0 && dev < 64) ? g_rt_sms[dev] : 0;
  if (sms == 0) {
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
    if (dev >= 0 && dev < 64) g_rt_sms[dev] = sms;
  }
  if (dev < 0 || dev >= 64 || !g_rt_attr[dev]) {
    if ((err = cudaFuncSetAttribute(router_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)RtGeo<1>::SMEM)) != cudaSuccess ||
        (err = cudaFuncSetAttribute(router_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)RtGeo<2>::SMEM)) != cudaSuccess)
      return err;
    if (dev >= 0 && dev < 64) g_rt_attr[dev] = 1;
  }
  const int tt = (T + RT_T - 1) / RT_T;
  const int et2 = (E + 2 * RT_E - 1) / (2 * RT_E);
  if (tt * et2 * ROUTER_KSPLIT >= sms) {  // two expert tiles per CTA still give every SM a CTA
    dim3 grid(tt, et2, ROUTER_KSPLIT);
    STRATA_LAUNCH(KID_ROUTER_TC, s, launch_pdl(router_tc_kernel<2>, grid, RT_THREADS, RtGeo<2>::SMEM, s, mh, ml, mw, T, E,
                                               parts, status));
  } else {
    dim3 grid(tt, (E + RT_E - 1) / RT_E, ROUTER_KSPLIT);
    STRATA_LAUNCH(KID_ROUTER_TC, s, launch_pdl(router_tc_kernel<1>, grid, RT_THREADS, RtGeo<1>::SMEM, s, mh, ml, mw, T, E,
                                               parts, status));
  }
  return cudaGetLastError();
}

}  // namespace strata
