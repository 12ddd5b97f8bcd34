// Router logits for prefill chunks on the tensor cores (tcgen05), sm_103a.
//
// zwxr.cn news/242664, section "一次路由的完整旅程": moe_route projects the normalised activation
// with a BF16 projection to 512 expert logits.  For a chunk of T tokens this is the GEMM
//   logits[T][E] = X[T][2560] * Wr[E][2560]^T (+ bias),
// run with the router rows (bf16, exact) as A (M = 128 experts) and the tokens as B (N = 128), so
// the accumulator's TMEM lanes are experts and the epilogue's stores are coalesced along experts.  The fp32 activations (times the
// token's 1/rms for residual layers) are split into bf16 x_hi = bf16(x) and x_lo = bf16(x - x_hi);
// both products accumulate into the same fp32 TMEM accumulator, so each term carries x to about 16
// significant bits (relative error ~2^-17).
// The contraction is split four ways over CTAs (ROUTER_KSPLIT; 640 columns each) and, inside a CTA,
// in two halves accumulated in separate TMEM columns; the CTA writes the sum of its two halves to
// its own slice of the partial-logit buffer and the top-k kernel adds the four slices in a fixed
// order (and the bias), so results do not depend on scheduling.  Short accumulation chains keep the
// tensor core's accumulation error (~1e-5 on a logit) far below the 1e-4 band within which tied
// logits may order either way.
// CTA tile: 128 tokens x 128 experts x 640 columns, 64-wide k-blocks double-buffered in
// 128B-swizzled shared memory, two CTAs per SM.
#include <cuda_bf16.h>

#include "tc_common.cuh"

namespace strata {
namespace {

constexpr int RT_T = 128;  // tokens per tile (MMA N)
constexpr int RT_E = 128;  // experts per tile (MMA M)
constexpr int RT_THREADS = 256;
constexpr uint32_t RT_TILE = 128 * 128;  // 128 rows x 64 bf16
constexpr uint32_t RT_STAGE = 3 * RT_TILE;  // x_hi, x_lo, router rows
constexpr int RT_KBS = KB_GU / ROUTER_KSPLIT;  // k-blocks per CTA
static_assert(KB_GU % ROUTER_KSPLIT == 0 && RT_KBS % 2 == 0, "even split of the contraction");

__host__ __device__ __forceinline__ uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__global__ void __launch_bounds__(RT_THREADS, 2) router_tc_kernel(const float* __restrict__ x,
                                                                  const float* __restrict__ inv_rms, int T,
                                                                  const uint16_t* __restrict__ wr, int E,
                                                                  float* __restrict__ parts, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[2], empty[2], done;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * RT_T, e0 = blockIdx.y * RT_E;
  const int kb0 = blockIdx.z * RT_KBS;
  if (warp == 1) tc::tmem_alloc(&tmem_base, 256);
  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&full[s], 8);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
    fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t idesc = idesc_bf16_f32(RT_E, RT_T);
  const int r = tid >> 1, c0 = 4 * (tid & 1);  // loader: row r, chunks c0 .. c0 + 3
  const float scale = (inv_rms && t0 + r < T) ? __ldg(inv_rms + t0 + r) : 1.f;
  bool ok = true;
  for (int kbl = 0; kbl < RT_KBS; ++kbl) {
    const int kb = kb0 + kbl;
    const int s = kbl & 1;
    uint8_t* st = smem + s * RT_STAGE;
    if (kbl >= 2) ok = ok && mbar_wait(&empty[s], (uint32_t)((kbl / 2 - 1) & 1), status);
    if (ok) {
      // token row r as bf16 hi and lo parts (MMA operand B)
      const int t = t0 + r;
#pragma unroll
      for (int c = c0; c < c0 + 4; ++c) {
        float v[8];
        if (t < T) {
          const float4 a = __ldg(reinterpret_cast<const float4*>(x + (size_t)t * H + kb * QK + 8 * c));
          const float4 b = __ldg(reinterpret_cast<const float4*>(x + (size_t)t * H + kb * QK + 8 * c + 4));
          v[0] = a.x * scale; v[1] = a.y * scale; v[2] = a.z * scale; v[3] = a.w * scale;
          v[4] = b.x * scale; v[5] = b.y * scale; v[6] = b.z * scale; v[7] = b.w * scale;
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = 0.f;
        }
        __nv_bfloat16 hi[8], lo[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          hi[i] = __float2bfloat16_rn(v[i]);
          lo[i] = __float2bfloat16_rn(v[i] - __bfloat162float(hi[i]));  // the difference is exact in fp32
        }
        *reinterpret_cast<uint4*>(st + tc::swz_off(r, c)) = *reinterpret_cast<uint4*>(hi);
        *reinterpret_cast<uint4*>(st + RT_TILE + tc::swz_off(r, c)) = *reinterpret_cast<uint4*>(lo);
      }
      // router row e0 + r (MMA operand A)
      const int e = e0 + r;
#pragma unroll
      for (int c = c0; c < c0 + 4; ++c) {
        uint4 w = make_uint4(0, 0, 0, 0);
        if (e < E) w = __ldg(reinterpret_cast<const uint4*>(wr + (size_t)e * H + kb * QK + 8 * c));
        *reinterpret_cast<uint4*>(st + 2 * RT_TILE + tc::swz_off(r, c)) = w;
      }
    }
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&full[s]);
    if (tid == 0) {
      ok = ok && mbar_wait(&full[s], (uint32_t)((kbl / 2) & 1), status);
      tc::fence_after_sync();
      if (ok) {
        const uint64_t ah = tc::smem_desc_sw128(smem_u32(st));
        const uint64_t al = tc::smem_desc_sw128(smem_u32(st + RT_TILE));
        const uint64_t bd = tc::smem_desc_sw128(smem_u32(st + 2 * RT_TILE));
        const int half = kbl >= RT_KBS / 2;
        const uint32_t acc_tmem = tmem + (half ? (uint32_t)RT_T : 0u);
        const bool first = kbl == (half ? RT_KBS / 2 : 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          tc::mma_f16(acc_tmem, bd + 2 * kk, ah + 2 * kk, idesc, (!first || kk > 0) ? 1u : 0u);
          tc::mma_f16(acc_tmem, bd + 2 * kk, al + 2 * kk, idesc, 1u);
        }
      }
      tc::mma_commit(&empty[s]);
    }
  }
  if (tid == 0) tc::mma_commit(&done);
  // epilogue: warps 0..3 own TMEM lane quadrants = expert rows; columns are tokens, so a warp's
  // stores for one token cover 32 consecutive experts
  if (warp < 4) {
    ok = mbar_wait(&done, 0u, status) && ok;
    tc::fence_after_sync();
    const int e = e0 + 32 * warp + lane;
#pragma unroll 1
    for (int ch = 0; ch < RT_T / 16; ++ch) {
      float v[16], v2[16];
      tc::tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + 16 * ch, v);
      tc::tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + RT_T + 16 * ch, v2);
      if (ok && e < E) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int t = t0 + 16 * ch + i;
          if (t < T) parts[((size_t)blockIdx.z * T + t) * EMAX + e] = v[i] + v2[i];
        }
      }
    }
  } else if (tid == 128) {
    mbar_wait(&done, 0u, status);  // every MMA has finished before TMEM is released
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::tmem_dealloc(tmem, 256);
    tc::tmem_relinquish();
  }
}

}  // namespace

cudaError_t launch_router_tc(const float* x, const float* inv_rms, int T, const uint16_t* w_router, int E,
                             float* parts, int* status, cudaStream_t s) {
  const size_t smem = 2 * RT_STAGE + 1024;
  cudaError_t err = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  dim3 grid((T + RT_T - 1) / RT_T, (E + RT_E - 1) / RT_E, ROUTER_KSPLIT);
  STRATA_LAUNCH(KID_ROUTER_TC, s,
                router_tc_kernel<<<grid, RT_THREADS, smem, s>>>(x, inv_rms, T, w_router, E, parts, status));
  return cudaGetLastError();
}

}  // namespace strata
