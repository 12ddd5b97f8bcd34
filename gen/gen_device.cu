// Seeded synthetic expert blobs on the GPU (input generation only; no arithmetic of the method).
//
// Philox4x32-10 (Salmon et al., "Parallel random numbers: as easy as 1, 2, 3", SC'11), restated
// from its definition, with the same keys and counters as gen/__init__.py:
//   block b of blob (layer l, expert e): codes  = philox(ctr=(b, 0, l, e),      key=(seed, 1)), 16 bytes LE
//                                        scale  = table[u16 #(b & 7) of philox(ctr=(b>>3, 0, l, e), key=(seed, 2))]
// The blob is written in the canonical Q2_0 layout: per block {fp16 d, 16 code bytes}, blocks
// numbered gate (FF x H row-major), then up, then down (H x FF row-major).  Only integer
// arithmetic and a table lookup are used, so the bytes equal the host generator's exactly.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr int kH = 2560;
constexpr int kFF = 640;
constexpr int kBlocks = 3 * kH * kFF / 64;  // 76,800 Q2_0 blocks per expert
constexpr int kBlockBytes = 18;

struct u32x4 { uint32_t v[4]; };

__device__ __forceinline__ u32x4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
  }
  return u32x4{{c0, c1, c2, c3}};
}

__global__ void gen_blobs_kernel(uint32_t seed, int32_t layer, int32_t e0, int32_t n,
                                 const uint16_t* __restrict__ table, uint8_t* __restrict__ out,
                                 int64_t blob_stride) {
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (int64_t)n * kBlocks) return;
  const int j = (int)(gid / kBlocks);
  const uint32_t b = (uint32_t)(gid % kBlocks);
  const uint32_t e = (uint32_t)(e0 + j);
  const u32x4 c = philox4x32_10(b, 0u, (uint32_t)layer, e, seed, 1u);
  const u32x4 s = philox4x32_10(b >> 3, 0u, (uint32_t)layer, e, seed, 2u);
  const uint32_t word = s.v[(b & 7) >> 1];
  const uint16_t u = (uint16_t)((b & 1) ? (word >> 16) : (word & 0xFFFFu));
  const uint16_t d = table[u];
  // 18-byte block at an even offset: nine 16-bit stores.
  uint16_t* dst = reinterpret_cast<uint16_t*>(out + (int64_t)j * blob_stride + (int64_t)b * kBlockBytes);
  dst[0] = d;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    dst[1 + 2 * q] = (uint16_t)(c.v[q] & 0xFFFFu);
    dst[2 + 2 * q] = (uint16_t)(c.v[q] >> 16);
  }
}

}  // namespace

// Fill n canonical blobs (layer, experts e0 .. e0+n-1) at out + j*blob_stride.
// table: device fp16[65536] scale table from gen/__init__.py.  Returns 0 or a cudaError_t.
extern "C" int strata_gen_canonical_blobs(uint32_t seed, int32_t layer, int32_t e0, int32_t n,
                                          const void* table, void* out, int64_t blob_stride,
                                          void* stream) {
  if (n <= 0) return 0;
  if (!table || !out || (blob_stride & 1) || blob_stride < (int64_t)kBlocks * kBlockBytes) return -1;
  if (((uintptr_t)out) & 1) return -1;
  const int64_t total = (int64_t)n * kBlocks;
  const int threads = 256;
  const int64_t grid = (total + threads - 1) / threads;
  gen_blobs_kernel<<<(unsigned)grid, threads, 0, (cudaStream_t)stream>>>(
      seed, layer, e0, n, (const uint16_t*)table, (uint8_t*)out, blob_stride);
  return (int)cudaGetLastError();
}
