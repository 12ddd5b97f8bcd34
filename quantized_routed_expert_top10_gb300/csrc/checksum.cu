// CRC-32 of packed expert blobs, on the host and on the device, for verifying an upload or a device
// pack against the bytes it came from (ABI: strata_blob_crc32, strata_blob_crc32_device).
//
// zwxr.cn news/242664, section "与静态 offload 方案的本质差异": every expert slot is read back and
// checked byte for byte after it is filled, and the engine refuses to run when a check fails.  Here
// the check is a checksum per blob: the one the host computes over the bytes it packed or uploaded
// must equal the one the device computes over the blob in HBM.
//
// The checksum is the common CRC-32 (IEEE 802.3 polynomial, reflected, register preset to all ones
// and inverted at the end).  In the reflected form bit 31 of a word is the coefficient of x^0 and bit
// 0 that of x^31; multiplying by x is a right shift, folding x^32 back as 0xEDB88320 (the polynomial
// without its x^32 term).  Feeding one byte b to the register c gives T[(c ^ b) & 0xFF] ^ (c >> 8),
// T[i] = i x^32 mod P.  The update is linear in (c, bytes), so the device splits a blob into chunks,
// takes each chunk's remainder from a zero register, moves it past the bytes that follow it by
// multiplying with x^(8n) mod P, and XORs the parts, adding the preset register moved past the whole
// blob.
#include <array>

#include "common.cuh"

namespace strata {
namespace {

constexpr uint32_t kCrcPoly = 0xEDB88320u;
constexpr int CRC_THREADS = 256;
constexpr int64_t CRC_CHUNK = BLOB / CRC_THREADS;  // 5,400 bytes per thread
static_assert(BLOB % CRC_THREADS == 0 && CRC_CHUNK % 8 == 0, "a blob splits into 8-byte aligned chunks");

__host__ __device__ __forceinline__ uint32_t crc_mulx(uint32_t a) { return (a >> 1) ^ ((a & 1u) ? kCrcPoly : 0u); }

// a(x) b(x) mod P, both reflected: sum over the set coefficients a_i of x^i b(x).
__host__ __device__ __forceinline__ uint32_t crc_mulmod(uint32_t a, uint32_t b) {
  uint32_t p = 0, t = b;  // t = x^i b(x)
  for (int i = 0; i < 32; ++i) {
    if ((a >> (31 - i)) & 1u) p ^= t;
    t = crc_mulx(t);
  }
  return p;
}

// x^(8 n) mod P, reflected, by square and multiply from x^8 (bit 31 - 8).
__host__ __device__ __forceinline__ uint32_t crc_x8n(uint64_t n) {
  uint32_t result = 0x80000000u;  // 1
  uint32_t base = 0x80000000u >> 8;
  while (n) {
    if (n & 1) result = crc_mulmod(result, base);
    base = crc_mulmod(base, base);
    n >>= 1;
  }
  return result;
}

__host__ __device__ __forceinline__ uint32_t crc_table_entry(uint32_t i) {
  uint32_t c = i;
  for (int k = 0; k < 8; ++k) c = crc_mulx(c);
  return c;
}

// One CTA per blob: thread i takes bytes [i CRC_CHUNK, (i + 1) CRC_CHUNK) from a zero register, moves
// the remainder past the (CRC_THREADS - 1 - i) chunks after it; the CTA XORs the parts.
__global__ void __launch_bounds__(CRC_THREADS) blob_crc32_kernel(const uint8_t* __restrict__ blobs, int64_t stride,
                                                                 uint32_t* __restrict__ crc) {
  __shared__ uint32_t table[256];
  __shared__ uint32_t part[CRC_THREADS / 32];
  const int tid = threadIdx.x;
  table[tid] = crc_table_entry((uint32_t)tid);
  __syncthreads();
  const uint2* src = reinterpret_cast<const uint2*>(blobs + (int64_t)blockIdx.x * stride + (int64_t)tid * CRC_CHUNK);
  uint32_t c = 0;
  for (int64_t w = 0; w < CRC_CHUNK / 8; ++w) {
    const uint2 v = __ldg(src + w);
#pragma unroll
    for (int b = 0; b < 4; ++b) c = table[(c ^ (v.x >> (8 * b))) & 0xFFu] ^ (c >> 8);
#pragma unroll
    for (int b = 0; b < 4; ++b) c = table[(c ^ (v.y >> (8 * b))) & 0xFFu] ^ (c >> 8);
  }
  uint32_t moved = crc_mulmod(c, crc_x8n((uint64_t)(CRC_THREADS - 1 - tid) * CRC_CHUNK));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) moved ^= __shfl_xor_sync(0xffffffffu, moved, o);
  if ((tid & 31) == 0) part[tid >> 5] = moved;
  __syncthreads();
  if (tid == 0) {
    uint32_t r = crc_mulmod(0xFFFFFFFFu, crc_x8n((uint64_t)BLOB));
    for (int w = 0; w < CRC_THREADS / 32; ++w) r ^= part[w];
    crc[blockIdx.x] = r ^ 0xFFFFFFFFu;
  }
}

}  // namespace

uint32_t blob_crc32_host(const uint8_t* data, int64_t n) {
  static const std::array<uint32_t, 256> table = [] {  // built once, thread-safe
    std::array<uint32_t, 256> t{};
    for (uint32_t i = 0; i < 256; ++i) t[i] = crc_table_entry(i);
    return t;
  }();
  uint32_t c = 0xFFFFFFFFu;
  for (int64_t i = 0; i < n; ++i) c = table[(c ^ data[i]) & 0xFFu] ^ (c >> 8);
  return c ^ 0xFFFFFFFFu;
}

cudaError_t launch_blob_crc32(const uint8_t* blobs, int64_t stride, int64_t n_blobs, uint32_t* crc, cudaStream_t s) {
  STRATA_LAUNCH(KID_BLOB_CRC32, s, blob_crc32_kernel<<<(unsigned)n_blobs, CRC_THREADS, 0, s>>>(blobs, stride, crc));
  return cudaGetLastError();
}

}  // namespace strata

extern "C" {

strata_status strata_blob_crc32(const uint8_t* blobs, int64_t stride, int64_t n_blobs, uint32_t* crc) {
  if (n_blobs < 0 || stride < strata::BLOB || (n_blobs > 0 && (!blobs || !crc))) return STRATA_E_INVAL;
  for (int64_t j = 0; j < n_blobs; ++j) crc[j] = strata::blob_crc32_host(blobs + j * stride, strata::BLOB);
  return STRATA_OK;
}

strata_status strata_blob_crc32_device(const void* blobs, int64_t stride, int64_t n_blobs, uint32_t* crc,
                                       void* stream) {
  if (n_blobs < 0 || n_blobs > 0x7FFFFFFF || stride < strata::BLOB || (n_blobs > 0 && (!blobs || !crc)))
    return STRATA_E_INVAL;
  if (n_blobs == 0) return STRATA_OK;
  if (((uintptr_t)blobs & 255) || (stride % 256) || ((uintptr_t)crc & 3)) return STRATA_E_ALIGN;
  return strata::launch_blob_crc32((const uint8_t*)blobs, stride, n_blobs, crc, (cudaStream_t)stream) == cudaSuccess
             ? STRATA_OK
             : STRATA_E_CUDA;
}

}  // extern "C"
