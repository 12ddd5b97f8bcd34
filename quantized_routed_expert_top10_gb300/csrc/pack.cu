// Blob packer: the canonical Q2_0 expert blob (gate, up, down; blocks {fp16 d, 16 code bytes}) to
// the GPU layout described in strata_moe.h, and back.  A pure byte permutation.
// ai.thesatyajit.com "Strata engine", section "The byte budget, in code": H = 2560, FF = 640,
// QK = 64, 18-byte blocks, 1,382,400 bytes per expert; momoyeyu.github.io "ai-infra-strata",
// section "权重映射": gate, up and down of an expert stored together.
#include <cstring>

#include "common.cuh"

namespace strata {
namespace {

constexpr int kBlocksPerMat = H * FF / QK;  // 25,600
constexpr int kBlocks = 3 * kBlocksPerMat;  // 76,800

// Where canonical block b's 16 code bytes and 2 scale bytes go in the packed blob.
__host__ __device__ inline void packed_offsets(int b, int64_t* codes_off, int64_t* scale_off) {
  if (b < 2 * kBlocksPerMat) {
    const int up = b >= kBlocksPerMat;
    const int bb = up ? b - kBlocksPerMat : b;
    const int r = bb / KB_GU, kb = bb % KB_GU;
    const int64_t piece = ((int64_t)(r / SLAB) * KB_GU + kb) * SLAB_KB;
    *codes_off = piece + (up ? 256 : 0) + 16 * (r % SLAB);
    *scale_off = piece + 512 + 4 * (r % SLAB) + (up ? 2 : 0);
  } else {
    const int bb = b - 2 * kBlocksPerMat;
    const int n = bb / KB_D, kb = bb % KB_D;
    const int64_t chunk = D_REGION + ((int64_t)(n / RT) * KB_D + kb) * D_CHUNK;
    *codes_off = chunk + 16 * (n % RT);
    *scale_off = chunk + 2048 + 2 * (n % RT);
  }
}

__global__ void pack_kernel(const uint8_t* __restrict__ canonical, int64_t src_stride, uint8_t* __restrict__ packed,
                            int64_t dst_stride, int64_t n_blobs) {
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= n_blobs * kBlocks) return;
  const int64_t j = gid / kBlocks;
  const int b = (int)(gid % kBlocks);
  const uint16_t* src = reinterpret_cast<const uint16_t*>(canonical + j * src_stride + (int64_t)b * 18);
  int64_t co, so;
  packed_offsets(b, &co, &so);
  uint8_t* dst = packed + j * dst_stride;
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) w[q] = (uint32_t)src[1 + 2 * q] | ((uint32_t)src[2 + 2 * q] << 16);
  *reinterpret_cast<uint4*>(dst + co) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint16_t*>(dst + so) = src[0];
}

}  // namespace

cudaError_t launch_pack_device(const uint8_t* canonical, int64_t src_stride, uint8_t* packed, int64_t dst_stride,
                               int64_t n_blobs, cudaStream_t s) {
  const int64_t total = n_blobs * kBlocks;
  STRATA_LAUNCH(KID_PACK, s,
                pack_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(canonical, src_stride, packed, dst_stride,
                                                                           n_blobs));
  return cudaGetLastError();
}

void pack_host(const uint8_t* canonical, uint8_t* packed, int64_t n_blobs) {
  for (int64_t j = 0; j < n_blobs; ++j) {
    const uint8_t* src = canonical + j * BLOB;
    uint8_t* dst = packed + j * BLOB;
    for (int b = 0; b < kBlocks; ++b) {
      int64_t co, so;
      packed_offsets(b, &co, &so);
      std::memcpy(dst + co, src + (int64_t)b * 18 + 2, 16);
      std::memcpy(dst + so, src + (int64_t)b * 18, 2);
    }
  }
}

void unpack_host(const uint8_t* packed, uint8_t* canonical, int64_t n_blobs) {
  for (int64_t j = 0; j < n_blobs; ++j) {
    const uint8_t* src = packed + j * BLOB;
    uint8_t* dst = canonical + j * BLOB;
    for (int b = 0; b < kBlocks; ++b) {
      int64_t co, so;
      packed_offsets(b, &co, &so);
      std::memcpy(dst + (int64_t)b * 18 + 2, src + co, 16);
      std::memcpy(dst + (int64_t)b * 18, src + so, 2);
    }
  }
}

}  // namespace strata
