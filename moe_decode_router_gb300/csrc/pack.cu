// One-time lossless repack of expert weights into the decode kernels' layout.
//
// "Day-0 Support for Flint on vLLM", section "Model architecture": the NVFP4
// checkpoint stores NVIDIA NVFP4 blocks in a different byte order and the
// loader repacks them losslessly.  The repack here starts from the plain
// NVFP4 layout (codes row-major, low nibble = even element; one E4M3 scale
// byte per 16 elements) and writes the slice layout described in
// flint_common.cuh: every byte is copied, none is changed or added.
//
// Each thread writes one 16-byte unit of the output.
#include "flint_common.cuh"
#include "flint_internal.h"

namespace flint {

namespace {

constexpr int F4_UNITS_SLICE = 128 + 16;  // 4 chunks x 32 lanes of codes + 16 scale units
constexpr int F4_UNITS_GU = GU_TILES * GU_SLICES * F4_UNITS_SLICE;  // 73728
constexpr int F4_UNITS_DN = DN_TILES * DN_SLICES * F4_UNITS_SLICE;  // 36864
constexpr int F4_UNITS_EXPERT = F4_UNITS_GU + F4_UNITS_DN;

constexpr int B16_UNITS_SLICE = 16 * 32;
constexpr int B16_UNITS_GU = GU_TILES * GU_SLICES * B16_UNITS_SLICE;
constexpr int B16_UNITS_DN = DN_TILES * DN_SLICES * B16_UNITS_SLICE;
constexpr int B16_UNITS_EXPERT = B16_UNITS_GU + B16_UNITS_DN;

// Plain row of tile row m: gate/up tiles interleave 8 gate rows and the 8 up
// rows of the same intermediate index; down tiles are 16 consecutive rows.
__device__ __forceinline__ int plain_row(bool gu, int tile, int m) {
  if (gu) return m < 8 ? tile * 8 + m : I + tile * 8 + (m - 8);
  return tile * 16 + m;
}

__global__ void pack_nvfp4_kernel(const uint8_t* __restrict__ gu_codes, const uint8_t* __restrict__ gu_scales,
                                  const uint8_t* __restrict__ dn_codes, const uint8_t* __restrict__ dn_scales,
                                  uint8_t* __restrict__ out, long long total_units) {
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= total_units) return;
  const int e = (int)(u / F4_UNITS_EXPERT);
  int r = (int)(u % F4_UNITS_EXPERT);
  const bool gu = r < F4_UNITS_GU;
  if (!gu) r -= F4_UNITS_GU;
  const int slices = gu ? GU_SLICES : DN_SLICES;
  const int tile = r / (slices * F4_UNITS_SLICE);
  const int rem = r % (slices * F4_UNITS_SLICE);
  const int slice = rem / F4_UNITS_SLICE;
  const int w = rem % F4_UNITS_SLICE;
  const int K = gu ? H : I;
  const size_t code_stride = K / 2, scale_stride = K / 16;
  const size_t rows = gu ? 2 * I : H;
  const uint8_t* codes = (gu ? gu_codes : dn_codes) + (size_t)e * rows * code_stride;
  const uint8_t* scales = (gu ? gu_scales : dn_scales) + (size_t)e * rows * scale_stride;
  const int kb0 = slice * 16;
  uint8_t b[16];
  size_t off;
  if (w < 128) {
    const int c = w / 32, L = w % 32, g = L / 4, t = L % 4;
    const size_t r0 = plain_row(gu, tile, g), r1 = plain_row(gu, tile, g + 8);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int kb = kb0 + 4 * c + j;
      b[4 * j + 0] = codes[r0 * code_stride + kb * 8 + t];
      b[4 * j + 1] = codes[r1 * code_stride + kb * 8 + t];
      b[4 * j + 2] = codes[r0 * code_stride + kb * 8 + t + 4];
      b[4 * j + 3] = codes[r1 * code_stride + kb * 8 + t + 4];
    }
    off = (size_t)c * 512 + (size_t)L * 16;
  } else {
    const int w2 = w - 128, hh = w2 / 8, g = w2 % 8;
    const size_t r0 = plain_row(gu, tile, g), r1 = plain_row(gu, tile, g + 8);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int kb = kb0 + 8 * hh + i;
      b[2 * i] = scales[r0 * scale_stride + kb];
      b[2 * i + 1] = scales[r1 * scale_stride + kb];
    }
    off = F4_CODES + (size_t)hh * 128 + (size_t)g * 16;
  }
  const size_t base = (size_t)e * F4_EXPERT + (gu ? (size_t)tile * F4_GU_TILE : F4_GU_BYTES + (size_t)tile * F4_DN_TILE) +
                      (size_t)slice * F4_SLICE + off;
  uint4 v;
  v.x = b[0] | (b[1] << 8) | (b[2] << 16) | ((uint32_t)b[3] << 24);
  v.y = b[4] | (b[5] << 8) | (b[6] << 16) | ((uint32_t)b[7] << 24);
  v.z = b[8] | (b[9] << 8) | (b[10] << 16) | ((uint32_t)b[11] << 24);
  v.w = b[12] | (b[13] << 8) | (b[14] << 16) | ((uint32_t)b[15] << 24);
  *reinterpret_cast<uint4*>(out + base) = v;
}

__global__ void pack_bf16_kernel(const uint16_t* __restrict__ gu_w, const uint16_t* __restrict__ dn_w,
                                 uint8_t* __restrict__ out, long long total_units) {
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= total_units) return;
  const int e = (int)(u / B16_UNITS_EXPERT);
  int r = (int)(u % B16_UNITS_EXPERT);
  const bool gu = r < B16_UNITS_GU;
  if (!gu) r -= B16_UNITS_GU;
  const int slices = gu ? GU_SLICES : DN_SLICES;
  const int tile = r / (slices * B16_UNITS_SLICE);
  const int rem = r % (slices * B16_UNITS_SLICE);
  const int slice = rem / B16_UNITS_SLICE;
  const int w = rem % B16_UNITS_SLICE;
  const int kb = w / 32, L = w % 32, g = L / 4, t = L % 4;
  const int K = gu ? H : I;
  const size_t rows = gu ? 2 * I : H;
  const uint16_t* W = (gu ? gu_w : dn_w) + (size_t)e * rows * K;
  const size_t r0 = plain_row(gu, tile, g), r1 = plain_row(gu, tile, g + 8);
  const int k = slice * 256 + kb * 16 + 2 * t;
  uint4 v;
  v.x = W[r0 * K + k] | ((uint32_t)W[r0 * K + k + 1] << 16);
  v.y = W[r1 * K + k] | ((uint32_t)W[r1 * K + k + 1] << 16);
  v.z = W[r0 * K + k + 8] | ((uint32_t)W[r0 * K + k + 9] << 16);
  v.w = W[r1 * K + k + 8] | ((uint32_t)W[r1 * K + k + 9] << 16);
  const size_t base = (size_t)e * B16_EXPERT +
                      (gu ? (size_t)tile * B16_GU_TILE : B16_GU_BYTES + (size_t)tile * B16_DN_TILE) +
                      (size_t)slice * B16_SLICE + (size_t)kb * 512 + (size_t)L * 16;
  *reinterpret_cast<uint4*>(out + base) = v;
}

}  // namespace

cudaError_t launch_pack(int fmt, const void* gate_up, const uint8_t* gu_scales, const void* down,
                        const uint8_t* dn_scales, void* packed, cudaStream_t st) {
  const int threads = 256;
  if (fmt == 0) {
    const long long total = (long long)NE * F4_UNITS_EXPERT;
    const unsigned blocks = (unsigned)((total + threads - 1) / threads);
    pack_nvfp4_kernel<<<blocks, threads, 0, st>>>(static_cast<const uint8_t*>(gate_up), gu_scales,
                                                  static_cast<const uint8_t*>(down), dn_scales,
                                                  static_cast<uint8_t*>(packed), total);
  } else {
    const long long total = (long long)NE * B16_UNITS_EXPERT;
    const unsigned blocks = (unsigned)((total + threads - 1) / threads);
    pack_bf16_kernel<<<blocks, threads, 0, st>>>(static_cast<const uint16_t*>(gate_up),
                                                 static_cast<const uint16_t*>(down), static_cast<uint8_t*>(packed),
                                                 total);
  }
  return cudaGetLastError();
}

}  // namespace flint
