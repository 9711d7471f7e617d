// Small-batch dense GEMV on packed NVFP4 weights, sm_103a.
//
// "Day-0 Support for Flint on vLLM", section "Optimizations": besides the MoE
// kernels, a small-batch dense GEMV on the same NVFP4 weights (used by the
// attention projections and the dense MLP of the first layers) cut its step by
// about a quarter.  The operation, for B <= 8 tokens:
//   y[t][n] = bf16( s * sum_k x[t][k] * e2m1(code[n][k]) * e4m3(scale[n][k/16]) )
// with fp32 accumulation, s the fp32 tensor scale, x and y bf16.
//
// Packed layout (flint_moe_pack_dense): [N/16 row tiles][K/256 slices], each
// slice the NVFP4 slice of flint_common.cuh over 16 consecutive rows, so the
// repack is lossless and adds no bytes.  The GEMV reads the slices of a tile in
// units of up to 8 (one TMA bulk copy each); 8 warps take one slice of a unit
// each, keep a running accumulator per tile, and a fixed-order sum over the
// warps gives each output.  Activations enter the tensor cores as f16 scaled by
// a per-token power of two (exact for bf16 inputs within 2^29 of the token's
// largest value), the same mapping as the decode kernels.
#include "decode_common.cuh"
#include "flint_internal.h"

namespace flint {

namespace {

constexpr int DG_CW = 8;                   // compute warps
constexpr int DG_THREADS = 32 * (DG_CW + 1);  // + producer warp
constexpr int DG_UNIT = 8 * F4_SLICE;      // one bulk copy: up to 8 slices of one tile
constexpr int DG_ST = 4;                   // unit ring

struct DenseParams {
  const uint8_t* w;   // packed tiles
  const __nv_bfloat16* x;  // [B][K]
  __nv_bfloat16* y;   // [B][N]
  float ts;           // tensor scale
  int N, K;
  unsigned* err;
};

// [ring][partials 8 x 128 fp32][full, empty, xbar][xmax 8][x rows, B x (2K + 16) bytes]
__host__ __device__ constexpr size_t dense_smem_fixed() {
  return (((size_t)DG_ST * DG_UNIT + 8 * 128 * 4 + (2 * DG_ST + 1) * 8 + 8 * 4) + 15) / 16 * 16;
}
// x rows are 16 bytes longer than K values so that the 8 tokens' fragment
// reads fall into different banks.
__host__ __device__ constexpr size_t dense_xrow_bytes(int K) { return (size_t)K * 2 + 16; }
__host__ __device__ constexpr size_t dense_smem_bytes(int B, int K) {
  return dense_smem_fixed() + (size_t)B * dense_xrow_bytes(K);
}
// Largest over B <= 8, B K <= DENSE_MAX_BK.
constexpr size_t DG_SMEM_MAX = dense_smem_fixed() + (size_t)DENSE_MAX_BK * 2 + 16 * 8;
static_assert(DG_SMEM_MAX <= 232448, "dense GEMV shared memory");

template <int NB>
__global__ void __launch_bounds__(DG_THREADS, 2) dense_gemv_kernel(const DenseParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ring = smem;
  float* red = reinterpret_cast<float*>(smem + (size_t)DG_ST * DG_UNIT);
  uint64_t* full = reinterpret_cast<uint64_t*>(red + 8 * 128);
  uint64_t* empty = full + DG_ST;
  uint64_t* xbar = empty + DG_ST;
  unsigned* xmax = reinterpret_cast<unsigned*>(xbar + 1);
  uint32_t* xs = reinterpret_cast<uint32_t*>(smem + dense_smem_fixed());  // x rows, bf16 pairs, then f16 pairs

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int KS = p.K / 256;              // slices per tile
  const int UPT = (KS + 7) / 8;          // units per tile
  const int NT = p.N / 16;               // row tiles
  const int n_tiles = c < NT ? (NT - c + G - 1) / G : 0;  // tiles c, c + G, ...
  const int n_units = n_tiles * UPT;
  constexpr int XL = 4 * NB;             // mma lanes carrying tokens
  if (tid == 0) {
    for (int s = 0; s < DG_ST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], DG_CW);
    }
    mbar_init(xbar, 1);
    fence_mbar_init();
  }
  if (tid < 8) xmax[tid] = 0u;
  __syncthreads();

  const uint64_t pol = l2_evict_first();
  auto unit_src = [&](int n, uint32_t& bytes) {
    const int tile = c + (n / UPT) * G, g = n % UPT;
    const int ns = min(8, KS - g * 8);
    bytes = (uint32_t)(ns * F4_SLICE);
    return p.w + ((size_t)tile * KS + (size_t)g * 8) * F4_SLICE;
  };
  int issued = 0;
  if (tid == DG_CW * 32) {
    // Weights are constants: the first units are requested before waiting on
    // the kernel that produces x.
    for (; issued < DG_ST && issued < n_units; ++issued) {
      uint32_t bytes;
      const uint8_t* src = unit_src(issued, bytes);
      mbar_arrive_expect_tx(&full[issued], bytes);
      bulk_g2s(ring + (size_t)issued * DG_UNIT, src, bytes, &full[issued], pol);
    }
  }
  pdl_wait();
  pdl_trigger();
  const int XW = (int)(dense_xrow_bytes(p.K) / 4);  // words per staged x row
  if (tid == DG_CW * 32) {
    // x: one bulk copy per token row (every CTA reads all of x).
    const uint64_t xpol = l2_evict_last();
    mbar_arrive_expect_tx(xbar, (uint32_t)(NB * p.K * 2));
    for (int t = 0; t < NB; ++t) bulk_g2s(xs + (size_t)t * XW, p.x + (size_t)t * p.K, (uint32_t)(p.K * 2), xbar, xpol);
  }

  if (warp == DG_CW) {
    if (lane == 0) {
      for (int n = issued; n < n_units; ++n) {
        const int s = n % DG_ST;
        if (!mbar_wait(&empty[s], ((n / DG_ST) - 1) & 1)) {
          atomicOr(p.err, ERR_WAIT_EMPTY);
          break;
        }
        uint32_t bytes;
        const uint8_t* src = unit_src(n, bytes);
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s(ring + (size_t)s * DG_UNIT, src, bytes, &full[s], pol);
        issued = n + 1;
      }
      for (int n = issued - DG_ST; n < issued; ++n) {
        if (n < 0) continue;
        if (!mbar_wait(&full[n % DG_ST], (n / DG_ST) & 1)) atomicOr(p.err, ERR_DRAIN);
      }
      if (!mbar_wait(xbar, 0)) atomicOr(p.err, ERR_DRAIN);
    }
    return;
  }

  // ---- x: warp w prepares the B fragments of the slices it multiplies
  // (w, w + 8, ...).  Lane L < 4 NB (token t = L >> 2, pair i = L & 3) holds
  //   word[kb][h] = x[t][256 s + 16 kb + 8 h + 2 i .. +1]   (kb < 16, h < 2),
  // converted to f16 scaled by 2^e(t) once every warp has added its part of
  // the token's largest magnitude.  With K <= 2048 a warp has one slice and
  // keeps it in registers; otherwise its columns of the staged rows are
  // converted in place (no other warp reads them) and re-read per tile.
  const bool in_regs = KS <= DG_CW;
  const int xt = lane >> 2, xi = lane & 3;
  auto xword = [&](int s, int kb, int h) -> uint32_t& { return xs[(size_t)xt * XW + s * 128 + kb * 8 + h * 4 + xi]; };
  uint32_t bfr[16][2];
#pragma unroll
  for (int kb = 0; kb < 16; ++kb) bfr[kb][0] = bfr[kb][1] = 0u;
  const bool x_ok = mbar_wait(xbar, 0);
  if (!x_ok && lane == 0) atomicOr(p.err, ERR_WAIT_FULL);
  {
    uint32_t mx = 0u;  // largest |x| of the token so far, as two bf16 magnitudes
    if (x_ok && lane < XL) {
      for (int s = warp; s < KS; s += DG_CW) {
#pragma unroll
        for (int kb = 0; kb < 16; ++kb) {
          const uint32_t v0 = xword(s, kb, 0), v1 = xword(s, kb, 1);
          mx = __vmaxu2(mx, v0 & 0x7FFF7FFFu);
          mx = __vmaxu2(mx, v1 & 0x7FFF7FFFu);
          if (in_regs) {
            bfr[kb][0] = v0;
            bfr[kb][1] = v1;
          }
        }
      }
    }
    mx = max(mx & 0xFFFFu, mx >> 16);
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    // As fp32 bits: the order of non-negative floats is that of their bits.
    if (lane < XL && xi == 0 && mx != 0u) atomicMax(&xmax[xt], mx << 16);
  }
  named_bar_sync(1, DG_CW * 32);
  if (x_ok && lane < XL) {
    const float sc = exp2i(f16_range_exp(__uint_as_float(xmax[xt])));
    auto to_f16 = [sc](uint32_t v) {
      const __half2 hv = __floats2half2_rn(__fmul_rn(__uint_as_float(v << 16), sc),
                                           __fmul_rn(__uint_as_float(v & 0xFFFF0000u), sc));
      return *reinterpret_cast<const uint32_t*>(&hv);
    };
    if (in_regs) {
#pragma unroll
      for (int kb = 0; kb < 16; ++kb) {
        bfr[kb][0] = to_f16(bfr[kb][0]);
        bfr[kb][1] = to_f16(bfr[kb][1]);
      }
    } else {
      for (int s = warp; s < KS; s += DG_CW) {
#pragma unroll
        for (int kb = 0; kb < 16; ++kb) {
          xword(s, kb, 0) = to_f16(xword(s, kb, 0));
          xword(s, kb, 1) = to_f16(xword(s, kb, 1));
        }
      }
    }
  }
  __syncwarp();

  // ---- tiles of this CTA
  int n = 0;
  for (int ti = 0; ti < n_tiles; ++ti) {
    const int tile = c + ti * G;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int g = 0; g < UPT; ++g, ++n) {
      const int s = n % DG_ST;
      const int slice = g * 8 + warp;
      if (mbar_wait(&full[s], (n / DG_ST) & 1)) {
        if (slice < KS) {
          if (!in_regs && lane < XL) {
#pragma unroll
            for (int kb = 0; kb < 16; ++kb) {
              bfr[kb][0] = xword(slice, kb, 0);
              bfr[kb][1] = xword(slice, kb, 1);
            }
          }
          nvfp4_slice_mma(ring + (size_t)s * DG_UNIT + warp * F4_SLICE, lane, bfr, acc);
        }
      } else {
        atomicOr(p.err, ERR_WAIT_FULL);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) red[warp * 128 + j * 32 + lane] = acc[j];
    named_bar_sync(1, DG_CW * 32);
    if (tid < 128) {
      // thread = (token tk, row): the 8 warps' partials in a fixed order
      const int row = tid & 15, tk = tid >> 4;
      if (tk < NB) {
        const int o = red_off(row, tk);
        float cc = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) cc += red[w * 128 + o];
        const float sc = __fmul_rn(p.ts, exp2i(-f16_range_exp(__uint_as_float(xmax[tk]))));
        p.y[(size_t)tk * p.N + tile * 16 + row] = __float2bfloat16_rn(__fmul_rn(cc, sc));
      }
    }
    named_bar_sync(1, DG_CW * 32);
  }
}

// Plain NVFP4 matrix [N][K] -> packed tiles.  Thread = one 16-byte unit.
constexpr int DP_UNITS_SLICE = 128 + 16;

__global__ void pack_dense_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                  uint8_t* __restrict__ out, int K, long long total_units) {
  const long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= total_units) return;
  const int KS = K / 256;
  const long long slice_id = u / DP_UNITS_SLICE;  // tile * KS + slice
  const int w = (int)(u % DP_UNITS_SLICE);
  const long long tile = slice_id / KS;
  const int slice = (int)(slice_id % KS);
  const size_t code_stride = (size_t)K / 2, scale_stride = (size_t)K / 16;
  const int kb0 = slice * 16;
  uint8_t b[16];
  size_t off;
  if (w < 128) {
    const int cc = w / 32, L = w % 32, g = L / 4, t = L % 4;
    const size_t r0 = (size_t)tile * 16 + g, r1 = r0 + 8;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int kb = kb0 + 4 * cc + j;
      b[4 * j + 0] = codes[r0 * code_stride + kb * 8 + t];
      b[4 * j + 1] = codes[r1 * code_stride + kb * 8 + t];
      b[4 * j + 2] = codes[r0 * code_stride + kb * 8 + t + 4];
      b[4 * j + 3] = codes[r1 * code_stride + kb * 8 + t + 4];
    }
    off = (size_t)cc * 512 + (size_t)L * 16;
  } else {
    const int w2 = w - 128, hh = w2 / 8, g = w2 % 8;
    const size_t r0 = (size_t)tile * 16 + g, r1 = r0 + 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int kb = kb0 + 8 * hh + i;
      b[2 * i] = scales[r0 * scale_stride + kb];
      b[2 * i + 1] = scales[r1 * scale_stride + kb];
    }
    off = F4_CODES + (size_t)hh * 128 + (size_t)g * 16;
  }
  uint4 v;
  v.x = b[0] | (b[1] << 8) | (b[2] << 16) | ((uint32_t)b[3] << 24);
  v.y = b[4] | (b[5] << 8) | (b[6] << 16) | ((uint32_t)b[7] << 24);
  v.z = b[8] | (b[9] << 8) | (b[10] << 16) | ((uint32_t)b[11] << 24);
  v.w = b[12] | (b[13] << 8) | (b[14] << 16) | ((uint32_t)b[15] << 24);
  *reinterpret_cast<uint4*>(out + (size_t)slice_id * F4_SLICE + off) = v;
}

}  // namespace

size_t dense_packed_bytes(int N, int K) { return (size_t)(N / 16) * (size_t)(K / 256) * F4_SLICE; }

cudaError_t dense_kernels_init() {
  const int bytes = (int)DG_SMEM_MAX;
  cudaError_t r[8] = {
      cudaFuncSetAttribute(dense_gemv_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
      cudaFuncSetAttribute(dense_gemv_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
      cudaFuncSetAttribute(dense_gemv_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
      cudaFuncSetAttribute(dense_gemv_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
      cudaFuncSetAttribute(dense_gemv_kernel<5>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
      cudaFuncSetAttribute(dense_gemv_kernel<6>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
      cudaFuncSetAttribute(dense_gemv_kernel<7>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
      cudaFuncSetAttribute(dense_gemv_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)};
  for (cudaError_t e : r)
    if (e != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t launch_pack_dense(const uint8_t* codes, const uint8_t* scales, int N, int K, void* packed,
                              cudaStream_t st) {
  const long long total = (long long)(N / 16) * (K / 256) * DP_UNITS_SLICE;
  const int threads = 256;
  pack_dense_kernel<<<(unsigned)((total + threads - 1) / threads), threads, 0, st>>>(
      codes, scales, static_cast<uint8_t*>(packed), K, total);
  return cudaGetLastError();
}

template <int NB>
static cudaError_t dense_launch_nb(const DenseParams& dp, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(DG_THREADS);
  cfg.dynamicSmemBytes = dense_smem_bytes(NB, dp.K);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, dense_gemv_kernel<NB>, dp);
}

cudaError_t launch_dense_gemv(const void* packed, int N, int K, float ts, const void* x, int B, void* y, int sm_count,
                              unsigned* err, cudaStream_t st) {
  DenseParams dp;
  dp.w = static_cast<const uint8_t*>(packed);
  dp.x = static_cast<const __nv_bfloat16*>(x);
  dp.y = static_cast<__nv_bfloat16*>(y);
  dp.ts = ts;
  dp.N = N;
  dp.K = K;
  dp.err = err;
  // Two CTAs per SM when their shared memory allows it (e.g. K = 2048 at any B).
  const int tiles = N / 16;
  const int per_sm = 2 * (dense_smem_bytes(B, K) + 1024) <= 233472 ? 2 : 1;
  const int grid = tiles < per_sm * sm_count ? tiles : per_sm * sm_count;
  switch (B) {
    case 1: return dense_launch_nb<1>(dp, grid, st);
    case 2: return dense_launch_nb<2>(dp, grid, st);
    case 3: return dense_launch_nb<3>(dp, grid, st);
    case 4: return dense_launch_nb<4>(dp, grid, st);
    case 5: return dense_launch_nb<5>(dp, grid, st);
    case 6: return dense_launch_nb<6>(dp, grid, st);
    case 7: return dense_launch_nb<7>(dp, grid, st);
    case 8: return dense_launch_nb<8>(dp, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace flint
