// Device helpers shared by the decode kernels: the 3-kernel chained path
// (decode.cu) and the persistent stack kernel (decode_fused.cu).
#pragma once

#include "flint_common.cuh"

namespace flint {

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// 2^e as a float for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((127 + e) << 23); }

// Exponent that maps a non-negative max |v| into [2^14, 2^15) (0 for 0/inf/nan).
__device__ __forceinline__ int f16_range_exp(float m) {
  if (!(m > 0.f) || !(m < INFINITY)) return 0;
  int e = ((__float_as_uint(m) >> 23) & 0xFF) - 127;
  if (e < -126) e = -126;  // subnormal max: scale as the smallest normal
  int s = 14 - e;
  if (s > 126) s = 126;
  if (s < -126) s = -126;
  return s;
}

// Reduce-scatter of V compensated sums across a warp (V a power of two <= 32).
// Lane L returns the total of value L >> (5 - log2 V); the lanes sharing a
// value hold the same total up to the low-order compensation term.
template <int V>
__device__ __forceinline__ CSum cs_reduce_scatter(CSum (&v)[V], int lane) {
#pragma unroll
  for (int st = 0; st < 5; ++st) {
    const int o = 16 >> st;
    const int n = V >> st;
    if (n >= 2) {
      const int h = n >> 1;
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < h; ++i) {
        CSum send = up ? v[i] : v[i + h];
        CSum mine = up ? v[i + h] : v[i];
        CSum recv;
        recv.s = __shfl_xor_sync(0xffffffffu, send.s, o);
        recv.c = __shfl_xor_sync(0xffffffffu, send.c, o);
        cs_merge(mine, recv);
        v[i] = mine;
      }
    } else {
      CSum recv;
      recv.s = __shfl_xor_sync(0xffffffffu, v[0].s, o);
      recv.c = __shfl_xor_sync(0xffffffffu, v[0].c, o);
      cs_merge(v[0], recv);
    }
  }
  return v[0];
}

template <int V>
struct Log2 {
  static constexpr int value = V <= 1 ? 0 : 1 + Log2<V / 2>::value;
};
template <>
struct Log2<1> {
  static constexpr int value = 0;
};
template <int V>
struct Pow2Ceil {
  static constexpr int value = V <= 1 ? 1 : V <= 2 ? 2 : V <= 4 ? 4 : V <= 8 ? 8 : V <= 16 ? 16 : 32;
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// ------------------------------------------------------------------ expert GEMV slices

// 16 weight rows x 256 columns (one packed slice in shared memory) times
// 256 x 8 activations (B fragments in registers), fp32 accumulate.  Four
// independent accumulator chains keep the tensor pipe busy.
__device__ __forceinline__ void nvfp4_slice_mma(const uint8_t* sl, int lane, const uint32_t (&bfr)[16][2],
                                                float (&acc)[4]) {
  const int g = lane >> 2;
  const uint4 s0 = *reinterpret_cast<const uint4*>(sl + F4_CODES + g * 16);
  const uint4 s1 = *reinterpret_cast<const uint4*>(sl + F4_CODES + 128 + g * 16);
  const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  float a4[4][4];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int j = 0; j < 4; ++j) a4[c][j] = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 cw = *reinterpret_cast<const uint4*>(sl + c * 512 + lane * 16);
    const uint32_t w4[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int kb = 4 * c + j;
      const uint32_t sc = e4m3x2_to_f16x2(sw[kb >> 1] >> ((kb & 1) * 16));
      uint32_t a0, a1, a2, a3;
      e2m1x8_to_f16x2(w4[j], a0, a1, a2, a3);
      a0 = hmul2_lo(a0, sc);
      a1 = hmul2_hi(a1, sc);
      a2 = hmul2_lo(a2, sc);
      a3 = hmul2_hi(a3, sc);
      mma_f16(a4[j], a0, a1, a2, a3, bfr[kb][0], bfr[kb][1]);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] += (a4[0][j] + a4[1][j]) + (a4[2][j] + a4[3][j]);
}

// nvfp4_slice_mma against two n8 blocks of activations (16 tokens): every
// dequantised A fragment feeds two mma, one per block.
__device__ __forceinline__ void nvfp4_slice_mma_n16(const uint8_t* sl, int lane, const uint32_t (&b0)[16][2],
                                                    const uint32_t (&b1)[16][2], float (&acc0)[4],
                                                    float (&acc1)[4]) {
  const int g = lane >> 2;
  const uint4 s0 = *reinterpret_cast<const uint4*>(sl + F4_CODES + g * 16);
  const uint4 s1 = *reinterpret_cast<const uint4*>(sl + F4_CODES + 128 + g * 16);
  const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  float a4[2][4][4];
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int j = 0; j < 4; ++j) a4[q][c][j] = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 cw = *reinterpret_cast<const uint4*>(sl + c * 512 + lane * 16);
    const uint32_t w4[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int kb = 4 * c + j;
      const uint32_t sc = e4m3x2_to_f16x2(sw[kb >> 1] >> ((kb & 1) * 16));
      uint32_t a0, a1, a2, a3;
      e2m1x8_to_f16x2(w4[j], a0, a1, a2, a3);
      a0 = hmul2_lo(a0, sc);
      a1 = hmul2_hi(a1, sc);
      a2 = hmul2_lo(a2, sc);
      a3 = hmul2_hi(a3, sc);
      mma_f16(a4[0][j], a0, a1, a2, a3, b0[kb][0], b0[kb][1]);
      mma_f16(a4[1][j], a0, a1, a2, a3, b1[kb][0], b1[kb][1]);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    acc0[j] += (a4[0][0][j] + a4[0][1][j]) + (a4[0][2][j] + a4[0][3][j]);
    acc1[j] += (a4[1][0][j] + a4[1][1][j]) + (a4[1][2][j] + a4[1][3][j]);
  }
}

// nvfp4_slice_mma on two slices at once (the same activations), their
// instruction streams interleaved for latency hiding.  Each slice keeps the
// four accumulator chains and the final summation order of nvfp4_slice_mma,
// so its result is bit for bit the same.
__device__ __forceinline__ void nvfp4_slice_mma2(const uint8_t* sa, const uint8_t* sb, int lane,
                                                 const uint32_t (&bfr)[16][2], float (&acc_a)[4],
                                                 float (&acc_b)[4]) {
  const int g = lane >> 2;
  uint32_t sw[2][8];
  {
    const uint4 a0 = *reinterpret_cast<const uint4*>(sa + F4_CODES + g * 16);
    const uint4 a1 = *reinterpret_cast<const uint4*>(sa + F4_CODES + 128 + g * 16);
    const uint4 b0 = *reinterpret_cast<const uint4*>(sb + F4_CODES + g * 16);
    const uint4 b1 = *reinterpret_cast<const uint4*>(sb + F4_CODES + 128 + g * 16);
    sw[0][0] = a0.x; sw[0][1] = a0.y; sw[0][2] = a0.z; sw[0][3] = a0.w;
    sw[0][4] = a1.x; sw[0][5] = a1.y; sw[0][6] = a1.z; sw[0][7] = a1.w;
    sw[1][0] = b0.x; sw[1][1] = b0.y; sw[1][2] = b0.z; sw[1][3] = b0.w;
    sw[1][4] = b1.x; sw[1][5] = b1.y; sw[1][6] = b1.z; sw[1][7] = b1.w;
  }
  float a4[2][4][4];
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int j = 0; j < 4; ++j) a4[q][c][j] = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 ca = *reinterpret_cast<const uint4*>(sa + c * 512 + lane * 16);
    const uint4 cb = *reinterpret_cast<const uint4*>(sb + c * 512 + lane * 16);
    const uint32_t w4[2][4] = {{ca.x, ca.y, ca.z, ca.w}, {cb.x, cb.y, cb.z, cb.w}};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int kb = 4 * c + j;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint32_t sc = e4m3x2_to_f16x2(sw[q][kb >> 1] >> ((kb & 1) * 16));
        uint32_t a0, a1, a2, a3;
        e2m1x8_to_f16x2(w4[q][j], a0, a1, a2, a3);
        a0 = hmul2_lo(a0, sc);
        a1 = hmul2_hi(a1, sc);
        a2 = hmul2_lo(a2, sc);
        a3 = hmul2_hi(a3, sc);
        mma_f16(a4[q][j], a0, a1, a2, a3, bfr[kb][0], bfr[kb][1]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    acc_a[j] += (a4[0][0][j] + a4[0][1][j]) + (a4[0][2][j] + a4[0][3][j]);
    acc_b[j] += (a4[1][0][j] + a4[1][1][j]) + (a4[1][2][j] + a4[1][3][j]);
  }
}

__device__ __forceinline__ void bf16_slice_mma(const uint8_t* sl, int lane, const uint32_t (&bfr)[16][2],
                                               float (&acc)[4]) {
  float a4[4][4];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int j = 0; j < 4; ++j) a4[c][j] = 0.f;
#pragma unroll
  for (int kb = 0; kb < 16; ++kb) {
    const uint4 a = *reinterpret_cast<const uint4*>(sl + kb * 512 + lane * 16);
    mma_bf16(a4[kb & 3], a.x, a.y, a.z, a.w, bfr[kb][0], bfr[kb][1]);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] += (a4[0][j] + a4[1][j]) + (a4[2][j] + a4[3][j]);
}

template <int FMT>
struct Fmt;
template <>
struct Fmt<0> {
  static constexpr int SLICE = F4_SLICE;
  static constexpr int GU_TILE = F4_GU_TILE;
  static constexpr int DN_TILE = F4_DN_TILE;
  static constexpr size_t EXPERT = F4_EXPERT;
  static constexpr size_t GU_BYTES = F4_GU_BYTES;
  __device__ static void slice(const uint8_t* sl, int lane, const uint32_t (&b)[16][2], float (&acc)[4]) {
    nvfp4_slice_mma(sl, lane, b, acc);
  }
};
template <>
struct Fmt<1> {
  static constexpr int SLICE = B16_SLICE;
  static constexpr int GU_TILE = B16_GU_TILE;
  static constexpr int DN_TILE = B16_DN_TILE;
  static constexpr size_t EXPERT = B16_EXPERT;
  static constexpr size_t GU_BYTES = B16_GU_BYTES;
  __device__ static void slice(const uint8_t* sl, int lane, const uint32_t (&b)[16][2], float (&acc)[4]) {
    bf16_slice_mma(sl, lane, b, acc);
  }
};

static_assert(sizeof(Routing) % 4 == 0, "Routing must keep 4-byte alignment");
static_assert(F4_GU_TILE % 128 == 0 && F4_DN_TILE % 128 == 0 && B16_GU_TILE % 128 == 0 &&
                  B16_DN_TILE % 128 == 0,
              "stage buffers must keep 16-byte (bulk copy) alignment");
static_assert(F4_SLICE % 16 == 0 && B16_SLICE % 16 == 0, "slices are read with 16-byte loads");

constexpr int HS_STRIDE = 520;  // halves per staged h row: 512 + 8 so rows land 4 banks apart

// Partial accumulators of one item, one warp: [4 registers][32 lanes] fp32.
// Register j of lane 4g+t holds row g (j < 2) or g + 8 (j >= 2), token 2t + (j & 1).
__device__ __forceinline__ int red_off(int row, int tk) {
  return ((row >> 3) * 2 + (tk & 1)) * 32 + 4 * (row & 7) + (tk >> 1);
}

}  // namespace flint
