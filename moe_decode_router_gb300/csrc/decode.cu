// Decode-path kernels of the Flint MoE sublayer (batch 1..8), sm_103a.
//
// One sublayer = three kernels chained with programmatic dependent launch
// ("Day-0 Support for Flint on vLLM", section "Optimizations": the
// low-latency path for up to 8 requests fuses routing and expert combination
// into the neighbouring GEMVs, and every kernel loads its weights while the
// previous one is still running):
//
//   router_kernel   RMSNorm (optional) + bf16 router GEMV over 256 experts;
//                   writes bf16 logits and the activation x_hat.  Its router
//                   weights are loaded before it waits on its predecessor.
//   gateup_kernel   every CTA derives the sigmoid top-6 routing from the
//                   logits, then streams the gate/up tiles of the shared
//                   expert and of the distinct selected experts only (TMA bulk
//                   copies into a shared-memory ring), dequantises NVFP4 in
//                   registers, runs mma.m16n8k16 with the batch as the N=8
//                   dimension and writes h = bf16(silu(g) * u).  Shared-expert
//                   tiles are requested before the dependency wait.
//   down_kernel     launched as soon as the routing is final; it requests its
//                   down-projection tiles before waiting for h, then computes
//                   the down GEMV of every selected expert for its 16 output
//                   rows and combines them with the routing weights (shared
//                   expert weight 1) in a fixed order, rounding once to bf16.
#include "flint_common.cuh"
#include "flint_internal.h"

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

// ------------------------------------------------------------------ router

struct RouterParams {
  const __nv_bfloat16* x;       // [B][H]
  const CSum* ss_in;            // [DN_TILES][8] sum-of-squares partials of x, or null
  const __nv_bfloat16* norm_w;  // [H] or null
  const __nv_bfloat16* wr;      // [E][H]
  float eps;
  int want_f16;
  __nv_bfloat16* logits;   // [B][E]
  __nv_bfloat16* xh_bf16;  // [B][H]
  __half* xh_f16;          // [B][H]
  int* xh_exp;             // [B]
};

// Router logits logit[t][e] = bf16( sum_k x_hat[t][k] * W_r[e][k] ).  The sum
// is accumulated error-free (products of bf16 values are exact in fp32) so
// the bf16 logit, which decides the top-6, is the correctly rounded value and
// does not depend on the order of accumulation.  Each CTA owns EPC experts;
// thread k owns columns [8k, 8k+8).
template <int EPC, int NB>
__global__ void __launch_bounds__(256) router_kernel(const RouterParams p) {
  constexpr int V = EPC * NB;
  constexpr int VP = Pow2Ceil<V>::value;
  constexpr int NBP = Pow2Ceil<NB>::value;
  __shared__ CSum red[8][VP];
  __shared__ CSum ssred[8][NBP];
  __shared__ float rscale[NB];
  __shared__ unsigned xmax[NB];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int e0 = blockIdx.x * EPC;
  const int k0 = tid * 8;
  if (tid < NB) xmax[tid] = 0u;

  // Before the dependency wait: the router and norm weights are constants.
  float wf[EPC][8];
#pragma unroll
  for (int j = 0; j < EPC; ++j)
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(p.wr + (size_t)(e0 + j) * H + k0)), wf[j]);
  float nw[8];
  const bool has_norm = p.norm_w != nullptr;
  if (has_norm) bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(p.norm_w + k0)), nw);

  pdl_trigger();
  pdl_wait();

  float xv[NB][8];
#pragma unroll
  for (int t = 0; t < NB; ++t)
    bf16x8_to_f32(__ldcg(reinterpret_cast<const uint4*>(p.x + (size_t)t * H + k0)), xv[t]);

  if (has_norm) {
    if (p.ss_in != nullptr) {
      // Partials written by the previous sublayer's down kernel.
      if (warp < NB) {
        CSum a = {0.f, 0.f};
        for (int j = lane; j < DN_TILES; j += 32) cs_merge(a, p.ss_in[j * BMAX + warp]);
        a = cs_warp_reduce(a);
        if (lane == 0) {
          const float ms = __fmul_rn(cs_value(a), 1.0f / (float)H);
          rscale[warp] = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, p.eps)));
        }
      }
    } else {
      CSum ss[NBP];
#pragma unroll
      for (int t = 0; t < NBP; ++t) ss[t] = CSum{0.f, 0.f};
#pragma unroll
      for (int t = 0; t < NB; ++t)
#pragma unroll
        for (int i = 0; i < 8; ++i) cs_add(ss[t], __fmul_rn(xv[t][i], xv[t][i]));
      const CSum tot = cs_reduce_scatter<NBP>(ss, lane);
      constexpr int SH = 5 - Log2<NBP>::value;
      if ((lane & ((1 << SH) - 1)) == 0) ssred[warp][lane >> SH] = tot;
      __syncthreads();
      if (tid < NB) {
        CSum a = ssred[0][tid];
#pragma unroll
        for (int w = 1; w < 8; ++w) cs_merge(a, ssred[w][tid]);
        const float ms = __fmul_rn(cs_value(a), 1.0f / (float)H);
        rscale[tid] = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, p.eps)));
      }
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < NB; ++t) {
      const float r = rscale[t];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        xv[t][i] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(__fmul_rn(xv[t][i], r), nw[i])));
    }
  }

  CSum d[VP];
#pragma unroll
  for (int v = 0; v < VP; ++v) d[v] = CSum{0.f, 0.f};
#pragma unroll
  for (int j = 0; j < EPC; ++j)
#pragma unroll
    for (int t = 0; t < NB; ++t)
#pragma unroll
      for (int i = 0; i < 8; ++i) cs_add(d[j * NB + t], __fmul_rn(xv[t][i], wf[j][i]));
  {
    const CSum tot = cs_reduce_scatter<VP>(d, lane);
    constexpr int SH = 5 - Log2<VP>::value;
    if ((lane & ((1 << SH) - 1)) == 0) red[warp][lane >> SH] = tot;
  }
  __syncthreads();
  if (tid < V) {
    CSum a = red[0][tid];
#pragma unroll
    for (int w = 1; w < 8; ++w) cs_merge(a, red[w][tid]);
    const int j = tid / NB, t = tid % NB;
    p.logits[(size_t)t * E + e0 + j] = __float2bfloat16_rn(cs_value(a));
  }

  if (blockIdx.x == 0) {
    // Every CTA computed the same x_hat; CTA 0 publishes it.
#pragma unroll
    for (int t = 0; t < NB; ++t) {
      uint32_t pk[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        pk[i] = (__float_as_uint(xv[t][2 * i]) >> 16) | (__float_as_uint(xv[t][2 * i + 1]) & 0xFFFF0000u);
      *reinterpret_cast<uint4*>(p.xh_bf16 + (size_t)t * H + k0) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
    if (p.want_f16) {
#pragma unroll
      for (int t = 0; t < NB; ++t) {
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(xv[t][i]));
        const unsigned wm = redux_max(__float_as_uint(m));
        if (lane == 0) atomicMax(&xmax[t], wm);
      }
      __syncthreads();
#pragma unroll
      for (int t = 0; t < NB; ++t) {
        const int ex = f16_range_exp(__uint_as_float(xmax[t]));
        const float sc = exp2i(ex);
        uint32_t pk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __half2 hv = __floats2half2_rn(__fmul_rn(xv[t][2 * i], sc), __fmul_rn(xv[t][2 * i + 1], sc));
          pk[i] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        *reinterpret_cast<uint4*>(p.xh_f16 + (size_t)t * H + k0) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        if (tid == 0) p.xh_exp[t] = ex;
      }
    }
  }
}

// ------------------------------------------------------------------ expert GEMV slices

// 16 weight rows x 256 columns of NVFP4 (one packed slice in shared memory)
// times 256 x 8 activations (B fragments in registers), fp32 accumulate.
__device__ __forceinline__ void nvfp4_slice_mma(const uint8_t* sl, int lane, const uint32_t (&bfr)[16][2],
                                                float (&acc)[4]) {
  const int g = lane >> 2;
  const uint4 s0 = *reinterpret_cast<const uint4*>(sl + F4_CODES + g * 16);
  const uint4 s1 = *reinterpret_cast<const uint4*>(sl + F4_CODES + 128 + g * 16);
  const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
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
      mma_f16(acc, a0, a1, a2, a3, bfr[kb][0], bfr[kb][1]);
    }
  }
}

__device__ __forceinline__ void bf16_slice_mma(const uint8_t* sl, int lane, const uint32_t (&bfr)[16][2],
                                               float (&acc)[4]) {
#pragma unroll
  for (int kb = 0; kb < 16; ++kb) {
    const uint4 a = *reinterpret_cast<const uint4*>(sl + kb * 512 + lane * 16);
    mma_bf16(acc, a.x, a.y, a.z, a.w, bfr[kb][0], bfr[kb][1]);
  }
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

// ------------------------------------------------------------------ gate/up
static_assert(sizeof(Routing) % 4 == 0, "Routing must keep 4-byte alignment");
static_assert(F4_GU_TILE % 128 == 0 && F4_DN_TILE % 128 == 0 && B16_GU_TILE % 128 == 0 &&
                  B16_DN_TILE % 128 == 0,
              "stage buffers must keep 16-byte (bulk copy) alignment");
static_assert(F4_SLICE % 16 == 0 && B16_SLICE % 16 == 0, "slices are read with 16-byte loads");


struct GateUpParams {
  const uint8_t* experts;
  const float* tscale;          // [NE][2] (NVFP4)
  const __nv_bfloat16* logits;  // [B][E]
  const void* xh;               // f16 [B][H] (NVFP4) or bf16 [B][H]
  const int* xh_exp;            // [B] (NVFP4)
  int B;
  __nv_bfloat16* h;             // [MAX_SLOTS][BMAX][I]
  float* hmax_part;             // [gridDim.x][BMAX]
  int32_t* ids_out;             // [B][6] or null
  float* w_out;                 // [B][6] or null
  unsigned* err;
};

constexpr int GU_THREADS = 288;  // 8 consumer warps (one K slice each) + 1 producer warp

template <int FMT, int STAGES>
__host__ __device__ constexpr size_t gateup_smem_bytes() {
  // [stages][red 2x8x128 fp32][full, empty barriers][abort flag, pad to 16][Routing]
  return (size_t)STAGES * Fmt<FMT>::GU_TILE + 2 * 8 * 128 * 4 + 2 * STAGES * 8 + 16 + sizeof(Routing);
}

template <int FMT, int STAGES>
__global__ void __launch_bounds__(GU_THREADS, 1) gateup_kernel(const GateUpParams p) {
  using F = Fmt<FMT>;
  constexpr int TILE = F::GU_TILE;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  float* red = reinterpret_cast<float*>(smem + (size_t)STAGES * TILE);  // [2][8][128], 16-byte aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(red + 2 * 8 * 128);
  uint64_t* empty = full + STAGES;
  int* abort_flag = reinterpret_cast<int*>(empty + STAGES);
  Routing& R = *reinterpret_cast<Routing*>(reinterpret_cast<uint8_t*>(abort_flag) + 16);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, bid = blockIdx.x;
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 8);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const uint64_t pol = l2_evict_first();
  int issued = 0;
  if (tid == 256) {
    // The shared expert's tiles do not depend on the routing: request them
    // while the router is still running.
    for (; issued < STAGES; ++issued) {
      const int i = bid + issued * G;
      if (i >= GU_TILES) break;
      mbar_arrive_expect_tx(&full[issued], TILE);
      bulk_g2s(stages + (size_t)issued * TILE, p.experts + (size_t)E * F::EXPERT + (size_t)i * TILE, TILE,
               &full[issued], pol);
    }
  }

  pdl_wait();
  compute_routing(p.logits, p.B, R);
  pdl_trigger();  // the down kernel may start: the routing inputs are final
  const int n_items = R.n_slots * GU_TILES;
  if (bid == 0 && tid < p.B * TOPK) {
    if (p.ids_out) p.ids_out[tid] = R.ids[tid / TOPK][tid % TOPK];
    if (p.w_out) p.w_out[tid] = R.w[tid / TOPK][tid % TOPK];
  }

  if (warp == 8) {
    if (lane == 0) {
      for (int n = issued;; ++n) {
        const int i = bid + n * G;
        if (i >= n_items) break;
        const int s = n % STAGES;
        if (n >= STAGES && !mbar_wait(&empty[s], ((n / STAGES) - 1) & 1)) {
          atomicOr(p.err, ERR_WAIT_EMPTY);
          break;
        }
        const int e = R.slot_expert[i / GU_TILES];
        mbar_arrive_expect_tx(&full[s], TILE);
        bulk_g2s(stages + (size_t)s * TILE, p.experts + (size_t)e * F::EXPERT + (size_t)(i % GU_TILES) * TILE,
                 TILE, &full[s], pol);
        issued = n + 1;
      }
      // Do not leave copies in flight: wait for the last use of every stage.
      for (int n = issued - STAGES; n < issued; ++n) {
        if (n < 0) continue;
        if (!mbar_wait(&full[n % STAGES], (n / STAGES) & 1)) atomicOr(p.err, ERR_DRAIN);
      }
    }
    return;
  }

  // ---- consumers: warp w multiplies K slice w of every tile
  const int g = lane >> 2, t = lane & 3;
  uint32_t bfr[16][2];
  if (g < p.B) {
    const uint32_t* xr = reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(p.xh) + (size_t)g * H +
                                                           warp * 256);
#pragma unroll
    for (int kb = 0; kb < 16; ++kb) {
      bfr[kb][0] = __ldcg(xr + kb * 8 + t);
      bfr[kb][1] = __ldcg(xr + kb * 8 + t + 4);
    }
  } else {
#pragma unroll
    for (int kb = 0; kb < 16; ++kb) bfr[kb][0] = bfr[kb][1] = 0u;
  }
  float xs[2] = {1.f, 1.f};  // 2^-exponent of tokens 2t, 2t+1 (NVFP4)
  if (FMT == 0) {
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if (2 * t + q < p.B) xs[q] = exp2i(-__ldcg(p.xh_exp + 2 * t + q));
  }
  float hm[2] = {0.f, 0.f};

  for (int n = 0;; ++n) {
    const int i = bid + n * G;
    if (i >= n_items) break;
    const int s = n % STAGES;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (mbar_wait(&full[s], (n / STAGES) & 1)) {
      F::slice(stages + (size_t)s * TILE + warp * F::SLICE, lane, bfr, acc);
    } else {
      atomicOr(p.err, ERR_WAIT_FULL);
      *abort_flag = 1;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    float* rb = red + (n & 1) * 1024;
    *reinterpret_cast<float4*>(rb + warp * 128 + lane * 4) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    named_bar_sync(1, 256);
    if (*abort_flag) break;
    if (warp == 0) {
      float c[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) c[j] = rb[lane * 4 + j];
#pragma unroll
      for (int w = 1; w < 8; ++w) {
        const float4 v = *reinterpret_cast<const float4*>(rb + w * 128 + lane * 4);
        c[0] += v.x;
        c[1] += v.y;
        c[2] += v.z;
        c[3] += v.w;
      }
      const int slot = i / GU_TILES, tile = i % GU_TILES;
      const int e = R.slot_expert[slot];
      const uint32_t mask = R.slot_mask[slot];
      const float ts = FMT == 0 ? __ldg(p.tscale + 2 * e) : 1.0f;
      const int j = tile * 8 + g;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int tk = 2 * t + q;
        if ((mask >> tk) & 1u) {
          const float f = __fmul_rn(xs[q], ts);
          const float gate = __fmul_rn(c[q], f);
          const float up = __fmul_rn(c[2 + q], f);
          const float silu = __fdiv_rn(gate, __fadd_rn(1.0f, expf(-gate)));
          const __nv_bfloat16 hv = __float2bfloat16_rn(__fmul_rn(silu, up));
          p.h[((size_t)slot * BMAX + tk) * I + j] = hv;
          hm[q] = fmaxf(hm[q], fabsf(__bfloat162float(hv)));
        }
      }
    }
  }
  if (warp == 0) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      float m = hm[q];
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
      if (g == 0) p.hmax_part[(size_t)bid * BMAX + 2 * t + q] = m;
    }
  }
}

// ------------------------------------------------------------------ down + combine

struct DownParams {
  const uint8_t* experts;
  const float* tscale;
  const __nv_bfloat16* logits;
  const __nv_bfloat16* h;
  const float* hmax_part;
  int n_hparts;
  int B;
  __nv_bfloat16* y;       // [B][H]
  __nv_bfloat16* y_copy;  // [B][H] or null
  CSum* ss_out;           // [DN_TILES][BMAX] or null
  unsigned* err;
};

constexpr int DN_THREADS = 288;
constexpr int HS_STRIDE = 520;  // halves per staged h row: 512 + 8 so rows land 4 banks apart

template <int FMT, int STAGES>
__host__ __device__ constexpr size_t down_smem_fixed() {
  // [stages][red 8x128 fp32][full, empty barriers][hexp 8, misc 8 ints][pidx][pair token][pair slot][Routing]
  return (size_t)STAGES * Fmt<FMT>::DN_TILE + 8 * 128 * 4 + 2 * STAGES * 8 + 64 + MAX_SLOTS * BMAX + 64 + 64 +
         sizeof(Routing);
}
template <int FMT, int STAGES>
size_t down_smem_bytes(int B) {
  return ((down_smem_fixed<FMT, STAGES>() + 15) / 16) * 16 + (size_t)(1 + TOPK) * B * HS_STRIDE * 2;
}

template <int FMT, int STAGES>
__global__ void __launch_bounds__(DN_THREADS, 1) down_kernel(const DownParams p) {
  using F = Fmt<FMT>;
  constexpr int TILE = F::DN_TILE;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  float* red = reinterpret_cast<float*>(smem + (size_t)STAGES * TILE);  // [8][128], 16-byte aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(red + 8 * 128);
  uint64_t* empty = full + STAGES;
  int* hexp = reinterpret_cast<int*>(empty + STAGES);    // [8]
  int* misc = hexp + 8;                                  // [0] abort, [1] n_pairs
  uint8_t* pidx = reinterpret_cast<uint8_t*>(misc + 8);  // [MAX_SLOTS][8]
  uint8_t* psrc_tok = pidx + MAX_SLOTS * BMAX;           // [<= 56] token of pair
  uint8_t* psrc_slot = psrc_tok + 64;                    // [<= 56] slot of pair
  Routing& R = *reinterpret_cast<Routing*>(psrc_slot + 64);
  uint16_t* hs = reinterpret_cast<uint16_t*>(smem + ((down_smem_fixed<FMT, STAGES>() + 15) / 16) * 16);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rt = blockIdx.x;
  const int B = p.B;
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 2);
    }
    misc[0] = 0;
    fence_mbar_init();
  }
  pdl_trigger();  // the next sublayer's router only prefetches constants before its wait
  __syncthreads();
  // The routing of this sublayer is final: this kernel is launched only after
  // every gate/up CTA passed its dependency wait on the router.
  compute_routing(p.logits, B, R);
  const int n_slots = R.n_slots;
  const uint64_t pol = l2_evict_first();
  int issued = 0;
  if (tid == 256) {
    for (; issued < STAGES && issued < n_slots; ++issued) {
      const int e = R.slot_expert[issued];
      mbar_arrive_expect_tx(&full[issued], TILE);
      bulk_g2s(stages + (size_t)issued * TILE, p.experts + (size_t)e * F::EXPERT + F::GU_BYTES + (size_t)rt * TILE,
               TILE, &full[issued], pol);
    }
  }
  if (warp == 0) {
    // compact (slot, token) pairs: pair index = prefix over slots of popc(mask)
    int base = 0;
    for (int c0 = 0; c0 < n_slots; c0 += 32) {
      const int u = c0 + lane;
      const uint32_t m = u < n_slots ? R.slot_mask[u] : 0u;
      const int cnt = __popc(m);
      int incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      int pi = base + incl - cnt;
      if (u < n_slots) {
#pragma unroll
        for (int tk = 0; tk < BMAX; ++tk) {
          if ((m >> tk) & 1u) {
            pidx[u * BMAX + tk] = (uint8_t)pi;
            psrc_tok[pi] = (uint8_t)tk;
            psrc_slot[pi] = (uint8_t)u;
            ++pi;
          }
        }
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) misc[1] = base;
  }

  pdl_wait();  // gate/up of this sublayer is complete: h and hmax_part are final

  if (FMT == 0 && warp < B) {
    float m = 0.f;
    for (int j = lane; j < p.n_hparts; j += 32) m = fmaxf(m, __ldcg(p.hmax_part + (size_t)j * BMAX + warp));
    const unsigned mb = redux_max(__float_as_uint(m));
    if (lane == 0) hexp[warp] = f16_range_exp(__uint_as_float(mb));
  }
  __syncthreads();
  {
    const int n_pairs = misc[1];
    for (int idx = tid; idx < n_pairs * 64; idx += DN_THREADS) {
      const int pr = idx >> 6, ch = idx & 63;
      const int tk = psrc_tok[pr], u = psrc_slot[pr];
      const uint4 raw =
          __ldcg(reinterpret_cast<const uint4*>(p.h + ((size_t)u * BMAX + tk) * I) + ch);
      uint4 outv = raw;
      if (FMT == 0) {
        float f[8];
        bf16x8_to_f32(raw, f);
        const float sc = exp2i(hexp[tk]);
        uint32_t pk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __half2 hv = __floats2half2_rn(__fmul_rn(f[2 * i], sc), __fmul_rn(f[2 * i + 1], sc));
          pk[i] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        outv = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      *reinterpret_cast<uint4*>(hs + (size_t)pr * HS_STRIDE + ch * 8) = outv;
    }
  }
  __syncthreads();

  if (warp == 8) {
    if (lane == 0) {
      for (int n = issued; n < n_slots; ++n) {
        const int s = n % STAGES;
        if (!mbar_wait(&empty[s], ((n / STAGES) - 1) & 1)) {
          atomicOr(p.err, ERR_WAIT_EMPTY);
          break;
        }
        const int e = R.slot_expert[n];
        mbar_arrive_expect_tx(&full[s], TILE);
        bulk_g2s(stages + (size_t)s * TILE, p.experts + (size_t)e * F::EXPERT + F::GU_BYTES + (size_t)rt * TILE,
                 TILE, &full[s], pol);
        issued = n + 1;
      }
      for (int n = issued - STAGES; n < issued; ++n) {
        if (n < 0) continue;
        if (!mbar_wait(&full[n % STAGES], (n / STAGES) & 1)) atomicOr(p.err, ERR_DRAIN);
      }
    }
    return;
  }

  const int g = lane >> 2, t = lane & 3;
  const int kh = warp & 1, grp = warp >> 1;
  float tot[4] = {0.f, 0.f, 0.f, 0.f};
  for (int u = grp; u < n_slots; u += 4) {
    const int s = u % STAGES;
    if (!mbar_wait(&full[s], (u / STAGES) & 1)) {
      atomicOr(p.err, ERR_WAIT_FULL);
      misc[0] = 1;
      break;
    }
    uint32_t bfr[16][2];
    const uint32_t mask = R.slot_mask[u];
    if (g < B && ((mask >> g) & 1u)) {
      const uint32_t* hr =
          reinterpret_cast<const uint32_t*>(hs + (size_t)pidx[u * BMAX + g] * HS_STRIDE + kh * 256);
#pragma unroll
      for (int kb = 0; kb < 16; ++kb) {
        bfr[kb][0] = hr[kb * 8 + t];
        bfr[kb][1] = hr[kb * 8 + t + 4];
      }
    } else {
#pragma unroll
      for (int kb = 0; kb < 16; ++kb) bfr[kb][0] = bfr[kb][1] = 0u;
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    F::slice(stages + (size_t)s * TILE + kh * F::SLICE, lane, bfr, acc);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    const int e = R.slot_expert[u];
    const float ts = FMT == 0 ? __ldg(p.tscale + 2 * e + 1) : 1.0f;
    const float w0 = __fmul_rn(R.slot_w[u][2 * t], ts);
    const float w1 = __fmul_rn(R.slot_w[u][2 * t + 1], ts);
    tot[0] = fmaf(w0, acc[0], tot[0]);
    tot[1] = fmaf(w1, acc[1], tot[1]);
    tot[2] = fmaf(w0, acc[2], tot[2]);
    tot[3] = fmaf(w1, acc[3], tot[3]);
  }
  *reinterpret_cast<float4*>(red + warp * 128 + lane * 4) = make_float4(tot[0], tot[1], tot[2], tot[3]);
  named_bar_sync(1, 256);
  if (warp == 0) {
    float c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) c[j] = red[lane * 4 + j];
#pragma unroll
    for (int w = 1; w < 8; ++w) {
      const float4 v = *reinterpret_cast<const float4*>(red + w * 128 + lane * 4);
      c[0] += v.x;
      c[1] += v.y;
      c[2] += v.z;
      c[3] += v.w;
    }
    CSum sq[2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int tk = 2 * t + q;
      if (tk < B) {
        const float sc = FMT == 0 ? exp2i(-hexp[tk]) : 1.0f;
        const __nv_bfloat16 y0 = __float2bfloat16_rn(__fmul_rn(c[q], sc));
        const __nv_bfloat16 y1 = __float2bfloat16_rn(__fmul_rn(c[2 + q], sc));
        const size_t o0 = (size_t)tk * H + rt * 16 + g;
        p.y[o0] = y0;
        p.y[o0 + 8] = y1;
        if (p.y_copy) {
          p.y_copy[o0] = y0;
          p.y_copy[o0 + 8] = y1;
        }
        const float f0 = __bfloat162float(y0), f1 = __bfloat162float(y1);
        cs_add(sq[q], __fmul_rn(f0, f0));
        cs_add(sq[q], __fmul_rn(f1, f1));
      }
    }
    if (p.ss_out) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        CSum a = sq[q];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          CSum b;
          b.s = __shfl_xor_sync(0xffffffffu, a.s, off);
          b.c = __shfl_xor_sync(0xffffffffu, a.c, off);
          cs_merge(a, b);
        }
        if (g == 0) p.ss_out[(size_t)rt * BMAX + 2 * t + q] = a;
      }
    }
  }
}

// ------------------------------------------------------------------ host side

constexpr int F4_GU_STAGES = 5;
constexpr int F4_DN_STAGES = 8;
constexpr int B16_GU_STAGES = 3;
constexpr int B16_DN_STAGES = 6;
constexpr int ROUTER_EPC = 2;

static size_t align256(size_t v) { return (v + 255) / 256 * 256; }

size_t decode_ws_bytes(int gu_grid) {
  size_t b = 0;
  b += align256((size_t)BMAX * E * 2);                  // logits
  b += align256((size_t)BMAX * H * 2);                  // xh_bf16
  b += align256((size_t)BMAX * H * 2);                  // xh_f16
  b += align256(BMAX * 4);                              // xh_exp
  b += align256((size_t)MAX_SLOTS * BMAX * I * 2);      // h
  b += align256((size_t)gu_grid * BMAX * 4);            // hmax_part
  b += align256((size_t)DN_TILES * BMAX * sizeof(CSum));  // ss_part
  b += align256((size_t)BMAX * H * 2);                  // y_mid
  return b;
}

DecodeWs carve_decode_ws(void* ws, int gu_grid) {
  uint8_t* p = static_cast<uint8_t*>(ws);
  DecodeWs w;
  w.logits = p;
  p += align256((size_t)BMAX * E * 2);
  w.xh_bf16 = p;
  p += align256((size_t)BMAX * H * 2);
  w.xh_f16 = p;
  p += align256((size_t)BMAX * H * 2);
  w.xh_exp = reinterpret_cast<int*>(p);
  p += align256(BMAX * 4);
  w.h = p;
  p += align256((size_t)MAX_SLOTS * BMAX * I * 2);
  w.hmax_part = reinterpret_cast<float*>(p);
  p += align256((size_t)gu_grid * BMAX * 4);
  w.ss_part = p;
  p += align256((size_t)DN_TILES * BMAX * sizeof(CSum));
  w.y_mid = p;
  return w;
}

template <typename... KArgs, typename... Args>
static cudaError_t launch(void (*k)(KArgs...), int grid, int block, size_t smem, cudaStream_t st, bool pdl,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}

template <int NB>
static cudaError_t launch_router_nb(const RouterParams& rp, cudaStream_t st, bool pdl) {
  return launch(router_kernel<ROUTER_EPC, NB>, E / ROUTER_EPC, 256, 0, st, pdl, rp);
}

static cudaError_t launch_router(int B, const RouterParams& rp, cudaStream_t st, bool pdl) {
  switch (B) {
    case 1: return launch_router_nb<1>(rp, st, pdl);
    case 2: return launch_router_nb<2>(rp, st, pdl);
    case 3: return launch_router_nb<3>(rp, st, pdl);
    case 4: return launch_router_nb<4>(rp, st, pdl);
    case 5: return launch_router_nb<5>(rp, st, pdl);
    case 6: return launch_router_nb<6>(rp, st, pdl);
    case 7: return launch_router_nb<7>(rp, st, pdl);
    case 8: return launch_router_nb<8>(rp, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t decode_kernels_init(int /*device*/) {
  cudaError_t e;
  e = cudaFuncSetAttribute(gateup_kernel<0, F4_GU_STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)gateup_smem_bytes<0, F4_GU_STAGES>());
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gateup_kernel<1, B16_GU_STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)gateup_smem_bytes<1, B16_GU_STAGES>());
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(down_kernel<0, F4_DN_STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)down_smem_bytes<0, F4_DN_STAGES>(BMAX));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(down_kernel<1, B16_DN_STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)down_smem_bytes<1, B16_DN_STAGES>(BMAX));
  return e;
}

cudaError_t launch_decode_layer(int fmt, const LayerArgs& L, const void* x, const void* ss_in, int B, float eps,
                                void* y, void* ys_copy, void* ss_out, int32_t* ids_out, float* w_out,
                                const DecodeWs& ws, int gu_grid, unsigned* err, cudaStream_t st, bool pdl_first) {
  RouterParams rp;
  rp.x = static_cast<const __nv_bfloat16*>(x);
  rp.ss_in = static_cast<const CSum*>(ss_in);
  rp.norm_w = static_cast<const __nv_bfloat16*>(L.norm_w);
  rp.wr = static_cast<const __nv_bfloat16*>(L.router_w);
  rp.eps = eps;
  rp.want_f16 = fmt == 0;
  rp.logits = static_cast<__nv_bfloat16*>(ws.logits);
  rp.xh_bf16 = static_cast<__nv_bfloat16*>(ws.xh_bf16);
  rp.xh_f16 = static_cast<__half*>(ws.xh_f16);
  rp.xh_exp = ws.xh_exp;
  cudaError_t e = launch_router(B, rp, st, pdl_first);
  if (e != cudaSuccess) return e;

  GateUpParams gp;
  gp.experts = L.experts;
  gp.tscale = L.tscale;
  gp.logits = rp.logits;
  gp.xh = fmt == 0 ? static_cast<const void*>(ws.xh_f16) : static_cast<const void*>(ws.xh_bf16);
  gp.xh_exp = ws.xh_exp;
  gp.B = B;
  gp.h = static_cast<__nv_bfloat16*>(ws.h);
  gp.hmax_part = ws.hmax_part;
  gp.ids_out = ids_out;
  gp.w_out = w_out;
  gp.err = err;
  if (fmt == 0)
    e = launch(gateup_kernel<0, F4_GU_STAGES>, gu_grid, GU_THREADS, gateup_smem_bytes<0, F4_GU_STAGES>(), st, true,
               gp);
  else
    e = launch(gateup_kernel<1, B16_GU_STAGES>, gu_grid, GU_THREADS, gateup_smem_bytes<1, B16_GU_STAGES>(), st,
               true, gp);
  if (e != cudaSuccess) return e;

  DownParams dp;
  dp.experts = L.experts;
  dp.tscale = L.tscale;
  dp.logits = rp.logits;
  dp.h = gp.h;
  dp.hmax_part = ws.hmax_part;
  dp.n_hparts = gu_grid;
  dp.B = B;
  dp.y = static_cast<__nv_bfloat16*>(y);
  dp.y_copy = static_cast<__nv_bfloat16*>(ys_copy);
  dp.ss_out = static_cast<CSum*>(ss_out);
  dp.err = err;
  if (fmt == 0)
    e = launch(down_kernel<0, F4_DN_STAGES>, DN_TILES, DN_THREADS, down_smem_bytes<0, F4_DN_STAGES>(B), st, true,
               dp);
  else
    e = launch(down_kernel<1, B16_DN_STAGES>, DN_TILES, DN_THREADS, down_smem_bytes<1, B16_DN_STAGES>(B), st,
               true, dp);
  return e;
}

}  // namespace flint
