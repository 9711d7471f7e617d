// Shared constants and sm_103a PTX helpers of the Flint MoE kernels.
//
// Packed expert layout (written by the packer, read by the decode kernels).
// An expert is [64 gate/up tiles][128 down tiles].  A tile is 16 weight rows
// cut into K-slices of 256 columns; one warp consumes one slice with 16
// mma.m16n8k16 steps (one 16-column NVFP4 block per step).
//   gate/up tile r: tile rows 0..7 = gate rows 8r..8r+7, rows 8..15 = up rows
//     8r..8r+7, so the accumulator thread holding gate row j holds up row j
//     too (SiLU*up needs no exchange); 8 slices cover K = 2048.
//   down tile r: rows 16r..16r+15, 2 slices cover K = 512.
// NVFP4 slice (2304 B): codes [4 chunks][32 lanes][16 B] + scales [2][8][16 B]
//   lane L = 4g + t of chunk c holds, for the 4 blocks kb = 4c + j, the bytes
//   {row g byte t, row g+8 byte t, row g byte t+4, row g+8 byte t+4} of block
//   kb -- exactly the A-fragment registers {a0a1, a2a3, a4a5, a6a7} of one
//   mma.m16n8k16 after an e2m1x2 -> f16x2 convert of each byte.
//   scales: half h, group g: 8 blocks x (row g, row g+8) E4M3 bytes.
// BF16 slice (8192 B): [16 blocks][32 lanes][16 B] A-fragment registers.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace flint {

constexpr int H = 2048;
constexpr int E = 256;
constexpr int NE = E + 1;  // routed + shared; expert E is the shared expert
constexpr int I = 512;
constexpr int TOPK = 6;
constexpr int BMAX = 8;
constexpr int MAX_SLOTS = 1 + BMAX * TOPK;  // shared + up to 48 unique routed

constexpr int GU_TILES = 2 * I / 16;  // 64
constexpr int DN_TILES = H / 16;      // 128
constexpr int GU_SLICES = H / 256;    // 8
constexpr int DN_SLICES = I / 256;    // 2

constexpr int F4_SLICE = 2304;
constexpr int F4_CODES = 2048;
constexpr int F4_GU_TILE = GU_SLICES * F4_SLICE;  // 18432
constexpr int F4_DN_TILE = DN_SLICES * F4_SLICE;  // 4608
constexpr size_t F4_GU_BYTES = (size_t)GU_TILES * F4_GU_TILE;  // 1179648
constexpr size_t F4_EXPERT = F4_GU_BYTES + (size_t)DN_TILES * F4_DN_TILE;  // 1769472

constexpr int B16_SLICE = 8192;
constexpr int B16_GU_TILE = GU_SLICES * B16_SLICE;  // 65536
constexpr int B16_DN_TILE = DN_SLICES * B16_SLICE;  // 16384
constexpr size_t B16_GU_BYTES = (size_t)GU_TILES * B16_GU_TILE;
constexpr size_t B16_EXPERT = B16_GU_BYTES + (size_t)DN_TILES * B16_DN_TILE;  // 6291456

// Error bits recorded in the device error word.
constexpr unsigned ERR_WAIT_FULL = 1u;
constexpr unsigned ERR_WAIT_EMPTY = 2u;
constexpr unsigned ERR_DRAIN = 4u;
// The prefill router's tensor-core logit of a candidate expert was further
// from the exact logit than a quarter of the error bound assumed for it; the
// token's routing was redone with every logit exact (results stay correct).
constexpr unsigned ERR_ROUTER_BOUND = 8u;
// A kernel found its dynamic shared memory misaligned for its layout and did
// no work.
constexpr unsigned ERR_LAYOUT = 16u;

// A wait of the persistent decode kernel for data written by another thread
// block gave up (its cycle limit ran out); the call was abandoned.
constexpr unsigned ERR_POLL = 32u;

// A bounded wait gives up after about one second at the maximum SM clock.
constexpr long long WAIT_LIMIT_CYCLES = 2000000000LL;

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity to complete; false after the limit.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > WAIT_LIMIT_CYCLES) return false;
  }
  return true;
}

// L2 policy for weights that are read once per step.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// L2 policy for small activations that every CTA reads.
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Requests `bytes` at gsrc into L2 (no destination, nothing to wait for).
// gsrc 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* gsrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gsrc), "r"(bytes) : "memory");
}

// One TMA bulk copy global -> shared, completion counted on `bar` in bytes.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* sdst, const void* gsrc, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(sdst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Four bytes of two E2M1 codes each -> four f16x2 (low nibble -> low half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t& h0, uint32_t& h1, uint32_t& h2,
                                                uint32_t& h3) {
  asm("{\n .reg .b8 a0, a1, a2, a3;\n mov.b32 {a0, a1, a2, a3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, a0;\n cvt.rn.f16x2.e2m1x2 %1, a1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, a2;\n cvt.rn.f16x2.e2m1x2 %3, a3;\n}\n"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(w));
}
// Two E4M3 bytes -> f16x2 (low byte -> low half).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t r;
  const uint16_t v = static_cast<uint16_t>(two_bytes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}
__device__ __forceinline__ uint32_t hmul2_lo(uint32_t a, uint32_t s) {
  __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), __low2half2(*reinterpret_cast<const __half2*>(&s)));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t hmul2_hi(uint32_t a, uint32_t s) {
  __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), __high2half2(*reinterpret_cast<const __half2*>(&s)));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ unsigned redux_max(unsigned v) {
  unsigned r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}
__device__ __forceinline__ unsigned redux_min(unsigned v) {
  unsigned r;
  asm volatile("redux.sync.min.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

// Asynchronous 16-byte global -> shared copies (L2 only), completed per thread.
__device__ __forceinline__ void cp_async16(void* sdst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(sdst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n cp.async.wait_all;" ::: "memory");
}

// Packed fp32 pairs (sm_100+): two IEEE round-to-nearest operations per instruction.
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ------------------------------------------------------- compensated summation
// Knuth's TwoSum: s + e == a + b exactly.  Used where a rounding decision
// (bf16 logits that feed top-k, the RMSNorm scale) must not depend on the
// order of accumulation: products of bf16 values are exact in fp32, and the
// compensated sum rounds to the same fp32 as the exact sum.
struct CSum {
  float s, c;
};
__device__ __forceinline__ void cs_add(CSum& x, float p) {
  const float s = __fadd_rn(x.s, p);
  const float z = __fsub_rn(s, x.s);
  const float e = __fadd_rn(__fsub_rn(x.s, __fsub_rn(s, z)), __fsub_rn(p, z));
  x.s = s;
  x.c = __fadd_rn(x.c, e);
}
__device__ __forceinline__ void cs_merge(CSum& x, const CSum& y) {
  cs_add(x, y.s);
  x.c = __fadd_rn(x.c, y.c);
}
__device__ __forceinline__ CSum cs_warp_reduce(CSum x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    CSum y;
    y.s = __shfl_xor_sync(0xffffffffu, x.s, off);
    y.c = __shfl_xor_sync(0xffffffffu, x.c, off);
    cs_merge(x, y);
  }
  return x;
}
__device__ __forceinline__ float cs_value(const CSum& x) { return __fadd_rn(x.s, x.c); }

// Two independent compensated sums in packed fp32 pairs (same TwoSum steps).
struct CSum2 {
  uint64_t s, c;
};
__device__ __forceinline__ void cs2_add(CSum2& x, uint64_t p) {
  const uint64_t s = f2add(x.s, p);
  const uint64_t z = f2sub(s, x.s);
  const uint64_t e = f2add(f2sub(x.s, f2sub(s, z)), f2sub(p, z));
  x.s = s;
  x.c = f2add(x.c, e);
}
__device__ __forceinline__ void cs2_split(const CSum2& x, CSum& lo, CSum& hi) {
  f2unpack(x.s, lo.s, hi.s);
  f2unpack(x.c, lo.c, hi.c);
}

// ---------------------------------------------------------------- routing
// Result of sigmoid top-6 for a batch, laid out for the expert kernels.
// Slot 0 is the shared expert; slots 1..n_slots-1 are the distinct routed
// experts chosen by any token, in ascending expert order.
struct Routing {
  int n_slots;
  int slot_expert[MAX_SLOTS];
  uint32_t slot_mask[MAX_SLOTS];  // bit t: token t uses the slot
  float slot_w[MAX_SLOTS][BMAX];  // routing weight of token t (shared: 1)
  int ids[BMAX][TOPK];
  float w[BMAX][TOPK];
  uint16_t lg[BMAX][TOPK];        // bf16 bits of the selected logits
  uint32_t umask[8];              // union of the selected experts, 256 bits
  int ubase[8];                   // exclusive prefix of popc(umask)
};

// Sigmoid top-6 of one token by one warp.  Lane l holds experts 8l..8l+7 of
// the bf16 logits row (global memory, written by the router kernel):
//   s = 1 / (1 + exp(-logit)) in fp32; top-6 by s, ties to the lower index;
//   w_j = s_j / sum of the 6 selected s (fp32, summed in selection order).
// Fast path: for bf16 logits v with 2^-12 <= |v|, -80 < v < 8, the correctly
// rounded fp32 sigmoid of v exceeds that of the next smaller bf16 value by at
// least 4 fp32 ulps (checked exhaustively over all bf16 values); outside that
// band fp32 scores of distinct logits can coincide (s rounds to 0.5 near 0,
// to 1 above ~17, underflows below ~-87).  So if all 7 best candidates by
// (logit desc, index asc) lie in the band, that order equals the order by
// (s desc, index asc) exactly, and a 32-bit key (order-preserving logit bits,
// then 255 - index) selects with one warp max per pick.  Otherwise the
// selection is redone on the fp32 scores.  Lanes 0..5 store ids and weights.
__device__ __forceinline__ uint4 load_logits(const __nv_bfloat16* __restrict__ row, int lane) {
  return __ldcg(reinterpret_cast<const uint4*>(row) + lane);
}
__device__ __forceinline__ float sigmoid_f32(float lg) { return __frcp_rn(__fadd_rn(1.0f, expf(-lg))); }

// Selection part of sigmoid top-6: every lane ends with the 6 selected expert
// indices (descending score, ties to the lower index) and the bf16 bits of
// their logits.
__device__ __forceinline__ void warp_top6_core(const uint4 raw, int lane, int (&sel_i)[TOPK],
                                               uint32_t (&sel_lg)[TOPK]) {
  const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t hb[8], key[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    hb[i] = (wv[i >> 1] >> ((i & 1) * 16)) & 0xFFFFu;
    const uint32_t ord = (hb[i] & 0x8000u) ? (~hb[i] & 0xFFFFu) : (hb[i] | 0x8000u);
    key[i] = (ord << 16) | (255u - (uint32_t)(lane * 8 + i));
  }
  // Fast path: top-7 by key (the 7th only to bound the candidates).  Each lane
  // sorts its 8 keys (descending, a 19-comparator network); the warp maximum of
  // the lane heads is the next key, and the lane that owned it pops its head.
  // Keys are distinct (they carry the expert index).
  {
#define FLINT_CAS(a, b)                              \
  {                                                  \
    const uint32_t hi_ = max(key[a], key[b]);        \
    key[b] = min(key[a], key[b]);                    \
    key[a] = hi_;                                    \
  }
    FLINT_CAS(0, 2) FLINT_CAS(1, 3) FLINT_CAS(4, 6) FLINT_CAS(5, 7)
    FLINT_CAS(0, 4) FLINT_CAS(1, 5) FLINT_CAS(2, 6) FLINT_CAS(3, 7)
    FLINT_CAS(0, 1) FLINT_CAS(2, 3) FLINT_CAS(4, 5) FLINT_CAS(6, 7)
    FLINT_CAS(2, 4) FLINT_CAS(3, 5)
    FLINT_CAS(1, 4) FLINT_CAS(3, 6)
    FLINT_CAS(1, 2) FLINT_CAS(3, 4) FLINT_CAS(5, 6)
#undef FLINT_CAS
  }
  uint32_t sel_key[TOPK + 1];
#pragma unroll
  for (int k = 0; k < TOPK + 1; ++k) {
    const uint32_t m = redux_max(key[0]);
    sel_key[k] = m;
    if (key[0] == m) {
#pragma unroll
      for (int i = 0; i < 7; ++i) key[i] = key[i + 1];
      key[7] = 0u;
    }
  }
  bool exact_by_logit = true;
#pragma unroll
  for (int k = 0; k < TOPK + 1; ++k) {
    const uint32_t ord = sel_key[k] >> 16;
    const uint32_t bits = (ord & 0x8000u) ? (ord & 0x7FFFu) : (~ord & 0xFFFFu);
    const uint32_t mag = bits & 0x7FFFu;  // 0x3980 = 2^-12, 0x4100 = 8, 0x42A0 = 80
    const bool in_band = mag >= 0x3980u && ((bits & 0x8000u) ? mag < 0x42A0u : mag < 0x4100u);
    exact_by_logit = exact_by_logit && in_band;
  }
  if (exact_by_logit) {
#pragma unroll
    for (int k = 0; k < TOPK; ++k) {
      const uint32_t ord = sel_key[k] >> 16;
      sel_lg[k] = (ord & 0x8000u) ? (ord & 0x7FFFu) : (~ord & 0xFFFFu);
      sel_i[k] = 255 - (int)(sel_key[k] & 0xFFu);
    }
  } else {
    uint32_t bits[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) bits[i] = __float_as_uint(sigmoid_f32(__uint_as_float(hb[i] << 16)));
    uint32_t tk2 = 0u;
#pragma unroll
    for (int k = 0; k < TOPK; ++k) {
      uint32_t best = 0u, bidx = 0xFFFFFFFFu;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (!((tk2 >> i) & 1u) && (bidx == 0xFFFFFFFFu || bits[i] > best)) {
          best = bits[i];
          bidx = lane * 8 + i;
        }
      }
      const uint32_t m = redux_max(best);
      const uint32_t win = redux_min(best == m ? bidx : 0xFFFFFFFFu);
      if ((win >> 3) == (uint32_t)lane) tk2 |= 1u << (win & 7u);
      uint32_t lb = 0u;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if ((int)(win & 7u) == i) lb = hb[i];
      sel_lg[k] = __shfl_sync(0xffffffffu, lb, (int)(win >> 3));
      sel_i[k] = (int)win;
    }
  }
}

// Weight part: s = fp32 sigmoid of each selected logit, w_j = s_j / sum of
// the 6 (fp32, summed in selection order); lanes 0..5 store w_out[lane].
__device__ __forceinline__ void warp_top6_weights(const uint32_t (&sel_lg)[TOPK], int lane, float* w_out) {
  float sel_s[TOPK];
#pragma unroll
  for (int k = 0; k < TOPK; ++k) sel_s[k] = sigmoid_f32(__uint_as_float(sel_lg[k] << 16));
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < TOPK; ++k) sum = __fadd_rn(sum, sel_s[k]);
  if (lane < TOPK) {
    float ws = 0.f;
#pragma unroll
    for (int k = 0; k < TOPK; ++k)
      if (k == lane) ws = sel_s[k];
    w_out[lane] = __fdiv_rn(ws, sum);
  }
}

// Lanes 0..5 store the selection (ids, logit bits) and mark it in umask.
__device__ __forceinline__ void warp_top6_store(const int (&sel_i)[TOPK], const uint32_t (&sel_lg)[TOPK], int lane,
                                                int* ids_out, uint16_t* lg_out, uint32_t* umask) {
  if (lane < TOPK) {
    int wi = 0;
    uint32_t wl = 0u;
#pragma unroll
    for (int k = 0; k < TOPK; ++k)
      if (k == lane) {
        wi = sel_i[k];
        wl = sel_lg[k];
      }
    ids_out[lane] = wi;
    if (lg_out) lg_out[lane] = (uint16_t)wl;
    atomicOr(&umask[wi >> 5], 1u << (wi & 31));
  }
}

__device__ __forceinline__ void warp_topk(const uint4 raw, int lane, int* ids_out, float* w_out,
                                          uint32_t* umask) {
  int sel_i[TOPK];
  uint32_t sel_lg[TOPK];
  warp_top6_core(raw, lane, sel_i, sel_lg);
  warp_top6_store(sel_i, sel_lg, lane, ids_out, nullptr, umask);
  warp_top6_weights(sel_lg, lane, w_out);
}

// Builds the slot table from the per-token selections (one warp).  Slot 0 is
// the shared expert; slots 1.. are the distinct routed experts in ascending
// order.  Experts part: n_slots, slot_expert, slot_mask (requires r.umask and
// r.ids complete and slot_mask zeroed).  Weights part: slot_w (requires r.w
// and slot_w zeroed).
__device__ __forceinline__ int slot_of(const Routing& r, int e) {
  const int wd = e >> 5;
  return 1 + r.ubase[wd] + __popc(r.umask[wd] & ((1u << (e & 31)) - 1u));
}

__device__ __forceinline__ void warp_slot_experts(Routing& r, int B, int lane) {
  const uint32_t m = lane < 8 ? r.umask[lane] : 0u;
  const int cnt = __popc(m);
  int incl = cnt;
#pragma unroll
  for (int off = 1; off < 8; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  const int base = incl - cnt;
  if (lane < 8) {
    r.ubase[lane] = base;
    uint32_t mm = m;
    int j = 0;
    while (mm) {
      const int b = __ffs(mm) - 1;
      mm &= mm - 1;
      r.slot_expert[1 + base + j] = lane * 32 + b;
      ++j;
    }
  }
  const int total = __shfl_sync(0xffffffffu, incl, 7);
  if (lane == 0) {
    r.n_slots = 1 + total;
    r.slot_expert[0] = E;
    r.slot_mask[0] = (1u << B) - 1u;
  }
  __syncwarp();
  for (int q = lane; q < B * TOPK; q += 32) {
    const int t = q / TOPK, j = q % TOPK;
    atomicOr(&r.slot_mask[slot_of(r, r.ids[t][j])], 1u << t);
  }
  __syncwarp();
}

__device__ __forceinline__ void warp_slot_weights(Routing& r, int B, int lane) {
  if (lane < B) r.slot_w[0][lane] = 1.0f;
  for (int q = lane; q < B * TOPK; q += 32) {
    const int t = q / TOPK, j = q % TOPK;
    r.slot_w[slot_of(r, r.ids[t][j])][t] = r.w[t][j];
  }
  __syncwarp();
}

__device__ __forceinline__ void warp_slot_table(Routing& r, int B, int lane) {
  warp_slot_experts(r, B, lane);
  warp_slot_weights(r, B, lane);
}

__device__ __forceinline__ void zero_routing(Routing& r, int tid, int nthreads) {
  for (int i = tid; i < MAX_SLOTS * (BMAX + 2); i += nthreads) {
    const int s = i / (BMAX + 2), k = i % (BMAX + 2);
    if (k < BMAX) r.slot_w[s][k] = 0.f;
    else if (k == BMAX) r.slot_mask[s] = 0u;
    else r.slot_expert[s] = -1;
  }
  if (tid < 8) r.umask[tid] = 0u;
}

}  // namespace flint
