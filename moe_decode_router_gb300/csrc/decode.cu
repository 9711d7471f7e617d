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
#include "decode_common.cuh"
#include "flint_internal.h"

namespace flint {

// ------------------------------------------------------------------ router

// x_hat in mma B-fragment order: [8 K-slices][32 lanes][16 blocks][2 regs]
// (u32 each, two 16-bit values), lane = 4 * token + t.  A consumer warp of
// slice w loads its 16 blocks' fragments with eight 16-byte loads.
constexpr int XFRAG_WORDS = 8 * 32 * 16 * 2;
static_assert(decode_ws_bytes(1) == ws_align256((size_t)BMAX * E * 2) + ws_align256((size_t)BMAX * H * 2) +
                                        2 * ws_align256((size_t)XFRAG_WORDS * 4) + ws_align256(BMAX * 4) +
                                        ws_align256((size_t)MAX_SLOTS * BMAX * I * 2) + ws_align256(BMAX * 4) +
                                        ws_align256((size_t)DN_TILES * BMAX * sizeof(CSum)) +
                                        ws_align256((size_t)BMAX * H * 2),
              "workspace size and carve-up must agree");

struct RouterParams {
  const __nv_bfloat16* x;       // [B][H]
  const CSum* ss_in;            // [DN_TILES][8] sum-of-squares partials of x, or null
  const __nv_bfloat16* norm_w;  // [H] or null
  const __nv_bfloat16* wr;      // [E][H]
  float eps;
  int want_f16;
  __nv_bfloat16* logits;   // [B][E]
  uint32_t* xfrag_f16;     // x_hat * 2^xh_exp[token] in f16, fragment order
  uint32_t* xfrag_bf16;    // x_hat in bf16, fragment order
  int* xh_exp;             // [B]
};

// Router logits logit[t][e] = bf16( sum_k x_hat[t][k] * W_r[e][k] ).  The sum
// is accumulated error-free (products of bf16 values are exact in fp32;
// TwoSum carries the rounding error), so the bf16 logit that decides the top-6
// is the correctly rounded value whatever the order of accumulation.  CTA e
// owns expert e; thread k owns columns [8k, 8k+8); token pairs share packed
// fp32x2 arithmetic.
template <int NB, int EPC>
__global__ void __launch_bounds__(256, 2) router_kernel(const RouterParams p) {
  constexpr int NP = (NB + 1) / 2;
  constexpr int VP = Pow2Ceil<NB * EPC>::value;
  constexpr int SH = 5 - Log2<VP>::value;
  __shared__ CSum red[8][VP];
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

  // Issue every dependent load before using any of them (one round trip).
  uint4 xraw[NB];
#pragma unroll
  for (int t = 0; t < NB; ++t) xraw[t] = __ldcg(reinterpret_cast<const uint4*>(p.x + (size_t)t * H + k0));
  const bool ss_given = has_norm && p.ss_in != nullptr;
  CSum ssp[DN_TILES / 32];
  if (ss_given && warp < NB) {
#pragma unroll
    for (int j = 0; j < DN_TILES / 32; ++j) {
      const float2 v = __ldcg(reinterpret_cast<const float2*>(p.ss_in + (lane + 32 * j) * BMAX + warp));
      ssp[j] = CSum{v.x, v.y};
    }
  }
  float xv[2 * NP][8];
#pragma unroll
  for (int t = 0; t < 2 * NP; ++t) {
    if (t < NB) {
      bf16x8_to_f32(xraw[t], xv[t]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) xv[t][i] = 0.f;
    }
  }

  if (has_norm) {
    if (ss_given) {
      // Partials written by the previous sublayer's down kernel.
      if (warp < NB) {
        CSum a = ssp[0];
#pragma unroll
        for (int j = 1; j < DN_TILES / 32; ++j) cs_merge(a, ssp[j]);
        a = cs_warp_reduce(a);
        if (lane == 0) {
          const float ms = __fmul_rn(cs_value(a), 1.0f / (float)H);
          rscale[warp] = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, p.eps)));
        }
      }
    } else {
      CSum2 ss2[NP];
#pragma unroll
      for (int q = 0; q < NP; ++q) ss2[q] = CSum2{0ull, 0ull};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int q = 0; q < NP; ++q) {
          const uint64_t v = f2pack(xv[2 * q][i], xv[2 * q + 1][i]);
          cs2_add(ss2[q], f2mul(v, v));
        }
      constexpr int VN = Pow2Ceil<NB>::value;
      constexpr int SHN = 5 - Log2<VN>::value;
      CSum ss[VN];
#pragma unroll
      for (int v = 0; v < VN; ++v) ss[v] = CSum{0.f, 0.f};
#pragma unroll
      for (int q = 0; q < NP; ++q) {
        CSum lo, hi;
        cs2_split(ss2[q], lo, hi);
        ss[2 * q] = lo;
        if (2 * q + 1 < VN) ss[2 * q + 1] = hi;
      }
      const CSum tot = cs_reduce_scatter<VN>(ss, lane);
      if ((lane & ((1 << SHN) - 1)) == 0) red[warp][lane >> SHN] = tot;
      __syncthreads();
      if (tid < NB) {
        CSum a = red[0][tid];
#pragma unroll
        for (int w = 1; w < 8; ++w) cs_merge(a, red[w][tid]);
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

  CSum2 d2[EPC][NP];
#pragma unroll
  for (int j = 0; j < EPC; ++j)
#pragma unroll
    for (int q = 0; q < NP; ++q) d2[j][q] = CSum2{0ull, 0ull};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
#pragma unroll
    for (int j = 0; j < EPC; ++j) {
      const uint64_t w2 = f2pack(wf[j][i], wf[j][i]);
#pragma unroll
      for (int q = 0; q < NP; ++q) cs2_add(d2[j][q], f2mul(f2pack(xv[2 * q][i], xv[2 * q + 1][i]), w2));
    }
  }
  {
    // value v = j * NB + t (expert e0 + j, token t)
    CSum d[VP];
#pragma unroll
    for (int v = 0; v < VP; ++v) d[v] = CSum{0.f, 0.f};
#pragma unroll
    for (int j = 0; j < EPC; ++j)
#pragma unroll
      for (int q = 0; q < NP; ++q) {
        CSum lo, hi;
        cs2_split(d2[j][q], lo, hi);
        d[j * NB + 2 * q] = lo;
        if (2 * q + 1 < NB) d[j * NB + 2 * q + 1] = hi;
      }
    const CSum tot = cs_reduce_scatter<VP>(d, lane);
    __syncthreads();  // red may still hold the norm partials
    if ((lane & ((1 << SH) - 1)) == 0) red[warp][lane >> SH] = tot;
  }
  __syncthreads();
  if (tid < NB * EPC) {
    CSum a = red[0][tid];
#pragma unroll
    for (int w = 1; w < 8; ++w) cs_merge(a, red[w][tid]);
    p.logits[(size_t)(tid % NB) * E + e0 + tid / NB] = __float2bfloat16_rn(cs_value(a));
  }

  // Every CTA computed the same x_hat.  CTA b < 8 publishes K-slice b
  // (columns 256 b .. 256 b + 255, held by its warp b) in mma fragment order:
  // columns 8k..8k+7 are block kb = (k % 32) / 2, register r = k % 2 of
  // K-slice k / 32, lanes 4t..4t+3 of token t.  BF16 weights take x_hat in
  // bf16; NVFP4 takes it in f16 scaled by 2^xh_exp[t], the exponent from the
  // token's largest |x_hat|, which each publishing CTA reduces itself.  (One
  // CTA publishing everything was the router's last CTA by 1.8 us at 8 tokens.)
  if (blockIdx.x < 8) {
    const int kb = (k0 & 255) >> 4, rr = (k0 >> 3) & 1;  // K-slice k0 >> 8 == warp
    const bool mine = warp == (int)blockIdx.x;
    if (!p.want_f16) {
      if (mine) {
#pragma unroll
        for (int t = 0; t < NB; ++t)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            p.xfrag_bf16[((warp * 32 + 4 * t + i) * 16 + kb) * 2 + rr] =
                (__float_as_uint(xv[t][2 * i]) >> 16) | (__float_as_uint(xv[t][2 * i + 1]) & 0xFFFF0000u);
      }
    } else {
#pragma unroll
      for (int t = 0; t < NB; ++t) {
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(xv[t][i]));
        const unsigned wm = redux_max(__float_as_uint(m));
        if (lane == 0) atomicMax(&xmax[t], wm);
      }
      __syncthreads();
      if (mine) {
#pragma unroll
        for (int t = 0; t < NB; ++t) {
          const int ex = f16_range_exp(__uint_as_float(xmax[t]));
          const float sc = exp2i(ex);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __half2 hv = __floats2half2_rn(__fmul_rn(xv[t][2 * i], sc), __fmul_rn(xv[t][2 * i + 1], sc));
            p.xfrag_f16[((warp * 32 + 4 * t + i) * 16 + kb) * 2 + rr] = *reinterpret_cast<const uint32_t*>(&hv);
          }
          if (blockIdx.x == 0 && lane == 0) p.xh_exp[t] = ex;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ gate/up

struct GateUpParams {
  const uint8_t* experts;
  const float* tscale;          // [NE][2] (NVFP4)
  const __nv_bfloat16* logits;  // [B][E]
  const uint32_t* xfrag;        // x_hat B fragments: f16 (NVFP4) or bf16
  const int* xh_exp;            // [B] (NVFP4)
  int B;
  __nv_bfloat16* h;             // [MAX_SLOTS][BMAX][I]
  float* hmax_part;             // [gridDim.x][BMAX]
  int32_t* ids_out;             // [B][6] or null
  float* w_out;                 // [B][6] or null
  unsigned* err;
};

// 8 compute warps (one K slice each), 1 TMA producer warp, 2 epilogue warps.
constexpr int GU_COMPUTE_WARPS = 8;
constexpr int GU_PRODUCER_WARP = 8;
constexpr int GU_THREADS = 32 * (GU_COMPUTE_WARPS + 1 + 2);  // 352
constexpr int GU_RED = 4;  // depth of the partial-sum ring between compute and epilogue warps
constexpr int TSCALE_WORDS = ((NE * 2 + 3) / 4) * 4;  // per-expert (gate/up, down) scales, padded

template <int FMT, int STAGES>
__host__ __device__ constexpr size_t gateup_smem_bytes() {
  // [stages][red ring GU_RED x 8 x 128 fp32][tensor scales][full, empty][rfull, rempty][pad 16][Routing]
  // [first pair of each slot]
  return (size_t)STAGES * Fmt<FMT>::GU_TILE + GU_RED * 8 * 128 * 4 + TSCALE_WORDS * 4 + 2 * STAGES * 8 +
         2 * GU_RED * 8 + 16 + (sizeof(Routing) + 15) / 16 * 16 + MAX_SLOTS * 4;
}

// Items are (slot, row tile) pairs, item i = slot * 64 + tile; CTA b takes
// items b, b + G, b + 2G, ...  One item is one 18 KiB (NVFP4) bulk copy.  The
// 8 compute warps each multiply one K-slice of it and pass their partial sums
// through a ring of GU_RED buffers to the 2 epilogue warps, which reduce them
// in a fixed order and apply SiLU*up.  Compute warps never wait on the
// epilogue unless the ring is full.
template <int FMT, int STAGES>
__global__ void __launch_bounds__(GU_THREADS, 1) gateup_kernel(const GateUpParams p) {
  using F = Fmt<FMT>;
  constexpr int TILE = F::GU_TILE;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  float* red = reinterpret_cast<float*>(smem + (size_t)STAGES * TILE);  // [GU_RED][8][128], 16-byte aligned
  float* ts_s = red + GU_RED * 8 * 128;                                   // [NE][2]
  uint64_t* full = reinterpret_cast<uint64_t*>(ts_s + TSCALE_WORDS);
  uint64_t* empty = full + STAGES;
  uint64_t* rfull = empty + STAGES;
  uint64_t* rempty = rfull + GU_RED;
  Routing& R = *reinterpret_cast<Routing*>(reinterpret_cast<uint8_t*>(rempty + GU_RED) + 16);
  int* slot_pair0 = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(&R) + (sizeof(Routing) + 15) / 16 * 16);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, bid = blockIdx.x;
  const int B = p.B;
  if (FMT == 0)
    for (int q = tid; q < NE * 2; q += GU_THREADS) ts_s[q] = __ldg(p.tscale + q);  // constants
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], GU_COMPUTE_WARPS);
    }
#pragma unroll
    for (int b = 0; b < GU_RED; ++b) {
      mbar_init(&rfull[b], GU_COMPUTE_WARPS);
      mbar_init(&rempty[b], 2);
    }
    fence_mbar_init();
  }
  zero_routing(R, tid, GU_THREADS);
  __syncthreads();

  const uint64_t pol = l2_evict_first();
  int issued = 0;
  if (tid == GU_PRODUCER_WARP * 32) {
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
  // The down kernel may start now: before its own dependency wait it reads
  // only the router's logits, which are final once this wait has returned.
  pdl_trigger();
  const int g = lane >> 2;
  // The routing input first, alone: the top-k waits on it.  The B fragments
  // (every CTA reads all of x_hat) are requested only after the routing, while
  // the first routed tiles are in flight.
  uint4 lraw = make_uint4(0u, 0u, 0u, 0u);
  if (warp < B) lraw = load_logits(p.logits + (size_t)warp * E, lane);
  if (warp < B) {
    // The selection alone decides which tiles to read; the routing weights are
    // only reported (CTA 0), so no other CTA computes them.
    int sel_i[TOPK];
    uint32_t sel_lg[TOPK];
    warp_top6_core(lraw, lane, sel_i, sel_lg);
    warp_top6_store(sel_i, sel_lg, lane, R.ids[warp], nullptr, R.umask);
    if (bid == 0 && p.w_out) warp_top6_weights(sel_lg, lane, R.w[warp]);
  }
  __syncthreads();
  int n_slots = 1;
#pragma unroll
  for (int i = 0; i < 8; ++i) n_slots += __popc(R.umask[i]);
  const int n_items = n_slots * GU_TILES;
  if (bid == 0 && tid < B * TOPK) {
    if (p.ids_out) p.ids_out[tid] = R.ids[tid / TOPK][tid % TOPK];
    if (p.w_out) p.w_out[tid] = R.w[tid / TOPK][tid % TOPK];
  }

  if (warp == GU_PRODUCER_WARP) {
    // The routed tiles are requested as soon as the selection is known.  Slot
    // k >= 1 is the (k-1)-th expert of the union in ascending order: the lane
    // holding that word of the union (lanes 0..7, a prefix count gives each
    // word's first slot) finds the bit.  The slot table itself is built by
    // the epilogue warps, its only readers.
    const uint32_t m = lane < 8 ? R.umask[lane] : 0u;
    const int cnt = __popc(m);
    int incl = cnt;
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    const int base = incl - cnt;
    issued = __shfl_sync(0xffffffffu, issued, 0);  // the prologue's copies (lane 0)
    for (int n = issued;; ++n) {
      const int i = bid + n * G;
      if (i >= n_items) break;
      const int slot = i / GU_TILES;
      int e = E;
      if (slot > 0) {
        const int k = slot - 1;
        const bool own = lane < 8 && k >= base && k < incl;
        uint32_t mm = m;
        for (int r = own ? k - base : 0; r > 0; --r) mm &= mm - 1u;
        const int el = own ? lane * 32 + __ffs(mm) - 1 : 0;
        e = __shfl_sync(0xffffffffu, el, __ffs(__ballot_sync(0xffffffffu, own)) - 1);
      }
      const int s = n % STAGES;
      int ok = 1;
      if (lane == 0) {
        if (n >= STAGES && !mbar_wait(&empty[s], ((n / STAGES) - 1) & 1)) {
          atomicOr(p.err, ERR_WAIT_EMPTY);
          ok = 0;
        } else {
          mbar_arrive_expect_tx(&full[s], TILE);
          bulk_g2s(stages + (size_t)s * TILE, p.experts + (size_t)e * F::EXPERT + (size_t)(i % GU_TILES) * TILE,
                   TILE, &full[s], pol);
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      issued = n + 1;
    }
    if (lane == 0) {
      // Do not leave copies in flight: wait for the last use of every stage.
      for (int n = issued - STAGES; n < issued; ++n) {
        if (n < 0) continue;
        if (!mbar_wait(&full[n % STAGES], (n / STAGES) & 1)) atomicOr(p.err, ERR_DRAIN);
      }
    }
    return;
  }

  uint32_t bfr[16][2];
  if (warp < GU_COMPUTE_WARPS) {
    if (g < B) {
      const uint4* src = reinterpret_cast<const uint4*>(p.xfrag + (size_t)(warp * 32 + lane) * 32);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint4 v = __ldcg(src + q);
        bfr[2 * q][0] = v.x;
        bfr[2 * q][1] = v.y;
        bfr[2 * q + 1][0] = v.z;
        bfr[2 * q + 1][1] = v.w;
      }
    } else {
#pragma unroll
      for (int kb = 0; kb < 16; ++kb) bfr[kb][0] = bfr[kb][1] = 0u;
    }
  }
  if (warp < GU_COMPUTE_WARPS) {
    // ---- compute warps: warp w multiplies K slice w of every tile
    for (int n = 0;; ++n) {
      const int i = bid + n * G;
      if (i >= n_items) break;
      const int s = n % STAGES;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (mbar_wait(&full[s], (n / STAGES) & 1)) {
        F::slice(stages + (size_t)s * TILE + warp * F::SLICE, lane, bfr, acc);
      } else {
        atomicOr(p.err, ERR_WAIT_FULL);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      const int b = n % GU_RED;
      if (n >= GU_RED && !mbar_wait(&rempty[b], ((n / GU_RED) - 1) & 1)) atomicOr(p.err, ERR_WAIT_EMPTY);
      float* rb = red + b * 1024;
#pragma unroll
      for (int j = 0; j < 4; ++j) rb[warp * 128 + j * 32 + lane] = acc[j];
      __syncwarp();
      if (lane == 0) mbar_arrive(&rfull[b]);
    }
    return;
  }

  // ---- epilogue warps: thread = (token ep_tk, gate/up row ep_row of the tile)
  const int et = tid - (GU_PRODUCER_WARP + 1) * 32;
  // The slot table (experts and token masks; this kernel needs no weights),
  // built while the first tiles are in flight, and the first pair of each
  // slot: h is stored by pair (slot, token), numbered slot by slot and token
  // by token, so the down kernel stages all of it with one copy.
  if (et < 32) {
    warp_slot_experts(R, B, lane);
    const int n_slots_w = R.n_slots;
    int run = 0;
    for (int c0 = 0; c0 < n_slots_w; c0 += 32) {
      const int u = c0 + lane;
      const int cnt = u < n_slots_w ? __popc(R.slot_mask[u]) : 0;
      int incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      if (u < n_slots_w) slot_pair0[u] = run + incl - cnt;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  named_bar_sync(1, 64);
  const int ep_tk = et >> 3, ep_row = et & 7;
  float xs = 1.f;  // 2^-exponent of token ep_tk (NVFP4)
  if (FMT == 0 && ep_tk < B) xs = exp2i(-__ldcg(p.xh_exp + ep_tk));
  float hm = 0.f;
  const int og = red_off(ep_row, ep_tk), ou = red_off(ep_row + 8, ep_tk);
  for (int n = 0;; ++n) {
    const int i = bid + n * G;
    if (i >= n_items) break;
    const int b = n % GU_RED;
    if (!mbar_wait(&rfull[b], (n / GU_RED) & 1)) {
      atomicOr(p.err, ERR_WAIT_FULL);
      break;
    }
    const float* rb = red + b * 1024;
    const int slot = i / GU_TILES, tile = i % GU_TILES;
    const uint32_t mask = slot == 0 ? ((1u << B) - 1u) : R.slot_mask[slot];
    if (ep_tk < B && ((mask >> ep_tk) & 1u)) {
      const int e = slot == 0 ? E : R.slot_expert[slot];
      float gsum = 0.f, usum = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        gsum += rb[w * 128 + og];
        usum += rb[w * 128 + ou];
      }
      const float f = FMT == 0 ? __fmul_rn(xs, ts_s[2 * e]) : 1.0f;
      const float gate = __fmul_rn(gsum, f);
      const float up = __fmul_rn(usum, f);
      const float silu = __fdiv_rn(gate, __fadd_rn(1.0f, expf(-gate)));
      const __nv_bfloat16 hv = __float2bfloat16_rn(__fmul_rn(silu, up));
      const int pair = slot_pair0[slot] + __popc(mask & ((1u << ep_tk) - 1u));
      p.h[(size_t)pair * I + tile * 8 + ep_row] = hv;
      hm = fmaxf(hm, fabsf(__bfloat162float(hv)));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&rempty[b]);
  }
  hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, 1));
  hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, 2));
  hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, 4));
  if (ep_row == 0) p.hmax_part[(size_t)bid * BMAX + ep_tk] = hm;
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

constexpr int MAX_HPARTS = 512;

template <int NG>
struct DnCfg {
  static constexpr int COMPUTE_WARPS = 2 * NG;  // NG slot groups x 2 K halves
  static constexpr int THREADS = 32 * (COMPUTE_WARPS + 1);
};

template <int FMT, int STAGES, int NG>
__host__ __device__ constexpr size_t down_smem_fixed() {
  // [stages][red (2NG) x 128 fp32][tensor scales][full, empty barriers, h barrier][hexp 8, misc 8 ints]
  // [pidx][pair token][Routing]
  return (size_t)STAGES * Fmt<FMT>::DN_TILE + DnCfg<NG>::COMPUTE_WARPS * 128 * 4 + TSCALE_WORDS * 4 +
         2 * STAGES * 8 + 8 + 64 + MAX_SLOTS * BMAX + 64 + sizeof(Routing);
}
template <int FMT, int STAGES, int NG>
size_t down_smem_bytes(int B) {
  return ((down_smem_fixed<FMT, STAGES, NG>() + 15) / 16) * 16 + (size_t)(1 + TOPK) * B * I * 2;
}

// CTA r owns output rows 16r..16r+15.  Slot u is consumed by warp group
// u % NG (two warps: the two 256-column halves of K) and lands in stage
// u % STAGES.  The parity wait on a stage's barrier is only sound if every use
// of a stage is consumed by the same group, in order; hence STAGES % NG == 0.
template <int FMT, int STAGES, int NG>
__global__ void __launch_bounds__(DnCfg<NG>::THREADS, 1) down_kernel(const DownParams p) {
  static_assert(STAGES % NG == 0, "each stage must belong to one consumer group");
  using F = Fmt<FMT>;
  constexpr int TILE = F::DN_TILE;
  constexpr int NCW = DnCfg<NG>::COMPUTE_WARPS;
  constexpr int NT = DnCfg<NG>::THREADS;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  float* red = reinterpret_cast<float*>(smem + (size_t)STAGES * TILE);  // [NCW][128], 16-byte aligned
  float* ts_s = red + NCW * 128;                                         // [NE][2]
  uint64_t* full = reinterpret_cast<uint64_t*>(ts_s + TSCALE_WORDS);
  uint64_t* empty = full + STAGES;
  uint64_t* hbar = empty + STAGES;                       // the staged h rows
  int* hexp = reinterpret_cast<int*>(hbar + 1);          // [8]
  int* misc = hexp + 8;                                  // [1] n_pairs
  uint8_t* pidx = reinterpret_cast<uint8_t*>(misc + 8);  // [MAX_SLOTS][8]
  uint8_t* psrc_tok = pidx + MAX_SLOTS * BMAX;           // [<= 56] token of pair
  Routing& R = *reinterpret_cast<Routing*>(psrc_tok + 64);
  uint16_t* hs = reinterpret_cast<uint16_t*>(smem + ((down_smem_fixed<FMT, STAGES, NG>() + 15) / 16) * 16);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rt = blockIdx.x;
  const int B = p.B;
  pdl_trigger();  // the next sublayer's router only prefetches constants before its wait
  // The routing of this sublayer is final: this kernel is launched only after
  // every gate/up CTA passed its dependency wait on the router.  Issue every
  // independent load first (tensor scales, logits), then consume them.
  constexpr int TS_PER_T = (NE * 2 + NT - 1) / NT;
  float tsv[TS_PER_T];
#pragma unroll
  for (int j = 0; j < TS_PER_T; ++j) {
    const int q = tid + j * NT;
    tsv[j] = (FMT == 0 && q < NE * 2) ? __ldg(p.tscale + q) : 0.f;
  }
  uint4 lraw = make_uint4(0u, 0u, 0u, 0u);
  if (warp < B) lraw = load_logits(p.logits + (size_t)warp * E, lane);
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 2);
    }
    mbar_init(hbar, 1);
    fence_mbar_init();
  }
  zero_routing(R, tid, NT);
#pragma unroll
  for (int j = 0; j < TS_PER_T; ++j) {
    const int q = tid + j * NT;
    if (q < NE * 2) ts_s[q] = tsv[j];
  }
  __syncthreads();
  if (warp < B) warp_topk(lraw, lane, R.ids[warp], R.w[warp], R.umask);
  __syncthreads();
  if (warp == 0) {
    warp_slot_table(R, B, lane);
    // compact (slot, token) pairs: pair index = prefix over slots of popc(mask)
    const int n_slots_w = R.n_slots;
    int base = 0;
    for (int c0 = 0; c0 < n_slots_w; c0 += 32) {
      const int u = c0 + lane;
      const uint32_t m = u < n_slots_w ? R.slot_mask[u] : 0u;
      const int cnt = __popc(m);
      int incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      int pi = base + incl - cnt;
      if (u < n_slots_w) {
#pragma unroll
        for (int tk = 0; tk < BMAX; ++tk) {
          if ((m >> tk) & 1u) {
            pidx[u * BMAX + tk] = (uint8_t)pi;
            psrc_tok[pi] = (uint8_t)tk;
            ++pi;
          }
        }
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) misc[1] = base;
  }
  __syncthreads();
  const int n_pairs = misc[1];
  const int n_slots = R.n_slots;
  const uint64_t pol = l2_evict_first();
  int issued = 0;
  if (tid == NCW * 32) {
    for (; issued < STAGES && issued < n_slots; ++issued) {
      const int e = R.slot_expert[issued];
      mbar_arrive_expect_tx(&full[issued], TILE);
      bulk_g2s(stages + (size_t)issued * TILE, p.experts + (size_t)e * F::EXPERT + F::GU_BYTES + (size_t)rt * TILE,
               TILE, &full[issued], pol);
    }
  }

  pdl_wait();  // gate/up of this sublayer is complete: h and hmax_part are final
  // h is stored by pair in the order of pidx: all of it is one copy, issued
  // first.  Then, with HBM idle, every NVFP4 tile beyond the ring is asked
  // into L2 at once, so the ring refills at L2 latency (BF16's 16 KB tiles
  // would take most of L2 at 8 tokens; measured slower there).
  if (tid == NCW * 32) {
    mbar_arrive_expect_tx(hbar, (uint32_t)(n_pairs * I * 2));
    bulk_g2s(hs, p.h, (uint32_t)(n_pairs * I * 2), hbar, l2_evict_last());
    if (FMT == 0)
      for (int n = STAGES; n < n_slots; ++n)
        bulk_prefetch_l2(p.experts + (size_t)R.slot_expert[n] * F::EXPERT + F::GU_BYTES + (size_t)rt * TILE, TILE);
  }
  if (FMT == 0 && warp < B) {
    float v[MAX_HPARTS / 32];
#pragma unroll
    for (int j = 0; j < MAX_HPARTS / 32; ++j) {
      const int q = lane + 32 * j;
      v[j] = q < p.n_hparts ? __ldcg(p.hmax_part + (size_t)q * BMAX + warp) : 0.f;
    }
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < MAX_HPARTS / 32; ++j) m = fmaxf(m, v[j]);
    const unsigned mb = redux_max(__float_as_uint(m));
    if (lane == 0) hexp[warp] = f16_range_exp(__uint_as_float(mb));
  }
  if (!mbar_wait(hbar, 0) && tid == 0) atomicOr(p.err, ERR_WAIT_FULL);
  __syncthreads();
  if (FMT == 0) {
    // bf16 h -> f16 h * 2^hexp[token], in place (each thread its own chunks).
    for (int idx = tid; idx < n_pairs * 64; idx += NT) {
      const int pr = idx >> 6, ch = idx & 63;
      uint4* ptr = reinterpret_cast<uint4*>(hs + (size_t)pr * I + ch * 8);
      float f[8];
      bf16x8_to_f32(*ptr, f);
      const float sc = exp2i(hexp[psrc_tok[pr]]);
      uint32_t pk[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 hv = __floats2half2_rn(__fmul_rn(f[2 * i], sc), __fmul_rn(f[2 * i + 1], sc));
        pk[i] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      *ptr = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
    __syncthreads();
  }

  if (warp == NCW) {
    // NVFP4: lane j serves the slots u = j (mod NG), whose stages consumer
    // group j alone frees, so the lanes wait on their groups in parallel
    // instead of one thread waking once per 4.6 KB tile.  BF16 (16 KB tiles,
    // one stage per group): one lane in slot order was measured faster.
    constexpr int PL = FMT == 0 ? NG : 1;
    if (lane < PL) {
      // The prologue (lane 0, before the dependency wait) requested slots
      // 0 .. min(STAGES, n_slots) - 1.
      const int pro = n_slots < STAGES ? n_slots : STAGES;
      int n = lane;
      while (n < pro) n += PL;
      for (; n < n_slots; n += PL) {
        const int s = n % STAGES;
        if (!mbar_wait(&empty[s], ((n / STAGES) - 1) & 1)) {
          atomicOr(p.err, ERR_WAIT_EMPTY);
          break;
        }
        const int e = R.slot_expert[n];
        mbar_arrive_expect_tx(&full[s], TILE);
        bulk_g2s(stages + (size_t)s * TILE, p.experts + (size_t)e * F::EXPERT + F::GU_BYTES + (size_t)rt * TILE,
                 TILE, &full[s], pol);
      }
      // Do not leave copies in flight: this lane's last STAGES / PL slots
      // (earlier ones had their stage reused, so they have landed).
      for (int m = n - PL; m >= 0 && m > n - PL - STAGES; m -= PL)
        if (!mbar_wait(&full[m % STAGES], (m / STAGES) & 1)) atomicOr(p.err, ERR_DRAIN);
    }
    return;
  }

  const int g = lane >> 2, t = lane & 3;
  const int kh = warp & 1, grp = warp >> 1;
  float tot[4] = {0.f, 0.f, 0.f, 0.f};
  for (int u = grp; u < n_slots; u += NG) {
    const int s = u % STAGES;
    if (!mbar_wait(&full[s], (u / STAGES) & 1)) {
      atomicOr(p.err, ERR_WAIT_FULL);
      break;
    }
    uint32_t bfr[16][2];
    const uint32_t mask = R.slot_mask[u];
    if (g < B && ((mask >> g) & 1u)) {
      const uint32_t* hr =
          reinterpret_cast<const uint32_t*>(hs + (size_t)pidx[u * BMAX + g] * I + kh * 256);
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
    const float ts = FMT == 0 ? ts_s[2 * e + 1] : 1.0f;
    const float w0 = __fmul_rn(R.slot_w[u][2 * t], ts);
    const float w1 = __fmul_rn(R.slot_w[u][2 * t + 1], ts);
    tot[0] = fmaf(w0, acc[0], tot[0]);
    tot[1] = fmaf(w1, acc[1], tot[1]);
    tot[2] = fmaf(w0, acc[2], tot[2]);
    tot[3] = fmaf(w1, acc[3], tot[3]);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) red[warp * 128 + j * 32 + lane] = tot[j];
  named_bar_sync(1, NCW * 32);
  if (tid < 128) {
    // thread = (token tk, row): sum the warps' partials in a fixed order
    const int row = tid & 15, tk = tid >> 4;
    const int o = red_off(row, tk);
    float c = 0.f;
#pragma unroll
    for (int w = 0; w < NCW; ++w) c += red[w * 128 + o];
    CSum sq = {0.f, 0.f};
    if (tk < B) {
      const float sc = FMT == 0 ? exp2i(-hexp[tk]) : 1.0f;
      const __nv_bfloat16 yv = __float2bfloat16_rn(__fmul_rn(c, sc));
      const size_t oy = (size_t)tk * H + rt * 16 + row;
      p.y[oy] = yv;
      if (p.y_copy) p.y_copy[oy] = yv;
      const float f = __bfloat162float(yv);
      sq.s = __fmul_rn(f, f);
    }
    if (p.ss_out) {
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) {
        CSum b;
        b.s = __shfl_xor_sync(0xffffffffu, sq.s, off);
        b.c = __shfl_xor_sync(0xffffffffu, sq.c, off);
        cs_merge(sq, b);
      }
      if (row == 0) p.ss_out[(size_t)rt * BMAX + tk] = sq;
    }
  }
}

// ------------------------------------------------------------------ host side

constexpr int F4_GU_STAGES = 5;
constexpr int B16_GU_STAGES = 3;
// Down kernel: 4 slot groups, small enough to be resident beside a gate/up
// CTA so that its down tiles stream in while gate/up still runs.  With 8
// tokens the staged h rows take 58 KB, so the tile ring shrinks to 8 stages.
constexpr int DN_GROUPS = 4;
constexpr int F4_DN_STAGES_S = 12, F4_DN_STAGES_L = 8;  // B <= 4 / B > 4
constexpr int B16_DN_STAGES = 4;
constexpr int DN_SMALL_MAX_B = 4;

static size_t align256(size_t v) { return ws_align256(v); }

DecodeWs carve_decode_ws(void* ws, int gu_grid) {
  uint8_t* p = static_cast<uint8_t*>(ws);
  DecodeWs w;
  w.logits = p;
  p += align256((size_t)BMAX * E * 2);
  w.xh_bf16 = p;
  p += align256((size_t)BMAX * H * 2);
  w.xfrag_f16 = p;
  p += align256((size_t)XFRAG_WORDS * 4);
  w.xfrag_bf16 = p;
  p += align256((size_t)XFRAG_WORDS * 4);
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

// One expert per CTA (256 CTAs) while the per-thread state is small; two
// experts per CTA (128 CTAs, one wave beside the waiting gate/up CTAs) when
// the batch makes every CTA register-heavy.
template <int NB>
struct RouterEpc {
  static constexpr int value = NB <= 2 ? 1 : 2;
};

template <int NB>
static cudaError_t launch_router_nb(const RouterParams& rp, cudaStream_t st, bool pdl) {
  constexpr int EPC = RouterEpc<NB>::value;
  return launch(router_kernel<NB, EPC>, E / EPC, 256, 0, st, pdl, rp);
}

template <int NB>
static cudaError_t router_carveout() {
  return cudaFuncSetAttribute(router_kernel<NB, RouterEpc<NB>::value>,
                              cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
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

// Every kernel asks for the maximal shared-memory carveout: an SM can only
// host CTAs of kernels with the same L1/shared split, and the chained kernels
// of a sublayer are meant to be resident together (a dependent kernel's
// prologue prefetches while its predecessor runs).
template <typename K>
static cudaError_t set_smem(K k, size_t bytes) {
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

cudaError_t decode_kernels_init(int /*device*/) {
  cudaError_t e;
  if ((e = set_smem(gateup_kernel<0, F4_GU_STAGES>, gateup_smem_bytes<0, F4_GU_STAGES>())) != cudaSuccess) return e;
  if ((e = set_smem(gateup_kernel<1, B16_GU_STAGES>, gateup_smem_bytes<1, B16_GU_STAGES>())) != cudaSuccess) return e;
  if ((e = set_smem(down_kernel<0, F4_DN_STAGES_S, DN_GROUPS>,
                    down_smem_bytes<0, F4_DN_STAGES_S, DN_GROUPS>(DN_SMALL_MAX_B))) != cudaSuccess)
    return e;
  if ((e = set_smem(down_kernel<0, F4_DN_STAGES_L, DN_GROUPS>, down_smem_bytes<0, F4_DN_STAGES_L, DN_GROUPS>(BMAX))) !=
      cudaSuccess)
    return e;
  if ((e = set_smem(down_kernel<1, B16_DN_STAGES, DN_GROUPS>, down_smem_bytes<1, B16_DN_STAGES, DN_GROUPS>(BMAX))) !=
      cudaSuccess)
    return e;
  cudaError_t r[8] = {router_carveout<1>(), router_carveout<2>(), router_carveout<3>(), router_carveout<4>(),
                      router_carveout<5>(), router_carveout<6>(), router_carveout<7>(), router_carveout<8>()};
  for (cudaError_t x : r)
    if (x != cudaSuccess) return x;
  return cudaSuccess;
}

cudaError_t launch_decode_chain(int fmt, const LayerArgs& L, const void* x, const void* ss_in, int B, float eps,
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
  rp.xfrag_f16 = static_cast<uint32_t*>(ws.xfrag_f16);
  rp.xfrag_bf16 = static_cast<uint32_t*>(ws.xfrag_bf16);
  rp.xh_exp = ws.xh_exp;
  cudaError_t e = launch_router(B, rp, st, pdl_first);
  if (e != cudaSuccess) return e;

  GateUpParams gp;
  gp.experts = L.experts;
  gp.tscale = L.tscale;
  gp.logits = rp.logits;
  gp.xfrag = fmt == 0 ? rp.xfrag_f16 : rp.xfrag_bf16;
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
  constexpr int NT = DnCfg<DN_GROUPS>::THREADS;
  if (fmt == 0) {
    if (B <= DN_SMALL_MAX_B)
      e = launch(down_kernel<0, F4_DN_STAGES_S, DN_GROUPS>, DN_TILES, NT,
                 down_smem_bytes<0, F4_DN_STAGES_S, DN_GROUPS>(B), st, true, dp);
    else
      e = launch(down_kernel<0, F4_DN_STAGES_L, DN_GROUPS>, DN_TILES, NT,
                 down_smem_bytes<0, F4_DN_STAGES_L, DN_GROUPS>(B), st, true, dp);
  } else {
    e = launch(down_kernel<1, B16_DN_STAGES, DN_GROUPS>, DN_TILES, NT, down_smem_bytes<1, B16_DN_STAGES, DN_GROUPS>(B),
               st, true, dp);
  }
  return e;
}

}  // namespace flint
