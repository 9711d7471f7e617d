// Medium-batch decode path (9..64 tokens) of the Flint MoE sublayer, sm_103a.
//
// "Day-0 Support for Flint on vLLM", section "Optimizations": the low-latency
// decode kernels cover up to 8 requests; larger batches leave that path.  Past
// 8 tokens the selected experts overlap less and less (about 199 distinct
// experts at 64 tokens), so splitting the batch into groups of 8 would read
// most experts several times (649 MB instead of 355 MB per sublayer at 64
// tokens).  This path reads every selected expert's weights once per
// slot-chunk: the tokens of one expert, up to 8 at a time, ride as the mma n8
// block on each dequantised weight fragment.  Kernels, chained with
// programmatic dependent launch:
//
//   mnorm_kernel    one CTA per token: RMSNorm, x_hat in bf16 and in f16
//                   scaled by a per-token power of two (first sublayer of a
//                   call only; inside a stack the previous sublayer's combine
//                   does this step for the next one).
//   mlogits_kernel  bf16 router logits (error-free accumulation) over units
//                   (chunk of 8 tokens, expert), one wave of CTAs.
//   mroute_kernel   one CTA: sigmoid top-6 per token, then the slot-chunk
//                   table (expert, up to 8 tokens, first pair) with the
//                   shared expert first and the routed experts in ascending
//                   order, and the pair of every (token, expert).
//   mgateup_kernel  items (slot-chunk, 16-row gate/up tile); each CTA walks a
//                   contiguous range of items with two groups of compute
//                   warps taking alternate items, so the activations of a
//                   slot-chunk are loaded once per group; h = bf16(silu(g) * u)
//                   per pair.
//   mdown_kernel    items (slot-chunk, 64 output rows); h in f16 scaled by a
//                   per-pair power of two (from the pair's largest |h|, which
//                   the two K-half warps of a row tile find together); writes
//                   the pair's down projection times its tensor scale, fp32.
//   mcombine_kernel one CTA per token: y = bf16(sum_j w_j d_j + d_shared), j
//                   in selection order; inside a stack also the next
//                   sublayer's x_hat from y.
#include <algorithm>

#include "decode_common.cuh"
#include "flint_internal.h"

namespace flint {

namespace {

constexpr int XFRAG_WORDS_M = 8 * 32 * 32;  // one chunk of 8 tokens (router fragment layout)

// ------------------------------------------------------------------ common item walk

// Items [lo, hi) of this CTA: a contiguous range, so that consecutive items
// mostly share a slot-chunk.
__device__ __forceinline__ void item_range(int n_items, int& lo, int& hi) {
  const int G = gridDim.x;
  const int q = (n_items + G - 1) / G;
  lo = min(n_items, (int)blockIdx.x * q);
  hi = min(n_items, lo + q);
}

// ------------------------------------------------------------------ x_hat

// Where x_hat goes: bf16 in the natural layout (the logits read it), f16
// times 2^xh_exp[t] in the mma fragment order of its chunk of 8 tokens (the
// gate/up kernel reads it), and the exponent itself.
struct XhatOut {
  __nv_bfloat16* xh;  // [T][H]
  uint32_t* xfrag;    // [chunks][XFRAG_WORDS_M]
  int* xh_exp;        // [T]
};

// x_hat of token t by a CTA of 256 threads; thread k holds columns 8k..8k+7
// of the token's input (bf16 values as fp32) in v.  With a norm weight
// (RMSNorm, "Day-0 Support for Flint on vLLM", section "Model architecture"):
// r = 1 / sqrt(sum(x^2) / H + eps) from a compensated sum of squares, so r is
// the one the exact sum gives whatever the order; x_hat = bf16(x * r * w).
// Without one, x_hat = x.  xh_exp[t] puts max |x_hat| into [2^14, 2^15).
__device__ __forceinline__ void publish_xhat(float (&v)[8], bool has_norm, const float (&nw)[8], float eps, int t,
                                             const XhatOut& o) {
  __shared__ CSum s_ss[8];
  __shared__ unsigned s_mx[8];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, k0 = tid * 8;
  if (has_norm) {
    CSum2 a2 = {0ull, 0ull};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint64_t q = f2pack(v[2 * i], v[2 * i + 1]);
      cs2_add(a2, f2mul(q, q));
    }
    CSum a, b;
    cs2_split(a2, a, b);
    cs_merge(a, b);
    a = cs_warp_reduce(a);
    if (lane == 0) s_ss[warp] = a;
    __syncthreads();
    a = s_ss[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) cs_merge(a, s_ss[w]);
    const float ms = __fmul_rn(cs_value(a), 1.0f / (float)H);
    const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(__fmul_rn(v[i], r), nw[i])));
  }
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
  const unsigned wm = redux_max(__float_as_uint(m));
  if (lane == 0) s_mx[warp] = wm;
  uint32_t pk[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) pk[i] = (__float_as_uint(v[2 * i]) >> 16) | (__float_as_uint(v[2 * i + 1]) & 0xFFFF0000u);
  *reinterpret_cast<uint4*>(o.xh + (size_t)t * H + k0) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  __syncthreads();
  unsigned mx = s_mx[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) mx = max(mx, s_mx[w]);
  const int ex = f16_range_exp(__uint_as_float(mx));
  const float sc = exp2i(ex);
  // Columns 8k..8k+7: K-slice k / 32, block (k % 32) / 2, register k % 2 of
  // the lanes 4 (t % 8) .. 4 (t % 8) + 3.
  const int ws = k0 >> 8, kb = (k0 & 255) >> 4, rr = (k0 >> 3) & 1;
  uint32_t* fr = o.xfrag + (size_t)(t >> 3) * XFRAG_WORDS_M;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 hv = __floats2half2_rn(__fmul_rn(v[2 * i], sc), __fmul_rn(v[2 * i + 1], sc));
    fr[((ws * 32 + 4 * (t & 7) + i) * 16 + kb) * 2 + rr] = *reinterpret_cast<const uint32_t*>(&hv);
  }
  if (tid == 0) o.xh_exp[t] = ex;
}

struct MNormParams {
  const __nv_bfloat16* x;       // [T][H]
  const __nv_bfloat16* norm_w;  // [H] or null
  float eps;
  XhatOut o;
};

__global__ void __launch_bounds__(256) mnorm_kernel(const MNormParams p) {
  const int t = blockIdx.x, k0 = threadIdx.x * 8;
  const bool has_norm = p.norm_w != nullptr;
  float nw[8] = {};
  if (has_norm) bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(p.norm_w + k0)), nw);
  pdl_trigger();
  pdl_wait();
  float v[8];
  bf16x8_to_f32(__ldcg(reinterpret_cast<const uint4*>(p.x + (size_t)t * H + k0)), v);
  publish_xhat(v, has_norm, nw, p.eps, t, p.o);
}

// ------------------------------------------------------------------ logits

// logit[t][e] = bf16(sum_k x_hat[t][k] W_r[e][k]), accumulated error-free
// (bf16 products are exact in fp32, TwoSum carries every rounding error), so
// it is the correctly rounded value whatever the order.  Units u = (chunk c =
// u / E, expert e = u % E); each CTA takes a contiguous range of units, so it
// keeps a chunk's 8 rows of x_hat in registers over many experts and reads
// one 4 KB router row per unit.  Thread k owns columns 8k..8k+7; token pairs
// share packed fp32x2 arithmetic.
struct MLogitsParams {
  const __nv_bfloat16* wr;  // [E][H]
  const __nv_bfloat16* xh;  // [T][H]
  int T;
  __nv_bfloat16* logits;    // [T][E]
};

__device__ __forceinline__ void load_xhat_chunk(const MLogitsParams& p, int c, int k0, uint4 (&xr)[8]) {
#pragma unroll
  for (int t = 0; t < 8; ++t)
    xr[t] = 8 * c + t < p.T ? __ldcg(reinterpret_cast<const uint4*>(p.xh + (size_t)(8 * c + t) * H + k0))
                            : make_uint4(0u, 0u, 0u, 0u);
}

__global__ void __launch_bounds__(256, 2) mlogits_kernel(const MLogitsParams p) {
  __shared__ CSum red[2][8][8];  // [unit parity][warp][token]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, k0 = tid * 8;
  const int NC = (p.T + 7) >> 3;
  int lo, hi;
  item_range(E * NC, lo, hi);
  // Router rows are constants: ask this CTA's rows into L2 before the wait.
  if (tid == 0)
    for (int u = lo; u < hi; ++u) bulk_prefetch_l2(p.wr + (size_t)(u % E) * H, H * 2);
  uint4 wnext = lo < hi ? __ldg(reinterpret_cast<const uint4*>(p.wr + (size_t)(lo % E) * H + k0)) : make_uint4(0u, 0u, 0u, 0u);
  pdl_trigger();
  pdl_wait();
  if (lo >= hi) return;
  uint4 xa[8], xb[8];
  int ca = lo / E;
  const int c_last = (hi - 1) / E;
  load_xhat_chunk(p, ca, k0, xa);
  if (ca + 1 <= c_last) load_xhat_chunk(p, ca + 1, k0, xb);
  for (int u = lo; u < hi; ++u) {
    const int c = u / E, e = u % E;
    if (c != ca) {
#pragma unroll
      for (int t = 0; t < 8; ++t) xa[t] = xb[t];
      ca = c;
      if (ca + 1 <= c_last) load_xhat_chunk(p, ca + 1, k0, xb);
    }
    const uint4 wcur = wnext;
    if (u + 1 < hi) wnext = __ldg(reinterpret_cast<const uint4*>(p.wr + (size_t)((u + 1) % E) * H + k0));
    float wf[8];
    bf16x8_to_f32(wcur, wf);
    CSum2 d2[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) d2[q] = CSum2{0ull, 0ull};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint64_t w2 = f2pack(wf[i], wf[i]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t a = (&xa[2 * q].x)[i >> 1], b = (&xa[2 * q + 1].x)[i >> 1];
        const float x0 = __uint_as_float((i & 1) ? (a & 0xFFFF0000u) : (a << 16));
        const float x1 = __uint_as_float((i & 1) ? (b & 0xFFFF0000u) : (b << 16));
        cs2_add(d2[q], f2mul(f2pack(x0, x1), w2));
      }
    }
    CSum d[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) cs2_split(d2[q], d[2 * q], d[2 * q + 1]);
    const CSum tot = cs_reduce_scatter<8>(d, lane);  // lanes 4t..4t+3: token t
    CSum(*rb)[8] = red[(u - lo) & 1];
    if ((lane & 3) == 0) rb[warp][lane >> 2] = tot;
    __syncthreads();
    if (tid < 8 && 8 * c + tid < p.T) {
      CSum a = rb[0][tid];
#pragma unroll
      for (int w = 1; w < 8; ++w) cs_merge(a, rb[w][tid]);
      p.logits[(size_t)(8 * c + tid) * E + e] = __float2bfloat16_rn(cs_value(a));
    }
  }
}

// ------------------------------------------------------------------ routing tables

struct MRouteParams {
  const __nv_bfloat16* logits;  // [T][E]
  int T;
  MedRoute* rt;
  int32_t* ids_out;             // [T][6] or null
  float* w_out;                 // [T][6] or null
};

constexpr int MR_THREADS = 1024;

__global__ void __launch_bounds__(MR_THREADS, 1) mroute_kernel(const MRouteParams p) {
  __shared__ int s_ids[MT_MAX][TOPK];
  __shared__ float s_w[MT_MAX][TOPK];
  __shared__ unsigned s_cnt[NE];
  __shared__ unsigned long long s_mask[NE];
  __shared__ int s_pbase[NE];  // first pair of expert e
  __shared__ int s_cbase[NE];  // first slot-chunk of expert e
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = p.T;
  for (int e = tid; e < NE; e += MR_THREADS) {
    s_cnt[e] = 0u;
    s_mask[e] = 0ull;
  }
  pdl_trigger();
  pdl_wait();
  __syncthreads();
  if (tid == 0) {
    s_cnt[E] = (unsigned)T;
    s_mask[E] = T == 64 ? ~0ull : ((1ull << T) - 1ull);
  }
  // Top-6 of tokens warp and warp + 32; both logits rows are requested first.
  static_assert(MT_MAX <= 64, "two tokens per warp");
  uint4 raw[2];
#pragma unroll
  for (int h = 0; h < 2; ++h)
    if (warp + 32 * h < T) raw[h] = load_logits(p.logits + (size_t)(warp + 32 * h) * E, lane);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int t = warp + 32 * h;
    if (t >= T) break;
    int sel_i[TOPK];
    uint32_t sel_lg[TOPK];
    warp_top6_core(raw[h], lane, sel_i, sel_lg);
    warp_top6_weights(sel_lg, lane, s_w[t]);
    if (lane < TOPK) {
      int wi = 0;
#pragma unroll
      for (int k = 0; k < TOPK; ++k)
        if (k == lane) wi = sel_i[k];
      s_ids[t][lane] = wi;
      atomicAdd(&s_cnt[wi], 1u);
      atomicOr(&s_mask[wi], 1ull << t);
    }
  }
  __syncthreads();
  // Exclusive scans of pairs and slot-chunks over the expert order
  // (shared, 0, 1, ..., 255): ordinal o -> expert o == 0 ? E : o - 1.
  if (warp == 0) {
    constexpr int PER = (NE + 31) / 32;  // 9
    int pc[PER], cc[PER];
    int ps = 0, cs = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int o = lane * PER + j;
      const int c = o < NE ? (int)s_cnt[o == 0 ? E : o - 1] : 0;
      pc[j] = c;
      cc[j] = (c + MCH - 1) / MCH;
      ps += pc[j];
      cs += cc[j];
    }
    int pin = ps, cin = cs;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, pin, d), b = __shfl_up_sync(0xffffffffu, cin, d);
      if (lane >= d) {
        pin += a;
        cin += b;
      }
    }
    int pb = pin - ps, cb = cin - cs;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int o = lane * PER + j;
      if (o < NE) {
        const int e = o == 0 ? E : o - 1;
        s_pbase[e] = pb;
        s_cbase[e] = cb;
      }
      pb += pc[j];
      cb += cc[j];
    }
    if (lane == 31) {
      p.rt->n_sc = cin;
      p.rt->n_pairs = pin;
    }
  }
  __syncthreads();
  // Every (token t, selection j) in one pass: its rank among the expert's
  // tokens (ascending) gives its pair, its slot-chunk and its place there; the
  // first token of a slot-chunk also writes the slot-chunk's entry.
  for (int q = tid; q < T * (TOPK + 1); q += MR_THREADS) {
    const int t = q / (TOPK + 1), j = q % (TOPK + 1);
    const int e = j < TOPK ? s_ids[t][j] : E;
    const unsigned long long before = t == 0 ? 0ull : (s_mask[e] & ((1ull << t) - 1ull));
    const int rank = __popcll(before);
    const int pr = s_pbase[e] + rank;
    const int c = s_cbase[e] + rank / MCH;
    p.rt->pidx[t][j] = pr;
    p.rt->sc_tok[c][rank % MCH] = (uint8_t)t;
    if (rank % MCH == 0) {
      p.rt->sc_e[c] = e;
      p.rt->sc_pair[c] = pr;
      p.rt->sc_n[c] = min(MCH, (int)s_cnt[e] - rank);
    }
  }
  for (int q = tid; q < T * TOPK; q += MR_THREADS) {
    const int t = q / TOPK, j = q % TOPK;
    p.rt->w[t][j] = s_w[t][j];
    if (p.ids_out) p.ids_out[q] = s_ids[t][j];
    if (p.w_out) p.w_out[q] = s_w[t][j];
  }
}

constexpr int M_TILE = 18432;  // one item's weights: 16 gate/up rows or 64 down rows, all of K
static_assert(M_TILE == F4_GU_TILE && M_TILE == 4 * F4_DN_TILE, "item size");
constexpr int MG_STAGES = 4;  // ring stages: measured faster than 6, 8 or 10 (fewer copies in flight)
constexpr int MG_CW = 8;                      // compute warps of a group (one K-slice each)
constexpr int MG_GROUPS = 2;                  // gate/up: compute groups taking alternate items
constexpr int MG_PW = MG_GROUPS * MG_CW;      // gate/up producer warp
constexpr int MG_EW = 4;                      // epilogue warps
constexpr int MG_RED = MG_EW;                 // partial-sum ring: buffer q belongs to epilogue warp q
constexpr int MG_THREADS = 32 * (MG_PW + 1 + MG_EW);
// Item n uses stage n % MG_STAGES and ring buffer n % MG_RED: each belongs to
// one compute group, which consumes it in order, as the parity waits require.
static_assert(MG_STAGES % MG_GROUPS == 0 && MG_RED % MG_GROUPS == 0, "stage and buffer ownership");
constexpr int MD_THREADS = 32 * (MG_CW + 1);
constexpr int TS_WORDS = ((NE * 2 + 3) / 4) * 4;

// Producer: one bulk copy per item, weights of expert sc_e[item / per] at
// byte offset base + (item % per) * M_TILE.  Waits for every copy to land.
__device__ __forceinline__ void produce_items(const uint8_t* experts, const MedRoute* rt, size_t base, int per,
                                              int lo, int hi, uint8_t* stages, uint64_t* full, uint64_t* empty,
                                              unsigned* err) {
  const uint64_t pol = l2_evict_first();
  int issued = 0, cur = -1, e = 0;
  for (int n = 0; lo + n < hi; ++n) {
    const int s = n % MG_STAGES;
    const int i = lo + n;
    if (i / per != cur) {  // the expert is read once per slot-chunk, not per copy
      cur = i / per;
      e = __ldcg(&rt->sc_e[cur]);
    }
    if (n >= MG_STAGES && !mbar_wait(&empty[s], ((n / MG_STAGES) - 1) & 1)) {
      atomicOr(err, ERR_WAIT_EMPTY);
      break;
    }
    mbar_arrive_expect_tx(&full[s], M_TILE);
    bulk_g2s(stages + (size_t)s * M_TILE, experts + (size_t)e * F4_EXPERT + base + (size_t)(i % per) * M_TILE,
             M_TILE, &full[s], pol);
    issued = n + 1;
  }
  for (int n = issued - MG_STAGES; n < issued; ++n) {
    if (n < 0) continue;
    if (!mbar_wait(&full[n % MG_STAGES], (n / MG_STAGES) & 1)) atomicOr(err, ERR_DRAIN);
  }
}

// ------------------------------------------------------------------ gate/up

struct MGateUpParams {
  const uint8_t* experts;
  const float* tscale;      // [NE][2]
  const uint32_t* xfrag;    // [chunks of 8 tokens][XFRAG_WORDS_M], f16 x_hat * 2^xh_exp
  const int* xh_exp;        // [T]
  const MedRoute* rt;
  __nv_bfloat16* h;         // [pairs][I]
  unsigned* err;
};

__host__ __device__ constexpr size_t mgateup_smem_bytes() {
  // [stages][red MG_RED x 8 warps x 128][tensor scales][full, empty][rfull, rempty]
  return (size_t)MG_STAGES * M_TILE + (size_t)MG_RED * MG_CW * 128 * 4 + TS_WORDS * 4 + 2 * MG_STAGES * 8 +
         2 * MG_RED * 8;
}

// Activation fragments of slot-chunk sc for K-slice `slice`: lane column g is
// the chunk's token g (zeros past its end).
__device__ __forceinline__ void load_x_block(const MGateUpParams& p, int sc, int nt, int slice, int lane,
                                             uint32_t (&b)[16][2]) {
  const int g = lane >> 2, t4 = lane & 3;
  if (g < nt) {
    const int tok = __ldcg(&p.rt->sc_tok[sc][g]);
    const uint4* src = reinterpret_cast<const uint4*>(p.xfrag + (size_t)(tok >> 3) * XFRAG_WORDS_M +
                                                      (size_t)(slice * 32 + 4 * (tok & 7) + t4) * 32);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint4 v = __ldcg(src + q);
      b[2 * q][0] = v.x;
      b[2 * q][1] = v.y;
      b[2 * q + 1][0] = v.z;
      b[2 * q + 1][1] = v.w;
    }
  } else {
#pragma unroll
    for (int kb = 0; kb < 16; ++kb) b[kb][0] = b[kb][1] = 0u;
  }
}

__global__ void __launch_bounds__(MG_THREADS, 1) mgateup_kernel(const MGateUpParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  float* red = reinterpret_cast<float*>(smem + (size_t)MG_STAGES * M_TILE);  // [MG_RED][8][128]
  float* ts_s = red + MG_RED * MG_CW * 128;
  uint64_t* full = reinterpret_cast<uint64_t*>(ts_s + TS_WORDS);
  uint64_t* empty = full + MG_STAGES;
  uint64_t* rfull = empty + MG_STAGES;
  uint64_t* rempty = rfull + MG_RED;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  for (int q = tid; q < NE * 2; q += MG_THREADS) ts_s[q] = __ldg(p.tscale + q);  // constants
  if (tid == 0) {
    for (int s = 0; s < MG_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], MG_CW);
    }
    for (int b = 0; b < MG_RED; ++b) {
      mbar_init(&rfull[b], MG_CW);
      mbar_init(&rempty[b], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int n_items = __ldcg(&p.rt->n_sc) * GU_TILES;
  int lo, hi;
  item_range(n_items, lo, hi);

  if (warp == MG_PW) {
    if (lane == 0) produce_items(p.experts, p.rt, 0, GU_TILES, lo, hi, stages, full, empty, p.err);
    return;
  }

  if (warp < MG_PW) {
    // ---- compute group grp takes items n = grp (mod MG_GROUPS); its warp kw
    // multiplies K-slice kw of each.
    const int grp = warp / MG_CW, kw = warp % MG_CW;
    uint32_t bfr[16][2];
    int cur = -1, nt = 0;
    for (int n = grp; lo + n < hi; n += MG_GROUPS) {
      const int i = lo + n, sc = i / GU_TILES, s = n % MG_STAGES;
      if (sc != cur) {
        cur = sc;
        nt = __ldcg(&p.rt->sc_n[sc]);
        load_x_block(p, sc, nt, kw, lane, bfr);
      }
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (mbar_wait(&full[s], (n / MG_STAGES) & 1))
        nvfp4_slice_mma(stages + (size_t)s * M_TILE + kw * F4_SLICE, lane, bfr, acc);
      else
        atomicOr(p.err, ERR_WAIT_FULL);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      const int b = n % MG_RED;
      if (n >= MG_RED && !mbar_wait(&rempty[b], ((n / MG_RED) - 1) & 1)) atomicOr(p.err, ERR_WAIT_EMPTY);
      float* rb = red + (size_t)b * MG_CW * 128;
#pragma unroll
      for (int j = 0; j < 4; ++j) rb[kw * 128 + j * 32 + lane] = acc[j];
      __syncwarp();
      if (lane == 0) mbar_arrive(&rfull[b]);
    }
    return;
  }

  // ---- epilogue warps: warp q takes items n = q (mod MG_EW), whose partial
  // sums arrive in ring buffer q; lane = (token k = 4 h + lane / 8 for
  // h = 0, 1, gate/up row lane % 8 of the tile).
  const int q = warp - (MG_PW + 1);
  const int ep_tk = lane >> 3, ep_row = lane & 7;
  int cur = -1, nt = 0, pair0 = 0;
  float fk[2] = {0.f, 0.f};  // 2^-exponent x gate/up tensor scale of tokens 4 h + ep_tk
  for (int n = q; lo + n < hi; n += MG_EW) {
    const int i = lo + n, sc = i / GU_TILES, tile = i % GU_TILES;
    if (sc != cur) {  // before the wait: the table reads overlap the tile's arithmetic
      cur = sc;
      nt = __ldcg(&p.rt->sc_n[sc]);
      pair0 = __ldcg(&p.rt->sc_pair[sc]);
      const float ts = ts_s[2 * __ldcg(&p.rt->sc_e[sc])];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int k = 4 * h + ep_tk;
        fk[h] = k < nt ? __fmul_rn(exp2i(-__ldcg(p.xh_exp + __ldcg(&p.rt->sc_tok[sc][k]))), ts) : 0.f;
      }
    }
    if (!mbar_wait(&rfull[q], (n / MG_EW) & 1)) {
      atomicOr(p.err, ERR_WAIT_FULL);
      break;
    }
    const float* rb = red + (size_t)q * MG_CW * 128;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int k = 4 * h + ep_tk;
      if (k < nt) {
        const int og = red_off(ep_row, k), ou = red_off(ep_row + 8, k);
        float gsum = 0.f, usum = 0.f;
#pragma unroll
        for (int w = 0; w < MG_CW; ++w) {
          gsum += rb[w * 128 + og];
          usum += rb[w * 128 + ou];
        }
        const float gate = __fmul_rn(gsum, fk[h]);
        const float up = __fmul_rn(usum, fk[h]);
        const float silu = __fdiv_rn(gate, __fadd_rn(1.0f, expf(-gate)));
        const __nv_bfloat16 hv = __float2bfloat16_rn(__fmul_rn(silu, up));
        p.h[(size_t)(pair0 + k) * I + tile * 8 + ep_row] = hv;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&rempty[q]);
  }
}

// ------------------------------------------------------------------ down

struct MDownParams {
  const uint8_t* experts;
  const float* tscale;
  const MedRoute* rt;
  const __nv_bfloat16* h;   // [pairs][I]
  float* part;              // [pairs][H]
  unsigned* err;
};

constexpr int MD_BLOCKS = H / 64;  // 64-row items per expert

constexpr int MD_RED_SET = 2 * 4 * 128;  // floats: [2 items][4 row tiles][128]

__host__ __device__ constexpr size_t mdown_smem_bytes() {
  // [stages][red 2 sets][tensor scales][full, empty][hx 4 x 2 x 8]
  return (size_t)MG_STAGES * M_TILE + 2 * MD_RED_SET * 4 + TS_WORDS * 4 + 2 * MG_STAGES * 8 + 4 * 2 * 8 * 4;
}

// h of slot-chunk sc, K half kh, as f16 B fragments scaled by 2^e(pair), e
// from the pair's largest |h| over both K halves: each warp takes the maximum
// of its half, and the two warps of row tile rtile swap them through hx
// ([4 row tiles][2 halves][8 tokens]) on named barrier 1 + rtile.  Returns the
// exponent of this lane's token lane / 4.
__device__ __forceinline__ int load_h_block(const MDownParams& p, int pair0, int nt, int rtile, int kh, int lane,
                                            unsigned* hx, uint32_t (&b)[16][2]) {
  const int g = lane >> 2, t4 = lane & 3;
  uint32_t mx = 0u;  // largest |h| so far, as two bf16 magnitudes
  if (g < nt) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(p.h + (size_t)(pair0 + g) * I) + kh * 128 + t4;
#pragma unroll
    for (int kb = 0; kb < 16; ++kb) {
      b[kb][0] = __ldcg(src + kb * 8);
      b[kb][1] = __ldcg(src + kb * 8 + 4);
    }
#pragma unroll
    for (int kb = 0; kb < 16; ++kb) {
      mx = __vmaxu2(mx, b[kb][0] & 0x7FFF7FFFu);
      mx = __vmaxu2(mx, b[kb][1] & 0x7FFF7FFFu);
    }
  } else {
#pragma unroll
    for (int kb = 0; kb < 16; ++kb) b[kb][0] = b[kb][1] = 0u;
  }
  mx = max(mx & 0xFFFFu, mx >> 16);
  mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  if (t4 == 0) hx[(rtile * 2 + kh) * 8 + g] = mx;
  named_bar_sync(1 + rtile, 64);
  mx = max(mx, hx[(rtile * 2 + (kh ^ 1)) * 8 + g]);
  // As fp32 bits (<< 16) the order of non-negative values is that of their bits.
  const int ex = f16_range_exp(__uint_as_float(mx << 16));
  const float sc = exp2i(ex);
#pragma unroll
  for (int kb = 0; kb < 16; ++kb)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const uint32_t v = b[kb][r];
      const __half2 hv = __floats2half2_rn(__fmul_rn(__uint_as_float(v << 16), sc),
                                           __fmul_rn(__uint_as_float(v & 0xFFFF0000u), sc));
      b[kb][r] = *reinterpret_cast<const uint32_t*>(&hv);
    }
  return ex;
}

// Warp w: row tile rt = w / 2 of the item's 64 rows, K half kh = w % 2.  The
// two warps of a row tile meet on named barrier 1 + rt: the kh = 1 warp hands
// its sums over, the kh = 0 warp adds them and stores.  Buffer sets alternate
// between exchanges, so a set is rewritten only after the barrier that follows
// its last read.
__global__ void __launch_bounds__(MD_THREADS, 1) mdown_kernel(const MDownParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  float* red = reinterpret_cast<float*>(smem + (size_t)MG_STAGES * M_TILE);  // [2 sets][MD_RED_SET]
  float* ts_s = red + 2 * MD_RED_SET;
  uint64_t* full = reinterpret_cast<uint64_t*>(ts_s + TS_WORDS);
  uint64_t* empty = full + MG_STAGES;
  unsigned* hx = reinterpret_cast<unsigned*>(empty + MG_STAGES);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  for (int q = tid; q < NE * 2; q += MD_THREADS) ts_s[q] = __ldg(p.tscale + q);
  if (tid == 0) {
    for (int s = 0; s < MG_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], MG_CW);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int n_items = __ldcg(&p.rt->n_sc) * MD_BLOCKS;
  int lo, hi;
  item_range(n_items, lo, hi);

  if (warp == MG_CW) {
    if (lane == 0) produce_items(p.experts, p.rt, F4_GU_BYTES, MD_BLOCKS, lo, hi, stages, full, empty, p.err);
    return;
  }

  const int rtile = warp >> 1, kh = warp & 1;
  const int g = lane >> 2, t4 = lane & 3;
  uint32_t b0[16][2];
  int cur = -1, nt = 0, pair0 = 0;
  float fsc[2] = {0.f, 0.f};  // tensor scale x 2^-e of this lane's output columns 2 t4 + j
  for (int n = 0, u = 0; lo + n < hi;) {
    const int i = lo + n, sc = i / MD_BLOCKS, blk = i % MD_BLOCKS, s = n % MG_STAGES;
    if (sc != cur) {
      cur = sc;
      nt = __ldcg(&p.rt->sc_n[sc]);
      pair0 = __ldcg(&p.rt->sc_pair[sc]);
      const int ex = load_h_block(p, pair0, nt, rtile, kh, lane, hx, b0);
      const float ts = ts_s[2 * __ldcg(&p.rt->sc_e[sc]) + 1];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int k = 2 * t4 + j;  // output column: the token of lanes 4 k ..
        const int e = __shfl_sync(0xffffffffu, ex, k * 4);
        fsc[j] = k < nt ? __fmul_rn(ts, exp2i(-e)) : 0.f;
      }
    }
    // One exchange between the two warps of the row tile: one item, or two
    // consecutive items of the slot-chunk through the interleaved two-slice
    // product.  Exchange u uses buffer set u & 1.
    const bool two = lo + n + 1 < hi && (i + 1) / MD_BLOCKS == sc;
    const int s1 = (n + 1) % MG_STAGES;
    const int sl_off = (rtile * 2 + kh) * F4_SLICE;
    float acc[2][4] = {};  // [item][4]
    if (two) {
      if (mbar_wait(&full[s], (n / MG_STAGES) & 1) && mbar_wait(&full[s1], ((n + 1) / MG_STAGES) & 1))
        nvfp4_slice_mma2(stages + (size_t)s * M_TILE + sl_off, stages + (size_t)s1 * M_TILE + sl_off, lane, b0,
                         acc[0], acc[1]);
      else
        atomicOr(p.err, ERR_WAIT_FULL);
    } else if (mbar_wait(&full[s], (n / MG_STAGES) & 1)) {
      nvfp4_slice_mma(stages + (size_t)s * M_TILE + sl_off, lane, b0, acc[0]);
    } else {
      atomicOr(p.err, ERR_WAIT_FULL);
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&empty[s]);
      if (two) mbar_arrive(&empty[s1]);
    }
    const int items = two ? 2 : 1;
    float* rset = red + (size_t)(u & 1) * MD_RED_SET;  // [2 items][4 row tiles][128]
    if (kh == 1) {
      for (int it = 0; it < items; ++it)
        *reinterpret_cast<float4*>(rset + (it * 4 + rtile) * 128 + lane * 4) =
            make_float4(acc[it][0], acc[it][1], acc[it][2], acc[it][3]);
    }
    named_bar_sync(1 + rtile, 64);
    if (kh == 0) {
      for (int it = 0; it < items; ++it) {
        const int row = (blk + it) * 64 + rtile * 16 + g;
        const float4 o = *reinterpret_cast<const float4*>(rset + (it * 4 + rtile) * 128 + lane * 4);
        const float v[4] = {acc[it][0] + o.x, acc[it][1] + o.y, acc[it][2] + o.z, acc[it][3] + o.w};
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int k = 2 * t4 + j;
          if (k < nt) {
            float* dst = p.part + (size_t)(pair0 + k) * H + row;
            dst[0] = __fmul_rn(v[j], fsc[j]);
            dst[8] = __fmul_rn(v[2 + j], fsc[j]);
          }
        }
      }
    }
    n += items;
    ++u;
  }
}

// ------------------------------------------------------------------ combine

struct MCombineParams {
  const MedRoute* rt;
  const float* part;
  __nv_bfloat16* y;                  // [T][H]
  int publish;                       // also x_hat of the next sublayer from y
  const __nv_bfloat16* next_norm_w;  // its norm weight, or null
  float eps;
  XhatOut o;
};

// One CTA per token t; thread k covers columns 8k..8k+7.
__global__ void __launch_bounds__(256) mcombine_kernel(const MCombineParams p) {
  const int t = blockIdx.x, k0 = threadIdx.x * 8;
  const bool has_norm = p.publish && p.next_norm_w != nullptr;
  float nw[8] = {};
  if (has_norm) bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(p.next_norm_w + k0)), nw);
  pdl_wait();
  pdl_trigger();
  float acc[8] = {};
#pragma unroll
  for (int j = 0; j < TOPK; ++j) {
    const float w = __ldcg(&p.rt->w[t][j]);
    const float4* d = reinterpret_cast<const float4*>(p.part + (size_t)__ldcg(&p.rt->pidx[t][j]) * H + k0);
    const float4 d0 = __ldcg(d), d1 = __ldcg(d + 1);
    const float dv[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = __fmaf_rn(w, dv[i], acc[i]);
  }
  const float4* ds = reinterpret_cast<const float4*>(p.part + (size_t)__ldcg(&p.rt->pidx[t][TOPK]) * H + k0);
  const float4 s0 = __ldcg(ds), s1 = __ldcg(ds + 1);
  const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  float v[8];
  uint32_t pk[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b2 =
        __floats2bfloat162_rn(__fadd_rn(acc[2 * i], sv[2 * i]), __fadd_rn(acc[2 * i + 1], sv[2 * i + 1]));
    pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
    v[2 * i] = __low2float(b2);
    v[2 * i + 1] = __high2float(b2);
  }
  *reinterpret_cast<uint4*>(p.y + (size_t)t * H + k0) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  if (p.publish) publish_xhat(v, has_norm, nw, p.eps, t, p.o);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*k)(KArgs...), int grid, int block, size_t smem, cudaStream_t st, bool pdl,
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

}  // namespace

MediumWs carve_medium_ws(void* ws) {
  uint8_t* q = static_cast<uint8_t*>(ws);
  MediumWs w;
  w.logits = q;
  q += ws_align256((size_t)MT_MAX * E * 2);
  w.xh_bf16 = q;
  q += ws_align256((size_t)MT_MAX * H * 2);
  w.xfrag_f16 = q;
  q += ws_align256((size_t)(MT_MAX / 8) * XFRAG_WORDS_M * 4);
  w.xh_exp = reinterpret_cast<int*>(q);
  q += ws_align256(MT_MAX * 4);
  w.rt = reinterpret_cast<MedRoute*>(q);
  q += ws_align256(sizeof(MedRoute));
  w.h = q;
  q += ws_align256((size_t)MPAIRS * I * 2);
  w.part = reinterpret_cast<float*>(q);
  q += ws_align256((size_t)MPAIRS * H * 4);
  w.y_mid = q;
  return w;
}
static_assert(medium_ws_bytes() == ws_align256((size_t)MT_MAX * E * 2) + ws_align256((size_t)MT_MAX * H * 2) +
                                       ws_align256((size_t)(MT_MAX / 8) * XFRAG_WORDS_M * 4) +
                                       ws_align256(MT_MAX * 4) + ws_align256(sizeof(MedRoute)) +
                                       ws_align256((size_t)MPAIRS * I * 2) + ws_align256((size_t)MPAIRS * H * 4) + ws_align256((size_t)MT_MAX * H * 2),
              "medium workspace size and carve-up must agree");

cudaError_t medium_kernels_init() {
  cudaError_t e = cudaFuncSetAttribute(mgateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)mgateup_smem_bytes());
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mdown_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mdown_smem_bytes());
}

cudaError_t launch_medium_chain(const LayerArgs& L, const void* x, const LayerArgs* next, int T, float eps, void* y,
                                int32_t* ids_out, float* w_out, const MediumWs& ws, int sm_count, unsigned* err,
                                cudaStream_t st, bool pdl_first) {
  XhatOut xo;
  xo.xh = static_cast<__nv_bfloat16*>(ws.xh_bf16);
  xo.xfrag = static_cast<uint32_t*>(ws.xfrag_f16);
  xo.xh_exp = ws.xh_exp;
  cudaError_t e;
  bool pdl = pdl_first;
  if (x != nullptr) {
    MNormParams np;
    np.x = static_cast<const __nv_bfloat16*>(x);
    np.norm_w = static_cast<const __nv_bfloat16*>(L.norm_w);
    np.eps = eps;
    np.o = xo;
    if ((e = launch_pdl(mnorm_kernel, T, 256, 0, st, pdl, np)) != cudaSuccess) return e;
    pdl = true;
  }

  MLogitsParams lp;
  lp.wr = static_cast<const __nv_bfloat16*>(L.router_w);
  lp.xh = xo.xh;
  lp.T = T;
  lp.logits = static_cast<__nv_bfloat16*>(ws.logits);
  const int units = E * ((T + 7) / 8);
  if ((e = launch_pdl(mlogits_kernel, std::min(units, 2 * sm_count), 256, 0, st, pdl, lp)) != cudaSuccess) return e;

  MRouteParams rp;
  rp.logits = lp.logits;
  rp.T = T;
  rp.rt = ws.rt;
  rp.ids_out = ids_out;
  rp.w_out = w_out;
  if ((e = launch_pdl(mroute_kernel, 1, MR_THREADS, 0, st, true, rp)) != cudaSuccess) return e;

  MGateUpParams gp;
  gp.experts = L.experts;
  gp.tscale = L.tscale;
  gp.xfrag = xo.xfrag;
  gp.xh_exp = xo.xh_exp;
  gp.rt = ws.rt;
  gp.h = static_cast<__nv_bfloat16*>(ws.h);
  gp.err = err;
  if ((e = launch_pdl(mgateup_kernel, sm_count, MG_THREADS, mgateup_smem_bytes(), st, true, gp)) != cudaSuccess)
    return e;

  MDownParams dp;
  dp.experts = L.experts;
  dp.tscale = L.tscale;
  dp.rt = ws.rt;
  dp.h = gp.h;
  dp.part = ws.part;
  dp.err = err;
  if ((e = launch_pdl(mdown_kernel, sm_count, MD_THREADS, mdown_smem_bytes(), st, true, dp)) != cudaSuccess)
    return e;

  MCombineParams cp;
  cp.rt = ws.rt;
  cp.part = ws.part;
  cp.y = static_cast<__nv_bfloat16*>(y);
  cp.publish = next != nullptr;
  cp.next_norm_w = next ? static_cast<const __nv_bfloat16*>(next->norm_w) : nullptr;
  cp.eps = eps;
  cp.o = xo;
  return launch_pdl(mcombine_kernel, T, 256, 0, st, true, cp);
}

}  // namespace flint
