// Medium-batch decode path (9..64 tokens) of the Flint MoE sublayer, sm_103a.
//
// "Day-0 Support for Flint on vLLM", section "Optimizations": the low-latency
// decode kernels cover up to 8 requests; larger batches leave that path.  Past
// 8 tokens the selected experts overlap less and less (about 199 distinct
// experts at 64 tokens), so splitting the batch into groups of 8 would read
// most experts several times (649 MB instead of 355 MB per sublayer at 64
// tokens).  This path reads every selected expert's weights once per
// slot-chunk: the tokens of one expert, up to 8 at a time, ride as the mma n8
// block on each dequantised weight fragment.  Five kernels, chained with
// programmatic dependent launch:
//
//   router_kernel   (decode.cu) over chunks of 8 tokens: RMSNorm, bf16
//                   logits (error-free accumulation), x_hat fragments in f16
//                   scaled by a per-token power of two.
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
//   mcombine_kernel y = bf16(sum_j w_j d_j + d_shared), j in selection order.
#include "decode_common.cuh"
#include "flint_internal.h"

namespace flint {

namespace {

constexpr int XFRAG_WORDS_M = 8 * 32 * 32;  // one chunk of 8 tokens (router fragment layout)

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
  // Top-6 of token t by warp t % 32.
  for (int t = warp; t < T; t += 32) {
    const uint4 raw = load_logits(p.logits + (size_t)t * E, lane);
    int sel_i[TOPK];
    uint32_t sel_lg[TOPK];
    warp_top6_core(raw, lane, sel_i, sel_lg);
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
  // Slot-chunks of expert e, tokens in ascending order.
  if (tid < NE) {
    const int e = tid, n = (int)s_cnt[e];
    if (n > 0) {
      const int c0 = s_cbase[e], pb = s_pbase[e];
      for (int c = 0; c * MCH < n; ++c) {
        p.rt->sc_e[c0 + c] = e;
        p.rt->sc_pair[c0 + c] = pb + c * MCH;
        p.rt->sc_n[c0 + c] = min(MCH, n - c * MCH);
      }
      unsigned long long m = s_mask[e];
      for (int k = 0; m != 0ull; ++k) {
        const int t = __ffsll((long long)m) - 1;
        m &= m - 1ull;
        p.rt->sc_tok[c0 + k / MCH][k % MCH] = (uint8_t)t;
      }
    }
  }
  // Pair of (token t, selection j): the expert's base + the tokens before t.
  for (int q = tid; q < T * (TOPK + 1); q += MR_THREADS) {
    const int t = q / (TOPK + 1), j = q % (TOPK + 1);
    const int e = j < TOPK ? s_ids[t][j] : E;
    const unsigned long long before = t == 0 ? 0ull : (s_mask[e] & ((1ull << t) - 1ull));
    p.rt->pidx[t][j] = s_pbase[e] + __popcll(before);
  }
  for (int q = tid; q < T * TOPK; q += MR_THREADS) {
    const int t = q / TOPK, j = q % TOPK;
    p.rt->w[t][j] = s_w[t][j];
    if (p.ids_out) p.ids_out[q] = s_ids[t][j];
    if (p.w_out) p.w_out[q] = s_w[t][j];
  }
}

// ------------------------------------------------------------------ common item walk

// Items [lo, hi) of this CTA: a contiguous range, so that consecutive items
// mostly share a slot-chunk.
__device__ __forceinline__ void item_range(int n_items, int& lo, int& hi) {
  const int G = gridDim.x;
  const int q = (n_items + G - 1) / G;
  lo = min(n_items, (int)blockIdx.x * q);
  hi = min(n_items, lo + q);
}

constexpr int M_TILE = 18432;  // one item's weights: 16 gate/up rows or 64 down rows, all of K
static_assert(M_TILE == F4_GU_TILE && M_TILE == 4 * F4_DN_TILE, "item size");
constexpr int MG_STAGES = 8;
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
  int T;
  __nv_bfloat16* y;  // [T][H]
};

__global__ void __launch_bounds__(256) mcombine_kernel(const MCombineParams p) {
  pdl_wait();
  pdl_trigger();
  const int q = blockIdx.x * 256 + threadIdx.x;  // (token, 4 columns)
  if (q >= p.T * (H / 4)) return;
  const int t = q / (H / 4), c = (q % (H / 4)) * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int j = 0; j < TOPK; ++j) {
    const float w = __ldcg(&p.rt->w[t][j]);
    const float4 d = __ldcg(reinterpret_cast<const float4*>(p.part + (size_t)__ldcg(&p.rt->pidx[t][j]) * H + c));
    acc.x = __fmaf_rn(w, d.x, acc.x);
    acc.y = __fmaf_rn(w, d.y, acc.y);
    acc.z = __fmaf_rn(w, d.z, acc.z);
    acc.w = __fmaf_rn(w, d.w, acc.w);
  }
  const float4 d = __ldcg(reinterpret_cast<const float4*>(p.part + (size_t)__ldcg(&p.rt->pidx[t][TOPK]) * H + c));
  const __nv_bfloat162 lo = __floats2bfloat162_rn(__fadd_rn(acc.x, d.x), __fadd_rn(acc.y, d.y));
  const __nv_bfloat162 hi = __floats2bfloat162_rn(__fadd_rn(acc.z, d.z), __fadd_rn(acc.w, d.w));
  uint2 o;
  o.x = *reinterpret_cast<const uint32_t*>(&lo);
  o.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p.y + (size_t)t * H + c) = o;
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
  w.xfrag_bf16 = q;
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
                                       2 * ws_align256((size_t)(MT_MAX / 8) * XFRAG_WORDS_M * 4) +
                                       ws_align256(MT_MAX * 4) + ws_align256(sizeof(MedRoute)) +
                                       ws_align256((size_t)MPAIRS * I * 2) + ws_align256((size_t)MPAIRS * H * 4) + ws_align256((size_t)MT_MAX * H * 2),
              "medium workspace size and carve-up must agree");

cudaError_t medium_kernels_init() {
  cudaError_t e = cudaFuncSetAttribute(mgateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)mgateup_smem_bytes());
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mdown_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mdown_smem_bytes());
}

cudaError_t launch_medium_chain(const LayerArgs& L, const void* x, int T, float eps, void* y, int32_t* ids_out,
                                float* w_out, const MediumWs& ws, int sm_count, unsigned* err, cudaStream_t st,
                                bool pdl_first) {
  cudaError_t e = launch_router_chunks(L, x, T, eps, ws, st, pdl_first);
  if (e != cudaSuccess) return e;

  MRouteParams rp;
  rp.logits = static_cast<const __nv_bfloat16*>(ws.logits);
  rp.T = T;
  rp.rt = ws.rt;
  rp.ids_out = ids_out;
  rp.w_out = w_out;
  if ((e = launch_pdl(mroute_kernel, 1, MR_THREADS, 0, st, true, rp)) != cudaSuccess) return e;

  MGateUpParams gp;
  gp.experts = L.experts;
  gp.tscale = L.tscale;
  gp.xfrag = static_cast<const uint32_t*>(ws.xfrag_f16);
  gp.xh_exp = ws.xh_exp;
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
  cp.T = T;
  cp.y = static_cast<__nv_bfloat16*>(y);
  return launch_pdl(mcombine_kernel, (T * (H / 4) + 255) / 256, 256, 0, st, true, cp);
}

}  // namespace flint
