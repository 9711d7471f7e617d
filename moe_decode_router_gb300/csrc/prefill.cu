// Prefill-shaped MoE sublayer (T tokens, e.g. 8,192), sm_103a.
//
// "Day-0 Support for Flint on vLLM", section "Optimizations": the small-batch
// MoE kernels also gave the largest gain in the 8,192-token prefill, and the
// dense kernels run on the same packed NVFP4 weights as the large ones.  Here
// the sublayer over many tokens is one dense grouped contraction per expert,
// run on the 5th-generation tensor cores:
//
//   prep            per token: optional RMSNorm (exact), x_hat * 2^e in f16
//                   with a per-token power-of-two e, and an upper bound on
//                   ||x_hat||_2; 32 more blocks bound every ||W_r[e]||_2
//   gemm<router>    approximate fp32 logits S[t][e] on the tensor cores (bf16
//                   x_hat and W_r, fp32 accumulation), with an assumed error
//                   bound 2^-9 * ||x_hat|| * ||W_e|| checked online
//   route           per token, one warp: the experts whose bound interval can
//                   reach the 6th largest lower bound get their exact bf16
//                   logit (an fp32 dot product with a rigorous error interval,
//                   or an error-free TwoSum sum where that interval straddles
//                   a bf16 rounding boundary); every other logit is provably
//                   below the 6th; the top-6 then follows the decode path's
//                   sigmoid top-6 on the exact bf16 logits
//   scatter         tokens bucketed by expert (routed experts, then the shared
//                   expert over all tokens), offsets and work-item prefixes
//   gemm<gate/up>   tcgen05.mma kind::f16 (M=128 weight rows, N=256 tokens,
//                   fp32 accumulator in tensor memory); NVFP4 weights
//                   dequantised to f16 (exact) into 128-byte-swizzled shared
//                   memory, token rows gathered with cp.async; epilogue
//                   h = bf16(silu(g) * u)
//   gemm<down>      the same with bf16 operands (h is bf16); epilogue adds
//                   w_pair * d into an fp32 accumulator (shared expert w = 1)
//   finalize        y = bf16(accumulator)
#include "flint_common.cuh"
#include "flint_internal.h"
#include "tc05.cuh"

namespace flint {

namespace {

constexpr int PG_M = 128;  // weight rows per tile
constexpr int PG_N = 256;  // tokens per tile
constexpr int PG_KS = 64;  // K per pipeline step (one 128-byte swizzle row)
// Error model of the tensor-core router GEMM (bf16 products are exact, fp32
// accumulation): every one of the 2048 terms is assumed to add at most 2^-20
// of the sum of |products| to the error, 8 times the worst case of a
// truncating 24-bit adder.  |S - exact| <= 2048 * 2^-20 * sum|x_k w_k| <=
// 2^-9 * ||x|| * ||w|| (Cauchy-Schwarz).  The route kernel checks every
// candidate it recomputes against a quarter of this bound.
constexpr float GAMMA_TC = 1.953125e-3f;

__device__ __forceinline__ float exp2i_p(int e) { return __int_as_float((127 + e) << 23); }

__device__ __forceinline__ int f16_exp_of(float m) {
  if (!(m > 0.f) || !(m < INFINITY)) return 0;
  int e = ((__float_as_uint(m) >> 23) & 0xFF) - 127;
  if (e < -126) e = -126;
  int s = 14 - e;
  if (s > 126) s = 126;
  if (s < -126) s = -126;
  return s;
}

__device__ __forceinline__ void bf16x8_f32(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// ---------------------------------------------------------------- prep
// One CTA (256 threads, 8 columns each) per token.
// Upper bound on ||W_r[e]||_2 for experts 8 wb .. 8 wb + 7, one warp each.
__device__ __forceinline__ void wnorm_rows(const __nv_bfloat16* __restrict__ wr, float* __restrict__ wnorm, int wb) {
  const int e = wb * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (e >= E) return;
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float f[8];
    bf16x8_f32(__ldg(reinterpret_cast<const uint4*>(wr + (size_t)e * H) + lane + 32 * j), f);
#pragma unroll
    for (int i = 0; i < 8; ++i) s = fmaf(f[i], f[i], s);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) wnorm[e] = sqrtf(s) * 1.001f;
}

__global__ void __launch_bounds__(256) prefill_prep_kernel(const __nv_bfloat16* __restrict__ x,
                                                           const __nv_bfloat16* __restrict__ norm_w, float eps,
                                                           __nv_bfloat16* __restrict__ xh, __half* __restrict__ xh16,
                                                           int* __restrict__ xexp, float* __restrict__ xnorm,
                                                           int* __restrict__ rprefix, int* __restrict__ roffs,
                                                           int router_items, int T,
                                                           const __nv_bfloat16* __restrict__ wr, float* __restrict__ wnorm) {
  __shared__ CSum red[8];
  __shared__ float redf[8];
  __shared__ unsigned redm[8];
  __shared__ float rs;
  // The first E / 8 blocks bound the router rows' norms; the others handle
  // one token each.
  if (blockIdx.x < E / 8) {
    wnorm_rows(wr, wnorm, blockIdx.x);
    return;
  }
  const int t = blockIdx.x - E / 8, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k0 = tid * 8;
  if (t == 0)  // the router GEMM's work list: one entry holding every token
    for (int e = tid; e <= NE; e += 256) {
      rprefix[e] = e == 0 ? 0 : router_items;
      roffs[e] = e == 0 ? 0 : T;
    }
  float v[8];
  bf16x8_f32(__ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H + k0)), v);
  if (norm_w != nullptr) {
    float w[8];
    bf16x8_f32(__ldg(reinterpret_cast<const uint4*>(norm_w + k0)), w);
    CSum a = {0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 8; ++i) cs_add(a, __fmul_rn(v[i], v[i]));
    a = cs_warp_reduce(a);
    if (lane == 0) red[warp] = a;
    __syncthreads();
    if (tid == 0) {
      CSum b = red[0];
#pragma unroll
      for (int i = 1; i < 8; ++i) cs_merge(b, red[i]);
      const float ms = __fmul_rn(cs_value(b), 1.0f / (float)H);
      rs = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, eps)));
    }
    __syncthreads();
    const float r = rs;
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(__fmul_rn(v[i], r), w[i])));
    uint32_t pk[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) pk[i] = (__float_as_uint(v[2 * i]) >> 16) | (__float_as_uint(v[2 * i + 1]) & 0xFFFF0000u);
    *reinterpret_cast<uint4*>(xh + (size_t)t * H + k0) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
  float sq = 0.f, m = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    sq = fmaf(v[i], v[i], sq);
    m = fmaxf(m, fabsf(v[i]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
  const unsigned mb = redux_max(__float_as_uint(m));
  if (lane == 0) {
    redf[warp] = sq;
    redm[warp] = mb;
  }
  __syncthreads();
  if (tid == 0) {
    float s = 0.f;
    unsigned mm = 0u;
    for (int i = 0; i < 8; ++i) {
      s += redf[i];
      mm = max(mm, redm[i]);
    }
    // upper bound: the fp32 sum of 2048 squares is within 1e-3 (relative) of the exact one
    xnorm[t] = sqrtf(s) * 1.001f;
    const int e = f16_exp_of(__uint_as_float(mm));
    xexp[t] = e;
    redm[0] = (unsigned)(e + 1000);
  }
  __syncthreads();
  const float sc = exp2i_p((int)redm[0] - 1000);
  uint32_t pk[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 hv = __floats2half2_rn(__fmul_rn(v[2 * i], sc), __fmul_rn(v[2 * i + 1], sc));
    pk[i] = *reinterpret_cast<const uint32_t*>(&hv);
  }
  *reinterpret_cast<uint4*>(xh16 + (size_t)t * H + k0) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
}


// ---------------------------------------------------------------- route
// One warp per token.  Lane l holds experts 8l..8l+7.
__device__ __forceinline__ uint32_t ord_f32(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__global__ void __launch_bounds__(256, 4) prefill_route_kernel(
    const __nv_bfloat16* __restrict__ xh, const __nv_bfloat16* __restrict__ wr, const float* __restrict__ S,
    const float* __restrict__ xnorm, const float* __restrict__ wnorm, int T, int32_t* __restrict__ ids,
    float* __restrict__ wts, int* __restrict__ counts, int32_t* __restrict__ ids_out, float* __restrict__ w_out,
    unsigned* __restrict__ err, float* __restrict__ yacc) {
  __shared__ __align__(16) __nv_bfloat16 lrow[8][E];
  __shared__ int sids[8][TOPK];
  __shared__ float sw[8][TOPK];
  __shared__ uint32_t umask_dummy[8][8];
  __shared__ uint8_t clist[8][E];
  __shared__ uint8_t hlist[8][E];
  __shared__ int hcount[8];
  __shared__ __align__(16) __nv_bfloat16 xs[8][H];  // x_hat row of each warp's token
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const float xn = xnorm[t];
  // the x_hat row is needed later; its loads go out now, with the logits'
  uint4 xraw[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) xraw[j] = __ldg(reinterpret_cast<const uint4*>(xh + (size_t)t * H) + lane * 8 + j);
  float sv[8], eps[8], wn8[8];
  {
    const float4 a = __ldg(reinterpret_cast<const float4*>(S + (size_t)t * E + lane * 8));
    const float4 b = __ldg(reinterpret_cast<const float4*>(S + (size_t)t * E + lane * 8 + 4));
    const float4 na = __ldg(reinterpret_cast<const float4*>(wnorm + lane * 8));
    const float4 nb = __ldg(reinterpret_cast<const float4*>(wnorm + lane * 8 + 4));
    const float s8[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const float n8[8] = {na.x, na.y, na.z, na.w, nb.x, nb.y, nb.z, nb.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      sv[i] = s8[i];
      wn8[i] = n8[i];
      eps[i] = GAMMA_TC * xn * n8[i] * 1.01f;
    }
  }
  // L = 6th largest lower bound (S - eps); ties irrelevant for a bound
  uint32_t taken = 0u;
  float L = 0.f;
  for (int k = 0; k < TOPK; ++k) {
    uint32_t best = 0u;
    int bi = -1;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t o = ord_f32(sv[i] - eps[i]);
      if (!((taken >> i) & 1u) && (bi < 0 || o > best)) {
        best = o;
        bi = i;
      }
    }
    const uint32_t m = redux_max(best);
    const unsigned owner = __ballot_sync(0xffffffffu, best == m);
    const int ol = __ffs(owner) - 1;
    const int oi = __shfl_sync(0xffffffffu, bi, ol);
    if (lane == ol) taken |= 1u << oi;
    const uint32_t fb = (m & 0x80000000u) ? (m & 0x7FFFFFFFu) : ~m;
    L = __uint_as_float(fb);
  }
  // An expert can be selected only if its bf16 logit reaches bf16(L), so its
  // exact logit lies within 1.5 bf16 ulps of L (half an ulp either side of the
  // rounded value, the lower side possibly in the next binade); 2 ulps are kept.
  const float aL = fabsf(L);
  const float ulp = aL > 0.f ? __int_as_float(((int)((__float_as_uint(aL) >> 23) & 0xFF) - 7) << 23) : 0.f;
  const float thr = L - 2.0f * ulp;
  uint32_t cand = 0u;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (sv[i] + eps[i] >= thr) cand |= 1u << i;
  int total = __popc(cand);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) total += __shfl_xor_sync(0xffffffffu, total, off);
  // Outside the band where distinct bf16 logits give distinct fp32 scores, or with
  // too many candidates, every logit is computed exactly.
  const bool all = total > 32 || !(L > -80.f && L < 8.f) || fabsf(L) < 4.8828125e-4f;
  if (all) cand = 0xFFu;
  // x_hat row into the warp's shared-memory slot
#pragma unroll
  for (int j = 0; j < 8; ++j) reinterpret_cast<uint4*>(xs[warp])[lane * 8 + j] = xraw[j];
  __syncwarp();
  // Exact bf16 logits of the candidates; every other logit is set to -inf.
  // Four candidates at a time, one per group of 8 lanes: lane l of a group
  // takes columns 64 i + 8 l .. +7 for i = 0..31 (coalesced 128-byte pieces of
  // the weight row; x_hat from shared memory), in 8 fused multiply-add chains
  // of 32, then a 3-level tree over the chains and a 3-level tree over the
  // group (depth 38): the error is at most gamma_38 * sum|x_k w_k| <=
  // G38 * ||x|| * ||w||, plus 38 * 2^-150 should a step underflow (covered by
  // an absolute 1e-37).  If both ends of that interval round to the same
  // bf16 value, so does the exact logit (rounding is monotone, and the ends
  // are fp32 values obtained with directed rounding).  Only the rare
  // candidate whose interval straddles a bf16 rounding boundary is
  // recomputed error-free (TwoSum).  Returns whether a candidate's
  // tensor-core logit missed it by more than a quarter of the assumed bound.
  constexpr float G38 = 2.27e-6f;  // >= gamma_38 = 38 u / (1 - 38 u), u = 2^-24
  static_assert((double)G38 >= 38.0 / 16777216.0 / (1.0 - 38.0 / 16777216.0), "G38 must bound gamma_38");
  const int grp = lane >> 3, gl = lane & 7;
  auto exact_logits = [&](uint32_t cmask) -> bool {
    for (int i = lane; i < E; i += 32) lrow[warp][i] = __float2bfloat16_rn(-INFINITY);
    const int cnt = __popc(cmask);
    int incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    const int n = __shfl_sync(0xffffffffu, incl, 31);
    int pos = incl - cnt;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((cmask >> i) & 1u) {
        clist[warp][pos] = (uint8_t)(lane * 8 + i);
        ++pos;
      }
    if (lane == 0) hcount[warp] = 0;
    __syncwarp();
    bool off = false;
    // One lane: record candidate e's exact logit lam; check the tensor-core
    // logit s_e against the assumed bound (recomputed as in the candidate test).
    auto settle = [&](int e, float lam, float s_e, float wn_e) {
      lrow[warp][e] = __float2bfloat16_rn(lam);
      if (!(fabsf(s_e - lam) <= 0.25f * (GAMMA_TC * xn * wn_e * 1.01f))) off = true;
    };
    const uint4* xv = reinterpret_cast<const uint4*>(xs[warp]);
    for (int ci = 0; ci < n; ci += 4) {
      const int c = ci + grp;
      const int e = clist[warp][c < n ? c : ci];
      const float s_e = __ldg(S + (size_t)t * E + e), wn_e = __ldg(wnorm + e);
      const uint4* wrow = reinterpret_cast<const uint4*>(wr + (size_t)e * H);
      float pc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
      for (int i = 0; i < H / 64; ++i) {
        const uint4 wv = __ldg(wrow + i * 8 + gl);
        const uint4 x8 = xv[i * 8 + gl];
        const uint32_t wa[4] = {wv.x, wv.y, wv.z, wv.w};
        const uint32_t xa[4] = {x8.x, x8.y, x8.z, x8.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          pc[2 * q] = fmaf(__uint_as_float(xa[q] << 16), __uint_as_float(wa[q] << 16), pc[2 * q]);
          pc[2 * q + 1] =
              fmaf(__uint_as_float(xa[q] & 0xFFFF0000u), __uint_as_float(wa[q] & 0xFFFF0000u), pc[2 * q + 1]);
        }
      }
      float sum = __fadd_rn(__fadd_rn(__fadd_rn(pc[0], pc[1]), __fadd_rn(pc[2], pc[3])),
                            __fadd_rn(__fadd_rn(pc[4], pc[5]), __fadd_rn(pc[6], pc[7])));
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) sum = __fadd_rn(sum, __shfl_xor_sync(0xffffffffu, sum, o));
      if (gl == 0 && c < n) {
        const float err = fmaf(G38 * xn, wn_e, 1.0e-37f);
        const __nv_bfloat16 blo = __float2bfloat16_rn(__fsub_rd(sum, err));
        const __nv_bfloat16 bhi = __float2bfloat16_rn(__fadd_ru(sum, err));
        if (__bfloat16_as_ushort(blo) == __bfloat16_as_ushort(bhi)) settle(e, sum, s_e, wn_e);
        else hlist[warp][atomicAdd(&hcount[warp], 1)] = (uint8_t)c;
      }
    }
    __syncwarp();
    const int nh = hcount[warp];
    for (int hi = 0; hi < nh; ++hi) {  // straddling candidates: error-free sum over the whole warp
      const int c = hlist[warp][hi], e = clist[warp][c];
      const float s_e = __ldg(S + (size_t)t * E + e), wn_e = __ldg(wnorm + e);
      CSum a = {0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float f[8], xf[8];
        bf16x8_f32(__ldg(reinterpret_cast<const uint4*>(wr + (size_t)e * H) + lane * 8 + j), f);
        bf16x8_f32(xv[lane * 8 + j], xf);
#pragma unroll
        for (int i = 0; i < 8; ++i) cs_add(a, __fmul_rn(xf[i], f[i]));
      }
      a = cs_warp_reduce(a);
      if (lane == 0) settle(e, cs_value(a), s_e, wn_e);  // the rounding of the exact sum
    }
    __syncwarp();
    return __any_sync(0xffffffffu, off);
  };
  if (exact_logits(cand)) {
    if (lane == 0) atomicOr(err, ERR_ROUTER_BOUND);
    if (!all) exact_logits(0xFFu);
  }
  __syncwarp();
  if (lane < 8) umask_dummy[warp][lane] = 0u;
  __syncwarp();
  const uint4 raw = *reinterpret_cast<const uint4*>(&lrow[warp][lane * 8]);
  warp_topk(raw, lane, sids[warp], sw[warp], umask_dummy[warp]);
  __syncwarp();
  if (lane < TOPK) {
    const int e = sids[warp][lane];
    const float w = sw[warp][lane];
    ids[(size_t)t * TOPK + lane] = e;
    wts[(size_t)t * TOPK + lane] = w;
    if (ids_out) ids_out[(size_t)t * TOPK + lane] = e;
    if (w_out) w_out[(size_t)t * TOPK + lane] = w;
    atomicAdd(&counts[e], 1);
  }
  // The fp32 output accumulator of this token starts at zero (stores that
  // overlap this latency-bound kernel instead of a separate memset; issued
  // last so that they do not queue ahead of the loads above).
#pragma unroll
  for (int j = 0; j < H / 128; ++j)
    reinterpret_cast<float4*>(yacc + (size_t)t * H)[lane + 32 * j] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ---------------------------------------------------------------- scatter
// offsets[e]: start of expert e's pairs (experts 0..255 routed, 256 shared);
// prefix[kind][e]: first work item of expert e (items = tiles of 256 pairs x
// weight-row tiles of 128).  One thread per (token, expert) pair.  Each block
// scans the 257 counts itself (exclusive prefix in shared memory); block 0
// also publishes the offsets and the work-item prefixes of the two grouped
// GEMMs.
__global__ void __launch_bounds__(256) prefill_scatter_kernel(const int32_t* __restrict__ ids,
                                                              const float* __restrict__ wts,
                                                              const int* __restrict__ counts,
                                                              int* __restrict__ cursor, int T,
                                                              int* __restrict__ pair_token, float* __restrict__ pair_w,
                                                              int* __restrict__ offsets, int* __restrict__ gu_prefix,
                                                              int* __restrict__ dn_prefix) {
  __shared__ int c[NE + 1];
  __shared__ int warp_sum[9];
  const int tid = threadIdx.x, lane = tid & 31, wp = tid >> 5;
  // inclusive scan of the counts, 2 per thread (expert 2tid, 2tid+1; 256 = shared)
  const int e0 = 2 * tid, e1 = 2 * tid + 1;
  const int v0 = e0 < E ? __ldg(counts + e0) : (e0 == E ? T : 0);
  const int v1 = e1 < E ? __ldg(counts + e1) : (e1 == E ? T : 0);
  int incl = v0 + v1;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += u;
  }
  if (lane == 31) warp_sum[wp] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < wp; ++w) base += warp_sum[w];
  const int excl = base + incl - v0 - v1;  // offset of expert e0
  if (e0 <= NE) c[e0] = excl;
  if (e1 <= NE) c[e1] = excl + v0;
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int e = tid; e <= NE; e += blockDim.x) {
      offsets[e] = c[e];
    }
    // work-item prefixes: exclusive scan of each expert's tiles of PG_N pairs
    // (entry NE = the total), times the weight-row tiles of each GEMM
    const int n0 = e0 < NE ? (c[e0 + 1] - c[e0] + PG_N - 1) / PG_N : 0;
    const int n1 = e1 < NE ? (c[e1 + 1] - c[e1] + PG_N - 1) / PG_N : 0;
    int tin = n0 + n1;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, tin, off);
      if (lane >= off) tin += u;
    }
    __syncthreads();  // every thread has read warp_sum above
    if (lane == 31) warp_sum[wp] = tin;
    __syncthreads();
    int tbase = 0;
    for (int w = 0; w < wp; ++w) tbase += warp_sum[w];
    const int t0 = tbase + tin - n0 - n1;  // tiles before expert e0
    if (e0 <= NE) {
      gu_prefix[e0] = t0 * (2 * I / PG_M);
      dn_prefix[e0] = t0 * (H / PG_M);
    }
    if (e1 <= NE) {
      gu_prefix[e1] = (t0 + n0) * (2 * I / PG_M);
      dn_prefix[e1] = (t0 + n0) * (H / PG_M);
    }
  }
  const int q = blockIdx.x * blockDim.x + tid;
  if (q < T * TOPK) {
    const int t = q / TOPK, e = ids[q];
    const int pos = c[e] + atomicAdd(&cursor[e], 1);
    pair_token[pos] = t;
    pair_w[pos] = wts[q];
  } else if (q < T * (TOPK + 1)) {
    const int t = q - T * TOPK;
    pair_token[c[E] + t] = t;
    pair_w[c[E] + t] = 1.0f;
  }
}

// ---------------------------------------------------------------- grouped GEMM
// One persistent CTA per SM walks work items (expert, token tile, 128-row
// weight tile), interleaved over CTAs.  Item = D[128 x N] = W[128 x K] *
// Xg[N x K]^T with N = the tile's token count rounded up to 16, K = 2048
// (gate/up) or 512 (down), in steps of 64 along K.  Rings in shared memory:
// 4 operand stages, each the dequantised A tile (16 KB) and the gathered B
// tile (32 KB) of one step, with one "full" barrier (both written) and one
// "empty" barrier (the step's MMAs done) per stage; and 3 slots of raw
// packed weight bytes, one 2-step pass of the 8 row tiles each (9 KB).  The
// router GEMM uses the same kernel with bf16 router weights copied into A as
// they are.  Warp roles:
//   warps 0-3   B producers: producer i gathers the N token rows of every
//               step g = i (mod 4) into B stage i with cp.async (8 lanes per
//               128-byte row piece, L2 evict-last), waits for its own
//               copies, fences them for the tensor core and signals
//   warp 4      lane 0 issues the TMA copies of the raw weight bytes of a
//               pass (8 row tiles x (1024 code bytes + 128 scale bytes));
//               the warp owns the tensor-memory allocation
//   warp 5      issues tcgen05.mma (4 per step, one elected lane) into one of two
//               256-column fp32 accumulators in tensor memory: one wait and
//               one commit per step
//   warps 8-11, 20-23  epilogue, two sets of 4 warps taking alternate
//               32-column chunks: tensor memory -> registers (lane quadrant =
//               warp % 4), SiLU*up -> h (gate/up), weighted add into the fp32
//               output (down) or the router logits; overlaps the next item's
//               main loop
//   warps 12-19 dequantisers: warp 12+r turns row tile r of a step into f16
//               (gate/up) or bf16 (down) with stmatrix into the
//               128-byte-swizzled A stage
// Every mbarrier wait is bounded; one that runs out sets the device error
// word and an abort flag that ends every role's loop.
struct GemmParams {
  const uint8_t* experts;
  const float* tscale;     // [NE][2]
  const int* prefix;       // [NE + 1] first item of each expert
  const int* offsets;      // [NE + 1]
  const int* pair_token;   // [P]
  const float* pair_w;     // [P]
  const uint16_t* bsrc;    // gate/up: x_hat f16 [T][H]; down: h bf16 [P][I]
  const int* xexp;         // [T]
  uint16_t* h;             // gate/up output [P][I]
  float* yacc;             // down output [T][H]
  const uint16_t* asrc;    // router: W_r bf16 [E][H]
  float* S;                // router output fp32 [T][E]
  unsigned* err;
};

// KIND 0: gate/up (NVFP4 -> f16 A, x_hat f16 B), 1: down (NVFP4 -> bf16 A,
// h bf16 B), 2: router (W_r bf16 A copied as is, x_hat bf16 B, fp32 logits).
template <int KIND>
struct GemmCfg {
  static constexpr int K = KIND == 1 ? I : H;
  static constexpr int NT = KIND == 2 ? 128 : PG_N;  // tokens per item (router: smaller, more items)
  static constexpr int NKS = K / PG_KS;
  static constexpr int MT = (KIND == 0 ? 2 * I : KIND == 1 ? H : E) / PG_M;
  static constexpr int TILE = KIND == 0 ? F4_GU_TILE : F4_DN_TILE;
  static constexpr size_t BASE = KIND == 0 ? 0 : F4_GU_BYTES;
};

constexpr int NS = 4;                          // operand ring stages (A and B tile of one K-step), one B producer warp each
constexpr int RPS = 3;                         // raw ring slots, one dequantiser pass (2 K-steps) each
constexpr int G_THREADS = 768;                 // 24 warps
constexpr int G_RAW_TILE = 1152;               // per row tile and pass: 1024 code bytes + 128 scale bytes
constexpr int G_A = PG_M * PG_KS * 2;          // 16 KB
constexpr int G_B = PG_N * PG_KS * 2;          // 32 KB
constexpr int G_RAW = 8 * G_RAW_TILE;          // 9 KB
static_assert(G_A % 1024 == 0 && G_B % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
static_assert((H / PG_KS) % 2 == 0 && (I / PG_KS) % 2 == 0, "dequantisers take two steps per pass");
// No alignment slack: the dynamic shared memory base is 1024-byte aligned
// (checked at run time).
constexpr size_t G_TABLES = 2 * (NE + 1) * sizeof(int) + 8;  // item prefixes and pair offsets, copied per CTA
constexpr size_t G_SMEM = (size_t)NS * (G_A + G_B) + (size_t)RPS * G_RAW + 256 + G_TABLES;
static_assert(G_SMEM <= 232448, "shared memory per CTA");

// 16-byte cp.async with an L2 eviction policy (token rows are re-read by
// every weight-row tile of their expert: keep them in L2).
__device__ __forceinline__ void cp_async16_keep(void* sdst, const void* gsrc, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_u32(sdst)), "l"(gsrc),
               "l"(pol)
               : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void stmatrix_x4(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(r0), "r"(r1),
               "r"(r2), "r"(r3)
               : "memory");
}

// f16 (KIND 0) or bf16 (KIND 1) pair of dequantised weights: code pair (f16x2)
// times the block scale; both results are exact (at most 6 significant bits).
template <int KIND>
__device__ __forceinline__ uint32_t dq_pair(uint32_t f16pair, uint32_t scale16x2_lohalf, float scale_f) {
  if (KIND == 0) return hmul2_lo(f16pair, scale16x2_lohalf);
  const __half2 hv = *reinterpret_cast<const __half2*>(&f16pair);
  const float2 f = __half22float2(hv);
  const __nv_bfloat162 b = __floats2bfloat162_rn(__fmul_rn(f.x, scale_f), __fmul_rn(f.y, scale_f));
  return *reinterpret_cast<const uint32_t*>(&b);
}

struct ItemInfo {
  int e, mtile, pair0, nvalid, n;  // n = MMA width (nvalid rounded up to 16)
};
// prefix and offs are the CTA's shared-memory copies.
__device__ __forceinline__ ItemInfo decode_item(int item, const int* prefix, const int* offs, int MT, int NT = PG_N) {
  int lo = 0, hi = NE;  // largest e with prefix[e] <= item
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= item) lo = mid;
    else hi = mid;
  }
  ItemInfo it;
  it.e = lo;
  const int local = item - prefix[lo];
  it.mtile = local % MT;
  const int ntile = local / MT;
  it.pair0 = offs[lo] + ntile * NT;
  it.nvalid = min(NT, offs[lo + 1] - it.pair0);
  it.n = (it.nvalid + 15) & ~15;
  return it;
}

template <int KIND>
__global__ void __launch_bounds__(G_THREADS, 1) prefill_gemm_kernel(const GemmParams p) {
  using C = GemmCfg<KIND>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // the swizzled stages need 1024-byte alignment
    if (threadIdx.x == 0) atomicOr(p.err, ERR_LAYOUT);
    return;
  }
  uint8_t* sm = smem_raw;
  uint8_t* aring = sm;                        // [NS][16 KB]
  uint8_t* bring = sm + NS * G_A;             // [NS][32 KB]
  uint8_t* rawring = bring + NS * G_B;        // [RPS][9 KB]
  uint64_t* bars = reinterpret_cast<uint64_t*>(rawring + RPS * G_RAW);
  uint64_t* full = bars;                      // [NS] A tile written (8 warps) and B rows landed (32 lanes)
  uint64_t* empty = full + NS;                // [NS] MMAs reading the stage done (tcgen05.commit)
  uint64_t* rfull = empty + NS;               // [RPS] raw bytes landed (TMA transaction count)
  uint64_t* rempty = rfull + RPS;             // [RPS] raw slot consumed (8 dequant warps)
  uint64_t* accfull = rempty + RPS;           // [2] accumulator complete (tcgen05.commit)
  uint64_t* accempty = accfull + 2;           // [2] accumulator read out (8 epilogue warps)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(accempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  int* sprefix = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(bars) + 256);  // [NE + 1]
  int* soffs = sprefix + (NE + 1);                                                // [NE + 1]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 4) {
    tc05::tmem_alloc(tslot, 2 * PG_N);
    tc05::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 8 + 32);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < RPS; ++i) {
      mbar_init(&rfull[i], 1);
      mbar_init(&rempty[i], 8);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accfull[i], 1);
      mbar_init(&accempty[i], 8);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = tid; i <= NE; i += G_THREADS) {  // item decoding then searches shared memory
    sprefix[i] = __ldg(p.prefix + i);
    soffs[i] = __ldg(p.offsets + i);
  }
  tc05::fence_before_sync();
  __syncthreads();
  tc05::fence_after_sync();
  const uint32_t tmem = *tslot;
  const int n_items = sprefix[NE];
  // Bounded wait shared by every role.  Where a whole warp waits and then goes
  // on to warp-synchronous instructions (shuffles, stmatrix, tcgen05.ld), its
  // lanes agree on the result: the awaited phase cannot move on without a later
  // arrival of this same warp, so once one lane sees it complete every lane
  // does, and the time limit is judged on the clock all lanes read in the same
  // instruction.  (The MMA warp elects among __activemask() and needs no such
  // argument.)
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (mbar_try_wait(bar, parity)) return true;  // the usual case: one probe
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity)) return true;
    atomicOr(p.err, ERR_WAIT_FULL);
    *abort_flag = 1;
    return false;
  };

  if (warp < NS) {
    // ---------------- B producers: warp w owns the B tile of stage w (steps g = w mod NS)
    const int bp = warp;
    uint32_t g = 0;  // global step of this CTA
    bool ok = true;
    const uint64_t keep = l2_evict_last();
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const ItemInfo it = decode_item(item, sprefix, soffs, C::MT, C::NT);
      int rowid[8];  // source row of tile rows lane + 32 i
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int pr = it.pair0 + min(lane + 32 * i, it.nvalid - 1);
        rowid[i] = KIND == 0 ? __ldg(p.pair_token + pr) : pr;  // router: the token itself
      }
      const int ch = lane & 7;
      for (int ks = 0; ks < C::NKS; ++ks, ++g) {
        if ((int)(g % NS) != bp) continue;
        if (!wait(&empty[bp], ((g / NS) & 1) ^ 1)) {
          ok = false;
          break;
        }
        uint8_t* dst = bring + bp * G_B;
        // 8 lanes per row: one instruction moves 4 whole 128-byte row pieces
#pragma unroll
        for (int i = 0; i < PG_N / 4; ++i) {
          const int r = 4 * i + (lane >> 3);
          const int row = __shfl_sync(0xffffffffu, rowid[i >> 3], r & 31);
          if (4 * i < it.n)
            cp_async16_keep(dst + tc05::sw128_off(r, ch * 8), p.bsrc + (size_t)row * C::K + ks * PG_KS + ch * 8, keep);
        }
        asm volatile("cp.async.commit_group;\n cp.async.wait_group 0;" ::: "memory");
        tc05::fence_proxy_async_smem();
        mbar_arrive(&full[bp]);
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == 4) {
    // ---------------- raw weight producer: one slot per dequantiser pass (2 K-steps)
    if (KIND != 2 && lane == 0) {
      uint32_t pi = 0;  // global pass
      bool ok = true;
      const uint64_t pol = l2_evict_first();
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
        const ItemInfo it = decode_item(item, sprefix, soffs, C::MT, C::NT);
        const uint8_t* wbase = p.experts + (size_t)it.e * F4_EXPERT + C::BASE + (size_t)it.mtile * 8 * C::TILE;
        for (int ks = 0; ks < C::NKS; ks += 2, ++pi) {
          const uint32_t s = pi % RPS;
          if (!wait(&rempty[s], ((pi / RPS) & 1) ^ 1)) {
            ok = false;
            break;
          }
          uint8_t* dst = rawring + s * G_RAW;
          mbar_arrive_expect_tx(&rfull[s], G_RAW);
          const int q = ks >> 2, c4 = ks & 3;  // c4 is 0 or 2: both steps share one half of the scales
          for (int r = 0; r < 8; ++r) {
            const uint8_t* sl = wbase + (size_t)r * C::TILE + (size_t)q * F4_SLICE;
            bulk_g2s(dst + r * G_RAW_TILE, sl + c4 * 512, 1024, &rfull[s], pol);
            bulk_g2s(dst + r * G_RAW_TILE + 1024, sl + F4_CODES + (c4 >> 1) * 128, 128, &rfull[s], pol);
          }
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA exits
        for (uint32_t q = pi > RPS ? pi - RPS : 0; q < pi; ++q) (void)mbar_wait(&rfull[q % RPS], (q / RPS) & 1);
      }
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer.  The whole warp runs the loop, so that the
    // stage indices and descriptors are warp-uniform values; each tcgen05.mma
    // and tcgen05.commit is issued by the lane elect.sync picks among the
    // lanes still in the loop.  Normally that is the whole warp; a lane whose
    // wait runs out leaves on its own, and no elect.sync waits for it.
    // Every item has a multiple of NS K-steps, so it starts at
    // stage 0 and the loop is unrolled over the stages: each stage's
    // descriptors are fixed offsets from two base descriptors, and one wait
    // and one commit cover a step.
    {
      static_assert(C::NKS % NS == 0, "items must start at ring stage 0");
      uint32_t i_local = 0, ph = 0, steps = 0;
      bool ok = true;
      const uint64_t da0 = tc05::sw128_desc(smem_u32(aring)), db0 = tc05::sw128_desc(smem_u32(bring));
      for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++i_local) {
        const ItemInfo it = decode_item(item, sprefix, soffs, C::MT, C::NT);
        const uint32_t b = i_local & 1, u = i_local >> 1;
        if (!wait(&accempty[b], (u & 1) ^ 1)) break;
        tc05::fence_after_sync();
        const uint32_t idesc = tc05::idesc_f16(PG_M, it.n, KIND == 0 ? 0 : 1);
        const uint32_t d = tmem + b * PG_N;
        for (int ks = 0; ks < C::NKS && ok; ks += NS) {
#pragma unroll
          for (int s = 0; s < NS; ++s) {
            if (!wait(&full[s], ph)) {
              ok = false;
              break;
            }
            tc05::fence_after_sync();
            const uint32_t members = __activemask();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc05::mma_f16_elect(members, d, da0 + (uint64_t)(s * (G_A >> 4) + 2 * kk),
                                  db0 + (uint64_t)(s * (G_B >> 4) + 2 * kk), idesc, (ks + s > 0 || kk > 0) ? 1u : 0u);
            tc05::commit_elect(members, &empty[s]);
            ++steps;
          }
          ph ^= 1u;
        }
        if (ok) tc05::commit_elect(__activemask(), &accfull[b]);
      }
      if (steps > 0) (void)mbar_wait(&empty[(steps - 1) % NS], ((steps - 1) / NS) & 1);  // last MMAs retired
    }
  } else if ((warp >= 8 && warp < 12) || warp >= 20) {
    // ---------------- epilogue: two sets of 4 warps (8-11 and 20-23), each
    // covering the 4 TMEM lane quadrants; set s takes the 32-column chunks
    // s, s + 2, s + 4, ... of every item
    const int quad = warp & 3, eset = warp >= 20 ? 1 : 0;
    uint32_t i_local = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++i_local) {
      const ItemInfo it = decode_item(item, sprefix, soffs, C::MT, C::NT);
      const uint32_t b = i_local & 1, u = i_local >> 1;
      const float ts = KIND == 2 ? 1.0f : __ldg(p.tscale + 2 * it.e + KIND);
      if (!wait(&accfull[b], u & 1)) break;
      tc05::fence_after_sync();
      const int m = quad * 32 + lane;  // weight row within the tile
      for (int c0 = 32 * eset; c0 < it.n; c0 += 64) {
        // per-column token and factor, one column per lane, broadcast below
        const int pr = it.pair0 + min(c0 + lane, it.nvalid - 1);
        const int ctok = KIND == 2 ? pr : __ldg(p.pair_token + pr);
        const float cfac = KIND == 0   ? __fmul_rn(ts, exp2i_p(-__ldg(p.xexp + ctok)))
                           : KIND == 1 ? __ldg(p.pair_w + pr)
                                       : 1.0f;
        uint32_t v[32];
        tc05::ld_32x32b_x32(tmem + ((uint32_t)(quad * 32) << 16) + b * PG_N + (uint32_t)c0, v);
        tc05::wait_ld();
        if (KIND == 2) {
          // router logits: lanes hold consecutive experts of one token column
          const int e = it.mtile * PG_M + m;
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c0 + c < it.nvalid) p.S[(size_t)(it.pair0 + c0 + c) * E + e] = __uint_as_float(v[c]);
        } else if (KIND == 0) {
          // Lane pairs (tr, tr ^ 8) hold the gate and up rows of one
          // intermediate index j: the low lane finishes even columns, the high
          // lane odd ones, so every lane works; neighbours (j, j ^ 1) then
          // store one bf16x2.
          const int tr = m & 15;
          const bool lo = tr < 8;
          const int j = (it.mtile * 8 + (m >> 4)) * 8 + (tr & 7);
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const uint32_t send = lo ? v[c + 1] : v[c];
            const float recv = __uint_as_float(__shfl_xor_sync(0xffffffffu, send, 8));
            const int cc = c + (lo ? 0 : 1);
            const float f = __shfl_sync(0xffffffffu, cfac, cc);
            const float gate = __fmul_rn(lo ? __uint_as_float(v[c]) : recv, f);
            const float up = __fmul_rn(lo ? recv : __uint_as_float(v[c + 1]), f);
            const float silu = __fdividef(gate, 1.0f + __expf(-gate));
            const __nv_bfloat16 hv = __float2bfloat16_rn(silu * up);
            const uint32_t hb = *reinterpret_cast<const uint16_t*>(&hv);
            const uint32_t nb = __shfl_xor_sync(0xffffffffu, hb, 1);
            if ((tr & 1) == 0 && c0 + cc < it.nvalid)
              *reinterpret_cast<uint32_t*>(p.h + (size_t)(it.pair0 + c0 + cc) * I + j) = hb | (nb << 16);
          }
        } else {
          // 4 x 4 transposes among lane quads (two shuffle stages): lane l
          // ends with rows 4(l/4)..+3 of column 4k + l%4 and adds them with
          // one 16-byte reduction.
          const int i1 = lane & 1, p2 = (lane >> 1) & 1;
          const int orow = it.mtile * PG_M + quad * 32 + (lane & ~3);
#pragma unroll
          for (int b4 = 0; b4 < 32; b4 += 4) {
            const float x0 = __uint_as_float(v[b4]), x1 = __uint_as_float(v[b4 + 1]);
            const float x2 = __uint_as_float(v[b4 + 2]), x3 = __uint_as_float(v[b4 + 3]);
            const float ra = __shfl_xor_sync(0xffffffffu, i1 ? x0 : x1, 1);
            const float rb = __shfl_xor_sync(0xffffffffu, i1 ? x2 : x3, 1);
            // column (i1): rows (2p, 2p+1) of the quad; column (2 + i1) likewise
            const float q0a = i1 ? ra : x0, q0b = i1 ? x1 : ra;
            const float q1a = i1 ? rb : x2, q1b = i1 ? x3 : rb;
            const float sa = __shfl_xor_sync(0xffffffffu, p2 ? q0a : q1a, 2);
            const float sb = __shfl_xor_sync(0xffffffffu, p2 ? q0b : q1b, 2);
            float4 o;
            o.x = p2 ? sa : q0a;
            o.y = p2 ? sb : q0b;
            o.z = p2 ? q1a : sa;
            o.w = p2 ? q1b : sb;
            const int cl = b4 + (lane & 3);
            const int tok = __shfl_sync(0xffffffffu, ctok, cl);
            const float f = __fmul_rn(__shfl_sync(0xffffffffu, cfac, cl), ts);
            if (c0 + cl < it.nvalid) {
              float* dst = p.yacc + (size_t)tok * H + orow;
              asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(__fmul_rn(o.x, f)),
                           "f"(__fmul_rn(o.y, f)), "f"(__fmul_rn(o.z, f)), "f"(__fmul_rn(o.w, f))
                           : "memory");
            }
          }
        }
      }
      tc05::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accempty[b]);
    }
  } else if (KIND == 2 && warp >= 12 && warp < 20) {
    // ---------------- router A producers: warp 12 + r copies rows 16r..16r+15
    // of the 128-expert tile of W_r, two K-steps per pass
    const int r = warp - 12;
    uint32_t g = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const ItemInfo it = decode_item(item, sprefix, soffs, C::MT, C::NT);
      const uint16_t* arow0 = p.asrc + (size_t)(it.mtile * PG_M + r * 16) * H;
      for (int ks = 0; ks < C::NKS; ks += 2, g += 2) {
        if (!wait(&empty[g % NS], ((g / NS) & 1) ^ 1) || !wait(&empty[(g + 1) % NS], (((g + 1) / NS) & 1) ^ 1)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint8_t* dst = aring + ((g + h) % NS) * G_A;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int idx = lane + 32 * i, row = idx >> 3, ch = idx & 7;
            cp_async16(dst + tc05::sw128_off(r * 16 + row, ch * 8), arow0 + (size_t)row * H + (ks + h) * PG_KS + ch * 8);
          }
        }
        asm volatile("cp.async.commit_group;\n cp.async.wait_group 0;" ::: "memory");
        tc05::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&full[g % NS]);
          mbar_arrive(&full[(g + 1) % NS]);
        }
      }
    }
  } else if (KIND != 2 && warp >= 12 && warp < 20) {
    // ---------------- dequantisers: warp 12 + r owns row tile r of every step
    const int r = warp - 12;
    const int g8 = lane >> 2;
    const int mi = lane >> 3, rr = lane & 7;
    const int st_row = r * 16 + (mi & 1) * 8 + rr;  // stmatrix row address of this lane
    uint32_t g = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      for (int ks = 0; ks < C::NKS; ks += 2, g += 2) {  // two steps per pass (NKS is even)
        const uint32_t pi = g >> 1, rs = pi % RPS;
        if (!wait(&rfull[rs], (pi / RPS) & 1)) {
          ok = false;
          break;
        }
        uint32_t cwv[2][4], scv[2][2];
        const uint8_t* raw = rawring + rs * G_RAW + r * G_RAW_TILE;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint4 cw = *reinterpret_cast<const uint4*>(raw + h * 512 + lane * 16);
          const uint2 sc8 = *reinterpret_cast<const uint2*>(raw + 1024 + g8 * 16 + 8 * h);
          cwv[h][0] = cw.x;
          cwv[h][1] = cw.y;
          cwv[h][2] = cw.z;
          cwv[h][3] = cw.w;
          scv[h][0] = sc8.x;
          scv[h][1] = sc8.y;
        }
        // Each step's A stage is awaited and published on its own, so that the
        // dequantisation of a step overlaps the MMAs of the two before it.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (!wait(&empty[(g + h) % NS], (((g + h) / NS) & 1) ^ 1)) {
            ok = false;
            break;
          }
          const uint32_t a_base = smem_u32(aring + ((g + h) % NS) * G_A);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t pair16 = (scv[h][j >> 1] >> ((j & 1) * 16)) & 0xFFFFu;
            const uint32_t sc = e4m3x2_to_f16x2(pair16);
            float sg = 0.f, sg8 = 0.f;
            if (KIND == 1) {
              const float2 sf = __half22float2(*reinterpret_cast<const __half2*>(&sc));
              sg = sf.x;
              sg8 = sf.y;
            }
            uint32_t a0, a1, a2, a3;
            e2m1x8_to_f16x2(cwv[h][j], a0, a1, a2, a3);
            const uint32_t hi_sc = __byte_perm(sc, 0, 0x3232);
            // fragments: (row g, k 16j+2t), (row g+8, same k), (row g, k+8), (row g+8, k+8)
            const uint32_t v0 = dq_pair<KIND>(a0, sc, sg);
            const uint32_t v1 = dq_pair<KIND>(a1, hi_sc, sg8);
            const uint32_t v2 = dq_pair<KIND>(a2, sc, sg);
            const uint32_t v3 = dq_pair<KIND>(a3, hi_sc, sg8);
            stmatrix_x4(a_base + tc05::sw128_off(st_row, 16 * j + (mi >> 1) * 8), v0, v1, v2, v3);
          }
          tc05::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[(g + h) % NS]);
        }
        if (!ok) break;
        // the raw slot is released only now: every lane has consumed the
        // values it loaded from it (an earlier release let the next TMA copy
        // overwrite a slot under loads still in flight)
        if (lane == 0) mbar_arrive(&rempty[rs]);
      }
    }
  }

  tc05::fence_before_sync();
  __syncthreads();
  if (warp == 4) {
    tc05::fence_after_sync();
    tc05::tmem_dealloc(tmem, 2 * PG_N);
  }
}

__global__ void prefill_finalize_kernel(const float4* __restrict__ yacc, uint2* __restrict__ y, size_t n4) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const float4 v = yacc[i];
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  y[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

size_t a256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

// ---------------------------------------------------------------- workspace and launch

struct PrefillWs {
  __nv_bfloat16* xh;  // [T][H] (only with a norm)
  __half* xh16;       // [T][H]
  int* xexp;          // [T]
  float* xnorm;       // [T]
  float* wnorm;       // [E]
  float* S;           // [T][E]
  int32_t* ids;       // [T][6]
  float* wts;         // [T][6]
  int* counts;        // [E]
  int* cursor;        // [E]
  int* offsets;       // [NE + 1]
  int* gu_prefix;     // [NE + 1]
  int* dn_prefix;     // [NE + 1]
  int* pair_token;    // [7T]
  float* pair_w;      // [7T]
  uint16_t* h;        // [7T][I]
  float* yacc;        // [T][H]
  int* rprefix;       // [NE + 1] work items of the router GEMM (all under entry 0)
  int* roffs;         // [NE + 1] its token range: 0 .. T
};

static PrefillWs carve_prefill(void* ws, int T, size_t* total) {
  uint8_t* p = static_cast<uint8_t*>(ws);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* r = p ? p + off : nullptr;
    off += a256(bytes);
    return r;
  };
  PrefillWs w;
  const size_t P = (size_t)T * (TOPK + 1);
  w.xh = reinterpret_cast<__nv_bfloat16*>(take((size_t)T * H * 2));
  w.xh16 = reinterpret_cast<__half*>(take((size_t)T * H * 2));
  w.xexp = reinterpret_cast<int*>(take((size_t)T * 4));
  w.xnorm = reinterpret_cast<float*>(take((size_t)T * 4));
  w.wnorm = reinterpret_cast<float*>(take((size_t)E * 4));
  w.S = reinterpret_cast<float*>(take((size_t)T * E * 4));
  w.ids = reinterpret_cast<int32_t*>(take((size_t)T * TOPK * 4));
  w.wts = reinterpret_cast<float*>(take((size_t)T * TOPK * 4));
  w.counts = reinterpret_cast<int*>(take((size_t)E * 4));
  w.cursor = reinterpret_cast<int*>(take((size_t)E * 4));
  w.offsets = reinterpret_cast<int*>(take((size_t)(NE + 1) * 4));
  w.gu_prefix = reinterpret_cast<int*>(take((size_t)(NE + 1) * 4));
  w.dn_prefix = reinterpret_cast<int*>(take((size_t)(NE + 1) * 4));
  w.pair_token = reinterpret_cast<int*>(take(P * 4));
  w.pair_w = reinterpret_cast<float*>(take(P * 4));
  w.h = reinterpret_cast<uint16_t*>(take(P * I * 2));
  w.yacc = reinterpret_cast<float*>(take((size_t)T * H * 4));
  w.rprefix = reinterpret_cast<int*>(take((size_t)(NE + 1) * 4));
  w.roffs = reinterpret_cast<int*>(take((size_t)(NE + 1) * 4));
  if (total) *total = off;
  return w;
}

size_t prefill_ws_bytes(int T) {
  size_t total = 0;
  carve_prefill(nullptr, T, &total);
  return total;
}

cudaError_t prefill_kernels_init(int /*device*/) {
  cudaError_t e = cudaFuncSetAttribute(prefill_gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)G_SMEM);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(prefill_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)G_SMEM);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(prefill_gemm_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)G_SMEM);
}

cudaError_t launch_prefill(const LayerArgs& L, const void* x, int T, float eps, void* y, int32_t* ids_out,
                           float* w_out, void* ws, int sm_count, unsigned* err, cudaStream_t st) {
  PrefillWs w = carve_prefill(ws, T, nullptr);
  const __nv_bfloat16* xin = static_cast<const __nv_bfloat16*>(x);
  const __nv_bfloat16* norm = static_cast<const __nv_bfloat16*>(L.norm_w);
  const __nv_bfloat16* xh = norm ? w.xh : xin;
  cudaError_t e;
  if ((e = cudaMemsetAsync(w.counts, 0, E * 4, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(w.cursor, 0, E * 4, st)) != cudaSuccess) return e;
  const int router_items = ((T + GemmCfg<2>::NT - 1) / GemmCfg<2>::NT) * (E / PG_M);
  prefill_prep_kernel<<<E / 8 + T, 256, 0, st>>>(xin, norm, eps, w.xh, w.xh16, w.xexp, w.xnorm, w.rprefix, w.roffs,
                                                 router_items, T, static_cast<const __nv_bfloat16*>(L.router_w),
                                                 w.wnorm);
  GemmParams gp = {};
  gp.err = err;
  gp.prefix = w.rprefix;
  gp.offsets = w.roffs;
  gp.bsrc = reinterpret_cast<const uint16_t*>(xh);
  gp.asrc = static_cast<const uint16_t*>(L.router_w);
  gp.S = w.S;
  prefill_gemm_kernel<2><<<sm_count < router_items ? sm_count : router_items, G_THREADS, G_SMEM, st>>>(gp);
  prefill_route_kernel<<<(T + 7) / 8, 256, 0, st>>>(xh, static_cast<const __nv_bfloat16*>(L.router_w), w.S, w.xnorm,
                                                    w.wnorm, T, w.ids, w.wts, w.counts, ids_out, w_out, err, w.yacc);
  const int nq = T * (TOPK + 1);
  prefill_scatter_kernel<<<(nq + 255) / 256, 256, 0, st>>>(w.ids, w.wts, w.counts, w.cursor, T, w.pair_token,
                                                            w.pair_w, w.offsets, w.gu_prefix, w.dn_prefix);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gp = GemmParams{};
  gp.experts = L.experts;
  gp.tscale = L.tscale;
  gp.offsets = w.offsets;
  gp.pair_token = w.pair_token;
  gp.pair_w = w.pair_w;
  gp.xexp = w.xexp;
  gp.h = w.h;
  gp.yacc = w.yacc;
  gp.err = err;
  gp.prefix = w.gu_prefix;
  gp.bsrc = reinterpret_cast<const uint16_t*>(w.xh16);
  prefill_gemm_kernel<0><<<sm_count, G_THREADS, G_SMEM, st>>>(gp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gp.prefix = w.dn_prefix;
  gp.bsrc = w.h;
  prefill_gemm_kernel<1><<<sm_count, G_THREADS, G_SMEM, st>>>(gp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t n4 = (size_t)T * H / 4;
  prefill_finalize_kernel<<<(unsigned)((n4 + 255) / 256), 256, 0, st>>>(reinterpret_cast<const float4*>(w.yacc),
                                                                       static_cast<uint2*>(y), n4);
  return cudaGetLastError();
}

}  // namespace flint
