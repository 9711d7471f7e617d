// Persistent decode kernel for NVFP4 sublayer stacks (batch 1..8), sm_103a.
//
// "Day-0 Support for Flint on vLLM", section "Optimizations": for up to 8
// requests the low-latency path fuses routing and expert combination into the
// neighbouring GEMV kernels, and every kernel loads its weights while its
// predecessor still runs.  This kernel takes that to its end point on one
// GPU: ONE cooperative launch runs up to 64 chained sublayers, one CTA per SM.
// Each sublayer has three grid-wide data dependencies (all logits -> routing,
// all h -> down projection, all of y -> the next RMSNorm and router), and each
// is crossed through tagged data words instead of a kernel boundary: every
// 64-bit word holds 32 data bits and the number of the sublayer that wrote
// it, so a reader polls the words it needs until all carry the expected tag
// (one L2 round trip after the last writer, no fence, no counter).
//
// Work of sublayer l in CTA c of P:
//   route     every CTA computes the sigmoid top-6 of every token from the
//             tagged logits (the same decision everywhere, no extra hop);
//   gate/up   items (slot, 16-row tile), item i = slot * 64 + tile, go to the
//             CTA with i mod P == c; slot 0 is the shared expert, known before
//             the routing, so its tiles are in shared memory before the logits
//             are; 8 compute warps take one 256-column K-slice each, 2
//             epilogue warps reduce them and write h = bf16(silu(g) * u);
//   down      CTA r < 128 owns output rows 16r..16r+15 of every slot; its
//             tiles are requested together with the gate/up tiles, and it
//             combines the slots in a fixed order once all h it needs carry
//             tag l + 1;
//   router    every CTA reads all of y, forms x_hat of sublayer l + 1 (exact
//             RMSNorm) and the logits of its experts c and c + P; the router
//             rows and the next shared-expert tiles were prefetched during
//             sublayer l.
// A producer warp issues every weight copy (TMA bulk copies into shared-memory
// rings, completion on mbarriers) in the order the consumers use them.
//
// Arithmetic per step is that of the three-kernel path in decode.cu (same
// dequantisation, same f16 exponents, same fixed-order reductions), so both
// give the same results.
#include <cooperative_groups.h>

#include "decode_common.cuh"
#include "flint_internal.h"

namespace flint {

namespace cg = cooperative_groups;

namespace {

constexpr int FZ_CW = 8;                  // compute warps
constexpr int FZ_PW = 8;                  // producer warp
constexpr int FZ_EW0 = 9;                 // first of the two epilogue warps
constexpr int FZ_THREADS = 32 * 11;       // 352
constexpr int FZ_CT = 32 * FZ_CW;         // 256 compute threads
constexpr int FZ_RED = 4;                 // partial-sum ring between compute and epilogue warps
constexpr int FZ_NG = 4;                  // down slot groups (two K-half warps each)
constexpr int FZ_DN_ST = 12;              // down tile ring (a multiple of FZ_NG)
constexpr int FZ_ROW_BYTES = H * 2;       // one bf16 router row
constexpr int FZ_EPC = 2;                 // router experts per CTA at most (c and c + P)
constexpr int FZ_SMEM_LIMIT = 232448;     // 227 KB of dynamic shared memory per CTA
static_assert(FZ_DN_ST % FZ_NG == 0, "each down stage must belong to one slot group");

template <int NB>
struct FzCfg {
  static constexpr int GU_ST = NB <= 4 ? 5 : 4;
  static constexpr int PAIRS = (1 + TOPK) * NB;               // (slot, token) pairs: shared + 6 per token
  static constexpr int HS_BYTES = PAIRS * HS_STRIDE * 2;      // staged h of the down phase
  static constexpr int XF_LANES = 4 * NB;                     // mma lanes that carry tokens
  static constexpr int XF_BYTES = GU_SLICES * XF_LANES * 32 * 4;
  static constexpr int UNI = ((HS_BYTES > XF_BYTES ? HS_BYTES : XF_BYTES) + 127) / 128 * 128;
  static constexpr int R_BYTES = (int)((sizeof(Routing) + 15) / 16 * 16);
  static constexpr int O_GU = 0;
  static constexpr int O_DN = O_GU + GU_ST * F4_GU_TILE;
  static constexpr int O_RED = O_DN + FZ_DN_ST * F4_DN_TILE;
  static constexpr int O_DRED = O_RED + FZ_RED * 8 * 128 * 4;
  static constexpr int O_ROWS = O_DRED + 8 * 128 * 4;
  static constexpr int O_UNI = O_ROWS + FZ_EPC * FZ_ROW_BYTES;
  static constexpr int O_R = O_UNI + UNI;
  static constexpr int O_MISC = O_R + 2 * R_BYTES;
};

static_assert(FzCfg<BMAX>::PAIRS <= 64, "pair tables hold 64 entries");

struct FzMisc {
  uint64_t gu_full[5], gu_empty[5];
  uint64_t dn_full[FZ_DN_ST], dn_empty[FZ_DN_ST];
  uint64_t rfull[FZ_RED], rempty[FZ_RED];
  uint64_t rbar;            // router rows of the next sublayer landed
  uint64_t route_ready[2];  // routing of sublayer l published (index l & 1)
  CSum redn[8][16];         // per-warp compensated partials (norm, logits)
  float rscale[BMAX];
  unsigned xmax[BMAX];      // max |x_hat| bits per token
  unsigned hmax[BMAX];      // max |h| bits per token (down phase)
  int xexp[2][BMAX];        // f16 exponent of x_hat per token, by sublayer parity
  int npairs;
  int abort;                // this CTA gives up (a wait ran out, or another CTA gave up)
  uint8_t pidx[MAX_SLOTS][BMAX];
  uint8_t ptok[64];
  uint8_t pslot[64];
};

template <int NB>
__host__ __device__ constexpr int fz_smem_bytes() {
  return FzCfg<NB>::O_MISC + (int)sizeof(FzMisc);
}

// ------------------------------------------------------------------ tagged words

__device__ __forceinline__ uint64_t tagw(uint32_t data, uint32_t tag) { return ((uint64_t)tag << 32) | data; }

__device__ __forceinline__ void st_tagged(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// Two consecutive tagged words; true if both carry `tag`.  The words are read
// from L2 (volatile loads bypass L1); each 64-bit word is read atomically.
__device__ __forceinline__ bool ld_tagged2(const uint64_t* p, uint32_t tag, uint32_t& d0, uint32_t& d1) {
  uint64_t a, b;
  asm volatile("ld.volatile.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
  d0 = (uint32_t)a;
  d1 = (uint32_t)b;
  return (uint32_t)(a >> 32) == tag && (uint32_t)(b >> 32) == tag;
}
__device__ __forceinline__ unsigned ld_volatile_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.volatile.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_volatile_u32(unsigned* p, unsigned v) {
  asm volatile("st.volatile.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Barrier of the 256 compute threads that also ORs a flag across them, so that
// every compute warp takes the same decision after it.
__device__ __forceinline__ bool cbar_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, 256, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// ------------------------------------------------------------------ parameters

struct FzLayer {
  const __nv_bfloat16* router_w;  // [E][H]
  const uint8_t* experts;         // packed NVFP4 blob
  const float* tscale;            // [NE][2]
  const __nv_bfloat16* norm_w;    // [H] or null
};

struct FusedParams {
  const __nv_bfloat16* x;  // [B][H] input of the first sublayer
  __nv_bfloat16* y;        // [B][H] output of the last sublayer
  __nv_bfloat16* ys;       // [n_layers][B][H] every sublayer's output, or null
  int32_t* ids;            // [n_layers][B][6] or null
  float* w;                // [n_layers][B][6] or null
  uint64_t* logits_t;      // tagged [2][BMAX][E]
  uint64_t* y_t;           // tagged [2][BMAX][H / 2]
  uint64_t* h_t;           // tagged [MAX_SLOTS][BMAX][I / 2]
  unsigned* gabort;        // set when any CTA gives up
  unsigned* err;           // device error word
  long long poll_limit;    // cycles a wait on other CTAs' data may take
  float eps;
  int n_layers;
  FzLayer layers[FUSED_MAX_LAYERS];
};

// A wait on other CTAs' data: gives up after poll_limit cycles, or at once when
// another CTA has given up.  Returns 0 (keep waiting), 1 (abort seen), 2 (ran out).
struct Waiter {
  long long t0 = 0;
  bool armed = false;
  __device__ __forceinline__ int check(const FusedParams& p) {
    if (ld_volatile_u32(p.gabort) != 0u) return 1;
    const long long now = clock64();
    if (!armed) {
      armed = true;
      t0 = now;
      return 0;
    }
    return now - t0 > p.poll_limit ? 2 : 0;
  }
};

__device__ __forceinline__ void fz_give_up(const FusedParams& p, FzMisc& M, int why) {
  if (why == 2) {
    atomicOr(p.err, ERR_POLL);
    st_volatile_u32(p.gabort, 1u);
  }
  *reinterpret_cast<volatile int*>(&M.abort) = 1;
}

__device__ __forceinline__ bool cta_aborted(FzMisc& M) { return *reinterpret_cast<volatile int*>(&M.abort) != 0; }

// Bounded mbarrier wait of one thread that also gives up when this CTA aborts.
__device__ __forceinline__ bool wait_abort1(uint64_t* bar, uint32_t parity, FzMisc& M, unsigned* err, unsigned bit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (cta_aborted(M)) return false;
    if (clock64() - t0 > WAIT_LIMIT_CYCLES) {
      atomicOr(err, bit);
      *reinterpret_cast<volatile int*>(&M.abort) = 1;
      return false;
    }
  }
}
// The same, by every lane of a full warp; the result is the same for all lanes.
__device__ __forceinline__ bool wait_abort(uint64_t* bar, uint32_t parity, FzMisc& M, unsigned* err, unsigned bit) {
  const bool ok = wait_abort1(bar, parity, M, err, bit);
  return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------------ the kernel

template <int NB>
__global__ void __launch_bounds__(FZ_THREADS, 1) decode_fused_kernel(const __grid_constant__ FusedParams p) {
  using C = FzCfg<NB>;
  static_assert(fz_smem_bytes<NB>() <= FZ_SMEM_LIMIT, "shared memory layout too large");
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* gu_st = smem + C::O_GU;
  uint8_t* dn_st = smem + C::O_DN;
  float* red = reinterpret_cast<float*>(smem + C::O_RED);    // [FZ_RED][8 warps][128]
  float* dred = reinterpret_cast<float*>(smem + C::O_DRED);  // [8 warps][128]
  uint8_t* rows = smem + C::O_ROWS;                          // [FZ_EPC][H] bf16
  uint32_t* xf = reinterpret_cast<uint32_t*>(smem + C::O_UNI);  // x_hat B fragments
  uint16_t* hs = reinterpret_cast<uint16_t*>(smem + C::O_UNI);  // staged h (aliases xf)
  FzMisc& M = *reinterpret_cast<FzMisc*>(smem + C::O_MISC);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = gridDim.x, c = blockIdx.x;
  const int NL = p.n_layers;
  const bool dn_cta = c < DN_TILES;
  const int n_rexp = (c + P < E) ? 2 : 1;
  int i_first = c;  // first routed gate/up item of this CTA (items 0..63 are the shared expert's)
  while (i_first < GU_TILES) i_first += P;
  auto routing = [&](int l) -> Routing& { return *reinterpret_cast<Routing*>(smem + C::O_R + (l & 1) * C::R_BYTES); };

  if (tid == 0) {
    for (int s = 0; s < C::GU_ST; ++s) {
      mbar_init(&M.gu_full[s], 1);
      mbar_init(&M.gu_empty[s], FZ_CW);
    }
    for (int s = 0; s < FZ_DN_ST; ++s) {
      mbar_init(&M.dn_full[s], 1);
      mbar_init(&M.dn_empty[s], 2);
    }
    for (int b = 0; b < FZ_RED; ++b) {
      mbar_init(&M.rfull[b], FZ_CW);
      mbar_init(&M.rempty[b], 2);
    }
    mbar_init(&M.rbar, 1);
    mbar_init(&M.route_ready[0], 1);
    mbar_init(&M.route_ready[1], 1);
    M.abort = 0;
    fence_mbar_init();
  }
  if (tid < BMAX) M.xmax[tid] = 0u;
  __syncthreads();

  // Producer state (lane 0 of the producer warp): copies issued per ring.
  const uint64_t pol = l2_evict_first();
  uint32_t gq = 0, dq = 0, rq = 0;
  auto issue_rows = [&](int k) {
    mbar_arrive_expect_tx(&M.rbar, (uint32_t)(n_rexp * FZ_ROW_BYTES));
    for (int j = 0; j < n_rexp; ++j)
      bulk_g2s(rows + j * FZ_ROW_BYTES, p.layers[k].router_w + (size_t)(c + j * P) * H, FZ_ROW_BYTES, &M.rbar, pol);
    ++rq;
  };
  auto gu_issue = [&](const uint8_t* src) -> bool {
    const int s = gq % C::GU_ST;
    if (gq >= (uint32_t)C::GU_ST && !wait_abort1(&M.gu_empty[s], ((gq / C::GU_ST) - 1) & 1, M, p.err, ERR_WAIT_EMPTY))
      return false;
    mbar_arrive_expect_tx(&M.gu_full[s], F4_GU_TILE);
    bulk_g2s(gu_st + (size_t)s * F4_GU_TILE, src, F4_GU_TILE, &M.gu_full[s], pol);
    ++gq;
    return true;
  };
  // 1 = issued, 0 = the stage is still in use (non-blocking call), -1 = gave up.
  auto dn_issue = [&](const uint8_t* src, bool blocking) -> int {
    const int s = dq % FZ_DN_ST;
    if (dq >= (uint32_t)FZ_DN_ST) {
      const uint32_t par = ((dq / FZ_DN_ST) - 1) & 1;
      if (!blocking) {
        if (!mbar_test(&M.dn_empty[s], par)) return 0;
      } else if (!wait_abort1(&M.dn_empty[s], par, M, p.err, ERR_WAIT_EMPTY)) {
        return -1;
      }
    }
    mbar_arrive_expect_tx(&M.dn_full[s], F4_DN_TILE);
    bulk_g2s(dn_st + (size_t)s * F4_DN_TILE, src, F4_DN_TILE, &M.dn_full[s], pol);
    ++dq;
    return 1;
  };
  auto dn_src = [&](const FzLayer& Ly, int e) {
    return Ly.experts + (size_t)e * F4_EXPERT + F4_GU_BYTES + (size_t)c * F4_DN_TILE;
  };
  if (tid == FZ_PW * 32) {
    // Constants of the first sublayer: its router rows, the shared expert's
    // gate/up tiles of this CTA and (down CTAs) the shared expert's down tile.
    issue_rows(0);
    for (int t = c; t < GU_TILES; t += P)
      gu_issue(p.layers[0].experts + (size_t)E * F4_EXPERT + (size_t)t * F4_GU_TILE);
    if (dn_cta) dn_issue(dn_src(p.layers[0], E), true);
  }

  // Clear every tagged word of this call (tag 0 is never awaited) and meet.
  {
    const size_t n16 = ((size_t)2 * BMAX * E + (size_t)2 * BMAX * (H / 2) + (size_t)MAX_SLOTS * BMAX * (I / 2)) / 2;
    uint4* z = reinterpret_cast<uint4*>(p.logits_t);
    for (size_t i = (size_t)c * FZ_THREADS + tid; i < n16; i += (size_t)P * FZ_THREADS) z[i] = make_uint4(0u, 0u, 0u, 0u);
    if (c == 0 && tid == 0) *p.gabort = 0u;
  }
  cg::this_grid().sync();

  // ================================================================ producer
  if (warp == FZ_PW) {
    if (lane != 0) return;
    bool ok = true;
    for (int l = 0; l < NL && ok; ++l) {
      if (!wait_abort1(&M.route_ready[l & 1], (l >> 1) & 1, M, p.err, ERR_WAIT_FULL)) break;
      const Routing& R = routing(l);
      const FzLayer& Ly = p.layers[l];
      const int S = R.n_slots;
      if (l + 1 < NL) issue_rows(l + 1);
      int u = 1;  // slot 0's down tile was requested a sublayer ahead
      if (dn_cta)
        while (u < S && dn_issue(dn_src(Ly, R.slot_expert[u]), false) == 1) ++u;
      for (int i = i_first; i < S * GU_TILES && ok; i += P)
        ok = gu_issue(Ly.experts + (size_t)R.slot_expert[i / GU_TILES] * F4_EXPERT +
                      (size_t)(i % GU_TILES) * F4_GU_TILE);
      if (l + 1 < NL)
        for (int t = c; t < GU_TILES && ok; t += P)
          ok = gu_issue(p.layers[l + 1].experts + (size_t)E * F4_EXPERT + (size_t)t * F4_GU_TILE);
      if (dn_cta) {
        for (; u < S && ok; ++u) ok = dn_issue(dn_src(Ly, R.slot_expert[u]), true) == 1;
        if (ok && l + 1 < NL) ok = dn_issue(dn_src(p.layers[l + 1], E), true) == 1;
      }
    }
    // Leave no copy in flight: wait for the last fill of every stage.
    for (uint32_t n = gq > (uint32_t)C::GU_ST ? gq - C::GU_ST : 0; n < gq; ++n)
      if (!mbar_wait(&M.gu_full[n % C::GU_ST], (n / C::GU_ST) & 1)) atomicOr(p.err, ERR_DRAIN);
    for (uint32_t n = dq > (uint32_t)FZ_DN_ST ? dq - FZ_DN_ST : 0; n < dq; ++n)
      if (!mbar_wait(&M.dn_full[n % FZ_DN_ST], (n / FZ_DN_ST) & 1)) atomicOr(p.err, ERR_DRAIN);
    if (rq > 0 && !mbar_wait(&M.rbar, (rq - 1) & 1)) atomicOr(p.err, ERR_DRAIN);
    return;
  }

  // ================================================================ epilogue warps
  if (warp >= FZ_EW0) {
    const int et = tid - FZ_EW0 * 32;
    const int tk = et >> 3, row = et & 7;
    const int og = red_off(row, tk), ou = red_off(row + 8, tk);
    uint32_t n = 0;
    // One gate/up item: fixed-order sum of the 8 slice partials, SiLU*up, and
    // the tagged store of h (two bf16 values per word) for the tokens that
    // use the slot.
    auto epi = [&](int l, int slot, int tile, int e, uint32_t mask) -> bool {
      const int b = n % FZ_RED;
      if (!wait_abort(&M.rfull[b], (n / FZ_RED) & 1, M, p.err, ERR_WAIT_FULL)) return false;
      const float* rb = red + b * 1024;
      float gsum = 0.f, usum = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        gsum += rb[w * 128 + og];
        usum += rb[w * 128 + ou];
      }
      const bool act = tk < NB && ((mask >> tk) & 1u);
      uint32_t hb = 0u;
      if (act) {
        const float f = __fmul_rn(exp2i(-M.xexp[l & 1][tk]), __ldg(p.layers[l].tscale + 2 * e));
        const float gate = __fmul_rn(gsum, f);
        const float up = __fmul_rn(usum, f);
        const float silu = __fdiv_rn(gate, __fadd_rn(1.0f, expf(-gate)));
        hb = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(silu, up)));
      }
      const uint32_t other = __shfl_xor_sync(0xffffffffu, hb, 1);
      if (act && (row & 1) == 0)
        st_tagged(p.h_t + ((size_t)(slot * BMAX + tk) * (I / 2) + ((tile * 8 + row) >> 1)),
                  tagw(hb | (other << 16), (uint32_t)(l + 1)));
      __syncwarp();
      if (lane == 0) mbar_arrive(&M.rempty[b]);
      ++n;
      return true;
    };
    for (int l = 0; l < NL; ++l) {
      bool ok = true;
      for (int t = c; t < GU_TILES && ok; t += P) ok = epi(l, 0, t, E, 0xFFu);
      if (!ok) return;
      if (!wait_abort(&M.route_ready[l & 1], (l >> 1) & 1, M, p.err, ERR_WAIT_FULL)) return;
      const Routing& R = routing(l);
      for (int i = i_first; i < R.n_slots * GU_TILES && ok; i += P) {
        const int slot = i / GU_TILES;
        ok = epi(l, slot, i % GU_TILES, R.slot_expert[slot], R.slot_mask[slot]);
      }
      if (!ok) return;
    }
    return;
  }

  // ================================================================ compute warps (tid < 256)
  bool dead = false;
  uint32_t gn = 0;      // gate/up items consumed (same sequence as the producer's)
  uint32_t dn_seq = 0;  // down tiles consumed
  const int k0 = tid * 8;

  // One gate/up item: this warp's K-slice times the x_hat fragments, partial
  // sums handed to the epilogue warps.
  auto gu_item = [&](const uint32_t (&bfr)[16][2]) -> bool {
    const int s = gn % C::GU_ST;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (!wait_abort(&M.gu_full[s], (gn / C::GU_ST) & 1, M, p.err, ERR_WAIT_FULL)) return false;
    nvfp4_slice_mma(gu_st + (size_t)s * F4_GU_TILE + warp * F4_SLICE, lane, bfr, acc);
    __syncwarp();
    if (lane == 0) mbar_arrive(&M.gu_empty[s]);
    const int b = gn % FZ_RED;
    if (gn >= (uint32_t)FZ_RED && !wait_abort(&M.rempty[b], ((gn / FZ_RED) - 1) & 1, M, p.err, ERR_WAIT_EMPTY))
      return false;
    float* rb = red + b * 1024;
#pragma unroll
    for (int j = 0; j < 4; ++j) rb[warp * 128 + j * 32 + lane] = acc[j];
    __syncwarp();
    if (lane == 0) mbar_arrive(&M.rfull[b]);
    ++gn;
    return true;
  };

  // RMSNorm + x_hat + router logits of sublayer k (k = 0: plain input x;
  // otherwise the tagged y of sublayer k - 1).  Writes the x_hat fragments and
  // exponents for the gate/up items of sublayer k and the tagged logits of
  // this CTA's experts.  Same arithmetic as router_kernel in decode.cu.
  auto router_phase = [&](int k) -> bool {
    constexpr int NP = (NB + 1) / 2;
    constexpr int VP = Pow2Ceil<NB * FZ_EPC>::value;
    constexpr int SH = 5 - Log2<VP>::value;
    const FzLayer& Lk = p.layers[k];
    const bool has_norm = Lk.norm_w != nullptr;
    float nw[8];
    if (has_norm) bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(Lk.norm_w + k0)), nw);
    float xv[2 * NP][8];
#pragma unroll
    for (int t = 0; t < 2 * NP; ++t)
#pragma unroll
      for (int i = 0; i < 8; ++i) xv[t][i] = 0.f;
    if (k == 0) {
#pragma unroll
      for (int t = 0; t < NB; ++t) bf16x8_to_f32(__ldcg(reinterpret_cast<const uint4*>(p.x + (size_t)t * H + k0)), xv[t]);
    } else if (!dead) {
      const uint32_t tag = (uint32_t)k;
      const uint64_t* base = p.y_t + (size_t)((k - 1) & 1) * BMAX * (H / 2) + tid * 4;
      uint32_t pend = (1u << (2 * NB)) - 1u;
      Waiter wt;
      for (;;) {
#pragma unroll
        for (int t = 0; t < NB; ++t)
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2)
            if ((pend >> (2 * t + h2)) & 1u) {
              uint32_t d0, d1;
              if (ld_tagged2(base + (size_t)t * (H / 2) + 2 * h2, tag, d0, d1)) {
                xv[t][4 * h2 + 0] = __uint_as_float(d0 << 16);
                xv[t][4 * h2 + 1] = __uint_as_float(d0 & 0xFFFF0000u);
                xv[t][4 * h2 + 2] = __uint_as_float(d1 << 16);
                xv[t][4 * h2 + 3] = __uint_as_float(d1 & 0xFFFF0000u);
                pend &= ~(1u << (2 * t + h2));
              }
            }
        if (pend == 0u) break;
        const int why = wt.check(p);
        if (why) {
          fz_give_up(p, M, why);
          dead = true;
          break;
        }
      }
    }
    if (has_norm) {
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
      if ((lane & ((1 << SHN) - 1)) == 0) M.redn[warp][lane >> SHN] = tot;
      if (cbar_or(dead || cta_aborted(M))) return false;
      if (tid < NB) {
        CSum a = M.redn[0][tid];
#pragma unroll
        for (int w = 1; w < 8; ++w) cs_merge(a, M.redn[w][tid]);
        const float ms = __fmul_rn(cs_value(a), 1.0f / (float)H);
        M.rscale[tid] = __frcp_rn(__fsqrt_rn(__fadd_rn(ms, p.eps)));
      }
      if (cbar_or(dead || cta_aborted(M))) return false;
#pragma unroll
      for (int t = 0; t < NB; ++t) {
        const float r = M.rscale[t];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          xv[t][i] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(__fmul_rn(xv[t][i], r), nw[i])));
      }
    }
    // x_hat in f16 with a per-token power-of-two exponent, in B-fragment order.
#pragma unroll
    for (int t = 0; t < NB; ++t) {
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(xv[t][i]));
      const unsigned wm = redux_max(__float_as_uint(m));
      if (lane == 0) atomicMax(&M.xmax[t], wm);
    }
    if (cbar_or(dead || cta_aborted(M))) return false;
    {
      const int ws = k0 >> 8, kb = (k0 & 255) >> 4, rr = (k0 >> 3) & 1;
#pragma unroll
      for (int t = 0; t < NB; ++t) {
        const int ex = f16_range_exp(__uint_as_float(M.xmax[t]));
        const float sc = exp2i(ex);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __half2 hv = __floats2half2_rn(__fmul_rn(xv[t][2 * i], sc), __fmul_rn(xv[t][2 * i + 1], sc));
          xf[((ws * C::XF_LANES + 4 * t + i) * 16 + kb) * 2 + rr] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        if (tid == 0) M.xexp[k & 1][t] = ex;
      }
    }
    // Router logits of experts c and c + P: error-free accumulation (TwoSum).
    if (!wait_abort(&M.rbar, (uint32_t)k & 1, M, p.err, ERR_WAIT_FULL)) dead = true;
    float wf[FZ_EPC][8];
#pragma unroll
    for (int j = 0; j < FZ_EPC; ++j) {
      if (j < n_rexp && !dead) {
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(rows + j * FZ_ROW_BYTES + k0 * 2), wf[j]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) wf[j][i] = 0.f;
      }
    }
    CSum2 d2[FZ_EPC][NP];
#pragma unroll
    for (int j = 0; j < FZ_EPC; ++j)
#pragma unroll
      for (int q = 0; q < NP; ++q) d2[j][q] = CSum2{0ull, 0ull};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
      for (int j = 0; j < FZ_EPC; ++j) {
        const uint64_t w2 = f2pack(wf[j][i], wf[j][i]);
#pragma unroll
        for (int q = 0; q < NP; ++q) cs2_add(d2[j][q], f2mul(f2pack(xv[2 * q][i], xv[2 * q + 1][i]), w2));
      }
    }
    {
      CSum d[VP];
#pragma unroll
      for (int v = 0; v < VP; ++v) d[v] = CSum{0.f, 0.f};
#pragma unroll
      for (int j = 0; j < FZ_EPC; ++j)
#pragma unroll
        for (int q = 0; q < NP; ++q) {
          CSum lo, hi;
          cs2_split(d2[j][q], lo, hi);
          d[j * NB + 2 * q] = lo;
          if (2 * q + 1 < NB) d[j * NB + 2 * q + 1] = hi;
        }
      const CSum tot = cs_reduce_scatter<VP>(d, lane);
      if ((lane & ((1 << SH) - 1)) == 0) M.redn[warp][lane >> SH] = tot;
    }
    if (cbar_or(dead || cta_aborted(M))) return false;
    if (tid < NB * FZ_EPC && tid / NB < n_rexp) {
      CSum a = M.redn[0][tid];
#pragma unroll
      for (int w = 1; w < 8; ++w) cs_merge(a, M.redn[w][tid]);
      const int e = c + (tid / NB) * P, t = tid % NB;
      const uint32_t bits = __bfloat16_as_ushort(__float2bfloat16_rn(cs_value(a)));
      st_tagged(p.logits_t + ((size_t)((k & 1) * BMAX + t) * E + e), tagw(bits, (uint32_t)(k + 1)));
    }
    return !cbar_or(dead || cta_aborted(M));
  };

  auto load_bfr = [&](uint32_t (&bfr)[16][2]) {
    if (lane < C::XF_LANES) {
      const uint4* src = reinterpret_cast<const uint4*>(xf + (size_t)(warp * C::XF_LANES + lane) * 32);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint4 v = src[q];
        bfr[2 * q][0] = v.x;
        bfr[2 * q][1] = v.y;
        bfr[2 * q + 1][0] = v.z;
        bfr[2 * q + 1][1] = v.w;
      }
    } else {
#pragma unroll
      for (int kb = 0; kb < 16; ++kb) bfr[kb][0] = bfr[kb][1] = 0u;
    }
  };

  if (!router_phase(0)) return;

  for (int l = 0; l < NL; ++l) {
    const FzLayer& Ly = p.layers[l];
    const uint32_t tag = (uint32_t)(l + 1);
    Routing& R = routing(l);

    // A, B. the shared expert's items (requested a sublayer ahead), against the
    // x_hat fragments of sublayer l (lanes 4t..4t+3 carry token t).
    {
      uint32_t bfr[16][2];
      load_bfr(bfr);
      for (int t = c; t < GU_TILES && !dead; t += P) dead = !gu_item(bfr);
    }

    // C. routing: every CTA takes the same decision from the tagged logits.
    zero_routing(R, tid, FZ_CT);
    if (tid < NB) {
      M.hmax[tid] = 0u;
      M.xmax[tid] = 0u;
    }
    if (cbar_or(dead || cta_aborted(M))) return;
    if (warp < NB) {
      const uint64_t* src = p.logits_t + ((size_t)((l & 1) * BMAX + warp) * E + lane * 8);
      uint32_t d[8];
      Waiter wt;
      bool got = false;
      for (;;) {
        bool ok = true;
#pragma unroll
        for (int q = 0; q < 4; ++q) ok = ld_tagged2(src + 2 * q, tag, d[2 * q], d[2 * q + 1]) && ok;
        if (__all_sync(0xffffffffu, ok)) {
          got = true;
          break;
        }
        const int why = wt.check(p);
        const int any = __reduce_max_sync(0xffffffffu, (unsigned)why);
        if (any) {
          if (lane == 0) fz_give_up(p, M, any);
          break;
        }
      }
      if (got) {
        const uint4 raw = make_uint4((d[0] & 0xFFFFu) | (d[1] << 16), (d[2] & 0xFFFFu) | (d[3] << 16),
                                     (d[4] & 0xFFFFu) | (d[5] << 16), (d[6] & 0xFFFFu) | (d[7] << 16));
        warp_topk(raw, lane, R.ids[warp], R.w[warp], R.umask);
      } else {
        dead = true;
      }
    }
    if (cbar_or(dead || cta_aborted(M))) return;
    if (warp == 0) {
      warp_slot_table(R, NB, lane);
      // (slot, token) pairs of the down phase, slot-major.
      const int S = R.n_slots;
      int base = 0;
      for (int c0 = 0; c0 < S; c0 += 32) {
        const int u = c0 + lane;
        const uint32_t m = u < S ? R.slot_mask[u] : 0u;
        const int cnt = __popc(m);
        int incl = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += v;
        }
        int pi = base + incl - cnt;
        if (u < S) {
#pragma unroll
          for (int tk = 0; tk < BMAX; ++tk) {
            if ((m >> tk) & 1u) {
              M.pidx[u][tk] = (uint8_t)pi;
              M.ptok[pi] = (uint8_t)tk;
              M.pslot[pi] = (uint8_t)u;
              ++pi;
            }
          }
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) {
        // Every token adds one pair per selected expert and one for the shared
        // expert, so base <= C::PAIRS; a larger count would overrun the staging
        // area, so it ends the call instead.
        if (base > C::PAIRS) {
          atomicOr(p.err, ERR_LAYOUT);
          fz_give_up(p, M, 1);
          st_volatile_u32(p.gabort, 1u);
        }
        M.npairs = base;
        mbar_arrive(&M.route_ready[l & 1]);
      }
    }
    if (cbar_or(dead || cta_aborted(M))) return;
    if (c == 0 && tid < NB * TOPK) {
      if (p.ids) p.ids[(size_t)l * NB * TOPK + tid] = R.ids[tid / TOPK][tid % TOPK];
      if (p.w) p.w[(size_t)l * NB * TOPK + tid] = R.w[tid / TOPK][tid % TOPK];
    }
    const int S = R.n_slots;

    // D. the routed experts' gate/up items of this CTA (fragments reloaded: they
    // are not kept in registers across the routing).
    {
      uint32_t bfr[16][2];
      load_bfr(bfr);
      for (int i = i_first; i < S * GU_TILES && !dead; i += P) dead = !gu_item(bfr);
    }

    // E. down projection + weighted combine for rows 16c..16c+15.
    if (dn_cta) {
      constexpr int NJ = (C::PAIRS * 128 + FZ_CT - 1) / FZ_CT;
      static_assert(NJ <= 32, "pending chunks must fit a 32-bit mask");
      const int nch = M.npairs * 128;
      uint32_t pend = 0u;
#pragma unroll
      for (int j = 0; j < NJ; ++j)
        if (tid + j * FZ_CT < nch) pend |= 1u << j;
      unsigned tmax[NB];
#pragma unroll
      for (int q = 0; q < NB; ++q) tmax[q] = 0u;
      Waiter wt;
      while (pend != 0u && !dead) {
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          if ((pend >> j) & 1u) {
            const int kk = tid + j * FZ_CT, pr = kk >> 7, ch = kk & 127;
            const int tok = M.ptok[pr], slot = M.pslot[pr];
            uint32_t d0, d1;
            if (ld_tagged2(p.h_t + ((size_t)(slot * BMAX + tok) * (I / 2) + ch * 2), tag, d0, d1)) {
              *reinterpret_cast<uint2*>(hs + (size_t)pr * HS_STRIDE + ch * 4) = make_uint2(d0, d1);
              const unsigned a0 = (d0 & 0x7FFFu) << 16, a1 = d0 & 0x7FFF0000u;
              const unsigned a2 = (d1 & 0x7FFFu) << 16, a3 = d1 & 0x7FFF0000u;
              const unsigned am = max(max(a0, a1), max(a2, a3));
#pragma unroll
              for (int q = 0; q < NB; ++q)
                if (q == tok) tmax[q] = max(tmax[q], am);
              pend &= ~(1u << j);
            }
          }
        }
        if (pend == 0u) break;
        const int why = wt.check(p);
        if (why) {
          fz_give_up(p, M, why);
          dead = true;
        }
      }
#pragma unroll
      for (int q = 0; q < NB; ++q) {
        const unsigned m = redux_max(tmax[q]);
        if (lane == 0 && m != 0u) atomicMax(&M.hmax[q], m);
      }
      if (cbar_or(dead || cta_aborted(M))) return;
      // bf16 h -> f16 h * 2^hexp[token], in place (each thread its own chunks).
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const int kk = tid + j * FZ_CT;
        if (kk < nch) {
          const int pr = kk >> 7, ch = kk & 127;
          uint2* ptr = reinterpret_cast<uint2*>(hs + (size_t)pr * HS_STRIDE + ch * 4);
          const uint2 v = *ptr;
          const float sc = exp2i(f16_range_exp(__uint_as_float(M.hmax[M.ptok[pr]])));
          const __half2 h0 = __floats2half2_rn(__fmul_rn(__uint_as_float(v.x << 16), sc),
                                               __fmul_rn(__uint_as_float(v.x & 0xFFFF0000u), sc));
          const __half2 h1 = __floats2half2_rn(__fmul_rn(__uint_as_float(v.y << 16), sc),
                                               __fmul_rn(__uint_as_float(v.y & 0xFFFF0000u), sc));
          *ptr = make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
        }
      }
      if (cbar_or(dead || cta_aborted(M))) return;

      const int g = lane >> 2, t4 = lane & 3;
      const int kh = warp & 1, grp = warp >> 1;
      const int cgrp = (grp - (int)(dn_seq % FZ_NG) + FZ_NG) % FZ_NG;  // the slots u = cgrp mod 4
      float tot[4] = {0.f, 0.f, 0.f, 0.f};
      for (int u = cgrp; u < S; u += FZ_NG) {
        const uint32_t q = dn_seq + u;
        const int s = q % FZ_DN_ST;
        if (!wait_abort(&M.dn_full[s], (q / FZ_DN_ST) & 1, M, p.err, ERR_WAIT_FULL)) {
          dead = true;
          break;
        }
        uint32_t hb[16][2];
        const uint32_t mask = R.slot_mask[u];
        if (g < NB && ((mask >> g) & 1u)) {
          const uint32_t* hr = reinterpret_cast<const uint32_t*>(hs + (size_t)M.pidx[u][g] * HS_STRIDE + kh * 256);
#pragma unroll
          for (int kb = 0; kb < 16; ++kb) {
            hb[kb][0] = hr[kb * 8 + t4];
            hb[kb][1] = hr[kb * 8 + t4 + 4];
          }
        } else {
#pragma unroll
          for (int kb = 0; kb < 16; ++kb) hb[kb][0] = hb[kb][1] = 0u;
        }
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        nvfp4_slice_mma(dn_st + (size_t)s * F4_DN_TILE + kh * F4_SLICE, lane, hb, acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(&M.dn_empty[s]);
        const float ts = __ldg(Ly.tscale + 2 * R.slot_expert[u] + 1);
        const float w0 = __fmul_rn(R.slot_w[u][2 * t4], ts);
        const float w1 = __fmul_rn(R.slot_w[u][2 * t4 + 1], ts);
        tot[0] = fmaf(w0, acc[0], tot[0]);
        tot[1] = fmaf(w1, acc[1], tot[1]);
        tot[2] = fmaf(w0, acc[2], tot[2]);
        tot[3] = fmaf(w1, acc[3], tot[3]);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) dred[(2 * cgrp + kh) * 128 + j * 32 + lane] = tot[j];
      if (cbar_or(dead || cta_aborted(M))) return;
      if (tid < 128) {
        // thread = (token tk, row): the 8 warps' partials in a fixed order
        const int row = tid & 15, tk = tid >> 4;
        const int o = red_off(row, tk);
        float cc = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) cc += dred[w * 128 + o];
        uint32_t yb = 0u;
        if (tk < NB) {
          const float sc = exp2i(-f16_range_exp(__uint_as_float(M.hmax[tk])));
          const __nv_bfloat16 yv = __float2bfloat16_rn(__fmul_rn(cc, sc));
          yb = __bfloat16_as_ushort(yv);
          const size_t oy = (size_t)tk * H + c * 16 + row;
          if (l == NL - 1) p.y[oy] = yv;
          if (p.ys) p.ys[(size_t)l * NB * H + oy] = yv;
        }
        const uint32_t other = __shfl_xor_sync(0xffffffffu, yb, 1);
        if (tk < NB && l + 1 < NL && (row & 1) == 0)
          st_tagged(p.y_t + ((size_t)((l & 1) * BMAX + tk) * (H / 2) + ((c * 16 + row) >> 1)),
                    tagw(yb | (other << 16), tag));
      }
      dn_seq += S;
    }

    // F. RMSNorm and router of the next sublayer.
    if (l + 1 < NL && !router_phase(l + 1)) return;
  }
}

}  // namespace

// ------------------------------------------------------------------ host side

static size_t a256(size_t v) { return ws_align256(v); }

FusedWs carve_fused_ws(void* ws) {
  uint8_t* p = static_cast<uint8_t*>(ws);
  FusedWs w;
  w.logits_t = p;
  p += a256((size_t)2 * BMAX * E * 8);
  w.y_t = p;
  p += a256((size_t)2 * BMAX * (H / 2) * 8);
  w.h_t = p;
  p += a256((size_t)MAX_SLOTS * BMAX * (I / 2) * 8);
  w.gabort = reinterpret_cast<unsigned*>(p);
  p += 256;
  w.y_mid = p;
  return w;
}

template <int NB>
static cudaError_t fused_init_nb(int sm_count) {
  cudaError_t e = cudaFuncSetAttribute(decode_fused_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       fz_smem_bytes<NB>());
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_fused_kernel<NB>, FZ_THREADS,
                                                    fz_smem_bytes<NB>());
  if (e != cudaSuccess) return e;
  (void)sm_count;
  return per_sm >= 1 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

cudaError_t fused_kernels_init(int sm_count) {
  cudaError_t r[8] = {fused_init_nb<1>(sm_count), fused_init_nb<2>(sm_count), fused_init_nb<3>(sm_count),
                      fused_init_nb<4>(sm_count), fused_init_nb<5>(sm_count), fused_init_nb<6>(sm_count),
                      fused_init_nb<7>(sm_count), fused_init_nb<8>(sm_count)};
  for (cudaError_t x : r)
    if (x != cudaSuccess) return x;
  return cudaSuccess;
}

template <int NB>
static cudaError_t fused_launch_nb(const FusedParams& fp, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(FZ_THREADS);
  cfg.dynamicSmemBytes = fz_smem_bytes<NB>();
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_fused_kernel<NB>, fp);
}

cudaError_t launch_fused_stack(const LayerArgs* layers, int n_layers, const void* x, int B, float eps, void* y,
                               void* ys, int32_t* ids, float* w, const FusedWs& ws, int grid, unsigned* err,
                               long long poll_limit, cudaStream_t st) {
  if (B < 1 || B > BMAX || n_layers < 1 || grid < DN_TILES || grid > E) return cudaErrorInvalidValue;
  for (int l0 = 0; l0 < n_layers; l0 += FUSED_MAX_LAYERS) {
    const int n = n_layers - l0 < FUSED_MAX_LAYERS ? n_layers - l0 : FUSED_MAX_LAYERS;
    const bool last = l0 + n == n_layers;
    FusedParams fp;
    fp.x = static_cast<const __nv_bfloat16*>(l0 == 0 ? x : ws.y_mid);
    fp.y = static_cast<__nv_bfloat16*>(last ? y : ws.y_mid);
    fp.ys = ys ? static_cast<__nv_bfloat16*>(ys) + (size_t)l0 * B * H : nullptr;
    fp.ids = ids ? ids + (size_t)l0 * B * TOPK : nullptr;
    fp.w = w ? w + (size_t)l0 * B * TOPK : nullptr;
    fp.logits_t = static_cast<uint64_t*>(ws.logits_t);
    fp.y_t = static_cast<uint64_t*>(ws.y_t);
    fp.h_t = static_cast<uint64_t*>(ws.h_t);
    fp.gabort = ws.gabort;
    fp.err = err;
    fp.poll_limit = poll_limit;
    fp.eps = eps;
    fp.n_layers = n;
    for (int i = 0; i < n; ++i) {
      const LayerArgs& a = layers[l0 + i];
      fp.layers[i].router_w = static_cast<const __nv_bfloat16*>(a.router_w);
      fp.layers[i].experts = a.experts;
      fp.layers[i].tscale = a.tscale;
      fp.layers[i].norm_w = static_cast<const __nv_bfloat16*>(a.norm_w);
    }
    cudaError_t e;
    switch (B) {
      case 1: e = fused_launch_nb<1>(fp, grid, st); break;
      case 2: e = fused_launch_nb<2>(fp, grid, st); break;
      case 3: e = fused_launch_nb<3>(fp, grid, st); break;
      case 4: e = fused_launch_nb<4>(fp, grid, st); break;
      case 5: e = fused_launch_nb<5>(fp, grid, st); break;
      case 6: e = fused_launch_nb<6>(fp, grid, st); break;
      case 7: e = fused_launch_nb<7>(fp, grid, st); break;
      default: e = fused_launch_nb<8>(fp, grid, st); break;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace flint
