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
// it.  A writer CTA stores its words, then adds 1 to the dependency's arrival
// counter (relaxed, no fence); one thread of a reader CTA polls that counter
// until every writer has arrived, then the CTA reads the words once and
// checks their tags (re-reading any that have not landed yet).  Polling a
// counter instead of the data keeps the spin traffic to one word per CTA.
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
constexpr int FZ_RED_MAX = 8;             // partial-sum ring between compute and epilogue warps, deepest
constexpr int FZ_NG = 4;                  // down slot groups (two K-half warps each)
constexpr int FZ_DN_ST = 12;              // down tile ring (a multiple of FZ_NG)
constexpr int FZ_ROW_BYTES = H * 2;       // one bf16 router row
constexpr int FZ_EPC = 2;                 // router experts per CTA at most (c and c + P)
// Per-sublayer constants in shared memory, one copy with the router rows: the
// router rows of this CTA's experts, the RMSNorm weight, and the (gate/up,
// down) tensor scales of the 256 routed experts (2 KB, by sublayer parity; the
// shared expert's two scales are read separately: 2,056 bytes is not a whole
// number of 16-byte copy units).
constexpr int FZ_TS_BYTES = E * 2 * 4;                                   // 2048
constexpr int FZ_CONST_BYTES = FZ_EPC * FZ_ROW_BYTES + H * 2 + 2 * FZ_TS_BYTES;
constexpr int FZ_SMEM_LIMIT = 232448;     // 227 KB of dynamic shared memory per CTA
static_assert(FZ_DN_ST % FZ_NG == 0, "each down stage must belong to one slot group");

template <int NB>
struct FzCfg {
  // Small batches poll the tagged h and y words themselves (one L2 round trip
  // after the last writer).  Larger ones wait on arrival counters: y stays
  // tagged; h is stored as plain bf16, published by a release fence before
  // each epilogue warp's counter increment, and fetched by bulk copies (up to
  // 56 KB per down CTA) once the counter is acquired.
  static constexpr bool POLL_DATA = NB <= 2;
  static constexpr int GU_ST = NB <= 4 ? 5 : 4;
  // Epilogue: 8 threads (the 8 h rows of an item) per token, so an item needs
  // 8 * NBP threads (NBP = NB rounded up to a power of two) and the 64
  // epilogue threads take IPR items at once; the partial-sum ring holds RED.
  static constexpr int NBP = NB <= 1 ? 1 : NB <= 2 ? 2 : NB <= 4 ? 4 : 8;
  static constexpr int TPI = 8 * NBP;
  static constexpr int IPR = 64 / TPI;
  static constexpr int RED = IPR > 4 ? IPR : 4;
  static constexpr int PAIRS = (1 + TOPK) * NB;               // (slot, token) pairs: shared + 6 per token
  static constexpr int HS_BYTES = PAIRS * HS_STRIDE * 2;      // staged h of the down phase
  static constexpr int XF_LANES = 4 * NB;                     // mma lanes that carry tokens
  static constexpr int XF_BYTES = GU_SLICES * XF_LANES * 32 * 4;
  static constexpr int UNI = ((HS_BYTES > XF_BYTES ? HS_BYTES : XF_BYTES) + 127) / 128 * 128;
  static constexpr int R_BYTES = (int)((sizeof(Routing) + 15) / 16 * 16);
  static constexpr int O_GU = 0;
  static constexpr int O_DN = O_GU + GU_ST * F4_GU_TILE;
  static constexpr int O_RED = O_DN + FZ_DN_ST * F4_DN_TILE;
  static constexpr int O_DRED = O_RED + RED * 8 * 128 * 4;
  static constexpr int O_ROWS = O_DRED + 8 * 128 * 4;
  static constexpr int O_UNI = O_ROWS + FZ_CONST_BYTES;
  static constexpr int O_R = O_UNI + UNI;
  static constexpr int O_MISC = O_R + 2 * R_BYTES;
};

static_assert(FzCfg<BMAX>::PAIRS <= 64, "pair tables hold 64 entries");

struct FzMisc {
  uint64_t gu_full[5], gu_empty[5];
  uint64_t dn_full[FZ_DN_ST], dn_empty[FZ_DN_ST];
  uint64_t rfull[FZ_RED_MAX], rempty[FZ_RED_MAX];
  uint64_t rbar;            // router rows of the next sublayer landed
  uint64_t route_ready[2];  // routing of sublayer l published (index l & 1)
  uint64_t hbar;            // bulk copies of h into the staging area landed (batches above 2)
  CSum redn[8][16];         // per-warp compensated partials (norm, logits)
  float rscale[BMAX];
  unsigned xmax[BMAX];      // max |x_hat| bits per token
  unsigned hmax[BMAX];      // max |h| bits per token (down phase)
  int xexp[2][BMAX];        // f16 exponent of x_hat per token, by sublayer parity
  float ts_sh[2][2];        // the shared expert's (gate/up, down) tensor scales, by sublayer parity
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
// Two consecutive tagged words, read from L2 without a check (the caller issues
// a batch of these before looking at any, so the batch costs one round trip).
__device__ __forceinline__ void ld_v2(const uint64_t* p, uint64_t& a, uint64_t& b) {
  asm volatile("ld.volatile.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ bool has_tag(uint64_t w, uint32_t tag) { return (uint32_t)(w >> 32) == tag; }
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
  unsigned* cnt;           // arrival counters: [0] logits, [32] h, [64] y (128 bytes apart)
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

// Warp-uniform decision of a polling warp after round `it` (1, 2, ...): lane 0
// looks at the abort word and the clock after the first two rounds and then
// every 16th, so the spin adds one L2 word per warp and not per thread.
__device__ __forceinline__ int warp_give_up(Waiter& wt, int it, const FusedParams& p, int lane) {
  int why = 0;
  if (lane == 0 && (it <= 2 || (it & 15) == 0)) why = wt.check(p);
  return __shfl_sync(0xffffffffu, why, 0);
}

__device__ __forceinline__ void fz_give_up(const FusedParams& p, FzMisc& M, int why) {
  if (why == 2) {
    atomicOr(p.err, ERR_POLL);
    st_volatile_u32(p.gabort, 1u);
  }
  *reinterpret_cast<volatile int*>(&M.abort) = 1;
}

// One thread: waits until the arrival counter reaches `target`.  0 = reached,
// 1 = another CTA gave up, 2 = the wait ran out.
__device__ __forceinline__ int wait_count(const unsigned* cnt, unsigned target, const FusedParams& p) {
  Waiter wt;
  for (;;) {
    if ((int)(ld_volatile_u32(cnt) - target) >= 0) return 0;
    const int why = wt.check(p);
    if (why) return why;
  }
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async;" ::: "memory"); }
__device__ __forceinline__ void arrive_count(unsigned* cnt) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(cnt) : "memory");
}

__device__ __forceinline__ bool cta_aborted(FzMisc& M) { return *reinterpret_cast<volatile int*>(&M.abort) != 0; }

// Bounded mbarrier wait of one thread that also gives up when this CTA aborts.
__device__ __forceinline__ bool wait_abort1(uint64_t* bar, uint32_t parity, FzMisc& M, unsigned* err, unsigned bit) {
  if (mbar_test(bar, parity)) return true;
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
  float* red = reinterpret_cast<float*>(smem + C::O_RED);    // [RED][8 warps][128]
  float* dred = reinterpret_cast<float*>(smem + C::O_DRED);  // [8 warps][128]
  uint8_t* rows = smem + C::O_ROWS;                          // [FZ_EPC][H] bf16 router rows
  const __nv_bfloat16* nw_s = reinterpret_cast<const __nv_bfloat16*>(rows + FZ_EPC * FZ_ROW_BYTES);  // [H]
  const float* ts_s = reinterpret_cast<const float*>(rows + FZ_EPC * FZ_ROW_BYTES + H * 2);  // [2][E][2]
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
    for (int b = 0; b < C::RED; ++b) {
      mbar_init(&M.rfull[b], FZ_CW);
      mbar_init(&M.rempty[b], C::TPI == 64 ? 2 : 1);  // one arrival per epilogue warp of the item
    }
    mbar_init(&M.rbar, 1);
    mbar_init(&M.route_ready[0], 1);
    mbar_init(&M.route_ready[1], 1);
    mbar_init(&M.hbar, 1);
    M.abort = 0;
    fence_mbar_init();
  }
  if (tid < BMAX) M.xmax[tid] = 0u;
  __syncthreads();

  // Producer state (lane 0 of the producer warp): copies issued per ring.
  const uint64_t pol = l2_evict_first();
  uint32_t gq = 0, dq = 0, rq = 0;
  auto issue_rows = [&](int k) {
    const FzLayer& Lk = p.layers[k];
    const bool nrm = Lk.norm_w != nullptr;
    mbar_arrive_expect_tx(&M.rbar, (uint32_t)(n_rexp * FZ_ROW_BYTES + FZ_TS_BYTES + (nrm ? H * 2 : 0)));
    for (int j = 0; j < n_rexp; ++j)
      bulk_g2s(rows + j * FZ_ROW_BYTES, Lk.router_w + (size_t)(c + j * P) * H, FZ_ROW_BYTES, &M.rbar, pol);
    bulk_g2s(const_cast<float*>(ts_s) + (k & 1) * E * 2, Lk.tscale, FZ_TS_BYTES, &M.rbar, pol);
    if (nrm) bulk_g2s(const_cast<__nv_bfloat16*>(nw_s), Lk.norm_w, H * 2, &M.rbar, pol);
    ++rq;
  };
  auto dn_src = [&](const FzLayer& Ly, int e) {
    return Ly.experts + (size_t)e * F4_EXPERT + F4_GU_BYTES + (size_t)c * F4_DN_TILE;
  };
  if (warp == FZ_PW) {
    // Constants of the first sublayer: its router rows, the shared expert's
    // gate/up tiles of this CTA and (down CTAs) the shared expert's down tile.
    // The rings are empty, so no stage needs waiting for.
    static_assert(GU_TILES <= 128 * 5, "at most GU_ST shared tiles per CTA");
    if (lane == 0) {
      issue_rows(0);
      for (int t = c; t < GU_TILES; t += P) {
        const int s = gq % C::GU_ST;
        mbar_arrive_expect_tx(&M.gu_full[s], F4_GU_TILE);
        bulk_g2s(gu_st + (size_t)s * F4_GU_TILE, p.layers[0].experts + (size_t)E * F4_EXPERT + (size_t)t * F4_GU_TILE,
                 F4_GU_TILE, &M.gu_full[s], pol);
        ++gq;
      }
      if (dn_cta) {
        mbar_arrive_expect_tx(&M.dn_full[0], F4_DN_TILE);
        bulk_g2s(dn_st, dn_src(p.layers[0], E), F4_DN_TILE, &M.dn_full[0], pol);
        ++dq;
      }
    }
    gq = __shfl_sync(0xffffffffu, gq, 0);
    dq = __shfl_sync(0xffffffffu, dq, 0);
    rq = __shfl_sync(0xffffffffu, rq, 0);
  }

  // Clear every tagged word of this call (tag 0 is never awaited) and meet.
  {
    const size_t n16 = ((size_t)2 * BMAX * E + (size_t)2 * BMAX * (H / 2) + (size_t)MAX_SLOTS * BMAX * (I / 2)) / 2;
    uint4* z = reinterpret_cast<uint4*>(p.logits_t);
    for (size_t i = (size_t)c * FZ_THREADS + tid; i < n16; i += (size_t)P * FZ_THREADS) z[i] = make_uint4(0u, 0u, 0u, 0u);
    if (c == 0 && tid == 0) {
      *p.gabort = 0u;
      p.cnt[0] = 0u;
      p.cnt[32] = 0u;
      p.cnt[64] = 0u;
    }
  }
  cg::this_grid().sync();

  // ================================================================ producer
  // All 32 lanes: a burst of copies into consecutive ring stages is issued by
  // parallel lanes.  Stages free up in sequence order (their consumers take
  // them in order), so the free ones are a prefix of the next stages.
  if (warp == FZ_PW) {
    // Issues up to n copies src_of(k), k = 0.., into ring (full/empty, ST stages
    // of `tile` bytes at `base`), advancing q.  blocking: wait for stages as
    // needed; otherwise stop at the first stage still in use.  Returns the number
    // issued, or -1 when this CTA gives up.
    auto issue_ring = [&](uint32_t& q, int ST, uint64_t* full, uint64_t* empty, uint8_t* base, int tile, int n,
                          bool blocking, auto src_of) -> int {
      int k = 0;
      while (k < n) {
        const int want = min(ST, n - k);
        const uint32_t ql = q + lane;
        const bool fr = lane < want && (ql < (uint32_t)ST || mbar_test(&empty[ql % ST], ((ql / ST) - 1) & 1));
        const unsigned m = __ballot_sync(0xffffffffu, fr);
        int run = (m == 0xffffffffu) ? 32 : __ffs(~m) - 1;
        run = min(run, want);
        if (run == 0) {
          if (!blocking) break;
          bool ok = true;
          if (lane == 0) ok = wait_abort1(&empty[q % ST], ((q / ST) - 1) & 1, M, p.err, ERR_WAIT_EMPTY);
          if (!__shfl_sync(0xffffffffu, ok, 0)) return -1;
          continue;
        }
        if (lane < run) {
          const int s = (q + lane) % ST;
          mbar_arrive_expect_tx(&full[s], (uint32_t)tile);
          bulk_g2s(base + (size_t)s * tile, src_of(k + lane), (uint32_t)tile, &full[s], pol);
        }
        q += run;
        k += run;
      }
      return k;
    };
    bool ok = true;
    for (int l = 0; l < NL && ok; ++l) {
      ok = __all_sync(0xffffffffu, wait_abort1(&M.route_ready[l & 1], (l >> 1) & 1, M, p.err, ERR_WAIT_FULL));
      if (!ok) break;
      const Routing& R = routing(l);
      const FzLayer& Ly = p.layers[l];
      const int S = R.n_slots;
      if (l + 1 < NL && lane == 0) issue_rows(l + 1);
      const int n_gu = i_first < S * GU_TILES ? (S * GU_TILES - i_first + P - 1) / P : 0;
      auto gu_src = [&](int k) {
        const int i = i_first + k * P;
        return Ly.experts + (size_t)R.slot_expert[i / GU_TILES] * F4_EXPERT + (size_t)(i % GU_TILES) * F4_GU_TILE;
      };
      auto dn_src_u = [&](int k) { return dn_src(Ly, R.slot_expert[1 + k]); };  // slot 0 went a sublayer ahead
      // routed gate/up tiles first (the critical path), then down tiles, while stages are free
      int g_done = issue_ring(gq, C::GU_ST, M.gu_full, M.gu_empty, gu_st, F4_GU_TILE, n_gu, false, gu_src);
      int d_done = 0;
      if (dn_cta)
        d_done = issue_ring(dq, FZ_DN_ST, M.dn_full, M.dn_empty, dn_st, F4_DN_TILE, S - 1, false, dn_src_u);
      if (g_done < n_gu) {
        const int r = issue_ring(gq, C::GU_ST, M.gu_full, M.gu_empty, gu_st, F4_GU_TILE, n_gu - g_done, true,
                                 [&](int k) { return gu_src(g_done + k); });
        ok = r == n_gu - g_done;
      }
      if (ok && l + 1 < NL) {
        const FzLayer& Ln = p.layers[l + 1];
        const int n_sh = c < GU_TILES ? (GU_TILES - c + P - 1) / P : 0;
        ok = issue_ring(gq, C::GU_ST, M.gu_full, M.gu_empty, gu_st, F4_GU_TILE, n_sh, true, [&](int k) {
               return Ln.experts + (size_t)E * F4_EXPERT + (size_t)(c + k * P) * F4_GU_TILE;
             }) == n_sh;
      }
      if (ok && dn_cta) {
        if (d_done < S - 1)
          ok = issue_ring(dq, FZ_DN_ST, M.dn_full, M.dn_empty, dn_st, F4_DN_TILE, S - 1 - d_done, true,
                          [&](int k) { return dn_src_u(d_done + k); }) == S - 1 - d_done;
        if (ok && l + 1 < NL)
          ok = issue_ring(dq, FZ_DN_ST, M.dn_full, M.dn_empty, dn_st, F4_DN_TILE, 1, true,
                          [&](int) { return dn_src(p.layers[l + 1], E); }) == 1;
      }
    }
    // Leave no copy in flight: wait for the last fill of every stage.
    if (lane == 0) {
      for (uint32_t n = gq > (uint32_t)C::GU_ST ? gq - C::GU_ST : 0; n < gq; ++n)
        if (!mbar_wait(&M.gu_full[n % C::GU_ST], (n / C::GU_ST) & 1)) atomicOr(p.err, ERR_DRAIN);
      for (uint32_t n = dq > (uint32_t)FZ_DN_ST ? dq - FZ_DN_ST : 0; n < dq; ++n)
        if (!mbar_wait(&M.dn_full[n % FZ_DN_ST], (n / FZ_DN_ST) & 1)) atomicOr(p.err, ERR_DRAIN);
      if (rq > 0 && !mbar_wait(&M.rbar, (rq - 1) & 1)) atomicOr(p.err, ERR_DRAIN);
    }
    return;
  }

  // ================================================================ epilogue warps
  // Thread et: item io = et / TPI of the current round, token tk, h row `row`.
  if (warp >= FZ_EW0) {
    const int et = tid - FZ_EW0 * 32;
    const int io = et / C::TPI, loc = et % C::TPI;
    const int tk = loc >> 3, row = loc & 7;
    const int og = red_off(row, tk), ou = red_off(row + 8, tk);
    uint32_t n0 = 0;  // items taken so far (the compute warps' sequence)
    // One round: items k0 + io, k0 + io < count, of a list; slot/tile/expert of
    // item k from item_of(k).  Fixed-order sum of the 8 slice partials,
    // SiLU*up, and the tagged store of h (two bf16 values per word) for the
    // tokens that use the slot.
    auto round = [&](int l, int k0, int count, auto item_of) -> bool {
      const int k = k0 + io;
      const bool active = k < count;
      const uint32_t n = n0 + (uint32_t)k;
      const int b = n % C::RED;
      bool ok = true;
      if (active) ok = wait_abort1(&M.rfull[b], (n / C::RED) & 1, M, p.err, ERR_WAIT_FULL);
      if (!__all_sync(0xffffffffu, ok)) return false;
      int slot = 0, tile = 0, e = E;
      uint32_t mask = 0u;
      if (active) item_of(k, slot, tile, e, mask);
      const bool act = active && tk < NB && ((mask >> tk) & 1u);
      uint32_t hb = 0u;
      if (act) {
        const float* rb = red + b * 1024;
        float gsum = 0.f, usum = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          gsum += rb[w * 128 + og];
          usum += rb[w * 128 + ou];
        }
        const float tsg = e < E ? ts_s[(l & 1) * E * 2 + 2 * e] : M.ts_sh[l & 1][0];
        const float f = __fmul_rn(exp2i(-M.xexp[l & 1][tk]), tsg);
        const float gate = __fmul_rn(gsum, f);
        const float up = __fmul_rn(usum, f);
        const float silu = __fdiv_rn(gate, __fadd_rn(1.0f, expf(-gate)));
        hb = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(silu, up)));
      }
      const uint32_t other = __shfl_xor_sync(0xffffffffu, hb, 1);
      if (act && (row & 1) == 0) {
        if (C::POLL_DATA)
          st_tagged(p.h_t + ((size_t)(slot * BMAX + tk) * (I / 2) + ((tile * 8 + row) >> 1)),
                    tagw(hb | (other << 16), (uint32_t)(l + 1)));
        else
          *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(p.h_t) + (size_t)(slot * BMAX + tk) * I +
                                       tile * 8 + row) = hb | (other << 16);
      }
      __syncwarp();
      if (active && (C::TPI == 64 ? lane == 0 : loc == 0)) mbar_arrive(&M.rempty[b]);
      return true;
    };
    const int n_sh = c < GU_TILES ? (GU_TILES - c + P - 1) / P : 0;
    for (int l = 0; l < NL; ++l) {
      // The tensor scales of sublayer l came with constants copy l.  The
      // compute warps observed that copy's completion before releasing any
      // item of l (their partial-sum barrier arrive is a release, this warp's
      // wait an acquire), so the copy is visible here without waiting on it:
      // a wait here could see the next copy's phase instead.
      for (int k0 = 0; k0 < n_sh; k0 += C::IPR)
        if (!round(l, k0, n_sh, [&](int k, int& slot, int& tile, int& e, uint32_t& mask) {
              slot = 0;
              tile = c + k * P;
              e = E;
              mask = 0xFFu;
            }))
          return;
      n0 += n_sh;
      if (!__all_sync(0xffffffffu, wait_abort1(&M.route_ready[l & 1], (l >> 1) & 1, M, p.err, ERR_WAIT_FULL)))
        return;
      const Routing& R = routing(l);
      const int S = R.n_slots;
      const int n_gu = i_first < S * GU_TILES ? (S * GU_TILES - i_first + P - 1) / P : 0;
      for (int k0 = 0; k0 < n_gu; k0 += C::IPR)
        if (!round(l, k0, n_gu, [&](int k, int& slot, int& tile, int& e, uint32_t& mask) {
              const int i = i_first + k * P;
              slot = i / GU_TILES;
              tile = i % GU_TILES;
              e = R.slot_expert[slot];
              mask = R.slot_mask[slot];
            }))
          return;
      n0 += n_gu;
      __syncwarp();
      if (!C::POLL_DATA && lane == 0) {  // this warp's h of sublayer l is stored: publish it
        fence_acq_rel_gpu();
        arrive_count(p.cnt + 32);
      }
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
    const int b = gn % C::RED;
    if (gn >= (uint32_t)C::RED && !wait_abort(&M.rempty[b], ((gn / C::RED) - 1) & 1, M, p.err, ERR_WAIT_EMPTY))
      return false;
    float* rb = red + b * 1024;
#pragma unroll
    for (int j = 0; j < 4; ++j) rb[warp * 128 + j * 32 + lane] = acc[j];
    __syncwarp();
    if (lane == 0) mbar_arrive(&M.rfull[b]);
    ++gn;
    return true;
  };

  // Two consecutive gate/up items, their slices multiplied together (more
  // independent work per warp); the partial sums go to the epilogue in order.
  auto gu_item2 = [&](const uint32_t (&bfr)[16][2]) -> bool {
    const int s0 = gn % C::GU_ST, s1 = (gn + 1) % C::GU_ST;
    float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
    if (!wait_abort(&M.gu_full[s0], (gn / C::GU_ST) & 1, M, p.err, ERR_WAIT_FULL)) return false;
    if (!wait_abort(&M.gu_full[s1], ((gn + 1) / C::GU_ST) & 1, M, p.err, ERR_WAIT_FULL)) return false;
    nvfp4_slice_mma2(gu_st + (size_t)s0 * F4_GU_TILE + warp * F4_SLICE, gu_st + (size_t)s1 * F4_GU_TILE + warp * F4_SLICE,
                     lane, bfr, acc0, acc1);
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&M.gu_empty[s0]);
      mbar_arrive(&M.gu_empty[s1]);
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t n = gn + q;
      const int b = n % C::RED;
      if (n >= (uint32_t)C::RED && !wait_abort(&M.rempty[b], ((n / C::RED) - 1) & 1, M, p.err, ERR_WAIT_EMPTY))
        return false;
      float* rb = red + b * 1024;
#pragma unroll
      for (int j = 0; j < 4; ++j) rb[warp * 128 + j * 32 + lane] = q == 0 ? acc0[j] : acc1[j];
      __syncwarp();
      if (lane == 0) mbar_arrive(&M.rfull[b]);
    }
    gn += 2;
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
    float ts_tail[2] = {0.f, 0.f};
    if (tid == 0) {  // the shared expert's scales of sublayer k; used once the phase ends
      ts_tail[0] = __ldg(Lk.tscale + 2 * E);
      ts_tail[1] = __ldg(Lk.tscale + 2 * E + 1);
    }
    float xv[2 * NP][8];
#pragma unroll
    for (int t = 0; t < 2 * NP; ++t)
#pragma unroll
      for (int i = 0; i < 8; ++i) xv[t][i] = 0.f;
    if (k == 0) {
#pragma unroll
      for (int t = 0; t < NB; ++t) bf16x8_to_f32(__ldcg(reinterpret_cast<const uint4*>(p.x + (size_t)t * H + k0)), xv[t]);
    } else {
      // every down CTA has stored its rows of y (sublayer k - 1)
      if (!C::POLL_DATA) {
        if (tid == 0 && !dead) {
          const int why = wait_count(p.cnt + 64, (unsigned)(k * DN_TILES), p);
          if (why) {
            fz_give_up(p, M, why);
            dead = true;
          }
        }
        if (cbar_or(dead || cta_aborted(M))) return false;
      }
      const uint32_t tag = (uint32_t)k;
      const uint64_t* base = p.y_t + (size_t)((k - 1) & 1) * BMAX * (H / 2) + tid * 4;
      uint32_t pend = (1u << (2 * NB)) - 1u;
      Waiter wt;
      for (int it = 1; !dead; ++it) {
        // tokens in groups of 4: 8 loads in flight, then their checks
#pragma unroll
        for (int t0 = 0; t0 < NB; t0 += 4) {
          uint64_t wv[4][2][2];
#pragma unroll
          for (int t = t0; t < t0 + 4 && t < NB; ++t)
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
              if ((pend >> (2 * t + h2)) & 1u)
                ld_v2(base + (size_t)t * (H / 2) + 2 * h2, wv[t - t0][h2][0], wv[t - t0][h2][1]);
#pragma unroll
          for (int t = t0; t < t0 + 4 && t < NB; ++t)
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
              if (((pend >> (2 * t + h2)) & 1u) && has_tag(wv[t - t0][h2][0], tag) &&
                  has_tag(wv[t - t0][h2][1], tag)) {
                const uint32_t d0 = (uint32_t)wv[t - t0][h2][0], d1 = (uint32_t)wv[t - t0][h2][1];
                xv[t][4 * h2 + 0] = __uint_as_float(d0 << 16);
                xv[t][4 * h2 + 1] = __uint_as_float(d0 & 0xFFFF0000u);
                xv[t][4 * h2 + 2] = __uint_as_float(d1 << 16);
                xv[t][4 * h2 + 3] = __uint_as_float(d1 & 0xFFFF0000u);
                pend &= ~(1u << (2 * t + h2));
              }
        }
        if (__all_sync(0xffffffffu, pend == 0u)) break;
        const int why = warp_give_up(wt, it, p, lane);
        if (why) {
          if (lane == 0) fz_give_up(p, M, why);
          dead = true;
        }
      }
    }
    // constants copy k (router rows, norm weight, tensor scales), a sublayer ahead
    if (!dead && !wait_abort(&M.rbar, (uint32_t)k & 1, M, p.err, ERR_WAIT_FULL)) dead = true;
    float nw[8];
    if (has_norm) bf16x8_to_f32(*reinterpret_cast<const uint4*>(nw_s + k0), nw);
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
    if (tid == 0) {
      M.ts_sh[k & 1][0] = ts_tail[0];
      M.ts_sh[k & 1][1] = ts_tail[1];
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
    // With one token, warp 0 does all of it and one barrier publishes it.
    if (NB == 1) {
      if (warp == 0) {
        zero_routing(R, lane, 32);
        if (lane == 0) {
          M.hmax[0] = 0u;
          M.xmax[0] = 0u;
        }
        __syncwarp();
      }
    } else {
      zero_routing(R, tid, FZ_CT);
      if (tid < NB) {
        M.hmax[tid] = 0u;
        M.xmax[tid] = 0u;
      }
      if (cbar_or(dead || cta_aborted(M))) return;
    }
    // Selection first (expert ids and the slot table, which is all the
    // producer and the epilogue need), the routing weights while the first
    // copies are in flight.
    int sel_i[TOPK];
    uint32_t sel_lg[TOPK];
    if (warp < NB) {
      const uint64_t* src = p.logits_t + ((size_t)((l & 1) * BMAX + warp) * E + lane * 8);
      uint32_t d[8];
      Waiter wt;
      bool got = false;
      for (int it = 1;; ++it) {
        uint64_t wv[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) ld_v2(src + 2 * q, wv[2 * q], wv[2 * q + 1]);
        bool ok = true;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          ok = ok && has_tag(wv[i], tag);
          d[i] = (uint32_t)wv[i];
        }
        if (__all_sync(0xffffffffu, ok)) {
          got = true;
          break;
        }
        const int why = warp_give_up(wt, it, p, lane);
        if (why) {
          if (lane == 0) fz_give_up(p, M, why);
          break;
        }
      }
      if (got) {
        const uint4 raw = make_uint4((d[0] & 0xFFFFu) | (d[1] << 16), (d[2] & 0xFFFFu) | (d[3] << 16),
                                     (d[4] & 0xFFFFu) | (d[5] << 16), (d[6] & 0xFFFFu) | (d[7] << 16));
        warp_top6_core(raw, lane, sel_i, sel_lg);
        warp_top6_store(sel_i, sel_lg, lane, R.ids[warp], R.lg[warp], R.umask);
      } else {
        dead = true;
      }
    }
    if (NB > 1 && cbar_or(dead || cta_aborted(M))) return;
    if (warp == 0 && !(NB == 1 && dead)) {
      __syncwarp();
      warp_slot_experts(R, NB, lane);
      if (lane == 0) mbar_arrive(&M.route_ready[l & 1]);  // the producer and the epilogue may go
    }
    if (warp < NB && !dead) warp_top6_weights(sel_lg, lane, R.w[warp]);
    if (NB > 1 && cbar_or(dead || cta_aborted(M))) return;
    if (warp == 0 && !(NB == 1 && dead)) {
      __syncwarp();
      warp_slot_weights(R, NB, lane);
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
      const int n_gu = i_first < S * GU_TILES ? (S * GU_TILES - i_first + P - 1) / P : 0;
      for (int k = 0; k < n_gu && !dead; k += 2) dead = k + 1 < n_gu ? !gu_item2(bfr) : !gu_item(bfr);
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
      if (!C::POLL_DATA) {
        // Both epilogue warps of every CTA published their h: acquire the
        // counter, then bring every (slot, token) row of h in by bulk copy.
        if (tid == 0 && !dead) {
          const int why = wait_count(p.cnt + 32, (unsigned)((l + 1) * 2 * P), p);
          if (why) {
            fz_give_up(p, M, why);
            dead = true;
          } else {
            fence_acq_rel_gpu();
          }
        }
        if (cbar_or(dead || cta_aborted(M))) return;
        const int npairs = M.npairs;
        if (warp == 0) {
          if (lane == 0) mbar_arrive_expect_tx(&M.hbar, (uint32_t)(npairs * I * 2));
          __syncwarp();
          fence_proxy_async();  // the staging area was last read by generic loads; h by other SMs' stores
          const uint16_t* hp = reinterpret_cast<const uint16_t*>(p.h_t);
          for (int pr = lane; pr < npairs; pr += 32)
            bulk_g2s(hs + (size_t)pr * HS_STRIDE, hp + (size_t)(M.pslot[pr] * BMAX + M.ptok[pr]) * I, I * 2,
                     &M.hbar, pol);
        }
        if (!wait_abort(&M.hbar, (uint32_t)l & 1, M, p.err, ERR_WAIT_FULL)) dead = true;
        // per-token maxima of |h| (16-byte chunks of the staged rows)
        for (int kk = tid; kk < npairs * (I / 8) && !dead; kk += FZ_CT) {
          const int pr = kk / (I / 8), ch = kk % (I / 8);
          const uint4 v = *reinterpret_cast<const uint4*>(hs + (size_t)pr * HS_STRIDE + ch * 8);
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
          unsigned am = 0u;
#pragma unroll
          for (int q = 0; q < 4; ++q) am = max(am, max((w4[q] & 0x7FFFu) << 16, w4[q] & 0x7FFF0000u));
          const int tok = M.ptok[pr];
#pragma unroll
          for (int q = 0; q < NB; ++q)
            if (q == tok) tmax[q] = max(tmax[q], am);
        }
      } else {
        Waiter wt;
        for (int it = 1; !dead; ++it) {
          // chunks in groups of 8: 8 loads in flight, then their checks
#pragma unroll
          for (int j0 = 0; j0 < NJ; j0 += 8) {
            uint64_t wv[8][2];
#pragma unroll
            for (int j = j0; j < j0 + 8 && j < NJ; ++j) {
              if ((pend >> j) & 1u) {
                const int kk = tid + j * FZ_CT, pr = kk >> 7, ch = kk & 127;
                ld_v2(p.h_t + ((size_t)(M.pslot[pr] * BMAX + M.ptok[pr]) * (I / 2) + ch * 2), wv[j - j0][0],
                      wv[j - j0][1]);
              }
            }
#pragma unroll
            for (int j = j0; j < j0 + 8 && j < NJ; ++j) {
              if (((pend >> j) & 1u) && has_tag(wv[j - j0][0], tag) && has_tag(wv[j - j0][1], tag)) {
                const int kk = tid + j * FZ_CT, pr = kk >> 7, ch = kk & 127;
                const int tok = M.ptok[pr];
                const uint32_t d0 = (uint32_t)wv[j - j0][0], d1 = (uint32_t)wv[j - j0][1];
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
          if (__all_sync(0xffffffffu, pend == 0u)) break;
            const int why = warp_give_up(wt, it, p, lane);
          if (why) {
            if (lane == 0) fz_give_up(p, M, why);
            dead = true;
          }
        }
      }
#pragma unroll
      for (int q = 0; q < NB; ++q) {
        const unsigned m = redux_max(tmax[q]);
        if (lane == 0 && m != 0u) atomicMax(&M.hmax[q], m);
      }
      if (cbar_or(dead || cta_aborted(M))) return;
      const int g = lane >> 2, t4 = lane & 3;
      const int kh = warp & 1, grp = warp >> 1;
      const int cgrp = (grp - (int)(dn_seq % FZ_NG) + FZ_NG) % FZ_NG;  // the slots u = cgrp mod 4
      const float hsc = g < NB ? exp2i(f16_range_exp(__uint_as_float(M.hmax[g]))) : 1.0f;
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
          // bf16 h -> f16 h * 2^hexp[token] while forming the B fragments
          const uint32_t* hr = reinterpret_cast<const uint32_t*>(hs + (size_t)M.pidx[u][g] * HS_STRIDE + kh * 256);
          const float sc = hsc;
#pragma unroll
          for (int kb = 0; kb < 16; ++kb) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              const uint32_t v = hr[kb * 8 + t4 + 4 * r];
              const __half2 hv = __floats2half2_rn(__fmul_rn(__uint_as_float(v << 16), sc),
                                                   __fmul_rn(__uint_as_float(v & 0xFFFF0000u), sc));
              hb[kb][r] = *reinterpret_cast<const uint32_t*>(&hv);
            }
          }
        } else {
#pragma unroll
          for (int kb = 0; kb < 16; ++kb) hb[kb][0] = hb[kb][1] = 0u;
        }
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        nvfp4_slice_mma(dn_st + (size_t)s * F4_DN_TILE + kh * F4_SLICE, lane, hb, acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(&M.dn_empty[s]);
        const int eu = R.slot_expert[u];
        const float ts = eu < E ? ts_s[(l & 1) * E * 2 + 2 * eu + 1] : M.ts_sh[l & 1][1];
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
      if (!C::POLL_DATA && l + 1 < NL) {
        if (cbar_or(dead || cta_aborted(M))) return;
        if (tid == 0) arrive_count(p.cnt + 64);  // this CTA's rows of y are stored
      }
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
  w.cnt = reinterpret_cast<unsigned*>(p + 128);
  p += 512;
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
    fp.cnt = ws.cnt;
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
