// Host-side interface between the C-ABI layer and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "flint_common.cuh"

namespace flint {

// Workspace carve-up for the decode path (one sublayer in flight at a time;
// a stack reuses the same buffers for every sublayer, which the PDL ordering
// makes safe: every buffer is rewritten only after its last reader finished).
struct DecodeWs {
  void* logits;      // bf16 [8][256]
  void* xh_bf16;     // bf16 [8][2048]
  void* xfrag_f16;   // f16 x_hat * 2^xh_exp[token], mma B-fragment order
  void* xfrag_bf16;  // bf16 x_hat, mma B-fragment order
  int* xh_exp;       // [8]
  void* h;           // bf16 [49 slots][8 tokens][512]
  float* hmax_part;  // [gate/up grid][8]
  void* ss_part;     // CSum [128][8]: sum of squares of y per down tile
  void* y_mid;       // bf16 [8][2048] output of a non-final stack sublayer
};

constexpr size_t ws_align256(size_t v) { return (v + 255) / 256 * 256; }

// Largest gate/up grid of the three-kernel path (one CTA per SM).
constexpr int MAX_GU_GRID = 512;

constexpr size_t decode_ws_bytes(int gu_grid) {
  return ws_align256((size_t)BMAX * E * 2)                      // logits
         + ws_align256((size_t)BMAX * H * 2)                    // xh_bf16
         + 2 * ws_align256((size_t)(8 * 32 * 16 * 2) * 4)       // xfrag_f16, xfrag_bf16
         + ws_align256(BMAX * 4)                                // xh_exp
         + ws_align256((size_t)MAX_SLOTS * BMAX * I * 2)        // h
         + ws_align256((size_t)gu_grid * BMAX * 4)              // hmax_part
         + ws_align256((size_t)DN_TILES * BMAX * sizeof(CSum))  // ss_part
         + ws_align256((size_t)BMAX * H * 2);                   // y_mid
}
DecodeWs carve_decode_ws(void* ws, int gu_grid);

struct LayerArgs {
  const void* router_w;
  const uint8_t* experts;
  const float* tscale;
  const void* norm_w;
};

// Enqueues the three decode kernels of one sublayer (fmt 0 = NVFP4, 1 = BF16).
//   x: input rows; ss_in: sum-of-squares partials of x written by the previous
//   sublayer's down kernel (nullptr: the router computes them itself).
//   ss_out: where this sublayer's down kernel writes the partials of y (or nullptr).
cudaError_t launch_decode_chain(int fmt, const LayerArgs& L, const void* x, const void* ss_in, int B,
                                float eps, void* y, void* ys_copy, void* ss_out, int32_t* ids_out,
                                float* w_out, const DecodeWs& ws, int gu_grid, unsigned* err,
                                cudaStream_t st, bool pdl_first);

cudaError_t decode_kernels_init(int device);

// Persistent NVFP4 decode kernel (decode_fused.cu): one cooperative launch
// runs up to FUSED_MAX_LAYERS chained sublayers; longer stacks take several.
constexpr int FUSED_MAX_LAYERS = 64;

// Workspace of the persistent kernel: tagged words (32 data bits + the number
// of the sublayer that wrote them) through which the CTAs exchange logits, y
// and h, an abort flag, the arrival counters of the three exchanges, and the
// plain output of a stack chunk that feeds the next chunk.
struct FusedWs {
  void* logits_t;    // [2][8][256] u64
  void* y_t;         // [2][8][1024] u64
  void* h_t;         // [49][8][256] u64
  unsigned* gabort;  // [1]
  unsigned* cnt;     // arrival counters, 128 bytes apart: [0] logits, [32] h, [64] y
  void* y_mid;       // bf16 [8][2048]
};
constexpr size_t fused_ws_bytes() {
  return ws_align256((size_t)2 * BMAX * E * 8) + ws_align256((size_t)2 * BMAX * (H / 2) * 8) +
         ws_align256((size_t)MAX_SLOTS * BMAX * (I / 2) * 8) + 512 + ws_align256((size_t)BMAX * H * 2);
}
// Decode workspace: either path's layout, whichever is larger.
constexpr size_t decode_path_ws_bytes() {
  return decode_ws_bytes(MAX_GU_GRID) > fused_ws_bytes() ? decode_ws_bytes(MAX_GU_GRID) : fused_ws_bytes();
}
FusedWs carve_fused_ws(void* ws);
cudaError_t fused_kernels_init(int sm_count);
// grid: CTAs of the cooperative launch, one per SM, 128 <= grid <= 256.
cudaError_t launch_fused_stack(const LayerArgs* layers, int n_layers, const void* x, int B, float eps, void* y,
                               void* ys, int32_t* ids, float* w, const FusedWs& ws, int grid, unsigned* err,
                               long long poll_limit, cudaStream_t st);

// Prefill-shaped sublayer over T tokens (NVFP4 weights): workspace size and
// the enqueue of its kernels on `st`.
size_t prefill_ws_bytes(int T);
cudaError_t prefill_kernels_init(int device);
cudaError_t launch_prefill(const LayerArgs& L, const void* x, int T, float eps, void* y, int32_t* ids_out,
                           float* w_out, void* ws, int sm_count, unsigned* err, cudaStream_t st);

// Medium-batch decode path (medium.cu), 9..64 tokens, NVFP4 weights.  Tokens
// of one expert are processed in slot-chunks of up to MCH tokens (one mma n8
// block); pairs (token, expert) are numbered expert by expert, the shared
// expert first.
constexpr int MT_MAX = 64;
constexpr int MCH = 8;
constexpr int MPAIRS = (TOPK + 1) * MT_MAX;
constexpr int MSC_MAX = 320;  // >= 257 experts + 7 MT_MAX / MCH extra chunks
static_assert(MSC_MAX >= NE + MPAIRS / MCH, "slot-chunk table");
struct MedRoute {
  int n_sc;                        // slot-chunks
  int n_pairs;                     // 7 T
  int pad[2];
  int sc_e[MSC_MAX];               // expert (E = shared)
  int sc_pair[MSC_MAX];            // pair of its first token
  int sc_n[MSC_MAX];               // its tokens, 1..MCH
  uint8_t sc_tok[MSC_MAX][MCH];    // their ids, ascending
  int pidx[MT_MAX][TOPK + 1];      // pair of (token, j); j = TOPK: the shared expert
  float w[MT_MAX][TOPK];           // routing weights
};
struct MediumWs {
  void* logits;      // bf16 [64][256]
  void* xh_bf16;     // bf16 [64][2048] x_hat
  void* xfrag_f16;   // [8 chunks][8 K-slices][32 lanes][32 words]
  int* xh_exp;       // [64]
  MedRoute* rt;
  void* h;           // bf16 [MPAIRS][512]
  float* part;       // [MPAIRS][2048] scaled down-projection of each pair
  void* y_mid;       // bf16 [64][2048] output of a non-final stack sublayer
};
constexpr size_t medium_ws_bytes() {
  return ws_align256((size_t)MT_MAX * E * 2) + ws_align256((size_t)MT_MAX * H * 2) +
         ws_align256((size_t)(MT_MAX / 8) * 8 * 32 * 32 * 4) + ws_align256(MT_MAX * 4) +
         ws_align256(sizeof(MedRoute)) + ws_align256((size_t)MPAIRS * I * 2) +
         ws_align256((size_t)MPAIRS * H * 4) + ws_align256((size_t)MT_MAX * H * 2);
}
MediumWs carve_medium_ws(void* ws);
cudaError_t medium_kernels_init();
// Enqueues one medium sublayer.  x: the sublayer's input, normalised first
// (mnorm); null when the previous sublayer's combine already left this
// sublayer's x_hat in the workspace.  next: non-null when the combine is to
// leave x_hat for that sublayer (its norm weight, the same eps).
cudaError_t launch_medium_chain(const LayerArgs& L, const void* x, const LayerArgs* next, int T, float eps, void* y,
                                int32_t* ids_out, float* w_out, const MediumWs& ws, int sm_count, unsigned* err,
                                cudaStream_t st, bool pdl_first);

// Small-batch dense GEMV on packed NVFP4 weights (dense.cu): B * K at most
// DENSE_MAX_BK (the activations are staged in shared memory).
constexpr int DENSE_MAX_BK = 32768;
size_t dense_packed_bytes(int N, int K);
cudaError_t dense_kernels_init();
cudaError_t launch_pack_dense(const uint8_t* codes, const uint8_t* scales, int N, int K, void* packed,
                              cudaStream_t st);
cudaError_t launch_dense_gemv(const void* packed, int N, int K, float ts, const void* x, int B, void* y, int sm_count,
                              unsigned* err, cudaStream_t st);

cudaError_t launch_pack(int fmt, const void* gate_up, const uint8_t* gu_scales, const void* down,
                        const uint8_t* dn_scales, void* packed, cudaStream_t st);

}  // namespace flint
