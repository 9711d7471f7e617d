// Host-side interface between the C-ABI layer and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

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

size_t decode_ws_bytes(int gu_grid);
DecodeWs carve_decode_ws(void* ws, int gu_grid);

struct LayerArgs {
  const void* router_w;
  const uint8_t* experts;
  const float* tscale;
  const void* norm_w;
};

// Enqueues the three decode kernels of one sublayer.
//   x: input rows; ss_in: sum-of-squares partials of x written by the previous
//   sublayer's down kernel (nullptr: the router computes them itself).
//   ss_out: where this sublayer's down kernel writes the partials of y (or nullptr).
cudaError_t launch_decode_layer(int fmt, const LayerArgs& L, const void* x, const void* ss_in, int B,
                                float eps, void* y, void* ys_copy, void* ss_out, int32_t* ids_out,
                                float* w_out, const DecodeWs& ws, int gu_grid, unsigned* err,
                                cudaStream_t st, bool pdl_first);

cudaError_t decode_kernels_init(int device);

// Prefill-shaped sublayer over T tokens (NVFP4 weights): workspace size and
// the enqueue of its kernels on `st`.
size_t prefill_ws_bytes(int T);
cudaError_t prefill_kernels_init(int device);
cudaError_t launch_prefill(const LayerArgs& L, const void* x, int T, float eps, void* y, int32_t* ids_out,
                           float* w_out, void* ws, int sm_count, unsigned* err, cudaStream_t st);

cudaError_t launch_pack(int fmt, const void* gate_up, const uint8_t* gu_scales, const void* down,
                        const uint8_t* dn_scales, void* packed, cudaStream_t st);

}  // namespace flint
