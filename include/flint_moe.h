/*
 * flint_moe.h -- C ABI of the GB300 (sm_103a) Flint MoE sublayer library.
 *
 * The operation is the MoE sublayer of the Flint model as described in
 * "Day-0 Support for Flint on vLLM" (sections "Model architecture" and
 * "Optimizations"): a 2048-wide token x_hat is scored by a bf16 router over
 * 256 experts, the 6 experts with the largest sigmoid score are selected and
 * their scores renormalised to sum to 1, each selected expert and the
 * always-on shared expert compute down(bf16(silu(gate(x_hat)) * up(x_hat))),
 * and the outputs are combined with the routing weights (shared weight 1) and
 * rounded once to bf16.  Expert weights are NVFP4 (16 E2M1 codes + one E4M3
 * block scale per 16 weights + one fp32 per-tensor scale) used weight-only
 * with bf16 activations ("W4A16", same section), or plain bf16.
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers (the current CUDA device) owned
 *     by the caller; every pointer must be 16-byte aligned.  Row-major layouts.
 *   - Arguments are validated on the host before anything is enqueued; an
 *     invalid call returns a negative status and enqueues nothing.  A buffer
 *     the call writes (outputs, workspace) must not share a byte with any
 *     other buffer of the call, weights included (FLINT_MOE_ERR_INVALID_ARG);
 *     buffers that are only read may overlap.
 *   - Work is enqueued asynchronously on `stream` (NULL = legacy default
 *     stream); outputs are valid after the stream is synchronised.
 *   - The library allocates no device memory on the compute path: scratch
 *     space is the caller's workspace `ws` (size from flint_moe_workspace_bytes,
 *     256-byte aligned, no initialisation needed).  Calls that share one
 *     workspace must be ordered on one stream.
 *   - Only the Flint shapes are supported: hidden 2048, 256 routed experts,
 *     1 shared expert, intermediate 512, top-6.  Anything else returns
 *     FLINT_MOE_ERR_UNSUPPORTED (there is no generic fallback path).
 */
#ifndef FLINT_MOE_H
#define FLINT_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the runtime's stream handle type). */
typedef struct CUstream_st *flint_moe_stream_t;

/* Status codes returned by every int-returning entry point. */
enum {
    FLINT_MOE_OK = 0,
    FLINT_MOE_ERR_INVALID_ARG = -1, /* null, misaligned or overlapping
                                       buffers, bad count                   */
    FLINT_MOE_ERR_UNSUPPORTED = -2, /* shape or batch outside the fast path */
    FLINT_MOE_ERR_WORKSPACE = -3,   /* workspace or output buffer too small */
    FLINT_MOE_ERR_CUDA = -4,        /* a CUDA runtime call failed           */
    FLINT_MOE_ERR_TIMEOUT = -5      /* a bounded device wait gave up        */
};

/* Expert weight formats. */
enum { FLINT_MOE_W_NVFP4 = 0, FLINT_MOE_W_BF16 = 1 };

/* Largest batch of the low-latency decode path ("Optimizations": the
 * low-latency path serves up to 8 requests). */
#define FLINT_MOE_MAX_DECODE_BATCH 8

/* Largest batch of the decode calls.  9..64 tokens (NVFP4 weights only) take
 * the medium-batch kernels: past the low-latency cap of 8 requests, each
 * selected expert's weights are read once per group of up to 16 of the
 * tokens that chose it, instead of once per group of 8 tokens. */
#define FLINT_MOE_MAX_MEDIUM_BATCH 64

/* Decode kernels for NVFP4 weights (flint_moe_set_decode_kernel). */
enum { FLINT_MOE_DECODE_CHAINED = 0, FLINT_MOE_DECODE_PERSISTENT = 1 };

/* Model dimensions.  Must equal {2048, 256, 1, 512, 6, *, eps}. */
typedef struct {
    int hidden;       /* H = 2048                                   */
    int n_experts;    /* E = 256 routed experts                     */
    int n_shared;     /* 1 shared expert (index E in the blobs)     */
    int inter;        /* I = 512 expert intermediate size           */
    int top_k;        /* 6                                          */
    int weight_dtype; /* FLINT_MOE_W_NVFP4 or FLINT_MOE_W_BF16      */
    float rms_eps;    /* RMSNorm epsilon (1e-6 for Flint stacks)    */
} flint_moe_dims;

/* One MoE sublayer's weights (all device pointers, caller-owned). */
typedef struct {
    const void *router_w;       /* bf16 [E][H]                                   */
    const void *experts;        /* packed blob from flint_moe_pack_weights       */
    const float *tensor_scales; /* NVFP4: fp32 [E+1][2] = (gate/up, down) scale
                                   per expert; ignored (may be NULL) for BF16    */
    const void *norm_w;         /* bf16 [H] RMSNorm weight applied to this
                                   sublayer's input, or NULL for no norm         */
} flint_moe_layer;

/* Bytes of one sublayer's packed expert blob (E routed + 1 shared expert):
 * NVFP4 1,769,472 B per expert, BF16 6,291,456 B per expert (the same byte
 * count as the plain layout: the repack is lossless and adds no padding).
 * Returns 0 for unsupported dims. */
size_t flint_moe_packed_bytes(const flint_moe_dims *dims);

/* Workspace bytes for calls with at most `max_tokens` tokens (decode: 1..64,
 * of which 9..64 NVFP4 only; prefill: any T >= 1).  Returns 0 for
 * unsupported dims or token counts. */
size_t flint_moe_workspace_bytes(const flint_moe_dims *dims, int max_tokens);

/*
 * One-time lossless repack of one sublayer's experts from the plain layout
 * into the kernels' interleaved layout ("Model architecture": the NVFP4
 * checkpoint is repacked losslessly at load time).
 *
 * NVFP4 inputs (expert index E is the shared expert):
 *   gate_up        uint8 [E+1][2I][H/2]  rows 0..I-1 gate, I..2I-1 up; byte j
 *                  of a row holds element 2j in its low nibble, 2j+1 high
 *   gate_up_scales uint8 [E+1][2I][H/16] E4M3 scale of each 16-element block
 *   down           uint8 [E+1][H][I/2]
 *   down_scales    uint8 [E+1][H][I/16]
 * BF16 inputs: gate_up bf16 [E+1][2I][H], down bf16 [E+1][H][I]; the scale
 *   pointers must be NULL.
 * packed: output, flint_moe_packed_bytes(dims) bytes.  Runs one device kernel
 * on `stream`; inputs may be freed once the stream has passed it.
 */
int flint_moe_pack_weights(const flint_moe_dims *dims, const void *gate_up,
                           const uint8_t *gate_up_scales, const void *down,
                           const uint8_t *down_scales, void *packed,
                           size_t packed_bytes, flint_moe_stream_t stream);

/*
 * One MoE sublayer for a decode batch of 1..64 independent tokens.
 *   x        bf16 [B][H] input (RMSNorm'd first if layer->norm_w != NULL)
 *   y        bf16 [B][H] output
 *   topk_ids int32 [B][6] selected experts (descending score) or NULL
 *   topk_w   fp32  [B][6] their renormalised weights, or NULL
 * Three steps: the router GEMV with sigmoid top-6; the gate/up GEMV with
 * SiLU*up over the selected experts only; the down GEMV fused with the
 * weighted combine and the shared expert.  By default (and always for BF16
 * weights) they are three kernels chained with programmatic dependent launch;
 * with FLINT_MOE_DECODE_PERSISTENT selected (flint_moe_set_decode_kernel),
 * NVFP4 weights take one cooperative kernel, one thread block per SM (at
 * least 128 SMs, else FLINT_MOE_ERR_UNSUPPORTED), whose blocks exchange
 * logits, h and y through the workspace.  9 <= B <= 64 (NVFP4 only, else
 * FLINT_MOE_ERR_UNSUPPORTED) runs the medium-batch chain: one block per token
 * for the RMSNorm; the router logits over (chunk of 8 tokens, expert) units;
 * one block that selects every token's top-6 and builds the table of
 * slot-chunks (an expert with up to 8 of the tokens that selected it);
 * gate/up and down kernels that stream each selected expert's tiles once per
 * slot-chunk; and one block per token that adds the pairs' down projections
 * in a fixed order (inside a stack it also normalises the next sublayer's
 * input, so that sublayer skips the RMSNorm block).  Its
 * workspace is flint_moe_workspace_bytes(dims, 64) bytes (less returns
 * FLINT_MOE_ERR_WORKSPACE).  B > 64 returns FLINT_MOE_ERR_UNSUPPORTED.  The
 * result is deterministic: the same inputs and kernel choice give the same
 * bits on every call.
 */
int flint_moe_decode_layer(const flint_moe_dims *dims, const flint_moe_layer *layer,
                           const void *x, int B, void *y, int32_t *topk_ids,
                           float *topk_w, void *ws, size_t ws_bytes,
                           flint_moe_stream_t stream);

/*
 * n_layers chained sublayers for one decode batch: sublayer i+1 reads
 * sublayer i's output (through its own RMSNorm when layers[i+1].norm_w is
 * set; no residual is added).
 *   x, y            bf16 [B][H]
 *   ids_per_layer   int32 [n_layers][B][6] or NULL
 *   w_per_layer     fp32  [n_layers][B][6] or NULL
 *   ys_per_layer    bf16  [n_layers][B][H] every sublayer's output, or NULL
 * Chained kernels (the default, BF16 weights, and every 9..64-token batch):
 * the chain of 3 (5 past 8 tokens) kernels per sublayer is captured once
 * into a CUDA graph (cached per argument set; see
 * flint_moe_release) and replayed with one graph launch per call; the graph
 * bakes in every pointer, so buffer contents may change between calls,
 * addresses not.  Persistent kernel (NVFP4, flint_moe_set_decode_kernel): one
 * cooperative launch per 64 sublayers, which prefetches each sublayer's
 * router rows, norm weight, tensor scales and shared-expert tiles while the
 * sublayer before it runs.  A stack call gives the same bits as the chain of
 * flint_moe_decode_layer calls over the same sublayers with the same kernel
 * choice.
 */
int flint_moe_decode_stack(const flint_moe_dims *dims, const flint_moe_layer *layers,
                           int n_layers, const void *x, int B, void *y,
                           int32_t *ids_per_layer, float *w_per_layer,
                           void *ys_per_layer, void *ws, size_t ws_bytes,
                           flint_moe_stream_t stream);

/*
 * One MoE sublayer over T tokens (prefill shape, e.g. T = 8192; "Day-0
 * Support for Flint on vLLM", section "Optimizations": the MoE kernels also
 * serve the 8K prefill).  Same definition as flint_moe_decode_layer, token by
 * token: router logits (approximated on the tensor cores, then recomputed
 * exactly for every expert that can reach the top 6), sigmoid top-6, tokens
 * grouped by expert, grouped gate/up GEMM with SiLU*up and grouped down GEMM
 * on the tensor cores (tcgen05, fp32 accumulation), weighted combine plus the
 * shared expert.
 *   x        bf16 [T][H] (RMSNorm'd first if layer->norm_w != NULL)
 *   y        bf16 [T][H]; must not overlap x (nor either of them the workspace)
 *   topk_ids int32 [T][6] or NULL; topk_w fp32 [T][6] or NULL
 *   ws       flint_moe_workspace_bytes(dims, T) bytes, 256-byte aligned, no
 *            initialisation needed
 * NVFP4 weights only (BF16: FLINT_MOE_ERR_UNSUPPORTED); 1 <= T <= 2^20.
 * The combine adds the experts' fp32 contributions in completion order, so y
 * can differ between runs in its last bits; the routing is exact and
 * repeatable.  Seven kernels on `stream`, asynchronous.
 */
int flint_moe_prefill_layer(const flint_moe_dims *dims, const flint_moe_layer *layer,
                            const void *x, int T, void *y, int32_t *topk_ids,
                            float *topk_w, void *ws, size_t ws_bytes,
                            flint_moe_stream_t stream);

/* Size of the scratch area built into the library for
 * flint_moe_decode_layer_noalloc, and the largest batch it serves. */
#define FLINT_MOE_NOALLOC_SCRATCH_BYTES 1048576
#define FLINT_MOE_NOALLOC_MAX_TOKENS 8

/*
 * flint_moe_decode_layer without a workspace argument, for callers that
 * cannot allocate device memory: code that runs where cudaMalloc is not
 * allowed or not wanted (inside a host callback or another library's
 * allocator hook, under a strict memory budget, or from a runtime that owns
 * every device allocation itself).  The paper has no counterpart; this is a
 * convenience of this library.
 *
 * Scratch lives in one fixed array of FLINT_MOE_NOALLOC_SCRATCH_BYTES in the
 * library's device image: every GPU that loads the library holds it until the
 * process exits, and this call allocates nothing.  Inputs, outputs and
 * weights are as for flint_moe_decode_layer (caller-owned device memory).
 *   B > FLINT_MOE_NOALLOC_MAX_TOKENS returns FLINT_MOE_ERR_WORKSPACE (the
 *   built-in scratch holds at most 8 tokens) and enqueues nothing.
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture (a first
 * call on a capturing stream returns FLINT_MOE_ERR_INVALID_ARG).  Every
 * call on a device shares the one array and it keeps the previous call's
 * contents; each call clears what it must find cleared, and its kernels read
 * no other scratch word before writing it.  Calls whose work overlaps on the GPU
 * (different streams, or other threads) race on the array: order them.
 */
int flint_moe_decode_layer_noalloc(const flint_moe_dims *dims, const flint_moe_layer *layer,
                                   const void *x, int B, void *y, int32_t *topk_ids,
                                   float *topk_w, flint_moe_stream_t stream);

/*
 * Small-batch dense GEMV on NVFP4 weights ("Day-0 Support for Flint on vLLM",
 * section "Optimizations": a small-batch dense GEMV on the same NVFP4 weights
 * serves the attention projections and the dense MLP of the first layers):
 *   y[t][n] = bf16( tensor_scale * sum_k x[t][k] * W[n][k] ),  fp32 accumulation,
 * W[n][k] = e2m1(code) * e4m3(block scale of k / 16).  Shapes: N a multiple
 * of 16 (below 2^24), K a multiple of 256, at most 32768; otherwise
 * FLINT_MOE_ERR_UNSUPPORTED.
 *
 * flint_moe_dense_packed_bytes: bytes of the packed matrix, N * K * 9 / 16
 *   (the plain layout's count: the repack is lossless), or 0 for an
 *   unsupported shape.
 * flint_moe_pack_dense: one-time repack on `stream` of
 *   codes  uint8 [N][K/2] (byte j of a row: element 2j low nibble, 2j+1 high)
 *   scales uint8 [N][K/16] (E4M3 per 16-element block)
 *   into packed (flint_moe_dense_packed_bytes(N, K) bytes).
 * flint_moe_dense_gemv: x bf16 [B][K], y bf16 [B][N]; 1 <= B <= 8 and
 *   B * K <= 32768 (else FLINT_MOE_ERR_UNSUPPORTED).  One kernel on `stream`
 *   (programmatic dependent launch: it requests its first weight tiles before
 *   waiting for the kernel before it), deterministic.  No workspace.
 */
size_t flint_moe_dense_packed_bytes(int N, int K);
int flint_moe_pack_dense(const uint8_t *codes, const uint8_t *scales, int N, int K, void *packed,
                         size_t packed_bytes, flint_moe_stream_t stream);
int flint_moe_dense_gemv(const void *packed, int N, int K, float tensor_scale, const void *x, int B,
                         void *y, flint_moe_stream_t stream);

/* Frees cached CUDA graphs of every device the calling thread used.  Call
 * before freeing buffers whose addresses a cached stack graph holds. */
int flint_moe_release(void);

/* Reads (and with reset != 0 clears) the current device's error word.  Bits:
 * 1, 2, 4 = a bounded wait gave up (full / empty barrier / draining copies);
 * 8 = the prefill router's tensor-core logit of some expert was further from
 * the exact value than its assumed error bound allows, and that token's
 * routing was recomputed from all 256 exact logits (results stay correct);
 * 16 = a prefill kernel found its shared memory misaligned and did nothing;
 * 32 = a persistent decode kernel's wait for data of its other thread blocks
 * ran out (flint_moe_set_wait_limit) and the call was abandoned.
 * Synchronises the device.  Returns the word (0 = none) or a negative
 * status. */
int flint_moe_device_error(int reset);

/* The current device's error word as a status: FLINT_MOE_OK (no bit, or only
 * bit 8), FLINT_MOE_ERR_TIMEOUT (bits 1, 2, 4 or 32: a bounded device wait
 * gave up and the outputs of the calls since the last reset are undefined),
 * FLINT_MOE_ERR_CUDA (bit 16, or a CUDA failure).  Synchronises the device;
 * reset != 0 clears the word. */
int flint_moe_device_status(int reset);

/* Selects the decode kernels of later NVFP4 calls (decode layer, stack and
 * the no-allocation call): FLINT_MOE_DECODE_CHAINED (default: router,
 * gate/up and down kernels chained with programmatic dependent launch) or
 * FLINT_MOE_DECODE_PERSISTENT (one cooperative kernel per up to 64
 * sublayers).  Both compute the same sublayer and pass the same parity
 * tests; BF16 weights always use the chained kernels.  Process-wide; returns
 * FLINT_MOE_OK or FLINT_MOE_ERR_INVALID_ARG for an unknown value. */
int flint_moe_set_decode_kernel(int kernel);

/* Cycle limit (SM clock) of every later persistent decode call's device-side waits
 * for data that its other thread blocks write.  A wait that runs out sets bit
 * 32 of the error word and ends the whole call early, with every thread block
 * returning and no copy left in flight.  The default, restored by
 * cycles <= 0, is about one second at the maximum SM clock.  Process-wide;
 * returns FLINT_MOE_OK.  Waits on the library's own bulk copies keep the
 * default limit. */
int flint_moe_set_wait_limit(long long cycles);

/* Static text for a status code. */
const char *flint_moe_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FLINT_MOE_H */
