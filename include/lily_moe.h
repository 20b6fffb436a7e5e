/*
 * lily_moe.h -- C ABI of the GB300 (sm_103a) W4 MoE expert-layer library.
 *
 * The layer (page "Lily Beats MLX-LM 1.35x on Decode: Perplexity's Rust+Metal
 * Engine for Apple Silicon", section "Model structure and three workload
 * shapes"; page "Revolutionizing Local AI Inference on Apple Silicon",
 * section "Understanding the Qwen3.6-35B-A3B Model"): a router scores
 * E experts per token and keeps the top k, plus one shared expert that every
 * token uses.  Experts are SwiGLU FFNs, y_t = sum_j g_tj FFN_{e_tj}(x_t) +
 * FFN_shared(x_t), whose weights are groupwise-affine 4-bit: every 64
 * consecutive input-dim weights of a row share one bf16 scale and one bf16
 * bias, w = scale*q + bias, q in 0..15 (same section).  Prefill runs the
 * routing histogram, prefix scan, scatter and block map on the GPU with no
 * host synchronisation, and a grouped GEMM that rebuilds weights one tile at
 * a time on chip with FP32 accumulation (section "Prefill: fusing
 * dequantisation and keeping routing GPU-resident").  Batch-1 decode is
 * bandwidth-bound (section "Decode: eliminating per-token CPU round trips").
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers unless a parameter says "host".  The caller
 *     owns every buffer.  Apart from the *_host and profiling entry points,
 *     the library never allocates, frees or synchronises; it launches only on
 *     `stream` (a cudaStream_t passed as void*, NULL = legacy default stream).
 *   - All device pointers must be 16-byte aligned.
 *   - bf16 values are passed as their 16-bit patterns (uint16_t).
 *   - Return value: LILY_OK (0) or a negative LILY_ERR_* code.  On an argument
 *     error nothing is launched.  No C++ exception crosses the ABI.
 *   - Errors found on the device (a NaN router logit, a bounded wait that ran
 *     out) never trap: they set bits of a status word kept in the workspace,
 *     read (and cleared) by lily_moe_status().
 *   - Calls are thread-safe for distinct workspaces; calls that share a
 *     workspace must be ordered on one stream.
 */
#ifndef LILY_MOE_H
#define LILY_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------- error codes */
#define LILY_OK 0
#define LILY_ERR_INVALID_ARG (-1)        /* NULL pointer, non-positive size    */
#define LILY_ERR_UNSUPPORTED_SHAPE (-2)  /* dims outside the supported ranges  */
#define LILY_ERR_MISALIGNED (-3)         /* a pointer is not 16-byte aligned   */
#define LILY_ERR_WORKSPACE_TOO_SMALL (-4)
#define LILY_ERR_ARCH (-5)               /* current device is not CC 10.3      */
#define LILY_ERR_CUDA (-6)               /* a CUDA runtime call or launch failed */
#define LILY_ERR_DEVICE (-7)             /* lily_moe_status: device status bits set */

/* Device status bits (lily_moe_status). */
#define LILY_STATUS_NAN_LOGIT 0x1u       /* a router logit was NaN             */
#define LILY_STATUS_TIMEOUT 0x2u         /* a bounded on-chip wait gave up     */
#define LILY_STATUS_BAD_TILE 0x4u        /* a block-map entry was out of range */
#define LILY_STATUS_F16_RANGE 0x8u       /* a value above 65504, the fp16 range
                                            of the tensor-core operands and the
                                            intermediate rows: |x|, |silu(g)*u|,
                                            or an expert output row value of the
                                            grouped GEMM path                   */

/* ------------------------------------------------------------------ shapes
 * T          tokens (rows) of this call; 1 <= T <= 16384 (decode: 1..8)
 * d_model    model width d; multiple of 128, 128 <= d <= 4096
 * n_experts  routed experts E; 1 <= E <= 256
 * top_k      k; 1 <= k <= min(E, 8)
 * d_ff       expert SwiGLU width F; multiple of 128, 128 <= F <= 4096
 * group      quantisation group; must be 64
 * tile_rows  BM, rows of one block-map tile (the grouped GEMM's N tile);
 *            one of 16, 32, 64, 128
 * out_dtype  element type of the layer output y: LILY_DTYPE_F32 (the fp32
 *            accumulator itself) or LILY_DTYPE_BF16 (rounded once)
 */
#define LILY_DTYPE_BF16 0
#define LILY_DTYPE_F32 1
typedef struct {
  int32_t T, d_model, n_experts, top_k, d_ff, group, tile_rows, out_dtype;
} lily_moe_dims;

/* Weights of one layer.  Expert index E (the (E+1)-th) is the shared expert.
 *   router_w  fp32 [E][d]            router_bias fp32 [E] or NULL
 *   gate_q, up_q  uint8 [E+1][F][d/2]   rows = output features; byte j of a row
 *                                      holds element 2j in bits 0-3 and 2j+1
 *                                      in bits 4-7
 *   gate_s, gate_b, up_s, up_b  bf16 [E+1][F][d/64]  scale / bias per group
 *   down_q    uint8 [E+1][d][F/2]
 *   down_s, down_b  bf16 [E+1][d][F/64]
 *   router_w_split  optional bf16 [3][E][d], 16-byte aligned: router_w split
 *              exactly into three bf16 terms (hi + mid + lo == w) by
 *              lily_moe_router_split.  The router (T > 8) runs on tensor cores
 *              against this split; given here it is made once per set of
 *              weights, else every call splits router_w into the workspace.
 *              The logits are the same bits either way.
 */
typedef struct {
  const float* router_w;
  const float* router_bias;
  const uint8_t* gate_q;
  const uint16_t* gate_s;
  const uint16_t* gate_b;
  const uint8_t* up_q;
  const uint16_t* up_s;
  const uint16_t* up_b;
  const uint8_t* down_q;
  const uint16_t* down_s;
  const uint16_t* down_b;
  const void* router_w_split;  // optional, see lily_moe_router_split; NULL = split per call
} lily_moe_weights;

/* Routing outputs, caller-owned device buffers (P = T*k pairs, pair p = t*k+j).
 *   logits     fp32 [T][E]   router logits (input when logits_in is given)
 *   topk_ids   int32 [T][k]  experts by (logit desc, id asc)
 *   topk_gates fp32 [T][k]   softmax over the kept logits
 *   counts     int32 [E]     pairs per expert (histogram)
 *   offsets    int32 [E+1]   exclusive prefix scan of counts; offsets[E] = P
 *   perm       int32 [P]     perm[r] = pair at expert-sorted row r; within an
 *                            expert pairs keep ascending pair index
 *   inv_perm   int32 [P]     inv_perm[p] = row of pair p
 *   block_map  int32 [cap][2] (expert, first row) of each tile of at most
 *                            tile_rows rows, experts ascending; unused = -1;
 *                            cap = lily_moe_block_map_cap()
 *   n_tiles    int32 [1]     number of valid block_map entries
 */
typedef struct {
  float* logits;
  int32_t* topk_ids;
  float* topk_gates;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv_perm;
  int32_t* block_map;
  int32_t* n_tiles;
} lily_moe_routing;

/* Bytes of device workspace a call with these dims needs (0 on bad dims).
 * The workspace must be zero-filled once before its first use; the library
 * keeps it consistent afterwards (its counters return to zero after a call). */
size_t lily_moe_workspace_bytes(const lily_moe_dims* dims);

/* Entries of routing->block_map: ceil(T*k / tile_rows) + min(E, T*k). */
int64_t lily_moe_block_map_cap(const lily_moe_dims* dims);

/* Check dims against the supported ranges above: LILY_OK or an error code. */
int lily_moe_check_dims(const lily_moe_dims* dims);

/* Routing only: router logits (unless logits_in != NULL), top-k and gates,
 * histogram, prefix scan, stable scatter and block map, all on `stream`
 * without host synchronisation.
 *   x          bf16 [T][d] device (ignored when logits_in != NULL)
 *   logits_in  fp32 [T][E] device or NULL; when given, routing starts from
 *              these logits (they are copied to routing->logits)
 *   weights    only router_w / router_bias are read (may be NULL with logits_in) */
int lily_moe_route(const lily_moe_dims* dims, const void* x, const float* logits_in,
                   const lily_moe_weights* weights, lily_moe_routing* routing,
                   void* workspace, size_t workspace_bytes, void* stream);

/* The whole layer for prefill-sized T: routing as in lily_moe_route, then the
 * gate/up grouped GEMM (fused 4-bit dequant + SwiGLU) and the down grouped GEMM
 * (fused dequant; each expert output row is stored as fp16 in expert-sorted
 * order), then the combine of each token's k + 1 rows, weighted by their
 * routing gates, in a fixed order back into token order, so y is the same
 * bits on every run.
 *   x  bf16 [T][d] device in; y [T][d] device out, fp32 or bf16 per
 *   dims->out_dtype. */
int lily_moe_forward(const lily_moe_dims* dims, const void* x,
                     const lily_moe_weights* weights, lily_moe_routing* routing,
                     void* y, void* workspace, size_t workspace_bytes, void* stream);

/* The expert part of lily_moe_forward alone: the gate/up and down grouped
 * GEMMs (shared expert included) from routing already in `routing` --
 * topk_gates, offsets, perm, block_map and n_tiles as lily_moe_route writes
 * them, e.g. from that call or built by the caller (page "Revolutionizing
 * Local AI Inference on Apple Silicon", section "Enhanced Tile and Scan
 * Operations": the dispatch tables feed the expert GEMMs).  With the same
 * routing the result equals lily_moe_forward's.  A perm entry outside
 * [0, T*k) or a block-map tile outside the pairs sets LILY_STATUS_BAD_TILE
 * and is clamped, never read out of bounds.
 *   x  bf16 [T][d] device in; y [T][d] device out, fp32 or bf16 per
 *   dims->out_dtype. */
int lily_moe_experts(const lily_moe_dims* dims, const void* x,
                     const lily_moe_weights* weights, const lily_moe_routing* routing,
                     void* y, void* workspace, size_t workspace_bytes, void* stream);

/* Same result as lily_moe_forward for T = 1..8 rows (batch-1 decode and
 * speculative-verify sizes), through the bandwidth-bound W4 GEMV path that
 * streams each distinct active expert's weights once. */
int lily_moe_decode(const lily_moe_dims* dims, const void* x,
                    const lily_moe_weights* weights, lily_moe_routing* routing,
                    void* y, void* workspace, size_t workspace_bytes, void* stream);

/* lily_moe_decode without a caller workspace.  The Lily pages have no
 * counterpart to this call; it exists for callers that cannot allocate device
 * memory: a host application that passes this library only its activation
 * and weight buffers while keeping all other device memory under its own
 * accounting, or a token loop that must not enter the CUDA allocator between
 * tokens.  Same arguments and result as lily_moe_decode minus the workspace.
 *   - Scratch comes from one array of 1 MiB declared at file scope in the
 *     library; every device that loads the library holds it until the
 *     process exits.  T > 8 is refused with LILY_ERR_UNSUPPORTED_SHAPE, and
 *     dims whose workspace (lily_moe_workspace_bytes) exceeds 1 MiB with
 *     LILY_ERR_WORKSPACE_TOO_SMALL, both before any launch.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - Every call shares the one array, which keeps the previous call's
 *     contents; each call clears the part that must start at zero (the status
 *     and barrier words).  Calls that overlap on the GPU (other streams, other
 *     host threads) race on the array and must be ordered by the caller.
 *   - Device status bits are cleared at the start of each call and cannot be
 *     read back through this entry point. */
int lily_moe_decode_static(const lily_moe_dims* dims, const void* x,
                           const lily_moe_weights* weights, lily_moe_routing* routing,
                           void* y, void* stream);

/* End-to-end form of lily_moe_forward (T >= 9) / lily_moe_decode (T <= 8) for
 * callers holding activations in HOST memory: copies x_host (bf16 [T][d]) to
 * x_dev, runs the layer, copies y_dev back into y_host and synchronises
 * `stream` before returning.  x_dev/y_dev are device staging buffers of T*d
 * elements (bf16 for x, out_dtype for y).
 *   - Copies are cudaMemcpyAsync on `stream`; page-locked host buffers
 *     (cudaHostAlloc / cudaHostRegister) copy fastest.
 *   - With both host buffers page-locked, the first call with a given
 *     argument set (dims and every pointer, on the current device) runs
 *     eagerly and then captures the whole copy-layer-copy sequence as a CUDA
 *     graph on a stream of the library's own; later calls with the same
 *     arguments replay that graph on `stream`.  The graph reads every buffer
 *     by address: contents may change between calls, and a buffer freed and
 *     re-allocated at the same address is simply reused.  At most 128 graphs
 *     are kept (least recently used evicted); lily_moe_host_graphs(0) drops
 *     them all and turns the cache off.  Calls made while per-kernel
 *     profiling is enabled always run eagerly. */
int lily_moe_forward_host(const lily_moe_dims* dims, const void* x_host, void* x_dev,
                          const lily_moe_weights* weights, lily_moe_routing* routing,
                          void* y_dev, void* y_host, void* workspace,
                          size_t workspace_bytes, void* stream);

/* lily_moe_forward_host without the final wait: once the argument set's
 * graph is cached (page-locked host buffers, second and later calls), the
 * call only queues the copy-layer-copy graph on `stream` and returns; y_host
 * holds the result once `stream` has been synchronised.  Until then none of
 * x_host, x_dev, y_dev, y_host, the routing buffers or the workspace may be
 * reused or freed.  A first call (or a call while profiling is on, or with a
 * pageable host buffer) runs as lily_moe_forward_host does, synchronously.
 * Calls on different streams with disjoint buffers overlap one call's copies
 * with another's kernels.  Same arguments and errors as lily_moe_forward_host. */
int lily_moe_forward_host_async(const lily_moe_dims* dims, const void* x_host, void* x_dev,
                                const lily_moe_weights* weights, lily_moe_routing* routing,
                                void* y_dev, void* y_host, void* workspace,
                                size_t workspace_bytes, void* stream);

/* Turn the end-to-end graph cache on (enable != 0, the default) or off; either
 * way every cached graph is destroyed.  Returns the previous setting (0/1). */
int lily_moe_host_graphs(int enable);

/* The exact three-term bf16 split of a router weight matrix (see
 * lily_moe_weights.router_w_split), written to `split` on `stream`.
 *   router_w  fp32 [n_experts][d_model] device, 16-byte aligned
 *   split     device, lily_moe_router_split_bytes(n_experts, d_model) bytes,
 *             16-byte aligned, caller-owned
 * Weights are static between calls, so a caller splits once after loading
 * them (as it packs the 4-bit codes).  Errors: LILY_ERR_INVALID_ARG,
 * LILY_ERR_UNSUPPORTED_SHAPE (d_model not a multiple of 128 in [128, 4096],
 * n_experts > 256), LILY_ERR_MISALIGNED, LILY_ERR_CUDA. */
size_t lily_moe_router_split_bytes(int32_t n_experts, int32_t d_model);
int lily_moe_router_split(const float* router_w, int32_t n_experts, int32_t d_model,
                          void* split, void* stream);

/* Unit-weight RMSNorm, out = bf16(x / sqrt(mean(x^2) + eps)), x fp32 [T][d],
 * out bf16 [T][d].  The pre-norm of the stacked-layer prefill. */
int lily_moe_rmsnorm(int32_t T, int32_t d, const float* x, float eps, void* out_bf16,
                     void* stream);

/* Stacked prefill: n_layers MoE layers with residual, in chunks of `chunk`
 * tokens (dims->T is the chunk size; T_total a multiple of it):
 *   for each chunk, for l in 0..n_layers-1:
 *     x <- x + MoE_l(bf16(rmsnorm(x)))      (MoE output added in fp32)
 * x fp32 [T_total][d] device, updated in place.  layers[l] are the weights of
 * layer l.  layer_inputs (fp32 [n_layers][T_total][d]) and layer_logits
 * (fp32 [n_layers][T_total][E]) are optional device traces (NULL to skip).
 * Long prompts are run in bounded chunks (section "Prefill: fusing
 * dequantisation and keeping routing GPU-resident"). */
int lily_moe_stack_prefill(const lily_moe_dims* dims, int32_t T_total, int32_t n_layers,
                           const lily_moe_weights* layers, float* x, float eps,
                           float* layer_inputs, float* layer_logits,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes for lily_moe_stack_prefill with chunk size dims->T, and
 * for lily_moe_stack_decode with dims->T rows. */
size_t lily_moe_stack_workspace_bytes(const lily_moe_dims* dims);

/* Stacked decode step: n_layers MoE layers with residual for dims->T = 1..8
 * rows (one token per sequence, or a speculative-verify batch):
 *   for l in 0..n_layers-1:  x <- x + MoE_l(bf16(rmsnorm(x)))
 * x fp32 [T][d] device, updated in place; layers[l] are the weights of layer
 * l; dims->out_dtype is ignored (the layer output is added in fp32).  Each
 * layer is three launches -- the router (RMSNorm, logits and the routing, in
 * one cluster of CTAs), the gate/up GEMV and the down GEMV, which adds its
 * output into x -- every one chained to the previous with programmatic
 * dependent launch, so the whole step runs with no host work between layers
 * and can be captured in one CUDA graph (page "Lily Beats MLX-LM 1.35x on
 * Decode: Perplexity's Rust+Metal Engine for Apple Silicon", section
 * "Decode: eliminating per-token CPU round trips": a decode step recorded
 * once and replayed, its kernels ordered only by their real data
 * dependencies).  layer_inputs (fp32 [n_layers][T][d]) and layer_logits
 * (fp32 [n_layers][T][E]) are optional device traces (NULL to skip; the
 * input trace adds a copy per layer).  Workspace: lily_moe_stack_workspace_bytes. */
int lily_moe_stack_decode(const lily_moe_dims* dims, int32_t n_layers,
                          const lily_moe_weights* layers, float* x, float eps,
                          float* layer_inputs, float* layer_logits, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Synchronises `stream`, returns the device status bits accumulated in the
 * workspace since the last call (0 = none) and clears them; after a
 * LILY_STATUS_TIMEOUT it also zeroes the workspace's grid-barrier counters.
 * Negative on a CUDA error. */
int lily_moe_status(void* workspace, void* stream);

/* Give-up limit, in nanoseconds, of the one wait in the routing kernel that
 * spans blocks (its grid barrier, used when T > 32): 2 s by default.  Returns
 * the previous limit.  A block whose wait runs out sets LILY_STATUS_TIMEOUT and
 * writes none of its tokens' scatter outputs (perm, inv_perm; counts, offsets
 * and block_map too if it is block 0), so that call's routing is invalid.
 * For tests of the error path; 0 makes every waiting block give up at once.
 * Applies to calls issued after it; the waits of the GEMM kernels keep 2 s. */
uint64_t lily_moe_set_route_wait_ns(uint64_t ns);

/* Static text for an error code. */
const char* lily_moe_strerror(int code);

/* ---------------------------------------------------------------- profiling
 * Per-kernel device time of the calls above, measured with CUDA events
 * recorded on the launch stream around every kernel while enabled.  Kernel
 * kinds are numbered; lily_moe_kernel_name() names them. */
#define LILY_KERNEL_KINDS 16
int lily_moe_profile_enable(int enable);
/* Synchronises the recorded events; fills total_ms[kind] and launches[kind]
 * (arrays of LILY_KERNEL_KINDS) and resets the counters. */
int lily_moe_profile_read(double* total_ms, int64_t* launches);
const char* lily_moe_kernel_name(int kind);

/* Library version, e.g. "lily_moe 0.1 sm_103a". */
const char* lily_moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* LILY_MOE_H */
