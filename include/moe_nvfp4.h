/*
 * moe_nvfp4.h -- C ABI of the fused NVFP4 Mixture-of-Experts layer for one
 * GB300 GPU (sm_103a).
 *
 * The layer (pages: "vLLM on the NVIDIA DGX Spark: A Complete Technical
 * Guide", sections 4.3, 6.1 and 7.1; "Serving Solar Open 2 on DGX Spark",
 * "Solar Open 2 in brief" and "The fix"):
 *
 *   route     softmax over E routed experts, top-k, weights renormalised
 *   permute   (token, slot) pairs grouped by expert, stable
 *   quantise  BF16 -> NVFP4 (W4A4 only)
 *   GEMM 1    [gate | up] = x W13^T over NVFP4 weights, SwiGLU epilogue
 *   GEMM 2    y = h W2^T, routing weight in the epilogue
 *   combine   out[t] = sum_j y[(t, j)] + y_shared[t]
 *
 * NVFP4 ("vLLM on the NVIDIA DGX Spark", section 6.1): e2m1 elements packed
 * two per byte (element 2j in the low nibble of byte j), one FP8 E4M3 block
 * scale per 16 consecutive elements along K, one fp32 global scale per
 * tensor. Global scales cross this ABI in the *quant* convention
 * gs = (448 * 6) / amax ("GLM-5.3-Flash-NVFP4 #4" discussion, follow-up on
 * the MoE fault); a value decodes as e2m1 * e4m3 / gs.
 *
 * Conventions for every call:
 *  - Pointers are device pointers unless a comment says "host". The caller
 *    owns every buffer; no call allocates or frees device memory on the
 *    compute path. Scratch comes from a caller-provided workspace.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream). Argument errors are found on the host and returned
 *    before anything is enqueued. Anomalies only visible on the device
 *    (an expert id out of range, say) set an error word inside the
 *    workspace; moe_get_device_status() reads it. A workspace's first 256
 *    bytes must be zero before its first use; afterwards the library
 *    maintains them (the status word, scale slots and the single-kernel
 *    decode path's launch ticket and flags), so they need not be cleared
 *    again, and the rest of a workspace needs no initialisation. A
 *    workspace serves one call at a time: calls that may run at the same
 *    time (on different streams, say) need different workspaces.
 *  - Only sm_103 devices are supported; anything else returns
 *    MOE_ERR_UNSUPPORTED. No call traps or aborts the process.
 *  - Matrices are row-major with the contraction dimension K contiguous.
 *    bf16 values travel as uint16_t bit patterns.
 */
#ifndef MOE_NVFP4_H
#define MOE_NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* the same type as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* bad pointer, size, scale or layout */
  MOE_ERR_UNSUPPORTED = 2, /* size outside the kernels' limits, or not sm_103 */
  MOE_ERR_CUDA = 3,        /* a CUDA runtime call failed (see moe_last_cuda_error) */
  MOE_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required */
  MOE_ERR_TIMEOUT = 5,     /* a bounded device wait gave up */
  MOE_ERR_DEVICE = 6       /* the device flagged bad data (e.g. expert id out of range) */
} moe_status;

typedef enum {
  MOE_W4A16 = 0, /* NVFP4 weights, bf16 activations (weight-only) */
  MOE_W4A4 = 1,  /* NVFP4 weights and activations (block-scaled FP4 MMA) */
  MOE_MXFP4 = 2  /* MXFP4 weights and activations: e2m1 with one power-of-two
                    E8M0 scale per 32 along K, no global scale ("vLLM on the
                    NVIDIA DGX Spark", section 6.4 "NVFP4 vs MXFP4");
                    block-scaled FP4 MMA with UE8M0 scales */
} moe_mode;

/* Human-readable name of a status code (static string, never NULL). */
const char* moe_status_string(moe_status s);

/* The last CUDA error string seen by this library in this thread (static). */
const char* moe_last_cuda_error(void);

/* ------------------------------------------------------------------------
 * Router.  "Serving Solar Open 2 on DGX Spark", "Solar Open 2 in brief"
 * (top-k routing over routed experts); "vLLM on the NVIDIA DGX Spark",
 * section 7.1 ([Router] stage).
 *
 * logits   fp32 [T, E]
 * topk_ids int32 [T, k] out: experts by rank; higher logit first, equal
 *          logits by lower expert index
 * topk_w   fp32 [T, k] out: softmax probabilities of the chosen experts
 *          renormalised to sum to 1
 * Limits: 1 <= E <= 1024, 1 <= k <= min(E, 32), T >= 0 (T = 0 is a no-op).
 * NaN logits are outside the contract (results unspecified, no fault).
 */
moe_status moe_route_topk(const float* logits, int T, int E, int k,
                          int32_t* topk_ids, float* topk_w, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Router GEMM ahead of the top-k ("vLLM on the NVIDIA DGX Spark", section
 * 7.1, the [Router] stage): logits = x . W_router^T.
 *
 * x        bf16 [T, H], 16-byte aligned (device)
 * w_router bf16 [E, H], 16-byte aligned (device); the router matrix is kept
 *          16-bit, it is not one of the NVFP4 expert weights
 * logits   fp32 [T, E] out (device)
 * Products are exact in fp32 and summed in fp32 in an order fixed by the
 * shapes (the same bits on every run; the order differs from a sequential
 * sum, so values differ from one by accumulated fp32 rounding).
 * Errors: T < 0, H <= 0, E < 1, a NULL pointer -> MOE_ERR_INVALID_ARG;
 * H % 8 != 0 or misaligned rows -> MOE_ERR_INVALID_ARG; T = 0 -> MOE_OK with
 * nothing enqueued.
 */
moe_status moe_router_gemm(const uint16_t* x, const uint16_t* w_router, int T, int H, int E,
                           float* logits, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Permutation into expert-contiguous groups.  "vLLM on the NVIDIA DGX
 * Spark", section 4.3 (token dispatch) and section 7.1
 * ([Permute-Experts-Unpermute]).
 *
 * Pair p = t*k + j is routed to expert topk_ids[p]. Outputs:
 * counts   int32 [E]    pairs per expert
 * offsets  int32 [E+1]  exclusive prefix sum of counts; offsets[E] = T*k
 * perm     int32 [T*k]  sorted position -> pair; ascending p within a group
 * inv_perm int32 [T*k]  pair -> sorted position
 * ws       scratch of at least moe_permute_workspace_size(T, k, E) bytes
 * An id outside [0, E) sets MOE_ERR_DEVICE in the workspace status word
 * (read it with moe_get_device_status); such pairs are dropped.
 */
size_t moe_permute_workspace_size(int T, int k, int E);
moe_status moe_permute(const int32_t* topk_ids, int T, int k, int E,
                       int32_t* counts, int32_t* offsets, int32_t* perm,
                       int32_t* inv_perm, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/* ------------------------------------------------------------------------
 * BF16 -> NVFP4 quantisation with a dynamic per-tensor global scale.
 * "vLLM on the NVIDIA DGX Spark", sections 4.3 (BF16 input quantised to FP4
 * inside the fused kernel) and 6.1 (format); the 448 clamp of the block
 * scale is from "Serving Solar Open 2 on DGX Spark", "Supporting real NVFP4
 * checkpoints".
 *
 * Steps, each a correctly rounded fp32 operation:
 *   amax = max |x|; gs = 2688 / amax (gs = 1 when amax = 0)
 *   per 16-element block: s = (max|x_i| / 6) * gs; sf = E4M3(s), round to
 *   nearest even, saturating at 448; if sf = 0 the codes are 0, otherwise
 *   code_i = e2m1(x_i * (gs / sf)), nearest even, saturating at 6, sign kept.
 *
 * x      bf16 [rows, K], K % 16 == 0
 * q      uint8 [rows, K/2] out, packed codes (element 2j in the low nibble)
 * sf     uint8 [rows, K/16] out, E4M3 block scales
 * gs_out fp32 [1] out (device)
 * ws     scratch of at least moe_quantize_workspace_size() bytes
 */
size_t moe_quantize_workspace_size(void);
moe_status moe_nvfp4_quantize(const uint16_t* x, int rows, int K, uint8_t* q,
                              uint8_t* sf, float* gs_out, void* ws, size_t ws_bytes,
                              moe_stream_t stream);

/* The same quantisation with a static (calibrated) global scale gs in place
 * of the dynamic 2688 / amax ("Serving Solar Open 2 on DGX Spark", "The
 * fix": static and dynamic NVFP4 W4A4 paths; "GLM-5.3-Flash-NVFP4 #4":
 * calibrated per-projection input scales). gs is a host float in the quant
 * convention (moe_import_global_scale turns a checkpoint's stored value into
 * it). Blocks whose (max|x_i| / 6) * gs exceeds 448 saturate: the block scale
 * clamps at 448 and the codes at 6. Errors: gs <= 0 or non-finite, and the
 * size and pointer errors of moe_nvfp4_quantize -> MOE_ERR_INVALID_ARG.
 */
moe_status moe_nvfp4_quantize_static(const uint16_t* x, int rows, int K, float gs,
                                     uint8_t* q, uint8_t* sf, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * BF16 -> MXFP4 ("vLLM on the NVIDIA DGX Spark", section 6.4 "NVFP4 vs
 * MXFP4": e2m1 elements, blocks of 32 along K, one E8M0 power-of-two scale
 * per block, no per-tensor scale). Per block: e = floor(log2 max|x_i|) - 2,
 * clamped to [-127, 127] (so max|x_i| / 2^e lies in [4, 8)); an all-zero
 * block takes e = -127 and zero codes; sf = e + 127; code_i = e2m1(x_i *
 * 2^-e), nearest even, saturating at 6, sign kept (the multiply is exact).
 *
 * x  bf16 [rows, K], K % 32 == 0, 16-byte aligned
 * q  uint8 [rows, K/2] out, packed codes (element 2j in the low nibble),
 *    16-byte aligned
 * sf uint8 [rows, K/32] out, E8M0 scale codes
 * Errors: K % 32 != 0, a NULL or misaligned pointer -> MOE_ERR_INVALID_ARG;
 * rows = 0 -> MOE_OK with nothing enqueued.
 */
moe_status moe_mxfp4_quantize(const uint16_t* x, int rows, int K, uint8_t* q, uint8_t* sf,
                              moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Checkpoint import ("Serving Solar Open 2 on DGX Spark", "Supporting real
 * NVFP4 checkpoints"; "GLM-5.3-Flash-NVFP4 #4" discussion, follow-up on the
 * MoE fault).
 *
 * Checkpoints store a tensor's global scale in one of two conventions:
 * ModelOpt keeps the dequant scale amax / (448*6) (weight_scale_2,
 * input_scale), compressed-tensors the quant scale (448*6) / amax
 * (global_scale). This library takes the quant convention everywhere.
 *
 * moe_import_global_scale (host only, no GPU work): gs_out = stored for
 * MOE_SCALE_QUANT, the fp32 reciprocal 1 / stored (correctly rounded) for
 * MOE_SCALE_DEQUANT. stored <= 0 or non-finite -> MOE_ERR_INVALID_ARG (a zero
 * scale silently zeroes every expert, the fault of the GLM thread); an
 * unknown format -> MOE_ERR_INVALID_ARG.
 *
 * moe_nvfp4_fold_scales (one-time, synchronous): moves n E4M3 block scales
 * to another global scale, sf_out[i] = E4M3(e4m3[sf_in[i]] * ratio) with one
 * correctly rounded fp32 multiply, nearest even, clamped at 448; use ratio =
 * gs_new / gs_old to express a matrix in the global scale gs_new (for
 * example one scale shared by a fused gate/up pair). A scale that underflows
 * becomes 0 and zeroes its block. sf_in and sf_out are device arrays (they
 * may be the same array). Errors: a NULL pointer, ratio <= 0 or non-finite,
 * or any input code with its sign bit set or a NaN code (0x7F/0xFF) ->
 * MOE_ERR_INVALID_ARG (sf_out then holds the converted codes with the bad
 * ones copied unchanged). n = 0 -> MOE_OK. The call synchronises the stream.
 */
typedef enum {
  MOE_SCALE_QUANT = 0,   /* stored value is (448*6) / amax */
  MOE_SCALE_DEQUANT = 1  /* stored value is amax / (448*6) */
} moe_scale_format;

moe_status moe_import_global_scale(float stored, moe_scale_format format, float* gs_out);
moe_status moe_nvfp4_fold_scales(const uint8_t* sf_in, size_t n, float ratio, uint8_t* sf_out,
                                 moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Weight preparation (one-time, synchronous).  "Serving Solar Open 2 on DGX
 * Spark", "Supporting real NVFP4 checkpoints" (checkpoint weights are
 * converted once into the kernels' tile layout, with gate/up ordering).
 *
 * Converts one linear NVFP4 matrix into the opaque tile layout the GEMMs
 * read. codes uint8 [N, K/2] (packed), sf uint8 [N, K/16] (E4M3), both
 * device. gs is a HOST array of fp32 global scales (quant convention): one
 * entry for a plain matrix, two (gate, up) when gate_up != 0, in which case
 * the N rows are [gate (N/2 rows); up (N/2 rows)]. out must hold
 * moe_prepare_size(N, K, mode, gate_up) bytes, 256-byte aligned.
 * MOE_MXFP4: sf is uint8 [N, K/32] E8M0 codes (moe_mxfp4_quantize), gs is
 * not read (may be NULL), K % 256 == 0, and code 0xFF (NaN) is refused.
 * Errors: gs <= 0 or non-finite (a zero scale would silently zero every
 * expert output, the failure described in "GLM-5.3-Flash-NVFP4 #4"), a block
 * scale with its sign bit set or a NaN code, N % 128 != 0 (N/2 % 64 for
 * gate_up), K % 64 != 0 -> MOE_ERR_INVALID_ARG. The call synchronises the
 * stream.
 */
size_t moe_prepare_size(int N, int K, moe_mode mode, int gate_up);
moe_status moe_nvfp4_prepare_weights(const uint8_t* codes, const uint8_t* sf,
                                     const float* gs, int N, int K, moe_mode mode,
                                     int gate_up, void* out, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Grouped GEMM over prepared NVFP4 weights.  "vLLM on the NVIDIA DGX
 * Spark", section 4.3 (the two GEMMs of the fused MoE, SwiGLU and top-k
 * weight reduction fused) and section 6.1 (alpha = 1 / (gs_a * gs_w)).
 *
 * Output row r belongs to group g when group_offsets[g] <= r <
 * group_offsets[g+1]; group g multiplies by prepared block g of `weights`
 * (blocks are moe_prepare_size(N, K, mode, gate_up) bytes apart), except
 * that the last group uses `last_weights` when it is not NULL (the shared
 * expert). Row r reads A row a_row_index[r] (or r when NULL).
 *
 * gate_up = 1: the weights are a prepared [gate; up] pair (N = 2*I); the
 *   epilogue writes h = silu(x Wg^T / gs) * (x Wu^T / gs) as bf16 [rows, I].
 * gate_up = 0: the epilogue writes y = (x W^T / gs) * row_scale[r] as bf16
 *   [rows, N] (row_scale NULL means 1).
 * W4A16: a is bf16 [a_rows, K]. W4A4: a is packed NVFP4 [a_rows, K/2] with
 *   E4M3 scales a_sf [a_rows, K/16] and device global scale a_gs.
 * out_amax (nullable, device fp32, must start at 0): W4A4 gate/up only (the
 *   W4A16 kernels do not write it): atomically maxed with |out| (as stored),
 *   to feed the next quantisation.
 * rows: the number of output rows, group_offsets[num_groups], or 0. A call
 *   that gives it together with a workspace of at least
 *   moe_gemm_workspace_size_rows(num_groups, rows, K) bytes runs the kernels
 *   of moe_nvfp4_forward, which read the activations in group order as
 *   tensor-map tiles: W4A16 first copies the rows, gathered through
 *   a_row_index, into the workspace as f16 with a power-of-two scale per row
 *   (groups of more than 32 rows then run the TMA-fed tensor-core GEMM);
 *   W4A4 gathers the codes into the workspace (without a_row_index they are
 *   read in place) and assembles the scales into per-tile tcgen05 atoms.
 *   Otherwise (rows = 0 or a smaller workspace) the large groups run
 *   tensor-core kernels that gather rows inside the GEMM, at a lower rate.
 *   A larger rows value only costs workspace (rows past group_offsets[
 *   num_groups] are neither read nor computed); a smaller one makes the
 *   large-group GEMM record MOE_ERR_DEVICE in the workspace status word and
 *   write nothing.
 * ws: scratch of at least moe_gemm_workspace_size(num_groups) bytes.
 * Limits: K % 64 == 0, N % 128 == 0, num_groups <= 1025. MOE_MXFP4 ->
 * MOE_ERR_UNSUPPORTED here (MXFP4 layers run through moe_nvfp4_forward).
 */
typedef struct {
  moe_mode mode;
  int gate_up;
  int num_groups;
  int N, K;
  const void* weights;
  const void* last_weights;
  const int32_t* group_offsets;
  const void* a;
  const uint8_t* a_sf;
  const float* a_gs;
  const int32_t* a_row_index;
  const float* row_scale;
  uint16_t* out;
  float* out_amax;
  int rows;
} moe_gemm_args;

size_t moe_gemm_workspace_size(int num_groups);
/* Workspace bytes for the activation copies described under `rows` above,
 * enough for either mode (0 for a negative argument or K <= 0). */
size_t moe_gemm_workspace_size_rows(int num_groups, int rows, int K);
moe_status moe_nvfp4_grouped_gemm(const moe_gemm_args* args, void* ws, size_t ws_bytes,
                                  moe_stream_t stream);

/* ------------------------------------------------------------------------
 * SwiGLU on a materialised gate/up product ("vLLM on the NVIDIA DGX Spark",
 * section 4.3). gu fp32 [rows, 2*I] with gate in columns [0, I) and up in
 * [I, 2I); h bf16 [rows, I] = silu(gate) * up, silu(z) = z / (1 + e^-z).
 * The fused path does this inside GEMM 1's epilogue; this call is the
 * standalone step.
 */
moe_status moe_swiglu(const float* gu, int rows, int I, uint16_t* h,
                      moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Combine back to token order ("vLLM on the NVIDIA DGX Spark", section 7.1
 * [Combine]; section 4.3 top-k weight reduction). Deterministic: fp32 sums
 * in the fixed order j = 0..k-1, then the shared row, rounded once to bf16.
 *
 * y        bf16 [T*k, H]: the routed rows in sorted (grouped) order
 * inv_perm int32 [T*k] pair -> sorted row; a negative entry (a dropped pair)
 *          contributes nothing
 * topk_w   fp32 [T, k] or NULL: multiplies row (t, j) (NULL when GEMM 2
 *          already applied the routing weight)
 * y_shared fp32 [T, H] or NULL: the shared expert's rows, added with weight
 *          1 (kept in fp32: with weight 1 their bf16 rounding would be the
 *          largest single error term of the output)
 * out      bf16 [T, H]
 * Errors: T < 0, k < 1, H <= 0 or H % 8 != 0, a NULL y / inv_perm / out, or
 * a pointer that is not 16-byte aligned -> MOE_ERR_INVALID_ARG; T = 0 ->
 * MOE_OK with nothing enqueued.
 */
moe_status moe_combine(const uint16_t* y, const int32_t* inv_perm, const float* topk_w,
                       const float* y_shared, int T, int k, int H, uint16_t* out,
                       moe_stream_t stream);

/* ------------------------------------------------------------------------
 * The whole layer. Weights come prepared (moe_nvfp4_prepare_weights):
 * w13 holds E gate/up blocks, w2 E down blocks, back to back; the shared
 * expert's blocks are separate and may be NULL (no shared expert).
 *
 * w_router (nullable): bf16 [E, H] router matrix, 16-byte aligned. When it
 *   is set the forward computes the logits itself (moe_router_gemm) and its
 *   `logits` argument may be NULL (it is ignored).
 * x_global_scale, h_global_scale (W4A4 only; 0 = dynamic): static
 *   calibrated global scales (quant convention) for the two activation
 *   quantisations, x before GEMM 1 and h before GEMM 2, in place of the
 *   dynamic 2688 / amax. Must be 0 on W4A16 and MXFP4 layers.
 * expert_offset, local_experts (expert parallelism; "Serving Solar Open 2
 *   on DGX Spark", "Adding Expert Parallelism to b12x": each node holds a
 *   contiguous shard of the experts, global expert ids are remapped to
 *   shard-local ones and out-of-shard pairs are filtered out): the router
 *   still ranks all E experts (logits [T, E], topk_ids_out global ids), but
 *   only pairs routed to experts [expert_offset, expert_offset +
 *   local_experts) are computed, with w13 / w2 holding just those
 *   local_experts blocks. out is then this shard's partial output: the sum
 *   over the shard's pairs (with their routing weights) plus the shared
 *   expert if this shard carries one (give the shared expert to exactly one
 *   shard). Summing the shards' outputs gives the layer's output. With
 *   dynamic W4A4 scales the h scale is the shard's own (the amax of its rows).
 *   local_experts = 0 means all E experts (expert_offset must be 0).
 * mode MOE_MXFP4: weights prepared with MOE_MXFP4; x and h (rounded to bf16)
 *   are quantised to MXFP4 (moe_mxfp4_quantize's steps) and both GEMMs run
 *   block-scaled FP4 MMA with UE8M0 scales; H % 256 == 0 and I % 256 == 0.
 */
typedef struct {
  int T, H, I, I_shared, E, k;
  moe_mode mode;
  const void* w13;
  const void* w2;
  const void* w13_shared;
  const void* w2_shared;
  const uint16_t* w_router;
  float x_global_scale;
  float h_global_scale;
  int expert_offset;   /* expert parallelism: this forward computes experts  */
  int local_experts;   /* [expert_offset, expert_offset + local_experts) of E; */
                       /* 0 = all E (no sharding)                             */
} moe_layer_desc;

/* Workspace bytes moe_nvfp4_forward needs for this descriptor. */
size_t moe_workspace_size(const moe_layer_desc* L);

/* x bf16 [T, H], logits fp32 [T, E] (or NULL with L->w_router) -> out bf16
 * [T, H]; topk_ids_out (nullable) int32 [T, k] receives the routing. ws must
 * hold moe_workspace_size(L) bytes, 256-byte aligned. Errors: a scale in
 * x_global_scale / h_global_scale that is negative or non-finite, or nonzero
 * on a W4A16 layer -> MOE_ERR_INVALID_ARG; a misaligned w_router or H % 8 != 0
 * with it -> MOE_ERR_INVALID_ARG.
 *
 * Decode batches (W4A16, T <= 8) run as one kernel ("micro path", "Serving
 * Solar Open 2 on DGX Spark", "The fix"; "vLLM on the NVIDIA DGX Spark",
 * section 4.3): routing, permutation, both GEMMs and the combine in a single
 * cooperative launch of one CTA per SM, after one small memset of its
 * counters (plus the router GEMM first when w_router is set). It needs the
 * whole GPU: another kernel occupying SMs at launch time makes the launch
 * fail with MOE_ERR_CUDA rather than wait. Its output equals the
 * multi-kernel path's bit for bit. */
moe_status moe_nvfp4_forward(const moe_layer_desc* L, const uint16_t* x, const float* logits,
                             uint16_t* out, int32_t* topk_ids_out, void* ws, size_t ws_bytes,
                             moe_stream_t stream);

/* Synchronises `stream`, returns and clears the device status word kept in
 * the first bytes of a workspace used by the calls above. */
moe_status moe_get_device_status(void* ws, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Measurement hooks (no counterpart in the pages; used by the benchmark).
 *
 * moe_set_stage_events: `events` is a HOST array of n >= MOE_STAGE_COUNT
 * cudaEvent_t handles owned by the caller. The next moe_nvfp4_forward call
 * on this host thread records events[0] before its first kernel and
 * events[i] after stage i (route, permute, quantise x, GEMM 1, quantise h,
 * GEMM 2, combine; a stage the mode does not run records at the same point
 * as the previous one; with w_router the router GEMM belongs to the route
 * stage), all on the call's stream; the setting is then
 * cleared. Pass NULL to clear it explicitly. On the single-kernel decode
 * path events[0] is recorded right before that kernel and events[1..] right
 * after it, so stage 0 -> 1 times the kernel alone.
 *
 * moe_kernel_launches: number of kernels this library has launched in this
 * process so far (all threads).
 */
#define MOE_STAGE_COUNT 8
moe_status moe_set_stage_events(void* const* events, int n);
unsigned long long moe_kernel_launches(void);

/* ------------------------------------------------------------------------
 * Test hooks (no counterpart in the pages). Process-wide settings that let
 * the test suite reach paths a correct run never takes; production callers
 * leave them at their defaults.
 *
 * MOE_DEBUG_WAIT_LIMIT (default 4000000000): the number of GPU clock cycles
 *   after which a bounded device wait gives up (about 2 s at 2 GHz). On a
 *   timeout the kernel records MOE_ERR_TIMEOUT in the workspace status word,
 *   lets its copies and tensor-core work drain, frees its tensor memory and
 *   returns. value <= 0 restores the default.
 * MOE_DEBUG_EXTRA_ARRIVALS (default 0): the single-kernel decode path waits
 *   for this many more arrivals per gate/up tile than happen, so its down
 *   phase times out (exercises the timeout path without any fault).
 * MOE_DEBUG_DISABLE_DECODE_FUSED (default 0): nonzero makes
 *   moe_nvfp4_forward take the multi-kernel path for decode batches too.
 * MOE_DEBUG_DECODE_STAGE_KB (default 8, range 1..8; 0 restores the default):
 *   the largest number of 64-wide K blocks per streamed shared-memory stage
 *   of the W4A16 decode GEMMs (multi-kernel and single-kernel paths alike).
 *   It sets how the two halves of the MMA warps split K, so results can
 *   differ in the last bits from one setting to another (never between the
 *   two decode paths at one setting). Used to tune the stage size.
 * MOE_DEBUG_FP4_TILE (default 0 = the library's choice): the tile shape of
 *   the W4A4 / MXFP4 GEMMs as two decimal digits, tens for the gate/up GEMM
 *   and units for the down GEMM: 1 = one CTA per SM (two accumulators, six
 *   stages) with the weight rows on the MMA's M side; 2 = two CTAs per SM
 *   (one accumulator and three stages each), weight rows on M; 3 = two CTAs
 *   per SM with the group's rows on M; 4 = one CTA per SM, the group's rows
 *   on M and 256 weight rows per tile (two N = 128 halves with their own
 *   MMA issuers); 5 = the same tile as one N = 256 MMA per K block (one
 *   issuer); a GEMM whose N is not a multiple of 256 takes 3 instead of 4 or
 *   5; 0 keeps the library's choice for that GEMM. Results agree to the last bit
 *   across shapes. Used to compare them.
 * MOE_DEBUG_F16_TILE (default 0): 1 = the W4A16 tensor-core GEMMs compute
 *   every group above the small-group limit in tiles of 128 token rows (two
 *   CTAs per SM); 0 = groups of more than 128 rows in tiles of 256 (one CTA
 *   per SM). Results agree to the last bit across the two. Used to compare them.
 * Errors: an unknown key, or a value out of range -> MOE_ERR_INVALID_ARG.
 */
typedef enum {
  MOE_DEBUG_WAIT_LIMIT = 1,
  MOE_DEBUG_EXTRA_ARRIVALS = 2,
  MOE_DEBUG_DISABLE_DECODE_FUSED = 3,
  MOE_DEBUG_DECODE_STAGE_KB = 4,
  MOE_DEBUG_FP4_TILE = 5,
  MOE_DEBUG_F16_TILE = 6
} moe_debug_key;
moe_status moe_debug_set(int key, long long value);

/* ------------------------------------------------------------------------
 * moe_permute_noalloc: the permutation of moe_permute for callers that
 * cannot allocate device memory when they call it (the pages have no
 * counterpart). Some callers own all device memory themselves: a serving
 * engine that reserves one pool at start-up and hands kernels only fixed
 * buffers, or a plug-in running inside a host program that gives it no
 * allocator. Such callers cannot size and provide a workspace per call.
 *
 * This entry point allocates nothing (no cudaMalloc, cudaFree or any
 * allocating routine): its scratch is one fixed device array of 64 KiB
 * that every GPU loading the library holds until the process exits.
 * Inputs and outputs are as in moe_permute; device_status (nullable, device int32) receives MOE_OK or
 * MOE_ERR_DEVICE (an expert id outside [0, E); such pairs are dropped and
 * get inv_perm = -1). A problem whose scratch would exceed the array
 * (T*k above 8192 pairs with more than 16320 histogram entries, e.g. more
 * than about 200k pairs at E = 320) returns MOE_ERR_UNSUPPORTED before
 * anything is enqueued.
 *
 * The first call on a device looks up the array's device address for that
 * device (cudaGetSymbolAddress) and caches it for the life of the process;
 * make that first call before any stream capture. A device reset
 * (cudaDeviceReset) invalidates the cached address: after one, this entry
 * point must not be called again in the same process. Every call on a device shares the one array and
 * leaves its contents behind; each call clears the status word it needs.
 * Calls that overlap on the GPU (on different streams, say) race on the
 * array: order them on one stream or with events.
 */
moe_status moe_permute_noalloc(const int32_t* topk_ids, int T, int k, int E,
                               int32_t* counts, int32_t* offsets, int32_t* perm,
                               int32_t* inv_perm, int32_t* device_status,
                               moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_NVFP4_H */
