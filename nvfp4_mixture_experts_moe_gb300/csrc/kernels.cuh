// Internal launchers shared between the translation units of the library.
#pragma once

#include <utility>

#include "common.cuh"

namespace moe {

// Launches `kernel`, with programmatic dependent launch when `pdl` is set.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Records the CUDA error string for moe_last_cuda_error() and maps it.
moe_status cuda_ok(cudaError_t e);

// Adds n to the process-wide count of kernels this library launched.
void count_launches(int n);

constexpr int kPermSingleMax = 8192;  // pairs handled by the one-CTA permutation
constexpr int kFusedRoutePermuteMax = 2048;  // pairs routed and permuted by one CTA in one launch

// Programmatic dependent launch: a kernel launched with it may start before
// its predecessor in the stream finishes; it must call pdl_wait() before it
// reads anything the predecessor writes. Without the attribute the wait
// returns at once.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Expert sharding (expert parallelism): the permutations group only the
// pairs of experts [shard_lo, shard_lo + n) (n = the E they are given, the
// routing covering E_global experts); other valid pairs are dropped without
// an error and get inv_perm = -1; the kept routed rows come first
// (offsets[n] of them) and the shared rows follow at [offsets[n], offsets[n] + T).
moe_status launch_route_permute_small(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                                      int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                                      int* status, int32_t* row_token, float* row_weight, int32_t* gofs,
                                      cudaStream_t s, int shard_lo, int shard_n);

moe_status launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                             cudaStream_t s);

size_t permute_scratch_bytes(int T, int k, int E);
moe_status launch_permute(const int32_t* ids, int T, int k, int E, int32_t* counts, int32_t* offsets,
                          int32_t* perm, int32_t* inv_perm, int* status, void* scratch,
                          int32_t* row_token, float* row_weight, const float* topk_w, int32_t* gofs,
                          cudaStream_t s, bool pdl = false, int shard_lo = 0, int E_global = 0);

// Quantisation: amax into *amax (must be zeroed first), then codes. A
// gs_static > 0 replaces the dynamic 2688 / amax (amax is then not read).
moe_status launch_amax_bf16(const uint16_t* x, size_t n, float* amax, cudaStream_t s, bool pdl = false);
moe_status launch_quantize_bf16(const uint16_t* x, int rows, int K, const float* amax, uint8_t* q,
                                uint8_t* sf, float* gs_out, float gs_static, cudaStream_t s, bool pdl = false);

// E4M3 block scales re-rounded by a ratio (checkpoint import); sign-bit or
// NaN codes set *flag.
moe_status launch_fold_scales(const uint8_t* in, size_t n, float ratio, uint8_t* out, int* flag, cudaStream_t s);

// Router GEMM: logits fp32 [T, E] = x bf16 [T, H] . w bf16 [E, H]^T, fp32
// accumulation in a fixed order (H % 8 == 0, 16-byte aligned rows).
moe_status launch_router_gemm(const uint16_t* x, const uint16_t* w, int T, int H, int E, float* logits,
                              cudaStream_t s, bool pdl = false);

moe_status launch_swiglu(const float* gu, int rows, int I, uint16_t* h, cudaStream_t s);
moe_status launch_combine(const uint16_t* y, const int32_t* inv_perm, const float* topk_w,
                          const float* y_shared, int T, int k, int H, uint16_t* out, cudaStream_t s,
                          bool pdl = false);

// Weight preparation (device part; the host validates sizes and scales).
moe_status launch_prepare_w4a16(const uint8_t* codes, const uint8_t* sf, int N, int K, int gate_up,
                                uint8_t* out, int* flag, cudaStream_t s);
moe_status launch_prepare_w4a4(const uint8_t* codes, const uint8_t* sf, int N, int K, int gate_up,
                               uint8_t* out_data, uint8_t* out_sf, int* flag, cudaStream_t s, bool mx = false);
size_t prepare_w4a4_sf_bytes(int N, int K);

// Grouped GEMMs.
struct GemmPlan {
  moe_mode mode;
  int gate_up;
  int num_groups;           // G
  int N, K;
  const uint8_t* weights;   // block 0
  size_t weight_stride;     // bytes between blocks
  const uint8_t* last_weights;  // block used by group G-1 (may equal weights + (G-1)*stride)
  const int32_t* group_offsets; // [G+1]
  const void* a;
  const uint8_t* a_sf;
  const float* a_gs;
  const int32_t* a_row_index;
  const float* row_scale;
  uint16_t* out;
  float* out_last_f32;      // nullable: rows of the last group (the shared expert) are written here
                            // as fp32, row (r - group_offsets[G-1]), instead of bf16 into out
  float* out_amax;
  const uint16_t* a_f16;    // W4A16 large groups: f16 copy of the A rows in group order
                            // (row r of the grouped layout; rows_to_f16), or null
  const float* a_mul;       // its per-row multipliers 2^-s
  int a_rows;               // rows of a_f16
  int* status;
  int max_rows;             // upper bound of group_offsets[G] (sizes launches)
  bool pdl;                 // programmatic dependent launch (inside the fused forward)
  bool early_weights;       // group offsets are final before the predecessor ends: weights may
                            // stream before the dependency wait (only with pdl)
  int ctas_per_sm;          // W4A4 tile GEMM: 1 = one CTA per SM (two accumulators); otherwise
                            // two CTAs per SM with the group's rows on the MMA's M side
};

// Small-group path: mma.sync m16n8k16 over register-dequantised weights; one
// pass of up to 8 rows per weight tile. Handles groups with rows <= max_rows.
moe_status launch_gemm_small_w4a16(const GemmPlan& p, int rows_limit, cudaStream_t s);

// Large-group path: tcgen05 MMA with TMEM accumulators. Handles groups with
// rows > rows_min.
moe_status launch_gemm_tc_w4a16(const GemmPlan& p, int rows_min, cudaStream_t s);

// Large-group W4A16 path with the dequantised weights in TMEM; needs the f16
// copy of the activation rows (a_f16, a_mul). Computes the groups with
// rows_min < rows <= rows_max, in tiles of up to 128 token rows (two CTAs per
// SM) or, with `wide`, of up to 256 (one CTA per SM).
moe_status launch_gemm_tc_f16(const GemmPlan& p, int rows_min, int rows_max, bool wide, cudaStream_t s);
// The wide tiles' shared memory (which grows with the group count) fits a CTA.
bool gemm_tc_f16_wide_fits(int num_groups);
// MOE_DEBUG_F16_TILE: 1 = 128-row tiles for every group of the W4A16 GEMMs.
bool debug_f16_narrow_only();

// MXFP4: bf16 [rows, K] -> codes [rows, K/2] and E8M0 scales [rows, K/32]
// (K % 32 == 0).
moe_status launch_quantize_mx(const uint16_t* x, int rows, int K, uint8_t* q, uint8_t* sf, cudaStream_t s);
// Per-tile assembly of the block-scaled GEMMs' activation codes (gathered
// through src_row, or left in place when it is null) and scale atoms from
// row-by-row quantised codes and scales; one CTA per 128-row tile of a group.
// The atoms: per (tile, 256-wide K stage) four (NVFP4, E4M3 per 16) or two
// (MXFP4, E8M0 per 32) 512-byte tcgen05 scale-factor atoms; rows past a
// group's end carry scale 0.
// q has room for q_rows rows (codes of rows past it are not copied).
moe_status launch_tile_gather(const uint8_t* q_src, const uint8_t* sf_src, const int32_t* src_row, int K,
                              const int32_t* gofs, int G, int tiles_max, int q_rows, uint8_t* q, uint8_t* sf_tiles,
                              bool mx, cudaStream_t s);

// bf16 rows -> f16 rows scaled by a power of two so that each row's largest
// magnitude lies in [2^14, 2^15); mul[r] = 2^-s undoes it. Row r of dst is
// row src_index[r] of src (row r when src_index is null).
// rows_limit (nullable, device): rows at or past *rows_limit are skipped (a
// caller's row count that may exceed its arrays).
moe_status launch_rows_to_f16(const uint16_t* src, const int32_t* src_index, int rows, int K, uint16_t* dst,
                              float* mul, cudaStream_t s, bool pdl = false, const int32_t* rows_limit = nullptr);

// W4A4: block-scaled FP4 tcgen05 kernel (every non-empty group).
moe_status launch_gemm_tc_w4a4(const GemmPlan& p, cudaStream_t s);

// W4A4 GEMM of the fused forward: activation codes in group order (a, a_rows
// rows) loaded as tensor-map boxes, their scales as per-tile atoms (a_sf, from
// launch_tile_gather). The large-group GEMMs record MOE_ERR_DEVICE and compute
// nothing when group_offsets[G] exceeds a_rows.
moe_status launch_gemm_tc_fp4(const GemmPlan& p, cudaStream_t s);

// Groups with at most this many rows take the small-group path.
constexpr int kSmallGroupRows = 32;
// Groups of more than this many rows take the W4A16 GEMMs' 256-row tiles.
constexpr int kWideGroupRows = 128;

// Single-kernel decode path (W4A16, T <= kDecodeFusedMaxT): routing,
// permutation, both GEMMs and the combine in one cooperative launch.
constexpr int kDecodeFusedMaxT = 8;
struct DecodeFusedPlan {
  const float* logits;       // [T, E]
  const uint16_t* x;         // [T, H]
  const uint8_t* w13;        // E prepared gate/up blocks, s13 bytes apart
  size_t s13;
  const uint8_t* w13_shared; // nullable (no shared expert)
  const uint8_t* w2;
  size_t s2;
  const uint8_t* w2_shared;
  int T, H, I, E, k;
  uint16_t* out;             // [T, H]
  int32_t* topk_ids_out;     // nullable
  uint16_t* h;               // [T*k + T, I]
  uint16_t* y;               // [T*k, H] routed rows, bf16
  float* y_shared;           // [T, H] the shared expert's rows, fp32
  // Two counter sets of set_ints ints (counters, then set 1): each holds
  // gu_done [E+1], cmb_cnt [T * H/128], hmax [T*k + T] and the grid's item
  // counter (counter_ints ints). A launch uses one set, found zero, and
  // zeroes the other for the next launch; both sets are zeroed by the first
  // launch that finds *clean == 0.
  int* counters;
  int set_ints;
  int counter_ints;
  int* clean;                          // workspace header words
  unsigned long long* ticket;
  unsigned long long* gbar;
  int* status;
  long long wait_limit;      // cycles per bounded wait
  int extra_arrivals;        // test hook (0): extra arrivals a gate/up tile is expected to make
};
bool decode_fused_supported(int T, int H, int I, int E, int k);
moe_status launch_decode_fused(const DecodeFusedPlan& q, cudaStream_t s);

// Test hooks set through moe_debug_set (process-wide).
long long debug_wait_limit();     // cycles per bounded device wait (default 4e9, about 2 s)
int debug_extra_arrivals();       // 0 normally
bool debug_decode_fused_disabled();
int debug_fp4_tile(bool gate_up);   // W4A4/MXFP4 tile shape: 0 (library's choice), 1, 2 or 3
int decode_stage_kb();             // max 64-wide K blocks per ring stage of the decode GEMMs (1..8)

}  // namespace moe
