// C ABI entry points: argument validation on the host, workspace carving,
// and the launch sequence of the fused layer. Declarations and the contract
// of every call are in include/moe_nvfp4.h.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"
#include "router.cuh"

namespace moe {

static thread_local char g_last_cuda_error[256] = "no CUDA error";
constexpr long long kDefaultWaitLimit = 4ll * 1000 * 1000 * 1000;
static std::atomic<long long> g_wait_limit{kDefaultWaitLimit};
static std::atomic<int> g_extra_arrivals{0};
static std::atomic<int> g_fused_disabled{0};
constexpr int kDefaultDecodeStageKb = 8;
static std::atomic<int> g_decode_stage_kb{kDefaultDecodeStageKb};
static std::atomic<int> g_fp4_tile{0};
static std::atomic<int> g_f16_tile{0};


long long debug_wait_limit() { return g_wait_limit.load(std::memory_order_relaxed); }
int debug_extra_arrivals() { return g_extra_arrivals.load(std::memory_order_relaxed); }
bool debug_decode_fused_disabled() { return g_fused_disabled.load(std::memory_order_relaxed) != 0; }
int decode_stage_kb() { return g_decode_stage_kb.load(std::memory_order_relaxed); }
bool debug_f16_narrow_only() { return g_f16_tile.load(std::memory_order_relaxed) == 1; }
int debug_fp4_tile(bool gate_up) {
  const int v = g_fp4_tile.load(std::memory_order_relaxed);
  return gate_up ? v / 10 : v % 10;
}
static std::atomic<unsigned long long> g_launches{0};
static thread_local cudaEvent_t g_stage_events[MOE_STAGE_COUNT];
static thread_local bool g_stage_events_set = false;

void count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

// Records stage event i of the current forward, if the caller asked for them.
static void stage_mark(int i, cudaStream_t s) {
  if (g_stage_events_set && i < MOE_STAGE_COUNT) cudaEventRecord(g_stage_events[i], s);
}

moe_status cuda_ok(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", cudaGetErrorName(e),
                cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}

// sm_103 only. Checked once per device.
static moe_status check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_ok(e);
  static std::mutex mu;
  static int known[64] = {0};  // 0 unknown, 1 ok, 2 unsupported
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (known[dev] == 0) {
      int major = 0, minor = 0;
      e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
      if (e != cudaSuccess) return cuda_ok(e);
      e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
      if (e != cudaSuccess) return cuda_ok(e);
      known[dev] = (major == 10 && minor == 3) ? 1 : 2;
    }
    return known[dev] == 1 ? MOE_OK : MOE_ERR_UNSUPPORTED;
  }
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Carves consecutive 256-byte aligned pieces out of a workspace.
struct Carver {
  uint8_t* base;
  size_t off;
  template <class T>
  T* take(size_t count) {
    T* p = reinterpret_cast<T*>(base ? base + off : nullptr);
    off = align_up(off + count * sizeof(T));
    return p;
  }
};

// Everything the fused forward keeps in its workspace.
struct ForwardWs {
  WsHeader* hdr;
  int32_t* ids;
  float* w;
  float* logits;      // [T, E] when the forward runs the router GEMM
  int32_t* counts;
  int32_t* offsets;   // [E+1]
  int32_t* gofs;      // [E+2] group offsets: routed groups, then the shared rows [P, P+T)
  int32_t* perm;
  int32_t* inv_perm;
  int32_t* row_token;
  float* row_weight;
  void* perm_scratch;
  uint16_t* h;        // [rows, I]
  uint16_t* y;        // [T*k, H] routed rows of GEMM 2, bf16
  float* ys;          // [T, H] the shared expert's rows of GEMM 2, fp32 (null without one)
  uint16_t* xf;       // W4A16, T above the small-group limit: f16 copy of x [T, H]
  float* xmul;        // [T]
  uint16_t* hf;       // f16 copy of h [rows, I]
  float* hmul;        // [rows]
  uint8_t* xq;        // W4A4: [rows, H/2], x quantised in group order
  uint8_t* xsf;       // W4A4: scale atoms per (128-row tile, 256-wide K stage): [tiles, H/256, 2048]
  float* xgs;
  uint8_t* hq;        // W4A4: [rows, I/2]
  uint8_t* hsf;       // W4A4: [tiles, I/256, 2048]
  uint8_t* xq_tok;    // W4A4: x quantised token by token: codes [T, H/2]
  uint8_t* xsf_tok;   //   and scales [T, H/BLK] (BLK = 16 NVFP4, 32 MXFP4), before the per-tile assembly
  uint8_t* hsf_lin;   // W4A4: h's scales row by row [rows, I/BLK] (its codes go straight to hq)
  int tiles;          // W4A4: bound on the 128-row tiles of all groups
  float* hgs;
  int* fused_region;        // kFusedRegionInts ints right after the header (every shape)
  int* fused_counters;      // decode micro path: gu_done [E+1], cmb_cnt [T * H/128], hmax [rows], next item
  size_t fused_counter_ints;
  size_t bytes;
};

// Experts this forward computes (expert parallelism: a contiguous shard).
static int local_experts(const moe_layer_desc& L) { return L.local_experts > 0 ? L.local_experts : L.E; }

// The single-kernel decode path applies to this layer.
// gu_done [E+1], cmb_cnt [T * H/128], hmax [rows], next item
static size_t fused_counter_ints(const moe_layer_desc& L) {
  const size_t rows = (size_t)L.T * L.k + (L.w13_shared ? (size_t)L.T : 0);
  return (size_t)(L.E + 1) + (size_t)L.T * (L.H / 128) + rows + 1;
}

static bool use_decode_fused(const moe_layer_desc& L) {
  return L.mode == MOE_W4A16 && decode_fused_supported(L.T, L.H, L.I, local_experts(L), L.k) &&
         local_experts(L) == L.E && fused_counter_ints(L) <= kFusedSetInts;
}

static ForwardWs carve_forward(const moe_layer_desc& L, void* ws) {
  const size_t P = (size_t)L.T * L.k;
  const size_t shared = L.w13_shared ? (size_t)L.T : 0;
  const size_t rows = P + shared;
  Carver c{static_cast<uint8_t*>(ws), 0};
  ForwardWs f;
  f.hdr = c.take<WsHeader>(1);
  f.fused_region = c.take<int>(kFusedRegionInts);   // fixed place for every shape
  f.ids = c.take<int32_t>(P);
  f.w = c.take<float>(P);
  f.logits = L.w_router ? c.take<float>((size_t)L.T * L.E) : nullptr;
  f.counts = c.take<int32_t>(L.E);
  f.offsets = c.take<int32_t>(L.E + 1);
  f.gofs = c.take<int32_t>(L.E + 2);
  f.perm = c.take<int32_t>(P);
  f.inv_perm = c.take<int32_t>(P);
  f.row_token = c.take<int32_t>(P + L.T);   // routed rows, then one per token
  f.row_weight = c.take<float>(P + L.T);
  f.perm_scratch = c.take<uint8_t>(permute_scratch_bytes(L.T, L.k, L.E));
  f.h = c.take<uint16_t>(rows * L.I);
  f.y = c.take<uint16_t>(P * L.H);
  f.ys = shared ? c.take<float>(shared * L.H) : nullptr;
  if (L.mode == MOE_W4A16 && L.T > kSmallGroupRows) {
    f.xf = c.take<uint16_t>(rows * L.H);  // x rows in group order
    f.xmul = c.take<float>(rows);
    f.hf = c.take<uint16_t>(rows * L.I);
    f.hmul = c.take<float>(rows);
  } else {
    f.xf = f.hf = nullptr;
    f.xmul = f.hmul = nullptr;
  }
  if (L.mode == MOE_W4A4 || L.mode == MOE_MXFP4) {
    const size_t sf_stage = L.mode == MOE_MXFP4 ? 1024 : 2048;  // scale-atom bytes per (tile, 256-wide K stage)
    f.tiles = (int)(rows / 128) + L.E + 1;  // sum over groups of ceil(rows_g / 128)
    f.xq = c.take<uint8_t>(rows * L.H / 2);
    f.xsf = c.take<uint8_t>((size_t)f.tiles * (L.H / 256) * sf_stage);
    f.xgs = c.take<float>(1);
    f.hq = c.take<uint8_t>(rows * L.I / 2);
    f.hsf = c.take<uint8_t>((size_t)f.tiles * (L.I / 256) * sf_stage);
    f.hgs = c.take<float>(1);
    const int blk = L.mode == MOE_MXFP4 ? 32 : 16;
    f.xq_tok = c.take<uint8_t>((size_t)L.T * L.H / 2);
    f.xsf_tok = c.take<uint8_t>((size_t)L.T * (L.H / blk));
    f.hsf_lin = c.take<uint8_t>(rows * (L.I / blk));
  } else {
    f.xq_tok = f.xsf_tok = f.hsf_lin = nullptr;
    f.xq = f.xsf = f.hq = f.hsf = nullptr;
    f.xgs = f.hgs = nullptr;
    f.tiles = 0;
  }
  if (use_decode_fused(L)) {
    f.fused_counter_ints = fused_counter_ints(L);
    f.fused_counters = f.fused_region;
  } else {
    f.fused_counters = nullptr;
    f.fused_counter_ints = 0;
  }
  f.bytes = c.off;
  return f;
}

static size_t prep_size(int N, int K, moe_mode mode, int gate_up) {
  (void)gate_up;
  if (mode == MOE_W4A16) return sizeof(PrepHeader) + w4a16_bytes(N, K);
  if (mode == MOE_MXFP4) return sizeof(PrepHeader) + (size_t)N * K / 2 + (size_t)N * K / 32;
  return sizeof(PrepHeader) + (size_t)N * K / 2 + prepare_w4a4_sf_bytes(N, K);
}

static moe_status validate_layer(const moe_layer_desc* L) {
  if (!L) return MOE_ERR_INVALID_ARG;
  if (L->T < 0 || L->H <= 0 || L->I <= 0 || L->E < 1 || L->k < 1) return MOE_ERR_INVALID_ARG;
  if (L->mode != MOE_W4A16 && L->mode != MOE_W4A4 && L->mode != MOE_MXFP4) return MOE_ERR_INVALID_ARG;
  if (L->E > 1024 || L->k > 32 || L->k > L->E) return MOE_ERR_UNSUPPORTED;
  if (L->H % 128 || L->I % 64) return MOE_ERR_UNSUPPORTED;
  if (L->mode != MOE_W4A16 && (L->H % 256 || L->I % 256)) return MOE_ERR_UNSUPPORTED;
  if (L->w13 == nullptr || L->w2 == nullptr) return MOE_ERR_INVALID_ARG;
  if ((L->w13_shared == nullptr) != (L->w2_shared == nullptr)) return MOE_ERR_INVALID_ARG;
  if (L->w13_shared && L->I_shared != L->I) return MOE_ERR_UNSUPPORTED;
  if (!aligned(L->w13, kAlign) || !aligned(L->w2, kAlign)) return MOE_ERR_INVALID_ARG;
  if (L->w13_shared && (!aligned(L->w13_shared, kAlign) || !aligned(L->w2_shared, kAlign)))
    return MOE_ERR_INVALID_ARG;
  if ((long long)L->T * L->k > (1LL << 30)) return MOE_ERR_UNSUPPORTED;
  if (L->local_experts < 0 || L->expert_offset < 0) return MOE_ERR_INVALID_ARG;
  if (L->local_experts == 0 && L->expert_offset != 0) return MOE_ERR_INVALID_ARG;
  if ((long long)L->expert_offset + L->local_experts > L->E) return MOE_ERR_INVALID_ARG;
  if (L->w_router && !aligned(L->w_router, 16)) return MOE_ERR_INVALID_ARG;
  const float sx = L->x_global_scale, sh = L->h_global_scale;
  if (!(sx >= 0.0f) || !(sh >= 0.0f) || !std::isfinite(sx) || !std::isfinite(sh)) return MOE_ERR_INVALID_ARG;
  if (L->mode != MOE_W4A4 && (sx != 0.0f || sh != 0.0f)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
  }
  return "MOE_ERR_UNKNOWN";
}

const char* moe_last_cuda_error(void) { return g_last_cuda_error; }

moe_status moe_route_topk(const float* logits, int T, int E, int k, int32_t* topk_ids, float* topk_w,
                          moe_stream_t stream) {
  if (T < 0 || E < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || k > 32 || k > E) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  moe_status st = check_device();
  if (st != MOE_OK) return st;
  return launch_route_topk(logits, T, E, k, topk_ids, topk_w, (cudaStream_t)stream);
}

moe_status moe_router_gemm(const uint16_t* x, const uint16_t* w_router, int T, int H, int E, float* logits,
                           moe_stream_t stream) {
  if (T < 0 || H <= 0 || E < 1 || H % 8) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !logits) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_router, 16)) return MOE_ERR_INVALID_ARG;
  moe_status st = check_device();
  if (st != MOE_OK) return st;
  return launch_router_gemm(x, w_router, T, H, E, logits, (cudaStream_t)stream);
}

size_t moe_permute_workspace_size(int T, int k, int E) {
  if (T < 0 || k < 1 || E < 1) return 0;
  return sizeof(WsHeader) + permute_scratch_bytes(T, k, E);
}

moe_status moe_permute(const int32_t* topk_ids, int T, int k, int E, int32_t* counts, int32_t* offsets,
                       int32_t* perm, int32_t* inv_perm, void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (T < 0 || E < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || (long long)T * k > (1LL << 30)) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_ids || !perm || !inv_perm)) return MOE_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, kAlign)) return MOE_ERR_WORKSPACE;
  if (ws_bytes < moe_permute_workspace_size(T, k, E)) return MOE_ERR_WORKSPACE;
  moe_status st = check_device();
  if (st != MOE_OK) return st;
  auto* hdr = static_cast<WsHeader*>(ws);
  // the scratch below overlaps a forward workspace's decode counters: they
  // are no longer known to be zero
  st = cuda_ok(cudaMemsetAsync(&hdr->fused_clean, 0, sizeof(int), (cudaStream_t)stream));
  if (st != MOE_OK) return st;
  return launch_permute(topk_ids, T, k, E, counts, offsets, perm, inv_perm, &hdr->status,
                        static_cast<uint8_t*>(ws) + sizeof(WsHeader), nullptr, nullptr, nullptr, nullptr,
                        (cudaStream_t)stream);
}

size_t moe_quantize_workspace_size(void) { return sizeof(WsHeader); }

moe_status moe_nvfp4_quantize(const uint16_t* x, int rows, int K, uint8_t* q, uint8_t* sf, float* gs_out,
                              void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (rows < 0 || K <= 0 || K % 16) return MOE_ERR_INVALID_ARG;
  if (!gs_out) return MOE_ERR_INVALID_ARG;
  if (rows > 0 && (!x || !q || !sf)) return MOE_ERR_INVALID_ARG;
  if (rows > 0 && (!aligned(x, 16) || !aligned(q, 8))) return MOE_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, kAlign) || ws_bytes < moe_quantize_workspace_size()) return MOE_ERR_WORKSPACE;
  moe_status st = check_device();
  if (st != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  auto* hdr = static_cast<WsHeader*>(ws);
  st = cuda_ok(cudaMemsetAsync(&hdr->amax[0], 0, sizeof(float), s));
  if (st != MOE_OK) return st;
  st = launch_amax_bf16(x, (size_t)rows * K, &hdr->amax[0], s);
  if (st != MOE_OK) return st;
  return launch_quantize_bf16(x, rows, K, &hdr->amax[0], q, sf, gs_out, 0.0f, s);
}

moe_status moe_nvfp4_quantize_static(const uint16_t* x, int rows, int K, float gs, uint8_t* q, uint8_t* sf,
                                     moe_stream_t stream) {
  if (rows < 0 || K <= 0 || K % 16) return MOE_ERR_INVALID_ARG;
  if (!(gs > 0.0f) || !std::isfinite(gs)) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!x || !q || !sf || !aligned(x, 16) || !aligned(q, 8)) return MOE_ERR_INVALID_ARG;
  moe_status st = check_device();
  if (st != MOE_OK) return st;
  return launch_quantize_bf16(x, rows, K, nullptr, q, sf, nullptr, gs, (cudaStream_t)stream);
}

moe_status moe_mxfp4_quantize(const uint16_t* x, int rows, int K, uint8_t* q, uint8_t* sf, moe_stream_t stream) {
  if (rows < 0 || K <= 0 || K % 32) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!x || !q || !sf || !aligned(x, 16) || !aligned(q, 16)) return MOE_ERR_INVALID_ARG;
  moe_status st = check_device();
  if (st != MOE_OK) return st;
  return launch_quantize_mx(x, rows, K, q, sf, (cudaStream_t)stream);
}

moe_status moe_import_global_scale(float stored, moe_scale_format format, float* gs_out) {
  if (!gs_out) return MOE_ERR_INVALID_ARG;
  if (!(stored > 0.0f) || !std::isfinite(stored)) return MOE_ERR_INVALID_ARG;
  if (format == MOE_SCALE_QUANT) {
    *gs_out = stored;
  } else if (format == MOE_SCALE_DEQUANT) {
    *gs_out = 1.0f / stored;  // IEEE fp32 division, correctly rounded
  } else {
    return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

static __device__ int g_fold_flag;

moe_status moe_nvfp4_fold_scales(const uint8_t* sf_in, size_t n, float ratio, uint8_t* sf_out,
                                 moe_stream_t stream) {
  if (!(ratio > 0.0f) || !std::isfinite(ratio)) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (!sf_in || !sf_out) return MOE_ERR_INVALID_ARG;
  moe_status st = check_device();
  if (st != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  int* flag = nullptr;
  st = cuda_ok(cudaGetSymbolAddress(reinterpret_cast<void**>(&flag), g_fold_flag));
  if (st != MOE_OK) return st;
  st = cuda_ok(cudaMemsetAsync(flag, 0, sizeof(int), s));
  if (st != MOE_OK) return st;
  st = launch_fold_scales(sf_in, n, ratio, sf_out, flag, s);
  if (st != MOE_OK) return st;
  int hflag = 0;
  st = cuda_ok(cudaMemcpyAsync(&hflag, flag, sizeof(int), cudaMemcpyDeviceToHost, s));
  if (st != MOE_OK) return st;
  st = cuda_ok(cudaStreamSynchronize(s));
  if (st != MOE_OK) return st;
  return hflag ? MOE_ERR_INVALID_ARG : MOE_OK;
}

size_t moe_prepare_size(int N, int K, moe_mode mode, int gate_up) {
  if (N <= 0 || K <= 0) return 0;
  return prep_size(N, K, mode, gate_up);
}

static __device__ int g_prepare_flag;

moe_status moe_nvfp4_prepare_weights(const uint8_t* codes, const uint8_t* sf, const float* gs, int N, int K,
                                     moe_mode mode, int gate_up, void* out, moe_stream_t stream) {
  if (!codes || !sf || !out || (mode != MOE_MXFP4 && !gs)) return MOE_ERR_INVALID_ARG;
  if (mode != MOE_W4A16 && mode != MOE_W4A4 && mode != MOE_MXFP4) return MOE_ERR_INVALID_ARG;
  if (mode == MOE_MXFP4 && K % 256) return MOE_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || K % 64 || N % 128) return MOE_ERR_INVALID_ARG;
  if (gate_up && (N / 2) % 64) return MOE_ERR_INVALID_ARG;
  if (!aligned(out, kAlign)) return MOE_ERR_INVALID_ARG;
  const int ngs = mode == MOE_MXFP4 ? 0 : (gate_up ? 2 : 1);  // MXFP4 has no global scale
  for (int i = 0; i < ngs; ++i)
    if (!(gs[i] > 0.0f) || !std::isfinite(gs[i])) return MOE_ERR_INVALID_ARG;
  moe_status st = check_device();
  if (st != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  PrepHeader h;
  std::memset(&h, 0, sizeof(h));
  h.magic = kPrepMagic;
  h.mode = mode;
  h.gate_up = gate_up;
  h.N = N;
  h.K = K;
  h.alpha[0] = mode == MOE_MXFP4 ? 1.0f : 1.0f / gs[0];
  h.alpha[1] = gate_up ? (mode == MOE_MXFP4 ? 1.0f : 1.0f / gs[1]) : 0.0f;
  uint8_t* o = static_cast<uint8_t*>(out);
  st = cuda_ok(cudaMemcpyAsync(o, &h, sizeof(h), cudaMemcpyHostToDevice, s));
  if (st != MOE_OK) return st;
  int* flag = nullptr;
  st = cuda_ok(cudaGetSymbolAddress(reinterpret_cast<void**>(&flag), g_prepare_flag));
  if (st != MOE_OK) return st;
  st = cuda_ok(cudaMemsetAsync(flag, 0, sizeof(int), s));
  if (st != MOE_OK) return st;
  uint8_t* data = o + sizeof(PrepHeader);
  if (mode == MOE_W4A16)
    st = launch_prepare_w4a16(codes, sf, N, K, gate_up, data, flag, s);
  else
    st = launch_prepare_w4a4(codes, sf, N, K, gate_up, data, data + (size_t)N * K / 2, flag, s, mode == MOE_MXFP4);
  if (st != MOE_OK) return st;
  int hflag = 0;
  st = cuda_ok(cudaMemcpyAsync(&hflag, flag, sizeof(int), cudaMemcpyDeviceToHost, s));
  if (st != MOE_OK) return st;
  st = cuda_ok(cudaStreamSynchronize(s));
  if (st != MOE_OK) return st;
  return hflag ? MOE_ERR_INVALID_ARG : MOE_OK;
}

size_t moe_gemm_workspace_size(int num_groups) {
  (void)num_groups;
  return sizeof(WsHeader);
}

// Small groups (decode-sized) stream weights through registers into
// mma.sync; large groups go to the tcgen05 kernel. `max_group_rows` is an
// upper bound on any group's rows (skips the tcgen05 launch when small).
static moe_status run_gemm(const GemmPlan& p, long long max_group_rows, cudaStream_t s) {
  if (p.mode == MOE_W4A4) return launch_gemm_tc_w4a4(p, s);
  moe_status st = launch_gemm_small_w4a16(p, kSmallGroupRows, s);
  if (st != MOE_OK || max_group_rows <= kSmallGroupRows) return st;
  if (p.a_f16 != nullptr) {
    // groups of up to 128 rows in 128-row tiles, larger ones in 256-row tiles
    const bool wide = !debug_f16_narrow_only() && gemm_tc_f16_wide_fits(p.num_groups);
    const int narrow_max = wide ? kWideGroupRows : INT_MAX;
    st = launch_gemm_tc_f16(p, kSmallGroupRows, narrow_max, false, s);
    if (st != MOE_OK || !wide || max_group_rows <= kWideGroupRows) return st;
    return launch_gemm_tc_f16(p, kWideGroupRows, INT_MAX, true, s);
  }
  return launch_gemm_tc_w4a16(p, kSmallGroupRows, s);
}

// W4A4 calls with a row count: a bound on the groups' 128-row tiles
static int gemm_fp4_tiles(int num_groups, int rows) { return rows / 128 + num_groups; }

size_t moe_gemm_workspace_size_rows(int num_groups, int rows, int K) {
  if (num_groups < 0 || rows < 0 || K <= 0) return 0;
  // W4A16: the f16 rows [rows, K] and their power-of-two multipliers [rows]
  const size_t f16 = align_up((size_t)rows * K * 2) + align_up((size_t)rows * 4);
  // W4A4: the codes in group order [rows, K/2] and the scale atoms, 2048 bytes
  // per (128-row tile, 256-wide K stage)
  const size_t fp4 = K % 256 ? 0
                             : align_up((size_t)rows * (K / 2)) +
                                   align_up((size_t)gemm_fp4_tiles(num_groups, rows) * (K / 256) * 2048);
  return moe_gemm_workspace_size(num_groups) + std::max(f16, fp4);
}

moe_status moe_nvfp4_grouped_gemm(const moe_gemm_args* a, void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!a) return MOE_ERR_INVALID_ARG;
  if (a->mode == MOE_MXFP4) return MOE_ERR_UNSUPPORTED;  // the fused forward runs MXFP4 layers
  if (a->mode != MOE_W4A16 && a->mode != MOE_W4A4) return MOE_ERR_INVALID_ARG;
  if (a->num_groups < 0 || a->rows < 0) return MOE_ERR_INVALID_ARG;
  if (a->num_groups == 0) return MOE_OK;
  if (a->num_groups > 1025) return MOE_ERR_UNSUPPORTED;
  if (a->K <= 0 || a->N <= 0 || a->K % 64 || a->N % 128) return MOE_ERR_UNSUPPORTED;
  if (a->gate_up && (a->N / 2) % 64) return MOE_ERR_UNSUPPORTED;
  if (!a->weights || !a->group_offsets || !a->a || !a->out) return MOE_ERR_INVALID_ARG;
  if (a->mode == MOE_W4A4 && (!a->a_sf || !a->a_gs)) return MOE_ERR_INVALID_ARG;
  if (a->mode == MOE_W4A4 && a->K % 256) return MOE_ERR_UNSUPPORTED;
  if (!aligned(a->weights, kAlign) || (a->last_weights && !aligned(a->last_weights, kAlign)))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(a->a, 16)) return MOE_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, kAlign) || ws_bytes < moe_gemm_workspace_size(a->num_groups)) return MOE_ERR_WORKSPACE;
  moe_status st = check_device();
  if (st != MOE_OK) return st;
  GemmPlan p;
  std::memset(&p, 0, sizeof(p));
  p.mode = a->mode;
  p.gate_up = a->gate_up;
  p.num_groups = a->num_groups;
  p.N = a->N;
  p.K = a->K;
  p.weights = static_cast<const uint8_t*>(a->weights);
  p.weight_stride = prep_size(a->N, a->K, a->mode, a->gate_up);
  p.last_weights = static_cast<const uint8_t*>(a->last_weights);
  p.group_offsets = a->group_offsets;
  p.a = a->a;
  p.a_sf = a->a_sf;
  p.a_gs = a->a_gs;
  p.a_row_index = a->a_row_index;
  p.row_scale = a->row_scale;
  p.out = a->out;
  p.out_amax = a->out_amax;
  p.status = &static_cast<WsHeader*>(ws)->status;
  p.max_rows = 1 << 30;
  p.pdl = false;
  p.early_weights = false;
  p.a_f16 = nullptr;
  p.a_mul = nullptr;
  cudaStream_t s = (cudaStream_t)stream;
  const bool copy_path = a->rows > 0 && ws_bytes >= moe_gemm_workspace_size_rows(a->num_groups, a->rows, a->K);
  uint8_t* base = static_cast<uint8_t*>(ws) + moe_gemm_workspace_size(a->num_groups);
  if (a->mode == MOE_W4A4) {
    if (!copy_path) return run_gemm(p, 1LL << 30, s);
    // the forward's layout: codes in group order (gathered through the row
    // index, or read in place without one) and per-tile scale atoms
    const bool gather = a->a_row_index != nullptr;
    uint8_t* q = gather ? base : nullptr;
    uint8_t* atoms = base + align_up((size_t)a->rows * (a->K / 2));
    st = launch_tile_gather(gather ? static_cast<const uint8_t*>(a->a) : nullptr, a->a_sf, a->a_row_index, a->K,
                            a->group_offsets, a->num_groups, gemm_fp4_tiles(a->num_groups, a->rows), a->rows, q,
                            atoms, false, s);
    if (st != MOE_OK) return st;
    GemmPlan t = p;
    t.a = gather ? static_cast<const void*>(q) : a->a;
    t.a_sf = atoms;
    t.a_rows = a->rows;
    t.max_rows = a->rows;
    st = launch_gemm_tc_fp4(t, s);
    // a tile shape whose shared memory cannot hold this many groups: the
    // gather kernel instead (the copies above are then unused)
    return st == MOE_ERR_UNSUPPORTED ? run_gemm(p, 1LL << 30, s) : st;
  }
  // W4A16 with the row count and room for the f16 copy: the forward's kernels
  if (!copy_path || a->rows <= kSmallGroupRows) return run_gemm(p, 1LL << 30, s);
  uint16_t* xf = reinterpret_cast<uint16_t*>(base);
  float* xmul = reinterpret_cast<float*>(base + align_up((size_t)a->rows * a->K * 2));
  // (rows past group_offsets[G] are not read: the caller's arrays may end there)
  st = launch_rows_to_f16(static_cast<const uint16_t*>(a->a), a->a_row_index, a->rows, a->K, xf, xmul, s, false,
                          a->group_offsets + a->num_groups);
  if (st != MOE_OK) return st;
  p.a_f16 = xf;
  p.a_mul = xmul;
  p.a_rows = a->rows;
  p.max_rows = a->rows;
  return run_gemm(p, a->rows, s);
}

moe_status moe_swiglu(const float* gu, int rows, int I, uint16_t* h, moe_stream_t stream) {
  if (rows < 0 || I <= 0) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!gu || !h) return MOE_ERR_INVALID_ARG;
  moe_status st = check_device();
  if (st != MOE_OK) return st;
  return launch_swiglu(gu, rows, I, h, (cudaStream_t)stream);
}

moe_status moe_combine(const uint16_t* y, const int32_t* inv_perm, const float* topk_w, const float* y_shared,
                       int T, int k, int H, uint16_t* out, moe_stream_t stream) {
  if (T < 0 || k < 1 || H <= 0 || H % 8) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!y || !inv_perm || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(y, 16) || !aligned(out, 16) || (y_shared && !aligned(y_shared, 16))) return MOE_ERR_INVALID_ARG;
  moe_status st = check_device();
  if (st != MOE_OK) return st;
  return launch_combine(y, inv_perm, topk_w, y_shared, T, k, H, out, (cudaStream_t)stream);
}

size_t moe_workspace_size(const moe_layer_desc* L) {
  if (validate_layer(L) != MOE_OK) return 0;
  return carve_forward(*L, nullptr).bytes;
}

moe_status moe_nvfp4_forward(const moe_layer_desc* L, const uint16_t* x, const float* logits, uint16_t* out,
                             int32_t* topk_ids_out, void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status st = validate_layer(L);
  if (st != MOE_OK) return st;
  if (L->T == 0) return MOE_OK;
  if (!x || !out || (!logits && !L->w_router)) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
  if (L->w_router && L->H % 8) return MOE_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, kAlign)) return MOE_ERR_WORKSPACE;
  ForwardWs f = carve_forward(*L, ws);
  if (ws_bytes < f.bytes) return MOE_ERR_WORKSPACE;
  st = check_device();
  if (st != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  const bool mx = L->mode == MOE_MXFP4;
  const bool fp4 = L->mode == MOE_W4A4 || mx;   // FP4 activations, block-scaled FP4 MMA
  const int T = L->T, k = L->k, E = L->E, H = L->H, I = L->I;
  const int P = T * k;
  const bool has_shared = L->w13_shared != nullptr;
  const int rows = P + (has_shared ? T : 0);
  const int EL = local_experts(*L), lo = L->expert_offset;   // this forward's expert shard
  int32_t* ids = topk_ids_out ? topk_ids_out : f.ids;
  struct StageGuard {  // the events apply to one forward call only
    ~StageGuard() { g_stage_events_set = false; }
  } guard;

  // Kernels after the first use programmatic dependent launch (each waits for
  // its predecessor's results in-kernel) unless stage events are recorded.
  const bool pdl = !g_stage_events_set;
  stage_mark(0, s);
  if (L->w_router) {  // router GEMM: the logits come from x
    st = launch_router_gemm_status(x, L->w_router, T, H, E, f.logits, s, false, &f.hdr->status);
    if (st != MOE_OK) return st;
    logits = f.logits;
  }
  if (f.fused_counters != nullptr && !debug_decode_fused_disabled()) {
    // decode micro path: the whole layer in one cooperative kernel (its
    // counters alternate between two sets in the workspace; each launch
    // zeroes the set the next one uses, so no memset precedes it)
    DecodeFusedPlan q;
    q.logits = logits;
    q.x = x;
    q.w13 = static_cast<const uint8_t*>(L->w13);
    q.s13 = prep_size(2 * I, H, L->mode, 1);
    q.w13_shared = static_cast<const uint8_t*>(L->w13_shared);
    q.w2 = static_cast<const uint8_t*>(L->w2);
    q.s2 = prep_size(H, I, L->mode, 0);
    q.w2_shared = static_cast<const uint8_t*>(L->w2_shared);
    q.T = T;
    q.H = H;
    q.I = I;
    q.E = E;
    q.k = k;
    q.out = out;
    q.topk_ids_out = topk_ids_out;
    q.h = f.h;
    q.y = f.y;
    q.y_shared = f.ys;
    q.counters = f.fused_region;   // set 0; set 1 kFusedSetInts further
    q.set_ints = (int)kFusedSetInts;
    q.counter_ints = (int)f.fused_counter_ints;
    q.clean = &f.hdr->fused_clean;
    q.ticket = &f.hdr->fused_ticket;
    q.gbar = &f.hdr->fused_gbar;
    q.status = &f.hdr->status;
    q.wait_limit = debug_wait_limit();
    q.extra_arrivals = debug_extra_arrivals();
    st = launch_decode_fused(q, s);
    if (st != MOE_OK) return st;
    for (int i = 1; i < MOE_STAGE_COUNT; ++i) stage_mark(i, s);
    return MOE_OK;
  }
  if (P <= kFusedRoutePermuteMax) {  // route + permute in one CTA
    st = launch_route_permute_small(logits, T, E, k, ids, f.w, f.counts, f.offsets, f.perm, f.inv_perm,
                                    &f.hdr->status, f.row_token, f.row_weight, f.gofs, s, lo, EL);
    if (st != MOE_OK) return st;
    stage_mark(1, s);
  } else {
    st = launch_route_topk(logits, T, E, k, ids, f.w, s);
    if (st != MOE_OK) return st;
    stage_mark(1, s);
    st = launch_permute(ids, T, k, EL, f.counts, f.offsets, f.perm, f.inv_perm, &f.hdr->status, f.perm_scratch,
                        f.row_token, f.row_weight, f.w, f.gofs, s, pdl, lo, E);
    if (st != MOE_OK) return st;
  }
  stage_mark(2, s);
  const float x_static = L->x_global_scale, h_static = L->h_global_scale;

  if (fp4) {  // x -> FP4 in group order: W4A4 with a per-tensor scale (dynamic amax or static); MXFP4 per 32
    st = cuda_ok(cudaMemsetAsync(&f.hdr->amax[0], 0, 2 * sizeof(float), s));
    if (st != MOE_OK) return st;
    if (!mx && x_static == 0.0f) {
      st = launch_amax_bf16(x, (size_t)T * H, &f.hdr->amax[0], s, pdl);
      if (st != MOE_OK) return st;
    }
    // token by token (coalesced codes and scales), then per 128-row tile:
    // each token's codes to its grouped rows, the scale atoms assembled
    st = mx ? launch_quantize_mx(x, T, H, f.xq_tok, f.xsf_tok, s)
            : launch_quantize_bf16(x, T, H, &f.hdr->amax[0], f.xq_tok, f.xsf_tok, f.xgs, x_static, s, pdl);
    if (st != MOE_OK) return st;
    st = launch_tile_gather(f.xq_tok, f.xsf_tok, f.row_token, H, f.gofs, EL + (has_shared ? 1 : 0), f.tiles, rows,
                            f.xq, f.xsf, mx, s);
    if (st != MOE_OK) return st;
  }
  if (f.xf) {  // f16 copy of x, rows in group order, for the large-group tensor-core GEMM
    st = launch_rows_to_f16(x, f.row_token, rows, H, f.xf, f.xmul, s, pdl);
    if (st != MOE_OK) return st;
  }
  stage_mark(3, s);

  const int G = EL + (has_shared ? 1 : 0);
  GemmPlan g1;
  std::memset(&g1, 0, sizeof(g1));
  g1.mode = L->mode;
  g1.gate_up = 1;
  g1.num_groups = G;
  g1.N = 2 * I;
  g1.K = H;
  g1.weights = static_cast<const uint8_t*>(L->w13);
  g1.weight_stride = prep_size(2 * I, H, L->mode, 1);
  g1.last_weights = has_shared ? static_cast<const uint8_t*>(L->w13_shared) : nullptr;
  g1.group_offsets = f.gofs;
  g1.a = fp4 ? static_cast<const void*>(f.xq) : static_cast<const void*>(x);
  g1.a_sf = fp4 ? f.xsf : nullptr;
  g1.a_gs = fp4 ? f.xgs : nullptr;
  g1.a_row_index = f.row_token;
  g1.out = f.h;
  g1.out_amax = (fp4 && !mx && h_static == 0.0f) ? &f.hdr->amax[1] : nullptr;
  g1.a_f16 = f.xf;
  g1.a_mul = f.xmul;
  g1.a_rows = rows;
  g1.status = &f.hdr->status;
  g1.max_rows = rows;
  g1.pdl = pdl;
  g1.early_weights = false;
  st = fp4 ? launch_gemm_tc_fp4(g1, s) : run_gemm(g1, T, s);
  if (st != MOE_OK) return st;
  stage_mark(4, s);
  if (fp4) {  // h -> FP4: NVFP4 with one global scale over all rows (amax from GEMM 1's epilogue); MXFP4 per 32
    // row by row (h is in group order: the codes land in place), then the
    // scale atoms per 128-row tile
    st = mx ? launch_quantize_mx(f.h, rows, I, f.hq, f.hsf_lin, s)
            : launch_quantize_bf16(f.h, rows, I, &f.hdr->amax[1], f.hq, f.hsf_lin, f.hgs, h_static, s, pdl);
    if (st != MOE_OK) return st;
    st = launch_tile_gather(nullptr, f.hsf_lin, nullptr, I, f.gofs, G, f.tiles, 0, nullptr, f.hsf, mx, s);
    if (st != MOE_OK) return st;
  } else if (f.hf) {
    st = launch_rows_to_f16(f.h, nullptr, rows, I, f.hf, f.hmul, s, pdl);
    if (st != MOE_OK) return st;
  }
  stage_mark(5, s);

  GemmPlan g2 = g1;
  g2.gate_up = 0;
  g2.N = H;
  g2.K = I;
  g2.weights = static_cast<const uint8_t*>(L->w2);
  g2.weight_stride = prep_size(H, I, L->mode, 0);
  g2.last_weights = has_shared ? static_cast<const uint8_t*>(L->w2_shared) : nullptr;
  g2.a = fp4 ? static_cast<const void*>(f.hq) : static_cast<const void*>(f.h);
  g2.a_sf = fp4 ? f.hsf : nullptr;
  g2.a_gs = fp4 ? f.hgs : nullptr;
  g2.out_amax = nullptr;
  g2.a_f16 = f.hf;
  g2.a_mul = f.hmul;
  g2.early_weights = true;  // group offsets come from the permutation, two launches back
  g2.a_row_index = nullptr;
  g2.row_scale = f.row_weight;
  g2.out = f.y;
  g2.out_last_f32 = f.ys;  // the shared expert's rows stay fp32 until the combine
  st = fp4 ? launch_gemm_tc_fp4(g2, s) : run_gemm(g2, T, s);
  if (st != MOE_OK) return st;
  stage_mark(6, s);
  st = launch_combine(f.y, f.inv_perm, nullptr, f.ys, T, k, H, out, s, pdl);
  if (st != MOE_OK) return st;
  stage_mark(7, s);
  return MOE_OK;
}

moe_status moe_set_stage_events(void* const* events, int n) {
  if (events == nullptr) {
    g_stage_events_set = false;
    return MOE_OK;
  }
  if (n < MOE_STAGE_COUNT) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < MOE_STAGE_COUNT; ++i) {
    if (events[i] == nullptr) return MOE_ERR_INVALID_ARG;
    g_stage_events[i] = static_cast<cudaEvent_t>(events[i]);
  }
  g_stage_events_set = true;
  return MOE_OK;
}

unsigned long long moe_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

moe_status moe_debug_set(int key, long long value) {
  switch (key) {
    case MOE_DEBUG_WAIT_LIMIT:
      g_wait_limit.store(value > 0 ? value : kDefaultWaitLimit, std::memory_order_relaxed);
      return MOE_OK;
    case MOE_DEBUG_EXTRA_ARRIVALS:
      g_extra_arrivals.store(value > 0 ? (int)std::min<long long>(value, 1 << 20) : 0, std::memory_order_relaxed);
      return MOE_OK;
    case MOE_DEBUG_DISABLE_DECODE_FUSED:
      g_fused_disabled.store(value != 0 ? 1 : 0, std::memory_order_relaxed);
      return MOE_OK;
    case MOE_DEBUG_DECODE_STAGE_KB:
      if (value < 0 || value > kW16MaxStageKb) return MOE_ERR_INVALID_ARG;
      g_decode_stage_kb.store(value > 0 ? (int)value : kDefaultDecodeStageKb, std::memory_order_relaxed);
      return MOE_OK;
    case MOE_DEBUG_FP4_TILE:
      if (value < 0 || value > 55 || value % 10 > 5) return MOE_ERR_INVALID_ARG;
      g_fp4_tile.store((int)value, std::memory_order_relaxed);
      return MOE_OK;
    case MOE_DEBUG_F16_TILE:
      if (value < 0 || value > 1) return MOE_ERR_INVALID_ARG;
      g_f16_tile.store((int)value, std::memory_order_relaxed);
      return MOE_OK;

  }
  return MOE_ERR_INVALID_ARG;
}

moe_status moe_get_device_status(void* ws, moe_stream_t stream) {
  if (!ws || !aligned(ws, kAlign)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int v = 0;
  moe_status st = cuda_ok(cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, s));
  if (st != MOE_OK) return st;
  st = cuda_ok(cudaMemsetAsync(ws, 0, sizeof(int), s));
  if (st != MOE_OK) return st;
  st = cuda_ok(cudaStreamSynchronize(s));
  if (st != MOE_OK) return st;
  return (moe_status)v;
}

}  // extern "C"
