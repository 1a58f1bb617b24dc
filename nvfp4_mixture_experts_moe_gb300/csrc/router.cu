// Router GEMM ahead of the top-k: logits[t][e] = sum_h x[t][h] * W[e][h], bf16
// inputs, fp32 accumulation, fp32 logits.
//
// "vLLM on the NVIDIA DGX Spark: A Complete Technical Guide", section 7.1
// (the [Router] stage that precedes top-k and dispatch); the router matrix
// stays 16-bit (it is not one of the NVFP4 expert weights).
//
// The product is small next to the experts (E x H weights, T x E x H
// multiply-adds: 2.6 MB and 10.7 GFLOP for E = 320, H = 4096 at 4096 tokens),
// and two kernels cover it:
// * few tokens (T <= 16): the weight rows stream from HBM once; two expert
//   rows per CTA of eight warps, the threads striding over K in 16-byte
//   chunks with every load of a round (both rows' weights, every token's x)
//   issued before any is used, one fp32 sum per (row, token) per thread, and
//   the partial sums added in a fixed order (lanes by a shuffle tree, then
//   warps 0..7). The 2.7 MB at 8 tokens, E = 320, H = 4096 would take 0.4 us
//   at HBM speed; a launch is bound by its latency (one CTA per row with
//   four dependent rounds of x loads measured about 10 us);
// * more tokens: tcgen05.mma (bf16 in, fp32 accumulate in TMEM) over
//   128-expert x 128-token tiles, described below.
// Both reduce in an order fixed by the shapes, so the logits are the same
// bits on every run. Rows past T or E and the K tail past H are zero-filled
// by the copies; every store is bounds-checked.
#include "common.cuh"
#include "kernels.cuh"
#include "router.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using tc::smem_u32;

// ---------------------------------------------------------------------------
// Few tokens.
constexpr int kGemvMaxT = 16;
constexpr int kGemvWarps = 8;
constexpr int kGemvRows = 2;   // expert rows per CTA

__device__ __forceinline__ void bf16x8_to_float(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// MAXT tokens at most; BATCH 16-byte chunks of K per thread per round, whose
// weight loads (HBM) and x loads (L2) for every row and token are all issued
// before any is used, so a round costs one memory latency. Each thread keeps
// one fp32 sum per (row, token) over its chunks in increasing order; lanes
// are added by a shuffle tree, then warps 0..7 in order.
template <int MAXT, int BATCH>
__global__ void __launch_bounds__(kGemvWarps * 32) router_gemv_kernel(const uint16_t* __restrict__ x,
                                                                      const uint16_t* __restrict__ w, int T,
                                                                      int H, int E, float* __restrict__ logits) {
  pdl_wait();
  const int e0 = blockIdx.x * kGemvRows;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = H / 8;   // 16-byte chunks of a row
  float acc[kGemvRows][MAXT];
#pragma unroll
  for (int r = 0; r < kGemvRows; ++r)
#pragma unroll
    for (int t = 0; t < MAXT; ++t) acc[r][t] = 0.0f;
  for (int cb = tid; cb < C; cb += kGemvWarps * 32 * BATCH) {
    uint4 wv[kGemvRows][BATCH], xv[BATCH][MAXT];
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
      const int c = cb + kGemvWarps * 32 * u;
#pragma unroll
      for (int r = 0; r < kGemvRows; ++r)
        wv[r][u] = (c < C && e0 + r < E) ? ldg_stream(reinterpret_cast<const uint4*>(w + (size_t)(e0 + r) * H) + c)
                                         : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int t = 0; t < MAXT; ++t)
        xv[u][t] = (c < C && t < T) ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H) + c)
                                    : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < BATCH; ++u) {
#pragma unroll
      for (int r = 0; r < kGemvRows; ++r) {
        float wf[8];
        bf16x8_to_float(wv[r][u], wf);
#pragma unroll
        for (int t = 0; t < MAXT; ++t) {
          float xf[8];
          bf16x8_to_float(xv[u][t], xf);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[r][t] = fmaf(xf[i], wf[i], acc[r][t]);
        }
      }
    }
  }
  __shared__ float part[kGemvWarps][kGemvRows][MAXT];
#pragma unroll
  for (int r = 0; r < kGemvRows; ++r)
#pragma unroll
    for (int t = 0; t < MAXT; ++t) {
      float v = acc[r][t];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) part[warp][r][t] = v;
    }
  __syncthreads();
  if (tid < kGemvRows * MAXT) {
    const int r = tid / MAXT, t = tid % MAXT;
    if (t < T && e0 + r < E) {
      float v = part[0][r][t];
#pragma unroll
      for (int q = 1; q < kGemvWarps; ++q) v += part[q][r][t];
      logits[(size_t)t * E + e0 + r] = v;
    }
  }
}

// ---------------------------------------------------------------------------
// Many tokens on the 5th-generation tensor cores: one 128-expert x 128-token
// tile per CTA (swap-AB: router rows on the MMA's M side, so TMEM lane = expert
// and the epilogue's stores are coalesced along E). Warps 0-3 copy both
// operands with cp.async into a 6-deep ring of 128-byte-swizzled K-major
// tiles (64 K per stage; four stages in flight per thread, since the copy
// rate is set by the bytes in flight) and then read the accumulator back; lane 0 of warp 4
// issues tcgen05.mma kind::f16 (bf16 in, fp32 accumulate in TMEM), four per
// stage. Every wait is bounded: on a timeout the tile's logits are written as
// NaN, the status word (when given) gets MOE_ERR_TIMEOUT, copies and MMAs
// drain and TMEM is freed.
constexpr int kTcM = 128;                   // experts per tile
constexpr int kTcN = 128;                   // tokens per tile
constexpr int kTcStages = 6;
constexpr int kTcTile = 128 * 128;          // bytes of one operand tile (128 rows x 64 bf16)
constexpr int kTcStageBytes = 2 * kTcTile;  // A (router rows) then B (token rows)
constexpr int kTcLookahead = 4;             // stages a producer keeps in flight before publishing
constexpr int kTcThreads = 160;
constexpr int kTcCols = 128;                // TMEM columns (one fp32 accumulator of N <= 128)
constexpr long long kTcWaitLimit = 2ll * 1000 * 1000 * 1000;  // cycles (~1 s)
static_assert(kTcStages >= kTcLookahead + 1, "a producer must publish a stage before it reuses its slot");

struct TcSmem {
  uint64_t full[kTcStages];
  uint64_t empty[kTcStages];
  uint64_t done;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kTcSmemBytes = 1024 + (size_t)kTcStages * kTcStageBytes + sizeof(TcSmem);

__global__ void __launch_bounds__(kTcThreads, 1) router_tc_kernel(const uint16_t* __restrict__ x,
                                                                  const uint16_t* __restrict__ w, int T, int H,
                                                                  int E, float* __restrict__ logits,
                                                                  int* __restrict__ status) {
  using namespace tc;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  TcSmem* sm = reinterpret_cast<TcSmem*>(base + kTcStages * kTcStageBytes);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int e0 = blockIdx.x * kTcM, t0 = blockIdx.y * kTcN;
  const int C = H / 8, KT = (C + 7) / 8;
  const int bn = (min(kTcN, T - t0) + 15) & ~15;  // the MMA's N: tokens of the tile rounded up to 16
  pdl_wait();
  if (tid == 0) {
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(&sm->full[i], 128);
      mbar_init(&sm->empty[i], 1);
    }
    mbar_init(&sm->done, 1);
    sm->abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (warp == 4) tmem_alloc(&sm->tmem_base, kTcCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  volatile int* abort = &sm->abort;

  if (warp < 4) {
    // ------------------------------------------------ copies, then epilogue
    int issued = 0, fin = 0;
    for (int kt = 0; kt < KT; ++kt) {
      const int slot = kt % kTcStages;
      if (!mbar_wait(&sm->empty[slot], ((kt / kTcStages) & 1) ^ 1, abort, kTcWaitLimit)) break;
      const uint32_t a_s = smem_u32(base + slot * kTcStageBytes);
      const uint32_t b_s = a_s + kTcTile;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int idx = tid + 128 * j;
        const int row = idx >> 3, ch = idx & 7;
        const int kc = kt * 8 + ch;
        const bool kin = kc < C;
        const int ex = e0 + row, tok = t0 + row;
        const bool va = kin && ex < E, vb = kin && tok < T;
        const uint32_t off = (uint32_t)(row * 128 + ((ch ^ (row & 7)) << 4));
        cp_async_16(a_s + off, va ? (const void*)(w + (size_t)ex * H + (size_t)kc * 8) : (const void*)w,
                    va ? 16u : 0u);
        cp_async_16(b_s + off, vb ? (const void*)(x + (size_t)tok * H + (size_t)kc * 8) : (const void*)x,
                    vb ? 16u : 0u);
      }
      cp_async_commit();
      ++issued;
      if (issued - fin > kTcLookahead) {
        cp_async_wait<kTcLookahead>();
        fence_proxy_async_smem();
        mbar_arrive(&sm->full[fin % kTcStages]);
        ++fin;
      }
    }
    cp_async_wait_all();
    while (fin < issued) {
      fence_proxy_async_smem();
      mbar_arrive(&sm->full[fin % kTcStages]);
      ++fin;
    }
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&sm->done, 0, abort, kTcWaitLimit) && !*abort);
    tc_fence_after();
    const int ex = e0 + warp * 32 + lane;  // TMEM lane = router row
    for (int c0 = 0; c0 < bn; c0 += 16) {
      uint32_t r[16];
      if (ok) {
        tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, r);
        tmem_ld_wait();
      }
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int tok = t0 + c0 + c;
        if (ex < E && tok < T) logits[(size_t)tok * E + ex] = ok ? __uint_as_float(r[c]) : __int_as_float(0x7fc00000);
      }
    }
  } else if (lane == 0) {
    // ------------------------------------------------------------------ MMA
    const uint32_t idesc = idesc_f16(kTcM, bn, 1);
    for (int kt = 0; kt < KT; ++kt) {
      const int slot = kt % kTcStages;
      if (!mbar_wait(&sm->full[slot], (kt / kTcStages) & 1, abort, kTcWaitLimit)) break;
      tc_fence_after();
      const uint32_t as = smem_u32(base + slot * kTcStageBytes);
      const uint32_t bs = as + kTcTile;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = smem_desc(as + kk * 32, 16, 1024, kSwizzle128B);
        const uint64_t bd = smem_desc(bs + kk * 32, 16, 1024, kSwizzle128B);
        mma_f16(tmem, ad, bd, idesc, (kt | kk) != 0);
      }
      tc_commit(&sm->empty[slot]);
    }
    // `done` arrives once every MMA issued above has completed (also after an abort)
    tc_commit(&sm->done);
    const long long c0 = clock64();
    while (!mbar_try_wait(&sm->done, 0) && clock64() - c0 < kTcWaitLimit) {
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 4) tmem_dealloc(tmem, kTcCols);
  if (tid == 0 && sm->abort && status != nullptr) set_status(status, MOE_ERR_TIMEOUT);
}

}  // namespace

moe_status launch_router_gemm_status(const uint16_t* x, const uint16_t* w, int T, int H, int E, float* logits,
                                     cudaStream_t s, bool pdl, int* status) {
  if (T == 0) return MOE_OK;
  cudaError_t e;
  if (T <= kGemvMaxT) {
    const dim3 grid((E + kGemvRows - 1) / kGemvRows), block(kGemvWarps * 32);
    e = T <= 8 ? launch_ex(pdl, router_gemv_kernel<8, 2>, grid, block, 0, s, x, w, T, H, E, logits)
               : launch_ex(pdl, router_gemv_kernel<kGemvMaxT, 1>, grid, block, 0, s, x, w, T, H, E, logits);
  } else {
    const int ntiles = (T + kTcN - 1) / kTcN;
    if (ntiles > 65535) return MOE_ERR_UNSUPPORTED;
    e = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmemBytes);
    if (e != cudaSuccess) return cuda_ok(e);
    const dim3 grid((E + kTcM - 1) / kTcM, ntiles);
    e = launch_ex(pdl, router_tc_kernel, grid, dim3(kTcThreads), kTcSmemBytes, s, x, w, T, H, E, logits, status);
  }
  if (e != cudaSuccess) return cuda_ok(e);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

moe_status launch_router_gemm(const uint16_t* x, const uint16_t* w, int T, int H, int E, float* logits,
                              cudaStream_t s, bool pdl) {
  return launch_router_gemm_status(x, w, T, H, E, logits, s, pdl, nullptr);
}

}  // namespace moe
