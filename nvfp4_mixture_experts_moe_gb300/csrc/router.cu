// Router GEMM ahead of the top-k: logits[t][e] = sum_h x[t][h] * W[e][h], bf16
// inputs, fp32 accumulation, fp32 logits.
//
// "vLLM on the NVIDIA DGX Spark: A Complete Technical Guide", section 7.1
// (the [Router] stage that precedes top-k and dispatch); the router matrix
// stays 16-bit (it is not one of the NVFP4 expert weights).
//
// The product is small next to the experts (E x H weights, T x E x H
// multiply-adds: 2.6 MB and 10.7 GFLOP for E = 320, H = 4096 at 4096 tokens),
// so two plain kernels cover it:
// * few tokens (T <= 16): the weight rows stream from HBM once; one CTA per
//   expert row, its four warps take a quarter of K each, every lane holds one
//   fp32 sum per token (its chunks in a fixed order), and the partial sums
//   are added in a fixed order (lanes by a shuffle tree, then warps 0..3).
//   Measured at 8 tokens, E = 320, H = 4096: about 11 us per launch after an
//   L2 flush, far from the 0.4 us the 2.7 MB would take at HBM speed; the
//   kernel is latency-bound (sixteen warps per row measured no faster);
// * more tokens: mma.sync m16n8k16 (bf16 in, fp32 accumulate) over 64 x 64
//   (token x expert) tiles, K in 64-wide stages moved by cp.async into a
//   4-deep ring of XOR-swizzled shared-memory tiles read by ldmatrix.
// Both reduce in an order fixed by the shapes, so the logits are the same
// bits on every run. Rows past T or E and the K tail past H are zero-filled
// by the copies; every store is bounds-checked. Neither kernel waits on
// anything but its own copies.
#include "common.cuh"
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using tc::smem_u32;

// ---------------------------------------------------------------------------
// Few tokens.
constexpr int kGemvMaxT = 16;
constexpr int kGemvWarps = 4;
constexpr int kGemvBatch = 4;

__device__ __forceinline__ void bf16x8_to_float(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__global__ void __launch_bounds__(kGemvWarps * 32) router_gemv_kernel(const uint16_t* __restrict__ x,
                                                                      const uint16_t* __restrict__ w, int T,
                                                                      int H, int E, float* __restrict__ logits) {
  pdl_wait();
  const int e = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = H / 8;  // 16-byte chunks of a row
  const int per = (C + kGemvWarps - 1) / kGemvWarps;
  const int c0 = min(C, warp * per), c1 = min(C, c0 + per);
  float acc[kGemvMaxT];
#pragma unroll
  for (int t = 0; t < kGemvMaxT; ++t) acc[t] = 0.0f;
  const uint4* wrow = reinterpret_cast<const uint4*>(w + (size_t)e * H);
  // kGemvBatch chunks per lane per round: their weight loads (HBM) are issued
  // together; then, chunk by chunk, the matching x chunks of every token (L2)
  // are issued together before they are used, so a round costs one HBM
  // latency plus one L2 latency per chunk instead of one per chunk and token
  for (int cb = c0 + lane; cb < c1; cb += 32 * kGemvBatch) {
    uint4 wv[kGemvBatch];
#pragma unroll
    for (int u = 0; u < kGemvBatch; ++u) {
      const int c = cb + 32 * u;
      wv[u] = c < c1 ? ldg_stream(wrow + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kGemvBatch; ++u) {
      const int c = cb + 32 * u;
      if (c >= c1) break;
      uint4 xv[kGemvMaxT];
#pragma unroll
      for (int t = 0; t < kGemvMaxT; ++t)
        xv[t] = t < T ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H) + c) : make_uint4(0, 0, 0, 0);
      float wf[8];
      bf16x8_to_float(wv[u], wf);
#pragma unroll
      for (int t = 0; t < kGemvMaxT; ++t) {
        if (t < T) {
          float xf[8];
          bf16x8_to_float(xv[t], xf);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[t] = fmaf(xf[i], wf[i], acc[t]);
        }
      }
    }
  }
  __shared__ float part[kGemvWarps][kGemvMaxT];
#pragma unroll
  for (int t = 0; t < kGemvMaxT; ++t) {
    float v = acc[t];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) part[warp][t] = v;
  }
  __syncthreads();
  if ((int)threadIdx.x < T) {
    float v = part[0][threadIdx.x];
#pragma unroll
    for (int q = 1; q < kGemvWarps; ++q) v += part[q][threadIdx.x];
    logits[(size_t)threadIdx.x * E + e] = v;
  }
}

// ---------------------------------------------------------------------------
// Many tokens: 64 tokens x 64 experts per CTA, four warps of 32 x 32.
constexpr int kBM = 64;
constexpr int kBN = 64;
constexpr int kBK = 64;                    // bf16 per row per stage (128 bytes)
constexpr int kRing = 4;
constexpr int kMmaThreads = 128;
constexpr int kTileBytes = kBM * kBK * 2;  // 8 KB (A and B tiles are the same size)
constexpr int kSlotBytes = 2 * kTileBytes;
constexpr int kRouterSmem = kRing * kSlotBytes;  // 64 KB
static_assert(kBM == kBN, "A and B tiles share the copy loop");

// Byte offset of 16-byte chunk `ch` (0..7) of tile row `row`: the chunk index
// is XORed with the row's low three bits, so the eight rows an ldmatrix phase
// reads sit in eight different bank groups.
__device__ __forceinline__ uint32_t swz(int row, int ch) { return (uint32_t)(row * 128 + ((ch ^ (row & 7)) << 4)); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kMmaThreads) router_mma_kernel(const uint16_t* __restrict__ x,
                                                                 const uint16_t* __restrict__ w, int T, int H,
                                                                 int E, float* __restrict__ logits) {
  pdl_wait();
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int n0 = blockIdx.x * kBN;  // first expert of the tile
  const int m0 = blockIdx.y * kBM;  // first token of the tile
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wm = warp & 1, wn = warp >> 1;  // 32-token x 32-expert quarter of the tile
  const int C = H / 8;
  const int KT = (C + 7) / 8;

  // stage kt -> ring slot: A (x rows) at 0, B (router rows) at kTileBytes
  auto load = [&](int kt, int slot) {
    const uint32_t a_s = sbase + (uint32_t)(slot * kSlotBytes);
    const uint32_t b_s = a_s + kTileBytes;
#pragma unroll
    for (int j = 0; j < (kBM * 8) / kMmaThreads; ++j) {
      const int idx = tid + j * kMmaThreads;
      const int row = idx >> 3, ch = idx & 7;
      const int kc = kt * 8 + ch;
      const int tok = m0 + row, ex = n0 + row;
      const bool kin = kc < C;
      const bool va = kin && tok < T, vb = kin && ex < E;
      cp_async16(a_s + swz(row, ch), va ? (const void*)(x + (size_t)tok * H + (size_t)kc * 8) : (const void*)x, va);
      cp_async16(b_s + swz(row, ch), vb ? (const void*)(w + (size_t)ex * H + (size_t)kc * 8) : (const void*)w, vb);
    }
  };

  float acc[2][4][4];
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < 4; ++ni) acc[mi][ni][0] = acc[mi][ni][1] = acc[mi][ni][2] = acc[mi][ni][3] = 0.0f;

#pragma unroll
  for (int s = 0; s < kRing - 1; ++s) {
    if (s < KT) load(s, s);
    cp_async_commit();
  }
  for (int kt = 0; kt < KT; ++kt) {
    cp_async_wait<kRing - 2>();  // stage kt has landed (this thread's copies) ...
    __syncthreads();             // ... everyone's, and slot (kt - 1) % kRing is free again
    const int nk = kt + kRing - 1;
    if (nk < KT) load(nk, nk % kRing);
    cp_async_commit();
    const uint32_t a_s = sbase + (uint32_t)((kt % kRing) * kSlotBytes);
    const uint32_t b_s = a_s + kTileBytes;
#pragma unroll
    for (int ks = 0; ks < kBK / 16; ++ks) {
      uint32_t a[2][4], b[2][4];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        // matrices: rows 0-7 / 8-15 (lane bit 3) x k 0-7 / 8-15 (lane bit 4)
        const int row = wm * 32 + mi * 16 + (lane & 15);
        ldsm4(a_s + swz(row, ks * 2 + (lane >> 4)), a[mi]);
      }
#pragma unroll
      for (int nj = 0; nj < 2; ++nj) {
        // matrices: k 0-7 / 8-15 (lane bit 3) x experts 0-7 / 8-15 (lane bit 4)
        const int row = wn * 32 + nj * 16 + (lane & 7) + ((lane >> 4) << 3);
        ldsm4(b_s + swz(row, ks * 2 + ((lane >> 3) & 1)), b[nj]);
      }
#pragma unroll
      for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni)
          mma_bf16_16816(acc[mi][ni], a[mi], b[ni >> 1][(ni & 1) * 2], b[ni >> 1][(ni & 1) * 2 + 1]);
    }
  }
  cp_async_wait<0>();

#pragma unroll
  for (int mi = 0; mi < 2; ++mi) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int tok = m0 + wm * 32 + mi * 16 + (lane >> 2) + half * 8;
      if (tok >= T) continue;
      float* dst = logits + (size_t)tok * E;
#pragma unroll
      for (int ni = 0; ni < 4; ++ni) {
        const int ex = n0 + wn * 32 + ni * 8 + 2 * (lane & 3);
        if (ex < E) dst[ex] = acc[mi][ni][2 * half];
        if (ex + 1 < E) dst[ex + 1] = acc[mi][ni][2 * half + 1];
      }
    }
  }
}

}  // namespace

moe_status launch_router_gemm(const uint16_t* x, const uint16_t* w, int T, int H, int E, float* logits,
                              cudaStream_t s, bool pdl) {
  if (T == 0) return MOE_OK;
  cudaError_t e;
  if (T <= kGemvMaxT) {
    e = launch_ex(pdl, router_gemv_kernel, dim3(E), dim3(kGemvWarps * 32), 0, s, x, w, T, H, E, logits);
  } else {
    const int mtiles = (T + kBM - 1) / kBM;
    if (mtiles > 65535) return MOE_ERR_UNSUPPORTED;
    e = cudaFuncSetAttribute(router_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRouterSmem);
    if (e != cudaSuccess) return cuda_ok(e);
    const dim3 grid((E + kBN - 1) / kBN, mtiles);
    e = launch_ex(pdl, router_mma_kernel, grid, dim3(kMmaThreads), (size_t)kRouterSmem, s, x, w, T, H, E, logits);
  }
  if (e != cudaSuccess) return cuda_ok(e);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

}  // namespace moe
