// BF16 -> NVFP4 quantisation, standalone SwiGLU and the deterministic
// combine.
//
// Quantisation: "vLLM on the NVIDIA DGX Spark: A Complete Technical Guide",
// section 4.3 (BF16 input quantised to FP4 inside the fused kernel) and
// section 6.1 (e2m1 elements, one E4M3 scale per 16 along K, one fp32
// global scale); the 448 clamp of the block scale is named in "Serving
// Solar Open 2 on DGX Spark", "Supporting real NVFP4 checkpoints"; the
// global scale is the quant-convention (448*6)/amax ("GLM-5.3-Flash-NVFP4 #4"
// discussion, follow-up on the MoE fault).
// Combine: same guide, section 7.1 ([Combine]) and section 4.3 (top-k weight
// reduction).
#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// amax = max |x| over n bf16 values. 16-byte loads, grid-stride; one atomic
// per block on the float's bit pattern (exact and order-independent).
__global__ void __launch_bounds__(256) amax_bf16_kernel(const uint16_t* __restrict__ x, size_t n,
                                                        float* __restrict__ amax) {
  pdl_wait();
  uint32_t m = 0;  // running max of |x| as a bf16 bit pattern (monotonic in magnitude)
  const size_t nvec = n / 8;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nvec;
       i += (size_t)gridDim.x * blockDim.x) {
    const uint4 v = ldg_stream(xv + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      m = max(m, finite_mag(w[j] & 0x7fffu));
      m = max(m, finite_mag((w[j] >> 16) & 0x7fffu));
    }
  }
  for (size_t i = nvec * 8 + blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    m = max(m, finite_mag((uint32_t)(x[i] & 0x7fffu)));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
  __shared__ uint32_t red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) m = max(m, red[i]);
    atomic_max_nonneg(amax, __uint_as_float(m << 16));
  }
}

moe_status launch_amax_bf16(const uint16_t* x, size_t n, float* amax, cudaStream_t s, bool pdl) {
  if (n == 0) return MOE_OK;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  size_t want = (n / 8 + 255) / 256;
  size_t cap = (size_t)sms * 8;
  int blocks = (int)(want == 0 ? 1 : (want < cap ? want : cap));
  cudaError_t e = launch_ex(pdl, amax_bf16_kernel, dim3(blocks), dim3(256), 0, s, x, n, amax);
  if (e != cudaSuccess) return cuda_ok(e);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

// e2m1 codes of two fp32 values with the hardware conversion: round to
// nearest, ties to the even code, saturating at 6, the sign kept (also on a
// zero result); `lo` lands in bits 0-3 of the byte, `hi` in bits 4-7.
__device__ __forceinline__ uint32_t e2m1x2_rn(float lo, float hi) {
  uint16_t r;
  asm("{\n .reg .b8 b;\n cvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n cvt.u16.u8 %0, b;\n}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r & 0xffu;
}

// E4M3 (fn) encoding of a non-negative fp32, nearest-even, saturating at 448.
__device__ __forceinline__ uint32_t e4m3_encode_sat(float s) {
  uint16_t r;
  // both halves get s, so the byte order of the packed result does not matter
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(s), "f"(s));
  return r & 0xffu;
}

__device__ __forceinline__ float e4m3_decode(uint32_t code) {
  const uint32_t h2 = cvt_e4m3x2_f16x2((code & 0xffu) * 0x101u);  // same byte in both halves
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
}

// The global scale of a quantisation: a static (calibrated) one when
// gs_static > 0, else the dynamic 2688 / amax (1 when amax is 0).
__device__ __forceinline__ float global_scale_of(const float* amax_p, float gs_static) {
  if (gs_static > 0.0f) return gs_static;
  const float amax = *amax_p;
  return amax > 0.0f ? 2688.0f / amax : 1.0f;
}

// One thread per 16-element block: 32 bytes of bf16 in, 8 bytes of codes and
// 1 scale byte out.
__global__ void __launch_bounds__(256) quantize_bf16_kernel(const uint16_t* __restrict__ x, int rows, int K,
                                                            const float* __restrict__ amax_p,
                                                            uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                                            float* __restrict__ gs_out, float gs_static) {
  pdl_wait();
  const float gs = global_scale_of(amax_p, gs_static);
  const size_t nblk = (size_t)rows * (K / 16);
  const size_t b = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (b == 0 && gs_out != nullptr) *gs_out = gs;
  if (b >= nblk) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + b * 16);
  const uint4 v0 = ldg_stream(src), v1 = ldg_stream(src + 1);
  const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  float f[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    f[2 * j] = __uint_as_float(w[j] << 16);
    f[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
  }
  float bmax = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) bmax = fmaxf(bmax, fabsf(f[j]));
  const float s = __fmul_rn(__fdiv_rn(bmax, 6.0f), gs);
  const uint32_t code = e4m3_encode_sat(s);
  const float sval = e4m3_decode(code);
  uint32_t lo = 0, hi = 0;
  if (sval > 0.0f) {
    const float r = __fdiv_rn(gs, sval);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t b = e2m1x2_rn(__fmul_rn(f[2 * j], r), __fmul_rn(f[2 * j + 1], r));
      if (j < 4) lo |= b << (8 * j);
      else hi |= b << (8 * (j - 4));
    }
  }
  *reinterpret_cast<uint2*>(q + b * 8) = make_uint2(lo, hi);
  sf[b] = (uint8_t)code;
}

moe_status launch_quantize_bf16(const uint16_t* x, int rows, int K, const float* amax, uint8_t* q,
                                uint8_t* sf, float* gs_out, float gs_static, cudaStream_t s, bool pdl) {
  const size_t nblk = (size_t)rows * (K / 16);
  const int blocks = (int)((nblk + 255) / 256);
  cudaError_t e = launch_ex(pdl, quantize_bf16_kernel, dim3(blocks > 0 ? blocks : 1), dim3(256), 0, s, x, rows,
                            K, amax, q, sf, gs_out, gs_static);
  if (e != cudaSuccess) return cuda_ok(e);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

// ---------------------------------------------------------------------------
// MXFP4 ("vLLM on the NVIDIA DGX Spark", section 6.4 "NVFP4 vs MXFP4"): e2m1
// elements with one power-of-two E8M0 scale per 32 along K and no global
// scale. Per block: e = floor(log2 amax) - 2 (6 = 1.5 * 2^2 is e2m1's
// largest value, so amax / 2^e lies in [4, 8)), clamped to [-127, 127], an
// all-zero block takes e = -127 and zero codes; the scale code is e + 127 and
// code_i = e2m1(x_i * 2^-e), nearest even, saturating at 6, sign kept. The
// multiply by 2^-e is exact.

// floor(log2 a) for a positive finite fp32 a, from its bits (subnormals too).
__device__ __forceinline__ int floor_log2_pos(float a) {
  const uint32_t bits = __float_as_uint(a);
  const int ex = (int)((bits >> 23) & 0xffu);
  if (ex > 0) return ex - 127;
  return (31 - __clz((int)(bits & 0x7fffffu))) - 149;
}

// 32 bf16 values (64 bytes, 16-byte aligned) -> 16 bytes of codes and the
// E8M0 scale code.
__device__ __forceinline__ void quant_block32_mx(const uint16_t* src, uint4& codes, uint32_t& scale_code) {
  const uint4* v = reinterpret_cast<const uint4*>(src);
  uint32_t wv[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 q = ldg_stream(v + i);
    wv[4 * i] = q.x;
    wv[4 * i + 1] = q.y;
    wv[4 * i + 2] = q.z;
    wv[4 * i + 3] = q.w;
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i)
    amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(wv[i] << 16)), fabsf(__uint_as_float(wv[i] & 0xffff0000u))));
  if (!(amax > 0.0f)) {  // all zeros (a NaN block, outside the contract, also lands here)
    codes = make_uint4(0u, 0u, 0u, 0u);
    scale_code = 0u;
    return;
  }
  const int e = max(-127, min(127, floor_log2_pos(amax) - 2));
  const float mul = __int_as_float((127 - e) << 23);  // 2^-e, a normal float for e in [-127, 126]
  uint32_t out[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t word = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t x = wv[4 * w + b];
      word |= e2m1x2_rn(__fmul_rn(__uint_as_float(x << 16), mul), __fmul_rn(__uint_as_float(x & 0xffff0000u), mul))
              << (8 * b);
    }
    out[w] = word;
  }
  codes = make_uint4(out[0], out[1], out[2], out[3]);
  scale_code = (uint32_t)(e + 127);
}

// One thread per 32-element block: codes [rows, K/2], scales [rows, K/32].
__global__ void __launch_bounds__(256) quantize_mx_bf16_kernel(const uint16_t* __restrict__ x, int rows, int K,
                                                               uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  const size_t nblk = (size_t)rows * (K / 32);
  const size_t b = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (b >= nblk) return;
  uint4 codes;
  uint32_t code;
  quant_block32_mx(x + b * 32, codes, code);
  *reinterpret_cast<uint4*>(q + b * 16) = codes;
  sf[b] = (uint8_t)code;
}

moe_status launch_quantize_mx(const uint16_t* x, int rows, int K, uint8_t* q, uint8_t* sf, cudaStream_t s) {
  const size_t nblk = (size_t)rows * (K / 32);
  if (nblk == 0) return MOE_OK;
  const int blocks = (int)((nblk + 255) / 256);
  quantize_mx_bf16_kernel<<<blocks, 256, 0, s>>>(x, rows, K, q, sf);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

// ---------------------------------------------------------------------------
// Per-tile assembly of the block-scaled GEMMs' activation operands from rows
// quantised one by one (quantize_bf16_kernel / quantize_mx_bf16_kernel:
// codes [src_rows, K/2], scales [src_rows, K/BLK]). One CTA per 128-row tile
// of a group (tiles numbered group by group, ceil(rows_g / 128) each):
// * with `src_row` (the grouped row's source row: x's token), each tile row's
//   codes are copied from its source row — a token's codes reach its k+1
//   grouped rows; without it the codes are already in place (h, quantised in
//   group order) and only the scales move;
// * the tile's scale atoms (the tcgen05 scale-factor layout: one 512-byte
//   atom per four consecutive blocks, row m's 4 bytes at (m % 32) * 16 +
//   (m / 32) * 4) are assembled in shared memory, rows past the group's end
//   left 0, and written out whole, 16 bytes per thread.
// So the scattered 4-byte writes of a token-major pass become coalesced ones.
template <int BLK>
__global__ void __launch_bounds__(256) tile_gather_kernel(const uint8_t* __restrict__ q_src,
                                                          const uint8_t* __restrict__ sf_src,
                                                          const int32_t* __restrict__ src_row, int K,
                                                          const int32_t* __restrict__ gofs, int G, int q_rows,
                                                          uint8_t* __restrict__ q, uint8_t* __restrict__ sf_tiles) {
  pdl_wait();
  extern __shared__ __align__(16) uint8_t smem_tg[];
  const int atoms = K / (4 * BLK), NB = K / BLK, W = NB / 4;   // atoms per tile; scale bytes and words per row
  uint8_t* at = smem_tg;                                                   // [atoms * 512]
  int* s_tb = reinterpret_cast<int*>(smem_tg + (size_t)atoms * 512);     // [G + 1] first tile of each group
  const int tid = threadIdx.x;
  if (tid < 32) {  // exclusive prefix of ceil(rows / 128) over the groups
    int carry = 0;
    for (int g0 = 0; g0 <= G; g0 += 32) {
      const int g = g0 + tid;
      const int v = g < G ? (__ldg(gofs + g + 1) - __ldg(gofs + g) + 127) / 128 : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += t;
      }
      if (g <= G) s_tb[g] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  for (int i = tid; i < atoms * 32; i += 256) reinterpret_cast<uint4*>(at)[i] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  const int t = blockIdx.x;
  if (t >= s_tb[G]) return;   // past the tiles this routing has (the grid is an upper bound)
  int lo = 0, hi = G - 1;     // group of tile t: the last g with s_tb[g] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_tb[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int row0 = __ldg(gofs + lo) + (t - s_tb[lo]) * 128;
  const int nrows = min(128, __ldg(gofs + lo + 1) - row0);
  // scales: thread (row m, four words of it); consecutive threads take
  // consecutive rows, so their shared-memory words are 16 bytes apart
  const int W4 = (W + 3) / 4;
  for (int i = tid; i < 128 * W4; i += 256) {
    const int m = i & 127, c = i >> 7;
    if (m >= nrows) continue;
    const int src = src_row ? __ldg(src_row + row0 + m) : row0 + m;
    const uint8_t* rowp = sf_src + (size_t)src * NB;
    const int w0 = 4 * c;
    uint32_t wv[4];
    if (w0 + 4 <= W && (NB & 15) == 0) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(rowp) + c);
      wv[0] = v.x; wv[1] = v.y; wv[2] = v.z; wv[3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) wv[e] = w0 + e < W ? __ldg(reinterpret_cast<const uint32_t*>(rowp) + w0 + e) : 0u;
    }
    const int off = (m & 31) * 16 + (m >> 5) * 4;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (w0 + e < W) *reinterpret_cast<uint32_t*>(at + (size_t)(w0 + e) * 512 + off) = wv[e];
  }
  // codes: a warp per row, 16 bytes per lane
  if (src_row != nullptr) {
    const int n16 = K / 32;   // 16-byte pieces of a row's codes
    const int nq = min(nrows, q_rows - row0);   // rows q has room for
    for (int m = tid >> 5; m < nq; m += 8) {
      const uint4* from = reinterpret_cast<const uint4*>(q_src + (size_t)__ldg(src_row + row0 + m) * (K / 2));
      uint4* to = reinterpret_cast<uint4*>(q + (size_t)(row0 + m) * (K / 2));
      for (int j = tid & 31; j < n16; j += 32) to[j] = __ldg(from + j);   // read by up to k+1 tiles: keep in L2
    }
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(sf_tiles + (size_t)t * atoms * 512);
  for (int i = tid; i < atoms * 32; i += 256) dst[i] = reinterpret_cast<const uint4*>(at)[i];
}

moe_status launch_tile_gather(const uint8_t* q_src, const uint8_t* sf_src, const int32_t* src_row, int K,
                              const int32_t* gofs, int G, int tiles_max, int q_rows, uint8_t* q, uint8_t* sf_tiles,
                              bool mx, cudaStream_t s) {
  if (K % 256 || G <= 0) return MOE_ERR_UNSUPPORTED;
  if (tiles_max <= 0) return MOE_OK;
  const int atoms = K / (4 * (mx ? 32 : 16));
  const size_t smem = (size_t)atoms * 512 + (size_t)(G + 1) * sizeof(int);
  if (smem > 227 * 1024) return MOE_ERR_UNSUPPORTED;
  auto k = mx ? tile_gather_kernel<32> : tile_gather_kernel<16>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_ok(e);
  e = launch_ex(false, k, dim3(tiles_max), dim3(256), smem, s, q_src, sf_src, src_row, K, gofs, G, q_rows, q,
                sf_tiles);
  if (e != cudaSuccess) return cuda_ok(e);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}


// ---------------------------------------------------------------------------
// Re-rounding E4M3 block scales by a global-scale ratio (checkpoint import,
// "Serving Solar Open 2 on DGX Spark", "Supporting real NVFP4 checkpoints":
// reciprocal global scales folded into the FP8 block scales with
// re-rounding, clamped at 448): out = E4M3(e4m3[in] * ratio), one correctly
// rounded fp32 multiply, then nearest even with saturation at 448. A code
// with the sign bit set or a NaN code sets *flag and is copied unchanged.
// One code per thread, grid-stride.
// `in` and `out` may be the same array (no __restrict__): each element is read
// and then written by one thread.
__global__ void __launch_bounds__(256) fold_scales_kernel(const uint8_t* in, size_t n, float ratio, uint8_t* out,
                                                          int* flag) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += stride) {
    const uint32_t c = in[i];
    if ((c & 0x80u) || (c & 0x7fu) == 0x7fu) {
      atomicOr(flag, 1);
      out[i] = (uint8_t)c;
      continue;
    }
    out[i] = (uint8_t)e4m3_encode_sat(__fmul_rn(e4m3_decode(c), ratio));
  }
}

moe_status launch_fold_scales(const uint8_t* in, size_t n, float ratio, uint8_t* out, int* flag, cudaStream_t s) {
  if (n == 0) return MOE_OK;
  const size_t want = (n + 255) / 256;
  const int blocks = (int)(want < 152 * 8 ? want : 152 * 8);
  fold_scales_kernel<<<blocks, 256, 0, s>>>(in, n, ratio, out, flag);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

// ---------------------------------------------------------------------------
// bf16 rows -> f16 rows with a power-of-two row scale (one warp per row);
// dst row r comes from src row src_index[r] (r when src_index is null).
// With the row's largest magnitude in [2^14, 2^15) every bf16 value is exact
// in f16 except magnitudes below 2^-24 of that maximum, which flush.
// V > 0: the row (at most V 16-byte pieces per lane) stays in registers
// between the max and the conversion, so it is read once; V = 0 reads it twice.
template <int V>
__global__ void __launch_bounds__(256) rows_to_f16_kernel(const uint16_t* __restrict__ src,
                                                          const int32_t* __restrict__ src_index, int rows, int K,
                                                          uint16_t* __restrict__ dst, float* __restrict__ mul,
                                                          const int32_t* __restrict__ rows_limit) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int row = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  if (row >= rows || (rows_limit != nullptr && row >= __ldg(rows_limit))) return;
  const int srow = src_index ? __ldg(src_index + row) : row;
  const uint4* s = reinterpret_cast<const uint4*>(src + (size_t)srow * K);
  uint4* d = reinterpret_cast<uint4*>(dst + (size_t)row * K);
  const int n16 = K / 8;
  auto row_max = [](uint32_t m, const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) m = max(m, max(finite_mag(w[q] & 0x7fffu), finite_mag((w[q] >> 16) & 0x7fffu)));
    return m;
  };
  uint32_t m = 0;
  uint4 keep[V > 0 ? V : 1];
  if (V > 0) {
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const int i = lane + 32 * j;
      keep[j] = i < n16 ? __ldg(s + i) : make_uint4(0u, 0u, 0u, 0u);
      m = row_max(m, keep[j]);
    }
  } else {
    for (int i = lane; i < n16; i += 32) m = row_max(m, __ldg(s + i));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
  const int e = (int)(m >> 7);
  int sh = (m == 0) ? 0 : 141 - max(e, 1);
  sh = max(-113, min(sh, 126));
  const float up = __int_as_float((127 + sh) << 23);
  auto convert = [up](const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __half2 h = __floats2half2_rn(__uint_as_float(w[q] << 16) * up, __uint_as_float(w[q] & 0xffff0000u) * up);
      o[q] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  };
  if (V > 0) {
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const int i = lane + 32 * j;
      if (i < n16) d[i] = convert(keep[j]);
    }
  } else {
    for (int i = lane; i < n16; i += 32) d[i] = convert(__ldg(s + i));
  }
  if (lane == 0) mul[row] = __int_as_float((127 - sh) << 23);
}

moe_status launch_rows_to_f16(const uint16_t* src, const int32_t* src_index, int rows, int K, uint16_t* dst,
                              float* mul, cudaStream_t s, bool pdl, const int32_t* rows_limit) {
  if (rows == 0) return MOE_OK;
  const int blocks = (int)(((size_t)rows * 32 + 255) / 256);
  const int per = (K / 8 + 31) / 32;   // 16-byte pieces of a row per lane
  // (keeping up to 16 pieces per lane in registers halved the resident warps
  // and doubled the time at K = 4096; up to 8 pieces the single read pays)
  auto k = per <= 8 ? rows_to_f16_kernel<8> : rows_to_f16_kernel<0>;
  cudaError_t e = launch_ex(pdl, k, dim3(blocks), dim3(256), 0, s, src, src_index, rows, K, dst, mul, rows_limit);
  if (e != cudaSuccess) return cuda_ok(e);
  count_launches(1);
  return MOE_OK;
}

// ---------------------------------------------------------------------------
// h = silu(gate) * up, gate in columns [0, I), up in [I, 2I).
__global__ void swiglu_kernel(const float* __restrict__ gu, int rows, int I, uint16_t* __restrict__ h) {
  const size_t n = (size_t)rows * I;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t r = i / I, c = i % I;
    const float g = gu[r * 2 * I + c];
    const float u = gu[r * 2 * I + I + c];
    h[i] = float_to_bf16_bits(silu(g) * u);
  }
}

moe_status launch_swiglu(const float* gu, int rows, int I, uint16_t* h, cudaStream_t s) {
  const size_t n = (size_t)rows * I;
  if (n == 0) return MOE_OK;
  const size_t want = (n + 255) / 256;
  const int blocks = (int)(want < 152 * 16 ? want : 152 * 16);
  swiglu_kernel<<<blocks, 256, 0, s>>>(gu, rows, I, h);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

// ---------------------------------------------------------------------------
__device__ __forceinline__ void combine_token(const uint16_t* __restrict__ y, const int32_t* __restrict__ inv_perm,
                                              const float* __restrict__ topk_w, const float* __restrict__ y_shared,
                                              int k, int H, uint16_t* __restrict__ out, int t, int c8) {
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  // the token's rows eight at a time: every index, then every row load, is
  // issued before the first use (no chain of dependent loads per row); the
  // sum still runs j = 0, 1, ... in order
  for (int j0 = 0; j0 < k; j0 += 8) {
    int row[8];
    float wt[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + u;
      row[u] = j < k ? __ldg(inv_perm + (size_t)t * k + j) : -1;
      wt[u] = (j < k && topk_w != nullptr) ? __ldg(topk_w + (size_t)t * k + j) : 1.0f;
    }
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      v[u] = row[u] >= 0 ? ldg_stream(y + (size_t)row[u] * H + (size_t)c8 * 8) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (row[u] < 0) continue;
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] += __uint_as_float(w[i] << 16) * wt[u];
        acc[2 * i + 1] += __uint_as_float(w[i] & 0xffff0000u) * wt[u];
      }
    }
  }
  if (y_shared != nullptr) {
    const float4* ys = reinterpret_cast<const float4*>(y_shared + (size_t)t * H + (size_t)c8 * 8);
    const float4 a = __ldg(ys), b = __ldg(ys + 1);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += v[i];
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = (uint32_t)float_to_bf16_bits(acc[2 * i]) | ((uint32_t)float_to_bf16_bits(acc[2 * i + 1]) << 16);
  *reinterpret_cast<uint4*>(out + (size_t)t * H + (size_t)c8 * 8) = make_uint4(o[0], o[1], o[2], o[3]);
}

// out[t] = sum_j y[inv_perm[t*k + j]] (* topk_w[t, j]) + y_shared[t], fp32 in
// that fixed order, rounded once to bf16 (routed rows bf16, the shared
// expert's rows fp32). One thread per 8 outputs (16-byte loads and stores); a
// grid of (H/8/64) x min(T, 65535) blocks of 64 threads, the y blocks
// stepping over the tokens (grid.y is capped at 65535).
__global__ void __launch_bounds__(64) combine_kernel(const uint16_t* __restrict__ y,
                                                     const int32_t* __restrict__ inv_perm,
                                                     const float* __restrict__ topk_w,
                                                     const float* __restrict__ y_shared, int T, int k, int H,
                                                     uint16_t* __restrict__ out) {
  pdl_wait();
  const int c8 = blockIdx.x * blockDim.x + threadIdx.x;  // chunk of 8 columns
  if (c8 * 8 >= H) return;
  for (int t = blockIdx.y; t < T; t += gridDim.y) combine_token(y, inv_perm, topk_w, y_shared, k, H, out, t, c8);
}
moe_status launch_combine(const uint16_t* y, const int32_t* inv_perm, const float* topk_w,
                          const float* y_shared, int T, int k, int H, uint16_t* out, cudaStream_t s, bool pdl) {
  if (T == 0) return MOE_OK;
  const int chunks = H / 8;
  dim3 grid((chunks + 63) / 64, T < 65535 ? T : 65535);
  cudaError_t e = launch_ex(pdl, combine_kernel, grid, dim3(64), 0, s, y, inv_perm, topk_w, y_shared, T, k, H,
                            out);
  if (e != cudaSuccess) return cuda_ok(e);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

}  // namespace moe
