// Grouped NVFP4 GEMM for small groups (decode-sized: a handful of rows per
// expert), weight-only path (W4A16).
//
// "vLLM on the NVIDIA DGX Spark: A Complete Technical Guide", section 4.3
// (the two expert GEMMs of the fused MoE with SwiGLU and the top-k weight
// fused), section 5 (weight-only: 4-bit weights stay 4-bit in memory and
// are dequantised to 16-bit inside the GEMM) and section 6.1 (alpha = 1/gs).
//
// At a few rows per expert the layer is bound by the bytes of the touched
// experts' weights ("Seven Months of GB10 Field Notes": decode re-reads the
// active weights). So this kernel streams each weight tile from HBM exactly
// once, straight into registers (no shared-memory round trip), turns the
// e2m1 codes into f16 MMA fragments with the hardware e2m1x2 conversion,
// multiplies in the E4M3 block scale (e2m1 * e4m3 is exact in f16) and feeds
// mma.sync m16n8k16 with the group's rows (up to 8) as the N side.
//
// Activations enter as f16: each row is scaled by a power of two 2^s so
// that its largest magnitude lands in [2^14, 2^15); bf16 values are then
// exact in f16 (apart from magnitudes below 2^-24 of the row's maximum,
// which flush), and the epilogue multiplies by 2^-s again.
//
// Work item = (group, chunk of 8 rows, 128 weight rows). Each of the 8 warps
// of a CTA owns every 8th 64-wide K block (split-K inside the CTA) and all
// eight 16-row MMA tiles of the item; partial sums meet in shared memory.
// CTAs are persistent and take contiguous item ranges.
#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerPass = 8;
constexpr int kTileRows = 128;     // weight rows per item
constexpr int kMaxGroups = 1025;

struct SmallArgs {
  const uint8_t* weights;
  size_t stride;
  const uint8_t* last_weights;
  int G, N, K;
  const int32_t* group_offsets;
  const uint16_t* a;
  const int32_t* a_row_index;
  const float* row_scale;
  uint16_t* out;
  int rows_limit;
};

__device__ __forceinline__ int group_items(const int32_t* off, int g, int mt_count, int limit) {
  const int rows = off[g + 1] - off[g];
  if (rows <= 0 || rows > limit) return 0;
  return ((rows + kRowsPerPass - 1) / kRowsPerPass) * mt_count;
}

template <bool GATE_UP>
__global__ void __launch_bounds__(kThreads, 2) gemm_small_kernel(SmallArgs p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int K = p.K, N = p.N;
  const int xs_stride = K + 8;  // f16 elements per staged row (16-byte pad: no bank conflicts)
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem_raw);                                  // [8][K+8]
  float* red = reinterpret_cast<float*>(smem_raw + (size_t)kRowsPerPass * xs_stride * 2);  // [8][8][32][4]
  int* pref = reinterpret_cast<int*>(red + kWarps * 8 * 32 * 4);                          // [G+1]
  __shared__ float row_mul[kRowsPerPass];   // 2^-s per staged row
  __shared__ int row_out[kRowsPerPass];     // output row index, -1 if padding
  __shared__ int warp_tmp[32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int mt_count = N / kTileRows;
  const int G = p.G;

  // Item prefix sums over groups (each CTA computes its own copy).
  for (int g = tid; g < G; g += kThreads) pref[g + 1] = group_items(p.group_offsets, g, mt_count, p.rows_limit);
  if (tid == 0) pref[0] = 0;
  __syncthreads();
  if (tid < 32) {
    // serial-by-warp inclusive scan in chunks of 32
    int carry = 0;
    for (int base = 1; base <= G; base += 32) {
      const int i = base + lane;
      int v = i <= G ? pref[i] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
      }
      if (i <= G) pref[i] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();
  const int total = pref[G];
  const int i0 = (int)((long long)total * blockIdx.x / gridDim.x);
  const int i1 = (int)((long long)total * (blockIdx.x + 1) / gridDim.x);

  const int kblocks = K / 64;
  int cur_g = -1, cur_c = -1;
  for (int item = i0; item < i1; ++item) {
    // group of this item: last g with pref[g] <= item
    int lo = 0, hi = G - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pref[mid] <= item) lo = mid; else hi = mid - 1;
    }
    const int g = lo;
    const int local = item - pref[g];
    const int c = local / mt_count, mt = local % mt_count;
    const int row0 = p.group_offsets[g] + c * kRowsPerPass;
    const int nrows = min(kRowsPerPass, p.group_offsets[g + 1] - row0);

    if (g != cur_g || c != cur_c) {
      __syncthreads();  // everyone is done with the previous rows
      // warp w stages row w: max |x|, power-of-two scale, f16 conversion
      const int r = warp;
      uint16_t* dst = xs + (size_t)r * xs_stride;
      if (r < nrows) {
        const int orow = row0 + r;
        const int arow = p.a_row_index ? p.a_row_index[orow] : orow;
        const uint4* src = reinterpret_cast<const uint4*>(p.a + (size_t)arow * K);
        uint32_t m = 0;
        for (int i = lane; i < K / 8; i += 32) {
          const uint4 v = __ldg(src + i);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) m = max(m, max(w[j] & 0x7fffu, (w[j] >> 16) & 0x7fffu));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
        // m = bf16 bits of the row max; its exponent e gives max in [2^(e-127), 2^(e-126))
        const int e = (int)(m >> 7);  // biased exponent (0 for zero/subnormal rows)
        int sh = (m == 0) ? 0 : 141 - max(e, 1);  // 2^(e-127+sh) = 2^14
        sh = max(-113, min(sh, 126));             // keeps 2^sh and 2^-sh normal floats
        const float up = __int_as_float((127 + sh) << 23);
        for (int i = lane; i < K / 8; i += 32) {
          const uint4 v = __ldg(src + i);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
          uint32_t o[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float f0 = __uint_as_float(w[j] << 16) * up;
            const float f1 = __uint_as_float(w[j] & 0xffff0000u) * up;
            const __half2 h = __floats2half2_rn(f0, f1);
            o[j] = *reinterpret_cast<const uint32_t*>(&h);
          }
          *reinterpret_cast<uint4*>(dst + i * 8) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if (lane == 0) {
          row_mul[r] = __int_as_float((127 - sh) << 23);
          row_out[r] = orow;
        }
      } else {
        for (int i = lane; i < K / 8; i += 32) *reinterpret_cast<uint4*>(dst + i * 8) = make_uint4(0, 0, 0, 0);
        if (lane == 0) {
          row_mul[r] = 0.0f;
          row_out[r] = -1;
        }
      }
      cur_g = g;
      cur_c = c;
      __syncthreads();
    }

    const uint8_t* blk = (g == G - 1 && p.last_weights != nullptr) ? p.last_weights
                                                                  : p.weights + (size_t)g * p.stride;
    const PrepHeader* hdr = reinterpret_cast<const PrepHeader*>(blk);
    const uint8_t* data = blk + sizeof(PrepHeader);
    const uint8_t* sfp = data + w4a16_data_bytes(N, K);

    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;

    const int g8 = lane >> 2, t4 = lane & 3;
    const uint16_t* xrow = xs + (size_t)g8 * xs_stride + 2 * t4;
    for (int kb = warp; kb < kblocks; kb += kWarps) {
      uint4 wq[8];
      uint2 sq[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const size_t b = (size_t)(mt * 8 + i) * kblocks + kb;
        wq[i] = ldg_stream(data + b * 512 + lane * 16);
        sq[i] = ldg_stream2(sfp + b * 64 + g8 * 8);
      }
      uint32_t bf[4][2];
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        bf[s][0] = *reinterpret_cast<const uint32_t*>(xrow + kb * 64 + 16 * s);
        bf[s][1] = *reinterpret_cast<const uint32_t*>(xrow + kb * 64 + 16 * s + 8);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t wv[4] = {wq[i].x, wq[i].y, wq[i].z, wq[i].w};
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          uint32_t a[4];
          cvt_e2m1x8_f16(wv[s], a);
          // block scales of rows g and g+8 for k16 group s, each duplicated
          // into both halves so the MMA fragments multiply element-wise
          const uint32_t sg = cvt_e4m3x2_f16x2(__byte_perm(sq[i].x, 0, s | (s << 4)));
          const uint32_t s8 = cvt_e4m3x2_f16x2(__byte_perm(sq[i].y, 0, s | (s << 4)));
          a[0] = hmul2_u32(a[0], sg);
          a[1] = hmul2_u32(a[1], s8);
          a[2] = hmul2_u32(a[2], sg);
          a[3] = hmul2_u32(a[3], s8);
          mma_f16_16816(acc[i], a, bf[s][0], bf[s][1]);
        }
      }
    }

    // Cross-warp reduction of the split-K partial sums.
    float* my = red + ((size_t)warp * 8 * 32) * 4;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      *reinterpret_cast<float4*>(my + ((size_t)i * 32 + lane) * 4) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    __syncthreads();
    {
      const int i = tid >> 5;  // 16-row tile within the item
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float4 v = *reinterpret_cast<const float4*>(red + (((size_t)w * 8 + i) * 32 + lane) * 4);
        c[0] += v.x; c[1] += v.y; c[2] += v.z; c[3] += v.w;
      }
      const int mb = mt * 8 + i;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int n = 2 * t4 + q;  // staged row
        if (n >= nrows) continue;
        const int orow = row_out[n];
        const float rm = row_mul[n];
        if (GATE_UP) {
          const float gv = c[q] * rm * hdr->alpha[0];
          const float uv = c[2 + q] * rm * hdr->alpha[1];
          const int f = 8 * mb + g8;
          p.out[(size_t)orow * (N / 2) + f] = float_to_bf16_bits(silu(gv) * uv);
        } else {
          const float rs = p.row_scale ? p.row_scale[orow] : 1.0f;
          const int hr = 16 * mb + g8;
          p.out[(size_t)orow * N + hr] = float_to_bf16_bits(c[q] * rm * hdr->alpha[0] * rs);
          p.out[(size_t)orow * N + hr + 8] = float_to_bf16_bits(c[2 + q] * rm * hdr->alpha[0] * rs);
        }
      }
    }
    __syncthreads();
  }
  (void)warp_tmp;
}

}  // namespace

size_t gemm_small_smem_bytes(int K, int G) {
  return (size_t)kRowsPerPass * (K + 8) * 2 + (size_t)kWarps * 8 * 32 * 4 * 4 + (size_t)(G + 1) * 4;
}

moe_status launch_gemm_small_w4a16(const GemmPlan& pl, int rows_limit, cudaStream_t s) {
  if (pl.num_groups <= 0) return MOE_OK;
  if (pl.num_groups > kMaxGroups) return MOE_ERR_UNSUPPORTED;
  SmallArgs a;
  a.weights = pl.weights;
  a.stride = pl.weight_stride;
  a.last_weights = pl.last_weights;
  a.G = pl.num_groups;
  a.N = pl.N;
  a.K = pl.K;
  a.group_offsets = pl.group_offsets;
  a.a = static_cast<const uint16_t*>(pl.a);
  a.a_row_index = pl.a_row_index;
  a.row_scale = pl.row_scale;
  a.out = pl.out;
  a.rows_limit = rows_limit;
  const size_t smem = gemm_small_smem_bytes(pl.K, pl.num_groups);
  if (smem > 227 * 1024) return MOE_ERR_UNSUPPORTED;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int per_sm = smem <= 110 * 1024 ? 2 : 1;
  // upper bound on items: every row its own chunk
  const long long max_items = (long long)((pl.max_rows + kRowsPerPass - 1) / kRowsPerPass + pl.num_groups) *
                              (pl.N / kTileRows);
  const int grid = (int)std::max<long long>(1, std::min<long long>((long long)sms * per_sm, max_items));
  if (pl.gate_up) {
    auto k = gemm_small_kernel<true>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k<<<grid, kThreads, smem, s>>>(a);
    count_launches(1);
  } else {
    auto k = gemm_small_kernel<false>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    k<<<grid, kThreads, smem, s>>>(a);
    count_launches(1);
  }
  return cuda_ok(cudaGetLastError());
}

}  // namespace moe
