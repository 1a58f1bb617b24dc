// Grouped NVFP4 GEMM for large groups, weight-only path (W4A16), with the
// dequantised weights in tensor memory.
//
// "vLLM on the NVIDIA DGX Spark: A Complete Technical Guide", section 4.3
// (the fused MoE's two expert GEMMs, SwiGLU and the top-k weight in the
// epilogues), section 5 (weight-only NVFP4: 4-bit weights dequantised to
// 16-bit inside the GEMM) and section 6.1 (alpha = 1/gs).
//
// Swap-AB tile: 128 weight rows are the MMA's M side, up to 128 rows of one
// expert group its N side. Producer warp q (lanes 32q..32q+31 of TMEM) owns
// 32 weight rows: each thread copies its row's raw e2m1 codes and E4M3
// scales for a 64-wide K stage into shared memory (cp.async), rebuilds the
// row from the m16n8k16 fragment layout with one register exchange with its
// partner row (lane ^ 8), converts to f16 with the hardware e2m1x2
// conversion, multiplies by the block scale (exact in f16) and writes the 32
// columns straight into TMEM with tcgen05.st. The MMA (kind::f16) reads A
// from TMEM and the activation rows from 128B-swizzled shared memory, so the
// dequantised weights never cross shared memory.
//
// The activation rows are f16 with a power-of-two row scale (the f16 copy
// from rows_to_f16); the epilogue multiplies by the row's 2^-s, alpha, and
// the routing weight (GEMM 2) or applies SwiGLU (GEMM 1).
//
// Warps: 0-7 producers in two sets of four that take alternate stages (the
// dependent chain load -> exchange -> convert -> tcgen05.st of one stage is
// long; two warps per scheduler overlap it), 8-11 epilogue (TMEM lane
// quarters), 12 MMA. Eight pipeline stages, two accumulator buffers of 128
// columns, eight A stages of 32 columns in TMEM. Every wait
// is bounded; on a timeout the kernel records MOE_ERR_TIMEOUT, drains, frees
// TMEM and exits.
#include "common.cuh"
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kM = 128;
constexpr int kBK = 64;
constexpr int kRowBytes = 128;       // one B row per stage: 64 f16
constexpr int kStages = 8;
constexpr int kLookahead = 3;        // per producer set; two sets alternate stages
constexpr int kMaxBN = 128;
constexpr int kProducerWarps = 8;    // two sets of four (one TMEM lane quarter each)
constexpr int kEpiWarp0 = kProducerWarps;
constexpr int kMmaWarp = kProducerWarps + 4;
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr int kProducers = 128;      // threads per producer set
constexpr int kBTile = kMaxBN * kRowBytes;  // 16 KB
constexpr int kRawPerThread = 48;           // 32 B codes + 8 B scales, padded to 16
constexpr int kRawStage = kProducers * kRawPerThread;
static_assert(2 * kLookahead < kStages, "both sets' copies in flight must fit the ring");
constexpr uint32_t kAccCols = 128;
constexpr uint32_t kAcol0 = 256;            // A stages: columns [256, 256 + 32 * kStages)
constexpr long long kWaitLimit = 4ll * 1000 * 1000 * 1000;

struct Args {
  const uint8_t* weights;
  size_t stride;
  const uint8_t* last_weights;
  int G, N, K;
  const int32_t* group_offsets;
  const uint16_t* a;       // f16 rows [*, K]
  const float* a_mul;      // per A row multiplier (2^-s)
  const int32_t* a_row_index;
  const float* row_scale;
  uint16_t* out;
  int rows_min;
  int* status;
};

struct Smem {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

struct Item {
  int g, row0, rows, bn, mt;
};

__device__ __forceinline__ Item decode_item(int idx, const int* pref, int G, int MT, const int32_t* off) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pref[mid] <= idx) lo = mid; else hi = mid - 1;
  }
  Item it;
  it.g = lo;
  const int local = idx - pref[lo];
  const int nt = local / MT;
  it.mt = local % MT;
  const int grows = off[lo + 1] - off[lo];
  it.row0 = off[lo] + nt * kMaxBN;
  it.rows = min(kMaxBN, grows - nt * kMaxBN);
  it.bn = (it.rows + 15) & ~15;
  return it;
}

__device__ __forceinline__ uint32_t byte_of(uint32_t w, int b) { return (w >> (8 * b)) & 0xffu; }

template <bool GATE_UP>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_f16_kernel(Args p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* b_tiles = base;                               // kStages x 16 KB
  uint8_t* raw = b_tiles + kStages * kBTile;             // kStages x 6 KB
  Smem* sm = reinterpret_cast<Smem*>(raw + kStages * kRawStage);
  int* pref = reinterpret_cast<int*>(sm + 1);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.G, K = p.K, N = p.N;
  const int MT = N / kM;
  const int KS = K / kBK;
  pdl_wait();

  for (int g = tid; g < G; g += kThreads) {
    const int rows = p.group_offsets[g + 1] - p.group_offsets[g];
    pref[g + 1] = rows > p.rows_min ? ((rows + kMaxBN - 1) / kMaxBN) * MT : 0;
  }
  if (tid == 0) {
    pref[0] = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm->full[i], kProducers);
      mbar_init(&sm->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm->tfull[i], 1);
      mbar_init(&sm->tempty[i], 128);
    }
    mbar_init(&sm->drain, 1);
    sm->abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int b0 = 1; b0 <= G; b0 += 32) {
      const int i = b0 + lane;
      int v = i <= G ? pref[i] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
      }
      if (i <= G) pref[i] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  if (warp == kMmaWarp) tmem_alloc(&sm->tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  const int total = pref[G];
  volatile int* abort = &sm->abort;

  if (warp < kProducerWarps) {
    // ------------------------------------------------------------- producers
    const int set = warp >> 2;                   // this set takes the stages j with j % 2 == set
    const int tau = tid & (kProducers - 1);      // TMEM lane = weight row in the tile
    const int blk = tau >> 4, g8 = tau & 7, hi = (tau >> 3) & 1;
    const uint32_t lane_taddr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    // byte selectors: the partner needs bytes (1-hi) and (3-hi) of my two
    // fragment words, I keep bytes hi and 2+hi
    const uint32_t sel_send = (uint32_t)((1 - hi) | ((5 - hi) << 4) | ((3 - hi) << 8) | ((7 - hi) << 12));
    const uint32_t sel_keep = (uint32_t)(hi | ((4 + hi) << 4) | ((2 + hi) << 8) | ((6 + hi) << 12));
    int j = 0, fin = set, pending = 0;
    auto finalize = [&](int i) {
      const int slot = i % kStages;
      const uint8_t* rw = raw + slot * kRawStage + tau * kRawPerThread;
      const uint4 wa4 = *reinterpret_cast<const uint4*>(rw);        // fragment lane 4g + 2hi
      const uint4 wb4 = *reinterpret_cast<const uint4*>(rw + 16);   // fragment lane 4g + 2hi + 1
      const uint2 sc = *reinterpret_cast<const uint2*>(rw + 32);
      const uint32_t wa[4] = {wa4.x, wa4.y, wa4.z, wa4.w};
      const uint32_t wb[4] = {wb4.x, wb4.y, wb4.z, wb4.w};
      uint32_t col[32];
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint32_t keep = __byte_perm(wa[s], wb[s], sel_keep);
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, __byte_perm(wa[s], wb[s], sel_send), 8);
        // bytes of lanes t = 0..3 for k 16s + 2t (lo) and 16s + 8 + 2t (hi)
        const uint32_t lo = hi ? __byte_perm(recv, keep, 0x5410) : __byte_perm(keep, recv, 0x5410);
        const uint32_t hh = hi ? __byte_perm(recv, keep, 0x7632) : __byte_perm(keep, recv, 0x7632);
        const int sb = 2 * (s & 1) + hi;  // my scale byte of step s
        const uint32_t sw = s < 2 ? sc.x : sc.y;
        const uint32_t scale = cvt_e4m3x2_f16x2(__byte_perm(sw, 0, sb | (sb << 4)));
        uint32_t flo[4], fhi[4];
        cvt_e2m1x8_f16(lo, flo);
        cvt_e2m1x8_f16(hh, fhi);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          col[8 * s + t] = hmul2_u32(flo[t], scale);
          col[8 * s + 4 + t] = hmul2_u32(fhi[t], scale);
        }
      }
      tmem_st32(lane_taddr + kAcol0 + slot * 32, col);
      fence_proxy_async_smem();  // the cp.async activation rows of this stage, for the tensor core
      tc_fence_before();
      mbar_arrive(&sm->full[slot]);
    };
    for (int item = blockIdx.x; item < total && !*abort; item += gridDim.x) {
      const Item it = decode_item(item, pref, G, MT, p.group_offsets);
      const uint8_t* wblk = (it.g == G - 1 && p.last_weights != nullptr) ? p.last_weights
                                                                         : p.weights + (size_t)it.g * p.stride;
      const uint8_t* wdata = wblk + sizeof(PrepHeader);
      const uint8_t* wsf = wdata + w4a16_data_bytes(N, K);
      const uint16_t* asrc[kMaxBN / 16];
#pragma unroll
      for (int q = 0; q < kMaxBN / 16; ++q) {
        const int n = (tau >> 3) + 16 * q;
        asrc[q] = nullptr;
        if (n < it.rows) {
          const int r = it.row0 + n;
          const int arow = p.a_row_index ? __ldg(p.a_row_index + r) : r;
          asrc[q] = p.a + (size_t)arow * K + (tau & 7) * 8;
        }
      }
      for (int ks = 0; ks < KS; ++ks, ++j) {
        if ((j & 1) != set) continue;
        const int slot = j % kStages;
        if (!mbar_wait(&sm->empty[slot], ((j / kStages) & 1) ^ 1, abort, kWaitLimit)) break;
        uint8_t* rw = raw + slot * kRawStage + tau * kRawPerThread;
        const size_t bidx = (size_t)(it.mt * 8 + blk) * KS + ks;
        const uint8_t* src = wdata + bidx * 512 + (4 * g8 + 2 * hi) * 16;
        cp_async_16(smem_u32(rw), src, 16);
        cp_async_16(smem_u32(rw + 16), src + 16, 16);
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(rw + 32)),
                     "l"(wsf + bidx * 64 + g8 * 8)
                     : "memory");
        const uint32_t bt = smem_u32(b_tiles + slot * kBTile);
#pragma unroll
        for (int q = 0; q < kMaxBN / 16; ++q) {
          const int n = (tau >> 3) + 16 * q, ch = tau & 7;
          if (n < it.bn) {
            const uint32_t dst = bt + n * kRowBytes + ((ch ^ (n & 7)) << 4);
            if (asrc[q] != nullptr) cp_async_16(dst, asrc[q] + ks * kBK, 16);
            else cp_async_16(dst, p.a, 0);  // zero fill
          }
        }
        cp_async_commit();
        if (++pending > kLookahead) {
          cp_async_wait<kLookahead>();
          finalize(fin);
          fin += 2;
          --pending;
        }
      }
    }
    cp_async_wait_all();
    while (pending > 0) {
      finalize(fin);
      fin += 2;
      --pending;
    }
  } else if (warp < kMmaWarp) {
    // -------------------------------------------------------------- epilogue
    const int q = warp - kEpiWarp0;
    const int rho = q * 32 + lane;
    int itc = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++itc) {
      const Item it = decode_item(item, pref, G, MT, p.group_offsets);
      const int acc = itc & 1;
      // per-row factors of the tile: lane l holds rows l, l + 32, ...
      float mulv[kMaxBN / 32];
#pragma unroll
      for (int i = 0; i < kMaxBN / 32; ++i) {
        const int n = 32 * i + lane;
        float m = 0.0f;
        if (n < it.rows) {
          const int r = it.row0 + n;
          const int arow = p.a_row_index ? __ldg(p.a_row_index + r) : r;
          m = __ldg(p.a_mul + arow);
          if (!GATE_UP && p.row_scale) m *= __ldg(p.row_scale + r);
        }
        mulv[i] = m;
      }
      if (!mbar_wait(&sm->tfull[acc], (itc >> 1) & 1, abort, kWaitLimit)) break;
      tc_fence_after();
      const uint8_t* wblk = (it.g == G - 1 && p.last_weights != nullptr) ? p.last_weights
                                                                         : p.weights + (size_t)it.g * p.stride;
      const PrepHeader* hdr = reinterpret_cast<const PrepHeader*>(wblk);
      const float a0 = hdr->alpha[0], a1 = hdr->alpha[1];
      for (int c0 = 0; c0 < it.bn; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + acc * kAccCols + c0, r);
        tmem_ld_wait();
        float m_chunk = 0.0f;
#pragma unroll
        for (int i = 0; i < kMaxBN / 32; ++i)
          if ((c0 >> 5) == i) m_chunk = mulv[i];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int n = c0 + c;
          const float m = __shfl_sync(0xffffffffu, m_chunk, n & 31);
          const float v = __uint_as_float(r[c]) * m;
          if (GATE_UP) {
            const float up = __shfl_down_sync(0xffffffffu, v, 8);
            if ((rho & 15) < 8 && n < it.rows) {
              const int f = 64 * it.mt + 8 * (rho >> 4) + (rho & 7);
              p.out[(size_t)(it.row0 + n) * (N / 2) + f] = float_to_bf16_bits(silu(v * a0) * (up * a1));
            }
          } else if (n < it.rows) {
            p.out[(size_t)(it.row0 + n) * N + it.mt * kM + rho] = float_to_bf16_bits(v * a0);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm->tempty[acc]);
    }
  } else {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      int j = 0, itc = 0;
      for (int item = blockIdx.x; item < total && !*abort; item += gridDim.x, ++itc) {
        const Item it = decode_item(item, pref, G, MT, p.group_offsets);
        const int acc = itc & 1;
        if (!mbar_wait(&sm->tempty[acc], ((itc >> 1) & 1) ^ 1, abort, kWaitLimit)) break;
        tc_fence_after();
        const uint32_t idesc = idesc_f16(kM, it.bn, 0);
        const uint32_t d = tmem + acc * kAccCols;
        bool ok = true;
        for (int ks = 0; ks < KS; ++ks, ++j) {
          const int slot = j % kStages;
          if (!mbar_wait(&sm->full[slot], (j / kStages) & 1, abort, kWaitLimit)) { ok = false; break; }
          tc_fence_after();
          const uint32_t bs = smem_u32(b_tiles + slot * kBTile);
          const uint32_t a_t = tmem + kAcol0 + slot * 32;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = smem_desc(bs + kk * 32, 16, 1024, kSwizzle128B);
            mma_f16_tmem_a(d, a_t + kk * 8, bd, idesc, (ks | kk) != 0);
          }
          tc_commit(&sm->empty[slot]);
        }
        if (!ok) break;
        tc_commit(&sm->tfull[acc]);
      }
      tc_commit(&sm->drain);
      const long long t0 = clock64();
      while (!mbar_try_wait(&sm->drain, 0) && clock64() - t0 < kWaitLimit) {
      }
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
  if (tid == 0 && sm->abort) set_status(p.status, MOE_ERR_TIMEOUT);
}

}  // namespace

static size_t smem_bytes(int G) {
  return 1024 + (size_t)kStages * (kBTile + kRawStage) + sizeof(Smem) + (size_t)(G + 1) * 4;
}

moe_status launch_gemm_tc_f16(const GemmPlan& pl, int rows_min, cudaStream_t s) {
  if (pl.num_groups <= 0) return MOE_OK;
  if (pl.a_f16 == nullptr || pl.a_mul == nullptr) return MOE_ERR_INVALID_ARG;
  Args a;
  a.weights = pl.weights;
  a.stride = pl.weight_stride;
  a.last_weights = pl.last_weights;
  a.G = pl.num_groups;
  a.N = pl.N;
  a.K = pl.K;
  a.group_offsets = pl.group_offsets;
  a.a = pl.a_f16;
  a.a_mul = pl.a_mul;
  a.a_row_index = pl.a_row_index;
  a.row_scale = pl.row_scale;
  a.out = pl.out;
  a.rows_min = rows_min;
  a.status = pl.status;
  const size_t smem = smem_bytes(pl.num_groups);
  if (smem > 227 * 1024) return MOE_ERR_UNSUPPORTED;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  auto k = pl.gate_up ? gemm_tc_f16_kernel<true> : gemm_tc_f16_kernel<false>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaError_t e = launch_ex(pl.pdl, k, dim3(sms), dim3(kThreads), smem, s, a);
  if (e != cudaSuccess) return cuda_ok(e);
  count_launches(1);
  return MOE_OK;
}

}  // namespace moe
