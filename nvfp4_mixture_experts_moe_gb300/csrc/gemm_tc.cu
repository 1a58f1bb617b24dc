// Grouped NVFP4 GEMM for large groups on the 5th-generation tensor cores
// (tcgen05, accumulators in TMEM), weight-only path (W4A16).
//
// "vLLM on the NVIDIA DGX Spark: A Complete Technical Guide", section 4.3
// (the fused MoE's two expert GEMMs with SwiGLU and the top-k weight in the
// epilogues), section 5 (weight-only NVFP4: 4-bit weights dequantised to
// 16-bit inside the GEMM, the MMA runs in 16-bit) and section 6.1 (alpha =
// 1/gs).
//
// Tile: 128 weight rows (the MMA's M side) x up to 256 rows of one expert
// group (N side) x K. The weights stay e2m1 in HBM; producer warps copy the
// raw codes and E4M3 scales into shared memory with cp.async, turn them into
// bf16 (e2m1 * e4m3 is exact in bf16; the global scale 1/gs is applied in
// the epilogue) and write them in the 128-byte-swizzled K-major layout the
// MMA reads. The group's activation rows (gathered through the row -> token
// map) arrive the same way. One thread issues tcgen05.mma (kind::f16, bf16
// inputs, fp32 accumulate in TMEM); four epilogue warps read the
// accumulators back with tcgen05.ld and apply SwiGLU (GEMM 1) or the
// routing weight (GEMM 2).
//
// Warp roles (288 threads): 0-3 producers, 4-7 epilogue (TMEM lane quarters
// 0-3), 8 MMA issue + TMEM allocation. CTAs are persistent (one per SM) and
// walk the (group, N tile, M tile) items round-robin. Four pipeline stages,
// two accumulator buffers. Every wait is bounded; on a timeout the kernel
// records MOE_ERR_TIMEOUT, drains its copies and MMAs, frees TMEM and exits.
#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int kM = 128;            // weight rows per tile
constexpr int kRowBytes = 128;     // bytes per operand row per stage (64 bf16)
constexpr int kBK = 64;            // K elements per stage
constexpr int kStages = 6;
constexpr int kMaxBN = 128;
constexpr int kLookahead = 4;      // cp.async groups in flight per producer thread
constexpr int kThreads = 288;
constexpr int kProducers = 128;
constexpr int kAccCols = 128;      // TMEM columns per accumulator buffer
constexpr long long kWaitLimit = 4ll * 1000 * 1000 * 1000;  // cycles (~2 s) before giving up

constexpr int kATileBytes = kM * kRowBytes;              // 16 KB
constexpr int kBTileBytes = kMaxBN * kRowBytes;          // 32 KB
constexpr int kRawData = 8 * 512;                        // 8 blocks of 16 rows x 64 K codes
constexpr int kRawSf = kProducers * 8;                   // one 8-byte scale word per producer
constexpr int kRawBytes = kRawData + kRawSf;

struct TcArgs {
  const uint8_t* weights;
  size_t stride;
  const uint8_t* last_weights;
  int G, N, K;
  const int32_t* group_offsets;
  const uint16_t* a;
  const int32_t* a_row_index;
  const float* row_scale;
  uint16_t* out;
  int rows_min;   // groups with more rows than this are handled here
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

__device__ __forceinline__ int n_tiles(int rows) { return (rows + kMaxBN - 1) / kMaxBN; }

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

// bf16x2 of two e2m1 codes (one byte, low nibble first) times an E4M3 scale
// given as f16x2 with the scale in both halves. Exact: the product has at
// most 6 significant bits and lies in [2^-10, 2688].
__device__ __forceinline__ uint32_t dequant_pair_bf16(uint32_t byte, uint32_t s2) {
  const uint32_t h = hmul2_u32(cvt_e2m1x2_f16x2(byte), s2);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
  return *reinterpret_cast<const uint32_t*>(&b);
}

template <bool GATE_UP>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_w4a16_kernel(TcArgs p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a_tiles = base;                                   // kStages x 16 KB
  uint8_t* b_tiles = a_tiles + kStages * kATileBytes;        // kStages x 32 KB
  uint8_t* raw = b_tiles + kStages * kBTileBytes;            // kStages x kRawBytes
  Smem* sm = reinterpret_cast<Smem*>(raw + kStages * kRawBytes);
  int* pref = reinterpret_cast<int*>(sm + 1);                // [G + 1]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.G, K = p.K, N = p.N;
  const int MT = N / kM;
  const int KS = K / kBK;
  pdl_wait();

  // Item prefix over groups.
  for (int g = tid; g < G; g += kThreads) {
    const int rows = p.group_offsets[g + 1] - p.group_offsets[g];
    pref[g + 1] = rows > p.rows_min ? n_tiles(rows) * MT : 0;
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
  if (warp == 8) tmem_alloc(&sm->tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  const int total = pref[G];
  volatile int* abort = &sm->abort;

  if (warp < 4) {
    // ------------------------------------------------------------- producers
    const int tau = tid;                  // 0..127
    const int blk = tau >> 4;             // 16-row block of the tile
    const int L = 2 * (tau & 15);         // first of the two fragment lanes
    const int g8 = L >> 2, t4 = L & 3;    // row within block, k pair index (0 or 2)
    int j = 0, fin = 0;
    auto finalize = [&](int i) {
      const int slot = i % kStages;
      uint8_t* rw = raw + slot * kRawBytes;
      const uint4 d0 = *reinterpret_cast<const uint4*>(rw + blk * 512 + L * 16);
      const uint4 d1 = *reinterpret_cast<const uint4*>(rw + blk * 512 + L * 16 + 16);
      const uint2 sw = *reinterpret_cast<const uint2*>(rw + kRawData + tau * 8);
      const uint32_t wa[4] = {d0.x, d0.y, d0.z, d0.w};
      const uint32_t wb[4] = {d1.x, d1.y, d1.z, d1.w};
      const uint32_t at = smem_u32(a_tiles + slot * kATileBytes);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        // (scale of row g, scale of row g+8) for step s -> each in both halves
        const uint32_t pair = cvt_e4m3x2_f16x2(((s < 2 ? sw.x : sw.y) >> (16 * (s & 1))) & 0xffffu);
        const uint32_t sg = __byte_perm(pair, 0, 0x1010);
        const uint32_t s8 = __byte_perm(pair, 0, 0x3232);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const uint32_t scale = (b & 1) ? s8 : sg;
          const uint32_t lo = dequant_pair_bf16((wa[s] >> (8 * b)) & 0xffu, scale);
          const uint32_t hi = dequant_pair_bf16((wb[s] >> (8 * b)) & 0xffu, scale);
          const int row = blk * 16 + g8 + ((b & 1) ? 8 : 0);
          const int k = 16 * s + 2 * t4 + ((b & 2) ? 8 : 0);
          const uint32_t addr = at + row * kRowBytes + ((((k >> 3) ^ (row & 7)) << 4)) + ((k & 7) << 1);
          asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(lo), "r"(hi) : "memory");
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&sm->full[slot]);
    };
    for (int item = blockIdx.x; item < total && !*abort; item += gridDim.x) {
      const Item it = decode_item(item, pref, G, MT, p.group_offsets);
      const uint8_t* wblk = (it.g == G - 1 && p.last_weights != nullptr) ? p.last_weights
                                                                         : p.weights + (size_t)it.g * p.stride;
      const uint8_t* wdata = wblk + sizeof(PrepHeader);
      // this thread's activation rows of the tile (chunk tau & 7 of rows tau/8 + 16q), loaded once
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
        const int slot = j % kStages;
        if (!mbar_wait(&sm->empty[slot], ((j / kStages) & 1) ^ 1, abort, kWaitLimit)) break;
        uint8_t* rw = raw + slot * kRawBytes;
        const uint8_t* chunk = wdata + w4a16_chunk(it.mt, ks, KS);
        cp_async_16(smem_u32(rw + blk * 512 + L * 16), chunk + blk * 512 + L * 16, 16);
        cp_async_16(smem_u32(rw + blk * 512 + L * 16 + 16), chunk + blk * 512 + L * 16 + 16, 16);
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(rw + kRawData + tau * 8)),
                     "l"(chunk + kW16SfOff + blk * 64 + g8 * 8)
                     : "memory");
        const uint32_t bt = smem_u32(b_tiles + slot * kBTileBytes);
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
        if (j - fin >= kLookahead) {
          cp_async_wait<kLookahead>();
          finalize(fin++);
        }
      }
    }
    cp_async_wait_all();
    while (fin < j) finalize(fin++);
  } else if (warp < 8) {
    // -------------------------------------------------------------- epilogue
    const int q = warp - 4;               // TMEM lane quarter
    const int rho = q * 32 + lane;        // weight row within the tile
    int itc = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++itc) {
      const Item it = decode_item(item, pref, G, MT, p.group_offsets);
      const int acc = itc & 1;
      if (!mbar_wait(&sm->tfull[acc], (itc >> 1) & 1, abort, kWaitLimit)) break;
      tc_fence_after();
      const uint8_t* wblk = (it.g == G - 1 && p.last_weights != nullptr) ? p.last_weights
                                                                         : p.weights + (size_t)it.g * p.stride;
      const PrepHeader* hdr = reinterpret_cast<const PrepHeader*>(wblk);
      const float a0 = hdr->alpha[0], a1 = hdr->alpha[1];
      // routing weights of the tile's rows: lane l holds rows l, l + 32, ...
      float rsv[kMaxBN / 32];
#pragma unroll
      for (int i = 0; i < kMaxBN / 32; ++i) {
        const int n = 32 * i + lane;
        rsv[i] = (!GATE_UP && p.row_scale && n < it.rows) ? __ldg(p.row_scale + it.row0 + n) : 1.0f;
      }
      for (int c0 = 0; c0 < it.bn; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + acc * kAccCols + c0, r);
        tmem_ld_wait();
        float rs_chunk = 1.0f;
#pragma unroll
        for (int i = 0; i < kMaxBN / 32; ++i)
          if ((c0 >> 5) == i) rs_chunk = rsv[i];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float v = __uint_as_float(r[c]);
          const int n = c0 + c;
          if (GATE_UP) {
            const float up = __shfl_down_sync(0xffffffffu, v, 8);
            if ((rho & 15) < 8 && n < it.rows) {
              const int f = 64 * it.mt + 8 * (rho >> 4) + (rho & 7);
              const float h = silu(v * a0) * (up * a1);
              p.out[(size_t)(it.row0 + n) * (N / 2) + f] = float_to_bf16_bits(h);
            }
          } else {
            const float rs = __shfl_sync(0xffffffffu, rs_chunk, n & 31);
            if (n < it.rows)
              p.out[(size_t)(it.row0 + n) * N + it.mt * kM + rho] = float_to_bf16_bits(v * a0 * rs);
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
        const uint32_t idesc = idesc_f16(kM, it.bn, 1);
        const uint32_t d = tmem + acc * kAccCols;
        bool ok = true;
        for (int ks = 0; ks < KS; ++ks, ++j) {
          const int slot = j % kStages;
          if (!mbar_wait(&sm->full[slot], (j / kStages) & 1, abort, kWaitLimit)) { ok = false; break; }
          tc_fence_after();
          const uint32_t as = smem_u32(a_tiles + slot * kATileBytes);
          const uint32_t bs = smem_u32(b_tiles + slot * kBTileBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = smem_desc(as + kk * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(bs + kk * 32, 16, 1024, kSwizzle128B);
            mma_f16(d, ad, bd, idesc, (ks | kk) != 0);
          }
          tc_commit(&sm->empty[slot]);
        }
        if (!ok) break;
        tc_commit(&sm->tfull[acc]);
      }
      // all issued MMAs complete before TMEM is released
      tc_commit(&sm->drain);
      long long t0 = clock64();
      while (!mbar_try_wait(&sm->drain, 0) && clock64() - t0 < kWaitLimit) {
      }
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 8) tmem_dealloc(tmem, 512);
  if (tid == 0 && sm->abort) set_status(p.status, MOE_ERR_TIMEOUT);
}


// ===========================================================================
// W4A4: block-scaled FP4 x FP4 on tcgen05 (kind::mxf4nvf4, scale_vec::4X,
// UE4M3 scales), "vLLM on the NVIDIA DGX Spark", section 6.1 (NVFP4 needs
// block-scaled tensor-core MMA) and section 4.3 (BF16 input quantised to FP4
// before the expert GEMMs).
//
// Stage = 256 K elements = 128 bytes per operand row. The weights' prepared
// layout is the exact shared-memory image of each (128-row, 256-K) tile (128-
// byte swizzle) followed by its four 512-byte scale-factor atoms, so one
// thread moves a stage with two bulk copies. Activation rows (FP4 codes) are
// gathered with cp.async; their E4M3 scales are placed into the atoms by the
// producers. The MMA thread copies the atoms into TMEM (tcgen05.cp
// 32x128b.warpx4) and issues four block-scaled MMAs per stage.
//
// Scale-factor atom (one per 64-wide K step, 128 rows x 4 scales): byte
// m0 * 16 + m1 * 4 + j holds scale j of row m = 32 * m1 + m0.

constexpr int kFp4BK = 256;
constexpr int kFp4MaxBN = 128;
constexpr int kFp4BTile = kFp4MaxBN * kRowBytes;   // 16 KB
constexpr int kSfAtom = 512;
constexpr int kSfStage = 4 * kSfAtom;              // 2 KB per operand per stage
constexpr int kFp4StageBytes = kATileBytes + kFp4BTile + 2 * kSfStage;

struct TcFp4Args {
  const uint8_t* weights;
  size_t stride;
  const uint8_t* last_weights;
  int G, N, K;
  const int32_t* group_offsets;
  const uint8_t* a;       // packed FP4 rows [*, K/2]
  const uint8_t* a_sf;    // E4M3 [*, K/16]
  const float* a_gs;      // device global scale of the activations
  const int32_t* a_row_index;
  const float* row_scale;
  uint16_t* out;
  float* out_amax;
  int* status;
};

__device__ __forceinline__ Item decode_item_fp4(int idx, const int* pref, int G, int MT, const int32_t* off) {
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
  it.row0 = off[lo] + nt * kFp4MaxBN;
  it.rows = min(kFp4MaxBN, grows - nt * kFp4MaxBN);
  it.bn = (it.rows + 15) & ~15;
  return it;
}

template <bool GATE_UP>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_w4a4_kernel(TcFp4Args p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // per stage: A tile 16 KB | B tile 16 KB | SFA 2 KB | SFB 2 KB
  Smem* sm = reinterpret_cast<Smem*>(base + kStages * kFp4StageBytes);
  int* pref = reinterpret_cast<int*>(sm + 1);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.G, K = p.K, N = p.N;
  const int MT = N / kM;
  const int KS = K / kFp4BK;
  pdl_wait();

  for (int g = tid; g < G; g += kThreads) {
    const int rows = p.group_offsets[g + 1] - p.group_offsets[g];
    pref[g + 1] = rows > 0 ? ((rows + kFp4MaxBN - 1) / kFp4MaxBN) * MT : 0;
  }
  if (tid == 0) {
    pref[0] = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm->full[i], kProducers + 1);  // + the bulk copies' expect_tx arrival
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
  if (warp == 8) tmem_alloc(&sm->tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  const int total = pref[G];
  volatile int* abort = &sm->abort;
  constexpr uint32_t kAccColsFp4 = 128;   // accumulators: columns [0, 256)
  constexpr uint32_t kSfCol0 = 256;       // scale factors: 32 columns per stage slot

  if (warp < 4) {
    // ------------------------------------------------------------- producers
    const int tau = tid;
    int j = 0, fin = 0;
    auto finalize = [&](int i) {
      fence_proxy_async_smem();
      mbar_arrive(&sm->full[i % kStages]);
    };
    for (int item = blockIdx.x; item < total && !*abort; item += gridDim.x) {
      const Item it = decode_item_fp4(item, pref, G, MT, p.group_offsets);
      const uint8_t* wblk = (it.g == G - 1 && p.last_weights != nullptr) ? p.last_weights
                                                                         : p.weights + (size_t)it.g * p.stride;
      const uint8_t* wdata = wblk + sizeof(PrepHeader);
      const uint8_t* wsf = wdata + (size_t)N * K / 2;
      // this thread's activation rows (codes: chunk tau & 7 of rows tau/8 + 16q; scales: row tau)
      const uint8_t* asrc[kFp4MaxBN / 16];
#pragma unroll
      for (int q = 0; q < kFp4MaxBN / 16; ++q) {
        const int n = (tau >> 3) + 16 * q;
        asrc[q] = nullptr;
        if (n < it.rows) {
          const int r = it.row0 + n;
          const int arow = p.a_row_index ? __ldg(p.a_row_index + r) : r;
          asrc[q] = p.a + (size_t)arow * (K / 2) + (tau & 7) * 16;
        }
      }
      const uint8_t* sfsrc = nullptr;
      if (tau < it.rows) {
        const int r = it.row0 + tau;
        const int arow = p.a_row_index ? __ldg(p.a_row_index + r) : r;
        sfsrc = p.a_sf + (size_t)arow * (K / 16);
      }
      for (int ks = 0; ks < KS; ++ks, ++j) {
        const int slot = j % kStages;
        if (!mbar_wait(&sm->empty[slot], ((j / kStages) & 1) ^ 1, abort, kWaitLimit)) break;
        uint8_t* st = base + slot * kFp4StageBytes;
        uint8_t* a_t = st;
        uint8_t* b_t = st + kATileBytes;
        uint8_t* sfa = b_t + kFp4BTile;
        uint8_t* sfb = sfa + kSfStage;
        if (tau == 0) {
          const size_t tile = (size_t)it.mt * KS + ks;
          mbar_arrive_expect_tx(&sm->full[slot], kATileBytes + kSfStage);
          bulk_g2s(smem_u32(a_t), wdata + tile * kATileBytes, kATileBytes, &sm->full[slot]);
          bulk_g2s(smem_u32(sfa), wsf + tile * kSfStage, kSfStage, &sm->full[slot]);
        }
        // activation codes: bn rows x 8 chunks of 16 bytes
        const uint32_t bt = smem_u32(b_t);
#pragma unroll
        for (int q = 0; q < kFp4MaxBN / 16; ++q) {
          const int n = (tau >> 3) + 16 * q, ch = tau & 7;
          if (n < it.bn) {
            const uint32_t dst = bt + n * kRowBytes + ((ch ^ (n & 7)) << 4);
            if (asrc[q] != nullptr) cp_async_16(dst, asrc[q] + ks * kRowBytes, 16);
            else cp_async_16(dst, p.a, 0);
          }
        }
        // activation scales: 16 per row per stage, 4 bytes into each atom (async)
        if (tau < kFp4MaxBN) {
          const int off = (tau & 31) * 16 + (tau >> 5) * 4;
          if (sfsrc != nullptr) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(sfb + kk * kSfAtom + off)),
                           "l"(sfsrc + ks * 16 + 4 * kk)
                           : "memory");
          } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) *reinterpret_cast<uint32_t*>(sfb + kk * kSfAtom + off) = 0u;
          }
        }
        cp_async_commit();  // codes and scales of this stage form one group
        if (j - fin >= kLookahead) {
          cp_async_wait<kLookahead>();
          finalize(fin++);
        }
      }
    }
    cp_async_wait_all();
    while (fin < j) finalize(fin++);
  } else if (warp < 8) {
    // -------------------------------------------------------------- epilogue
    const int q = warp - 4;
    const int rho = q * 32 + lane;
    const float inv_gs_a = 1.0f / *p.a_gs;
    float amax = 0.0f;
    int itc = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++itc) {
      const Item it = decode_item_fp4(item, pref, G, MT, p.group_offsets);
      const int acc = itc & 1;
      if (!mbar_wait(&sm->tfull[acc], (itc >> 1) & 1, abort, kWaitLimit)) break;
      tc_fence_after();
      const uint8_t* wblk = (it.g == G - 1 && p.last_weights != nullptr) ? p.last_weights
                                                                         : p.weights + (size_t)it.g * p.stride;
      const PrepHeader* hdr = reinterpret_cast<const PrepHeader*>(wblk);
      const float a0 = hdr->alpha[0] * inv_gs_a, a1 = hdr->alpha[1] * inv_gs_a;
      float rsv[kFp4MaxBN / 32];
#pragma unroll
      for (int i = 0; i < kFp4MaxBN / 32; ++i) {
        const int n = 32 * i + lane;
        rsv[i] = (!GATE_UP && p.row_scale && n < it.rows) ? __ldg(p.row_scale + it.row0 + n) : 1.0f;
      }
      for (int c0 = 0; c0 < it.bn; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + acc * kAccColsFp4 + c0, r);
        tmem_ld_wait();
        float rs_chunk = 1.0f;
#pragma unroll
        for (int i = 0; i < kFp4MaxBN / 32; ++i)
          if ((c0 >> 5) == i) rs_chunk = rsv[i];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float v = __uint_as_float(r[c]);
          const int n = c0 + c;
          if (GATE_UP) {
            const float up = __shfl_down_sync(0xffffffffu, v, 8);
            if ((rho & 15) < 8 && n < it.rows) {
              const int f = 64 * it.mt + 8 * (rho >> 4) + (rho & 7);
              const uint16_t hb = float_to_bf16_bits(silu(v * a0) * (up * a1));
              p.out[(size_t)(it.row0 + n) * (N / 2) + f] = hb;
              amax = fmaxf(amax, fabsf(bf16_bits_to_float(hb)));
            }
          } else {
            const float rs = __shfl_sync(0xffffffffu, rs_chunk, n & 31);
            if (n < it.rows)
              p.out[(size_t)(it.row0 + n) * N + it.mt * kM + rho] = float_to_bf16_bits(v * a0 * rs);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm->tempty[acc]);
    }
    if (GATE_UP && p.out_amax != nullptr) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (lane == 0) atomic_max_nonneg(p.out_amax, amax);
    }
  } else {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      int j = 0, itc = 0;
      for (int item = blockIdx.x; item < total && !*abort; item += gridDim.x, ++itc) {
        const Item it = decode_item_fp4(item, pref, G, MT, p.group_offsets);
        const int acc = itc & 1;
        if (!mbar_wait(&sm->tempty[acc], ((itc >> 1) & 1) ^ 1, abort, kWaitLimit)) break;
        tc_fence_after();
        const uint32_t idesc = idesc_nvf4(kM, it.bn);
        const uint32_t d = tmem + acc * kAccColsFp4;
        bool ok = true;
        for (int ks = 0; ks < KS; ++ks, ++j) {
          const int slot = j % kStages;
          if (!mbar_wait(&sm->full[slot], (j / kStages) & 1, abort, kWaitLimit)) { ok = false; break; }
          tc_fence_after();
          uint8_t* st = base + slot * kFp4StageBytes;
          const uint32_t as = smem_u32(st);
          const uint32_t bs = smem_u32(st + kATileBytes);
          const uint32_t sfa = smem_u32(st + kATileBytes + kFp4BTile);
          const uint32_t sfb = sfa + kSfStage;
          const uint32_t sf_col = tmem + kSfCol0 + slot * 32;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            tc_cp_32x128b_warpx4(sf_col + kk * 4, smem_desc(sfa + kk * kSfAtom, 16, 128, kSwizzleNone));
            tc_cp_32x128b_warpx4(sf_col + 16 + kk * 4, smem_desc(sfb + kk * kSfAtom, 16, 128, kSwizzleNone));
          }
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = smem_desc(as + kk * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(bs + kk * 32, 16, 1024, kSwizzle128B);
            mma_nvf4(d, ad, bd, idesc, sf_col + kk * 4, sf_col + 16 + kk * 4, (ks | kk) != 0);
          }
          tc_commit(&sm->empty[slot]);
        }
        if (!ok) break;
        tc_commit(&sm->tfull[acc]);
      }
      tc_commit(&sm->drain);
      long long t0 = clock64();
      while (!mbar_try_wait(&sm->drain, 0) && clock64() - t0 < kWaitLimit) {
      }
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 8) tmem_dealloc(tmem, 512);
  if (tid == 0 && sm->abort) set_status(p.status, MOE_ERR_TIMEOUT);
}

}  // namespace

size_t gemm_tc_smem_bytes(int G) {
  return 1024 + (size_t)kStages * (kATileBytes + kBTileBytes + kRawBytes) + sizeof(Smem) + (size_t)(G + 1) * 4;
}

moe_status launch_gemm_tc_w4a16(const GemmPlan& pl, int rows_min, cudaStream_t s) {
  if (pl.num_groups <= 0) return MOE_OK;
  TcArgs a;
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
  a.rows_min = rows_min;
  a.status = pl.status;
  const size_t smem = gemm_tc_smem_bytes(pl.num_groups);
  if (smem > 227 * 1024) return MOE_ERR_UNSUPPORTED;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  auto k = pl.gate_up ? gemm_tc_w4a16_kernel<true> : gemm_tc_w4a16_kernel<false>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaError_t e = launch_ex(pl.pdl, k, dim3(sms), dim3(kThreads), smem, s, a);
  if (e != cudaSuccess) return cuda_ok(e);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

}  // namespace moe

namespace moe {

size_t gemm_tc_fp4_smem_bytes(int G) {
  return 1024 + (size_t)kStages * kFp4StageBytes + sizeof(Smem) + (size_t)(G + 1) * 4;
}

moe_status launch_gemm_tc_w4a4(const GemmPlan& pl, cudaStream_t s) {
  if (pl.num_groups <= 0) return MOE_OK;
  if (pl.K % kFp4BK) return MOE_ERR_UNSUPPORTED;
  TcFp4Args a;
  a.weights = pl.weights;
  a.stride = pl.weight_stride;
  a.last_weights = pl.last_weights;
  a.G = pl.num_groups;
  a.N = pl.N;
  a.K = pl.K;
  a.group_offsets = pl.group_offsets;
  a.a = static_cast<const uint8_t*>(pl.a);
  a.a_sf = pl.a_sf;
  a.a_gs = pl.a_gs;
  a.a_row_index = pl.a_row_index;
  a.row_scale = pl.row_scale;
  a.out = pl.out;
  a.out_amax = pl.out_amax;
  a.status = pl.status;
  const size_t smem = gemm_tc_fp4_smem_bytes(pl.num_groups);
  if (smem > 227 * 1024) return MOE_ERR_UNSUPPORTED;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  auto k = pl.gate_up ? gemm_tc_w4a4_kernel<true> : gemm_tc_w4a4_kernel<false>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaError_t e = launch_ex(pl.pdl, k, dim3(sms), dim3(kThreads), smem, s, a);
  if (e != cudaSuccess) return cuda_ok(e);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

}  // namespace moe
