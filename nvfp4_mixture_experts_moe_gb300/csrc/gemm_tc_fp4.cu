// Grouped NVFP4 x NVFP4 GEMM (W4A4) of the fused forward: block-scaled FP4
// tensor-core MMA with UE4M3 scales, both operands moved by the copy engine.
//
// "vLLM on the NVIDIA DGX Spark: A Complete Technical Guide", section 6.1
// (NVFP4 needs block-scaled tensor-core MMA: e2m1 values, one E4M3 scale per
// 16, fp32 global scales) and section 4.3 (the BF16 input quantised to FP4
// before the expert GEMMs; SwiGLU and the top-k weight in the epilogues).
//
// Swap-AB tile: 128 weight rows on the MMA's M side, up to 128 rows of one
// expert group on N, K in stages of 256 (four kind::mxf4nvf4 MMAs of K 64).
// * A weight-loader warp copies the stage's prepared weight tile (the exact
//   128-byte-swizzled shared-memory image, 16 KB) and its four scale-factor
//   atoms (2 KB) with two bulk copies.
// * An activation-loader warp copies the group's FP4 rows with one
//   tensor-map box (16/32/64/128 rows x 128 bytes, 128-byte swizzle) and the
//   tile's four scale-factor atoms, written in that layout by the quantiser
//   (rows past the group carry scale 0), with one bulk copy.
// * One thread moves the stage's eight atoms into tensor memory (tcgen05.cp
//   32x128b.warpx4) and commits them; another issues the four MMAs (each
//   tcgen05 instruction costs its issuing thread tens of cycles, so the two
//   streams run in parallel); four epilogue warps apply alpha and
//   the activations' 1/gs, SwiGLU (gate/up, with the amax of h for its
//   quantisation) or the routing weight (down), and store bf16.
// Two CTAs share an SM: each has one accumulator (128 TMEM columns) and
// three stages of scale factors (32 columns each), so while one drains its
// accumulator the other's MMAs run, and the two MMA issuers overlap their
// per-stage wait/commit latency. Every wait is bounded; on a timeout the
// kernel records MOE_ERR_TIMEOUT, lets its copies and MMAs drain, frees TMEM
// and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kM = 128;
constexpr int kBK = 256;                    // K per stage
constexpr int kRowBytes = 128;              // one operand row per stage: 256 FP4
constexpr int kMaxStages = 6;
constexpr int kMaxBN = 128;
constexpr int kTile = kM * kRowBytes;       // 16 KB (A; B at most the same)
constexpr int kSfStage = 4 * 512;           // four atoms
constexpr int kStageBytes = 2 * kTile + 2 * kSfStage;
constexpr int kEpiWarp0 = 0;                // warps 0..3
constexpr int kMmaWarp = 4;
constexpr int kALoadWarp = 5;
constexpr int kBLoadWarp = 6;
constexpr int kSfWarp = 7;
constexpr int kThreads = 8 * 32;
constexpr long long kWaitLimit = 4ll * 1000 * 1000 * 1000;

// Two shapes: two CTAs per SM, each with one accumulator and three stages
// (two independent MMA issuers; a CTA's MMAs stall while its accumulator
// drains), or one CTA per SM with two accumulators and six stages (the
// epilogue overlaps the next tile's MMAs). TMEM: accumulators of 128 columns,
// then 32 columns of scale factors per stage.
template <int CTAS>
struct Shape {
  static constexpr int kStages = CTAS == 2 ? 3 : 6;
  static constexpr int kAcc = CTAS == 2 ? 1 : 2;
  static constexpr int kTmemCols = CTAS == 2 ? 256 : 512;
  static constexpr uint32_t kSfCol0 = 128 * kAcc;
  static_assert(kSfCol0 + 32 * kStages <= kTmemCols, "TMEM columns");
  static_assert(kStages <= kMaxStages, "stages");
};

struct BoxMaps {
  CUtensorMap m[4];
};

struct Args {
  const uint8_t* weights;
  size_t stride;
  const uint8_t* last_weights;
  int G, N, K;
  const int32_t* group_offsets;
  const uint8_t* b_sf_tiles;   // activation scale atoms per (tile, stage)
  const float* b_gs;           // activation global scale
  const float* row_scale;
  uint16_t* out;
  float* out_last_f32;
  float* out_amax;
  int a_rows;                  // rows of the activation codes (group order)
  int* status;
  long long wait_limit;        // cycles per bounded wait (a timeout aborts the kernel)
};

struct Smem {
  uint64_t wready[kMaxStages];   // the weight loader's bytes of the stage landed
  uint64_t bready[kMaxStages];   // the activation loader's bytes of the stage landed
  uint64_t sf_full[kMaxStages];  // the stage's scale factors are in tensor memory
  uint64_t empty[kMaxStages];    // the stage's MMAs completed
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint64_t drain_sf;
  uint32_t tmem_base;
  int abort;
};

struct Item {
  int g, row0, rows, bn, mt, tile;
};

// pref[g]: first item of group g; tb[g]: its first 128-row activation tile
__device__ __forceinline__ Item decode_item(int idx, const int* pref, const int* tb, int G, int MT,
                                            const int32_t* off) {
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
  it.tile = tb[lo] + nt;
  return it;
}

__device__ __forceinline__ const uint8_t* weight_block(const Args& p, int g) {
  return (g == p.G - 1 && p.last_weights != nullptr) ? p.last_weights : p.weights + (size_t)g * p.stride;
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity) && clock64() - t0 < kWaitLimit) {
  }
}

// Drains one 128 x 128 accumulator whose lanes are the rows of the item's
// tile (lane rho = row rho) and whose columns are the rows of weight tile
// mt: SwiGLU to bf16 h (gate/up) or y = acc * fac to bf16 (down; the shared
// expert's rows to fp32), 32 columns at a time, 32-byte stores.
template <bool GATE_UP>
__device__ __forceinline__ void drain_rows(const Args& p, uint32_t tacc, const Item& it, int mt, int rho, int N,
                                           float a0, float a1, float fac, bool last_f32, int row_last0,
                                           float& amax) {
  const bool valid = rho < it.rows;
#pragma unroll 1
  for (int c0 = 0; c0 < kM; c0 += 32) {
    uint32_t r[32];
    tmem_ld32(tacc + c0, r);
    tmem_ld_wait();
    if (!valid) continue;
    if (GATE_UP) {
      // columns c0..c0+31: gate of features F0..F0+7, their up, gate of
      // F0+8..F0+15, their up (weight rows interleaved by 8)
      const int F0 = 64 * mt + (c0 >> 1);
      uint32_t hb[8];
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        float h2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = i + e, gc = j < 8 ? j : j + 8;
          h2[e] = silu(__uint_as_float(r[gc]) * a0) * (__uint_as_float(r[gc + 8]) * a1);
        }
        hb[i >> 1] = float2_to_bf16x2_bits(h2[0], h2[1]);
        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(hb[i >> 1] << 16)),
                                 fabsf(__uint_as_float(hb[i >> 1] & 0xffff0000u))));
      }
      stg_v8(p.out + (size_t)(it.row0 + rho) * (N / 2) + F0, hb);
    } else if (last_f32) {   // the shared expert's rows stay fp32
      float* o = p.out_last_f32 + (size_t)(it.row0 - row_last0 + rho) * N + mt * kM + c0;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = __float_as_uint(__uint_as_float(r[8 * v + e]) * fac);
        stg_v8(o + 8 * v, w);
      }
    } else {
      uint16_t* o = p.out + (size_t)(it.row0 + rho) * N + mt * kM + c0;
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        uint32_t yb[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          yb[e] = float2_to_bf16x2_bits(__uint_as_float(r[16 * v + 2 * e]) * fac,
                                        __uint_as_float(r[16 * v + 2 * e + 1]) * fac);
        stg_v8(o + 16 * v, yb);
      }
    }
  }
}

// The same drain with the whole 128-column row in registers first: the
// accumulator is read and converted, `release` hands it back to the next
// tile's MMAs, and only then the row is stored (bf16 outputs only).
template <bool GATE_UP, typename Release>
__device__ __forceinline__ void drain_rows_release(const Args& p, uint32_t tacc, const Item& it, int mt, int rho,
                                                   int N, float a0, float a1, float fac, float& amax,
                                                   Release release) {
  const bool valid = rho < it.rows;
  constexpr int kPk = GATE_UP ? 8 : 16;   // bf16 pairs per 32 columns
  uint32_t pk[4 * kPk];
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
    if (!GATE_UP) {   // 16 columns per load: the 64 packed words and one load fit the registers
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t r[16];
        tmem_ld16(tacc + 32 * ch + 16 * hf, r);
        tmem_ld_wait();
#pragma unroll
        for (int v = 0; v < 8; ++v)
          pk[ch * kPk + 8 * hf + v] =
              float2_to_bf16x2_bits(__uint_as_float(r[2 * v]) * fac, __uint_as_float(r[2 * v + 1]) * fac);
      }
      continue;
    }
    uint32_t r[32];
    tmem_ld32(tacc + 32 * ch, r);
    tmem_ld_wait();
    {
      // columns 32ch..32ch+31: gate of features 64 mt + 16 ch + 0..7, their
      // up, gate of the next 8, their up (weight rows interleaved by 8)
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        float h2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = i + e, gc = j < 8 ? j : j + 8;
          h2[e] = silu(__uint_as_float(r[gc]) * a0) * (__uint_as_float(r[gc + 8]) * a1);
        }
        const uint32_t hb = float2_to_bf16x2_bits(h2[0], h2[1]);
        pk[ch * kPk + (i >> 1)] = hb;
        if (valid)
          amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(hb << 16)), fabsf(__uint_as_float(hb & 0xffff0000u))));
      }
    }
  }
  release();
  if (!valid) return;
  uint16_t* o = GATE_UP ? p.out + (size_t)(it.row0 + rho) * (N / 2) + 64 * mt
                        : p.out + (size_t)(it.row0 + rho) * N + mt * kM;
#pragma unroll
  for (int v = 0; v < kPk / 2; ++v) {
    uint32_t w[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = pk[8 * v + e];
    stg_v8(o + 16 * v, w);
  }
}

// MX: MXFP4 operands (E8M0 scales per 32, kind::mxf4, two scale atoms per
// operand and stage, no global scales); otherwise NVFP4 (E4M3 per 16,
// kind::mxf4nvf4, four atoms per operand and stage).
// TOK_M: the group's rows on the MMA's M side (always 128: rows past the
// group only reach accumulator lanes that are never stored) and 128 weight
// rows on N, so each epilogue thread owns one row of the output tile and
// stores it in 32-byte pieces; otherwise (swap-AB) the weight rows on M and
// the group's rows on N (rounded up to 16), each thread owning one output
// column. The same stage images and scale atoms serve both.
template <bool GATE_UP, int CTAS, bool MX, bool TOK_M>
__global__ void __launch_bounds__(kThreads, CTAS) gemm_tc_fp4_kernel(const __grid_constant__ BoxMaps maps, Args p) {
  constexpr int kSfBytes = MX ? kSfStage / 2 : kSfStage;   // scale bytes per operand and stage
  constexpr int kAtoms = kSfBytes / 512;
  constexpr int kStages = Shape<CTAS>::kStages;
  constexpr int kAcc = Shape<CTAS>::kAcc;
  constexpr int kTmemCols = Shape<CTAS>::kTmemCols;
  constexpr uint32_t kSfCol0 = Shape<CTAS>::kSfCol0;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // per stage: A tile | B tile | SFA atoms | SFB atoms
  Smem* sm = reinterpret_cast<Smem*>(base + kStages * kStageBytes);
  int* pref = reinterpret_cast<int*>(sm + 1);   // [G + 1]
  int* tb = pref + (p.G + 1);                   // [G + 1]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.G, K = p.K, N = p.N;
  const int MT = N / kM;
  const int KS = K / kBK;
  pdl_wait();
  if (p.group_offsets[G] > p.a_rows) {   // the codes do not cover the groups: compute nothing
    if (tid == 0) set_status(p.status, MOE_ERR_DEVICE);
    return;
  }

  for (int g = tid; g < G; g += kThreads) {
    const int rows = p.group_offsets[g + 1] - p.group_offsets[g];
    const int nt = rows > 0 ? (rows + kMaxBN - 1) / kMaxBN : 0;
    pref[g + 1] = nt * MT;
    tb[g + 1] = nt;
  }
  if (tid == 0) {
    pref[0] = 0;
    tb[0] = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm->wready[i], 1);
      mbar_init(&sm->bready[i], 1);
      mbar_init(&sm->sf_full[i], 1);
      mbar_init(&sm->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm->tfull[i], 1);
      mbar_init(&sm->tempty[i], 128);
    }
    mbar_init(&sm->drain, 1);
    mbar_init(&sm->drain_sf, 1);
    sm->abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (warp < 2) {  // inclusive scans of pref (warp 0) and tb (warp 1)
    int* arr = warp == 0 ? pref : tb;
    int carry = 0;
    for (int b0 = 1; b0 <= G; b0 += 32) {
      const int i = b0 + lane;
      int v = i <= G ? arr[i] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
      }
      if (i <= G) arr[i] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  if (warp == kMmaWarp) tmem_alloc(&sm->tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  const int total = pref[G];
  volatile int* abort = &sm->abort;

  if (warp == kALoadWarp) {
    // --------------------------------------------------------- weight loader
    if (lane == 0) {
      int j = 0;
      for (int item = blockIdx.x; item < total && !*abort; item += gridDim.x) {
        const Item it = decode_item(item, pref, tb, G, MT, p.group_offsets);
        const uint8_t* wdata = weight_block(p, it.g) + sizeof(PrepHeader);
        const uint8_t* wsf = wdata + (size_t)N * K / 2;
        bool ok = true;
        for (int ks = 0; ks < KS; ++ks, ++j) {
          const int slot = j % kStages;
          if (!mbar_wait(&sm->empty[slot], ((j / kStages) & 1) ^ 1, abort, p.wait_limit)) { ok = false; break; }
          uint8_t* st = base + slot * kStageBytes;
          const size_t tile = (size_t)it.mt * KS + ks;
          mbar_arrive_expect_tx(&sm->wready[slot], kTile + kSfBytes);
          bulk_g2s(smem_u32(st), wdata + tile * kTile, kTile, &sm->wready[slot]);
          bulk_g2s(smem_u32(st + 2 * kTile), wsf + tile * kSfBytes, kSfBytes, &sm->wready[slot]);
        }
        if (!ok) break;
      }
      // the copies this warp issued land before the shared memory is released
      for (int i = max(0, j - kStages); i < j; ++i) drain_wait(&sm->wready[i % kStages], (i / kStages) & 1);
    }
    __syncwarp();
  } else if (warp == kBLoadWarp) {
    // ----------------------------------------------------- activation loader
    if (lane < 4) tma_prefetch_map(&maps.m[lane]);
    if (lane == 0) {
      int j = 0;
      for (int item = blockIdx.x; item < total && !*abort; item += gridDim.x) {
        const Item it = decode_item(item, pref, tb, G, MT, p.group_offsets);
        const int q = TOK_M ? 3 : 32 - __clz((it.bn >> 4) - 1);   // box of 16 << q >= bn rows
        const uint32_t bytes = (uint32_t)((16 << q) * kRowBytes + kSfBytes);
        bool ok = true;
        for (int ks = 0; ks < KS; ++ks, ++j) {
          const int slot = j % kStages;
          if (!mbar_wait(&sm->empty[slot], ((j / kStages) & 1) ^ 1, abort, p.wait_limit)) { ok = false; break; }
          uint8_t* st = base + slot * kStageBytes;
          mbar_arrive_expect_tx(&sm->bready[slot], bytes);
          tma_load_2d(smem_u32(st + kTile), &maps.m[q], ks * kRowBytes, it.row0, &sm->bready[slot]);
          bulk_g2s(smem_u32(st + 2 * kTile + kSfStage), p.b_sf_tiles + ((size_t)it.tile * KS + ks) * kSfBytes,
                   kSfBytes, &sm->bready[slot]);
        }
        if (!ok) break;
      }
      // the copies this warp issued land before the shared memory is released
      for (int i = max(0, j - kStages); i < j; ++i) drain_wait(&sm->bready[i % kStages], (i / kStages) & 1);
    }
    __syncwarp();
  } else if (warp == kSfWarp) {
    // ------------------------------------------------- scale factors -> TMEM
    if (lane == 0) {
      int j = 0;
      for (int item = blockIdx.x; item < total && !*abort; item += gridDim.x) {
        bool ok = true;
        for (int ks = 0; ks < KS; ++ks, ++j) {
          const int slot = j % kStages;
          // the slot's previous MMAs completed before its loads were issued, so
          // its TMEM columns are free once the new data has landed
          if (!mbar_wait(&sm->wready[slot], (j / kStages) & 1, abort, p.wait_limit) ||
              !mbar_wait(&sm->bready[slot], (j / kStages) & 1, abort, p.wait_limit)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa = smem_u32(base + slot * kStageBytes) + 2 * kTile;
          const uint32_t sfb = sfa + kSfStage;
          const uint32_t sf_col = tmem + kSfCol0 + slot * 32;
#pragma unroll
          for (int kk = 0; kk < kAtoms; ++kk) {
            tc_cp_32x128b_warpx4(sf_col + kk * 4, smem_desc(sfa + kk * 512, 16, 128, kSwizzleNone));
            tc_cp_32x128b_warpx4(sf_col + 16 + kk * 4, smem_desc(sfb + kk * 512, 16, 128, kSwizzleNone));
          }
          tc_commit(&sm->sf_full[slot]);
        }
        if (!ok) break;
      }
      tc_commit(&sm->drain_sf);
      drain_wait(&sm->drain_sf, 0);
    }
    __syncwarp();
  } else if (warp < kEpiWarp0 + 4) {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int rho = q * 32 + lane;   // this thread's TMEM lane
    const float inv_gs_b = MX ? 1.0f : 1.0f / *p.b_gs;
    const int row_last0 = p.out_last_f32 != nullptr ? p.group_offsets[G - 1] : 0;   // first shared row
    float amax = 0.0f;
    int itc = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++itc) {
      const Item it = decode_item(item, pref, tb, G, MT, p.group_offsets);
      const PrepHeader* hdr = reinterpret_cast<const PrepHeader*>(weight_block(p, it.g));
      const float a0 = hdr->alpha[0] * inv_gs_b, a1 = hdr->alpha[1] * inv_gs_b;
      const bool last_f32 = !GATE_UP && p.out_last_f32 != nullptr && it.g == G - 1;  // shared expert: fp32
      // down: y = acc * (alpha * routing weight), one factor per row of the group
      float fac[TOK_M ? 1 : kMaxBN / 32];
#pragma unroll
      for (int i = 0; i < (TOK_M ? 1 : kMaxBN / 32); ++i) {
        const int n = TOK_M ? rho : 32 * i + lane;
        fac[i] = (!GATE_UP && p.row_scale && n < it.rows) ? a0 * __ldg(p.row_scale + it.row0 + n) : a0;
      }
      const int acc = itc % kAcc;
      if (!mbar_wait(&sm->tfull[acc], (itc / kAcc) & 1, abort, p.wait_limit)) break;
      tc_fence_after();
      const uint32_t tacc = tmem + ((uint32_t)(q * 32) << 16) + acc * 128;
      if (TOK_M) {
        drain_rows<GATE_UP>(p, tacc, it, it.mt, rho, N, a0, a1, fac[0], last_f32, row_last0, amax);
      } else {
        // lane rho = weight row rho of tile mt; TMEM column n = row n of the tile
        const bool gate_lane = (rho & 8) == 0;  // rows 16j..16j+7 gate, 16j+8..16j+15 up (interleave by 8)
        const int f = 64 * it.mt + 8 * (rho >> 4) + (rho & 7);
        for (int c0 = 0; c0 < it.bn; c0 += 32) {  // columns past bn are read (within the buffer) and not stored
          uint32_t r[32];
          tmem_ld32(tacc + c0, r);
          tmem_ld_wait();
          if (GATE_UP) {
            // the gate lane finishes columns c0..c0+15, its up partner (lane ^ 8) c0+16..c0+31
            const int cb = gate_lane ? 0 : 16;
            float other[16];
#pragma unroll
            for (int c = 0; c < 16; ++c)
              other[c] = __shfl_xor_sync(0xffffffffu, __uint_as_float(gate_lane ? r[16 + c] : r[c]), 8);
#pragma unroll
            for (int c = 0; c < 16; c += 2) {  // two tokens per bf16 conversion
              float h2[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float own = __uint_as_float(gate_lane ? r[c + e] : r[16 + c + e]);
                const float g = gate_lane ? own : other[c + e];
                const float u = gate_lane ? other[c + e] : own;
                h2[e] = silu(g * a0) * (u * a1);
              }
              const uint32_t hb = float2_to_bf16x2_bits(h2[0], h2[1]);
              const int n = c0 + cb + c;
              uint16_t* o = p.out + (size_t)(it.row0 + n) * (N / 2) + f;
              if (n < it.rows) {
                o[0] = (uint16_t)(hb & 0xffffu);
                amax = fmaxf(amax, fabsf(__uint_as_float(hb << 16)));
              }
              if (n + 1 < it.rows) {
                o[N / 2] = (uint16_t)(hb >> 16);
                amax = fmaxf(amax, fabsf(__uint_as_float(hb & 0xffff0000u)));
              }
            }
          } else {
            float fac_chunk = fac[0];
#pragma unroll
            for (int i = 1; i < (TOK_M ? 1 : kMaxBN / 32); ++i)
              if ((c0 >> 5) == i) fac_chunk = fac[i];
#pragma unroll
            for (int c = 0; c < 32; c += 2) {  // two tokens per bf16 conversion
              const int n = c0 + c;
              const float v0 = __uint_as_float(r[c]) * __shfl_sync(0xffffffffu, fac_chunk, c);
              const float v1 = __uint_as_float(r[c + 1]) * __shfl_sync(0xffffffffu, fac_chunk, c + 1);
              if (last_f32) {
                float* o32 = p.out_last_f32 + (size_t)(it.row0 - row_last0 + n) * N + it.mt * kM + rho;
                if (n < it.rows) o32[0] = v0;
                if (n + 1 < it.rows) o32[N] = v1;
              } else {
                const uint32_t yb = float2_to_bf16x2_bits(v0, v1);
                uint16_t* o = p.out + (size_t)(it.row0 + n) * N + it.mt * kM + rho;
                if (n < it.rows) o[0] = (uint16_t)(yb & 0xffffu);
                if (n + 1 < it.rows) o[N] = (uint16_t)(yb >> 16);
              }
            }
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
        const Item it = decode_item(item, pref, tb, G, MT, p.group_offsets);
        const int acc = itc % kAcc;
        if (!mbar_wait(&sm->tempty[acc], ((itc / kAcc) & 1) ^ 1, abort, p.wait_limit)) break;
        const uint32_t d = tmem + acc * 128;
        tc_fence_after();
        const int mma_n = TOK_M ? kM : it.bn;
        const uint32_t idesc = idesc_nvf4(kM, mma_n);
        const uint32_t idesc_mx0 = idesc_mxf4(kM, mma_n, 0), idesc_mx2 = idesc_mxf4(kM, mma_n, 2);
        bool ok = true;
        for (int ks = 0; ks < KS; ++ks, ++j) {
          const int slot = j % kStages;
          if (!mbar_wait(&sm->sf_full[slot], (j / kStages) & 1, abort, p.wait_limit)) { ok = false; break; }
          tc_fence_after();
          // stage: weight tile | activation tile; TMEM: weight atoms at +0, activation atoms at +16
          const uint32_t ws_ = smem_u32(base + slot * kStageBytes);
          const uint32_t as = TOK_M ? ws_ + kTile : ws_;
          const uint32_t bs = TOK_M ? ws_ : ws_ + kTile;
          const uint32_t sf_col = tmem + kSfCol0 + slot * 32;
          const uint32_t sfa_col = sf_col + (TOK_M ? 16 : 0), sfb_col = sf_col + (TOK_M ? 0 : 16);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = smem_desc(as + kk * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(bs + kk * 32, 16, 1024, kSwizzle128B);
            if (MX)  // atom kk / 2, byte pair 2 * (kk % 2)
              mma_mxf4(d, ad, bd, (kk & 1) ? idesc_mx2 : idesc_mx0, sfa_col + (kk >> 1) * 4,
                       sfb_col + (kk >> 1) * 4, (ks | kk) != 0);
            else
              mma_nvf4(d, ad, bd, idesc, sfa_col + kk * 4, sfb_col + kk * 4, (ks | kk) != 0);
          }
          tc_commit(&sm->empty[slot]);
        }
        if (!ok) break;
        tc_commit(&sm->tfull[acc]);
      }
      tc_commit(&sm->drain);
      drain_wait(&sm->drain, 0);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
  if (tid == 0 && sm->abort) set_status(p.status, MOE_ERR_TIMEOUT);
}

// ---------------------------------------------------------------------------
// Wide tile: one CTA per SM, the group's rows on M (128) and 256 weight rows
// on N as two halves of 128 (weight tiles 2m and 2m+1), each half with its
// own accumulator (TMEM columns 0-127, 128-255), MMA-issuing thread and
// scale-copy thread. The activation tile and its scale atoms come into shared
// memory once per stage for both halves: 54 KB per 16.8 MFLOP instead of
// 36 KB per 8.4 MFLOP, a quarter fewer bytes per FLOP through the SM's
// L2 -> shared-memory path, which is what bounds the 128 x 128 tiles.
namespace wide {
constexpr int kWStages = 4;
constexpr int kSfSlot = kSfStage;                         // one operand's atoms per stage (NVFP4 size)
constexpr int kWStageBytes = 3 * kTile + 3 * kSfSlot;      // A | B0 | B1 | SFA | SFB0 | SFB1
constexpr uint32_t kWSfCol0 = 256;                         // after the two accumulators
constexpr int kSfCols = 48;                               // per stage: SFA, SFB0, SFB1 (16 columns each)
constexpr int kWTmemCols = 512;
static_assert(kWSfCol0 + kSfCols * kWStages <= kWTmemCols, "TMEM columns");
static_assert(kWStageBytes % 1024 == 0, "stage alignment");
constexpr int kEpiWarps = 8;    // warps 0..7: TMEM lane quarter w % 4, half w / 4
constexpr int kMmaWarp0 = 8;    // 8, 9: MMA issuer of half 0, 1
constexpr int kSfWarp0 = 10;    // 10, 11: scale copies of half 0, 1
constexpr int kWALoadWarp = 12;  // the group's rows
constexpr int kWBLoadWarp = 13;  // the two weight tiles
constexpr int kWThreads = 14 * 32;
static_assert(kEpiWarps == kMmaWarp0, "the epilogue warps are warps 0 .. kMmaWarp0 - 1");

struct WSmem {
  uint64_t aready[kWStages];   // the activation tile landed
  uint64_t bready[kWStages];   // both weight tiles landed
  uint64_t sfready[kWStages];  // the stage's scale atoms landed (copied first, so the
                               // moves into TMEM overlap the tiles' flight)
  uint64_t sf_full[kWStages];  // both halves' scale copies completed
  uint64_t empty[kWStages];    // both halves' MMAs completed
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;             // both MMA issuers' last commits
  uint64_t drain_sf;          // both scale-copy threads' last commits
  uint32_t tmem_base;
  int abort;
};
}  // namespace wide

// N256: one N = 256 MMA per K block into one 256-column accumulator (one
// issuing thread; three scale-copy threads: the activation atoms and each
// weight tile's atoms); otherwise two N = 128 halves, each with its own
// issuing thread, scale-copy thread and accumulator.
template <bool GATE_UP, bool MX, bool N256>
__global__ void __maxnreg__(128)
    gemm_tc_fp4_wide_kernel(const __grid_constant__ BoxMaps maps, Args p) {
  using namespace wide;
  constexpr int kSfBytes = MX ? kSfStage / 2 : kSfStage;   // scale bytes per operand tile and stage
  constexpr int kAtoms = kSfBytes / 512;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  WSmem* sm = reinterpret_cast<WSmem*>(base + kWStages * kWStageBytes);
  int* pref = reinterpret_cast<int*>(sm + 1);   // [G + 1]
  int* tb = pref + (p.G + 1);                   // [G + 1]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.G, K = p.K, N = p.N;
  const int MT2 = N / (2 * kM);   // items per 128-row tile of a group: pairs of weight tiles
  const int KS = K / kBK;
  pdl_wait();
  if (p.group_offsets[G] > p.a_rows) {   // the codes do not cover the groups: compute nothing
    if (tid == 0) set_status(p.status, MOE_ERR_DEVICE);
    return;
  }

  for (int g = tid; g < G; g += kWThreads) {
    const int rows = p.group_offsets[g + 1] - p.group_offsets[g];
    const int nt = rows > 0 ? (rows + kMaxBN - 1) / kMaxBN : 0;
    pref[g + 1] = nt * MT2;
    tb[g + 1] = nt;
  }
  if (tid == 0) {
    pref[0] = 0;
    tb[0] = 0;
    for (int i = 0; i < kWStages; ++i) {
      mbar_init(&sm->aready[i], 1);
      mbar_init(&sm->bready[i], 1);
      mbar_init(&sm->sfready[i], 2);
      mbar_init(&sm->sf_full[i], N256 ? 3 : 2);
      mbar_init(&sm->empty[i], N256 ? 1 : 2);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm->tfull[i], 1);
      mbar_init(&sm->tempty[i], N256 ? 256 : 128);
    }
    mbar_init(&sm->drain, N256 ? 1 : 2);
    mbar_init(&sm->drain_sf, N256 ? 3 : 2);
    sm->abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (warp < 2) {  // inclusive scans of pref (warp 0) and tb (warp 1)
    int* arr = warp == 0 ? pref : tb;
    int carry = 0;
    for (int b0 = 1; b0 <= G; b0 += 32) {
      const int i = b0 + lane;
      int v = i <= G ? arr[i] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
      }
      if (i <= G) arr[i] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  if (warp == kMmaWarp0) tmem_alloc(&sm->tmem_base, kWTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  const int total = pref[G];
  volatile int* abort = &sm->abort;

  if (warp == kWALoadWarp) {
    // ------------------------------------------------ activation (row) loader
    if (lane == 0) {
      tma_prefetch_map(&maps.m[3]);
      int j = 0;
      for (int item = blockIdx.x; item < total && !*abort; item += gridDim.x) {
        const Item it = decode_item(item, pref, tb, G, MT2, p.group_offsets);
        bool ok = true;
        for (int ks = 0; ks < KS; ++ks, ++j) {
          const int slot = j % kWStages;
          if (!mbar_wait(&sm->empty[slot], ((j / kWStages) & 1) ^ 1, abort, p.wait_limit)) { ok = false; break; }
          uint8_t* st = base + slot * kWStageBytes;
          mbar_arrive_expect_tx(&sm->sfready[slot], kSfBytes);
          bulk_g2s(smem_u32(st + 3 * kTile), p.b_sf_tiles + ((size_t)it.tile * KS + ks) * kSfBytes, kSfBytes,
                   &sm->sfready[slot]);
          mbar_arrive_expect_tx(&sm->aready[slot], kTile);
          tma_load_2d(smem_u32(st), &maps.m[3], ks * kRowBytes, it.row0, &sm->aready[slot]);
        }
        if (!ok) break;
      }
      for (int i = max(0, j - kWStages); i < j; ++i) {
        drain_wait(&sm->aready[i % kWStages], (i / kWStages) & 1);
        drain_wait(&sm->sfready[i % kWStages], (i / kWStages) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kWBLoadWarp) {
    // ------------------------------------------------------- weight loader
    if (lane == 0) {
      int j = 0;
      for (int item = blockIdx.x; item < total && !*abort; item += gridDim.x) {
        const Item it = decode_item(item, pref, tb, G, MT2, p.group_offsets);
        const uint8_t* wdata = weight_block(p, it.g) + sizeof(PrepHeader);
        const uint8_t* wsf = wdata + (size_t)N * K / 2;
        bool ok = true;
        for (int ks = 0; ks < KS; ++ks, ++j) {
          const int slot = j % kWStages;
          if (!mbar_wait(&sm->empty[slot], ((j / kWStages) & 1) ^ 1, abort, p.wait_limit)) { ok = false; break; }
          uint8_t* st = base + slot * kWStageBytes;
          mbar_arrive_expect_tx(&sm->sfready[slot], 2 * kSfBytes);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const size_t tile = (size_t)(2 * it.mt + h) * KS + ks;
            bulk_g2s(smem_u32(st + 3 * kTile + (1 + h) * kSfSlot), wsf + tile * kSfBytes, kSfBytes,
                     &sm->sfready[slot]);
          }
          mbar_arrive_expect_tx(&sm->bready[slot], 2 * kTile);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const size_t tile = (size_t)(2 * it.mt + h) * KS + ks;
            bulk_g2s(smem_u32(st + (1 + h) * kTile), wdata + tile * kTile, kTile, &sm->bready[slot]);
          }
        }
        if (!ok) break;
      }
      for (int i = max(0, j - kWStages); i < j; ++i) {
        drain_wait(&sm->bready[i % kWStages], (i / kWStages) & 1);
        drain_wait(&sm->sfready[i % kWStages], (i / kWStages) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kSfWarp0 || warp == kSfWarp0 + 1 || (N256 && warp == kMmaWarp0 + 1)) {
    // ------------------------- scale factors -> TMEM. Two halves: thread h
    // copies weight tile h's atoms and every other activation atom. N256:
    // thread h copies weight tile h's atoms, the third the activation atoms.
    const int h = warp == kMmaWarp0 + 1 ? 2 : warp - kSfWarp0;
    if (lane == 0) {
      int j = 0;
      for (int item = blockIdx.x; item < total && !*abort; item += gridDim.x) {
        bool ok = true;
        for (int ks = 0; ks < KS; ++ks, ++j) {
          const int slot = j % kWStages;
          // the slot's previous MMAs completed before its loads were issued,
          // so its TMEM columns are free once the atoms landed
          if (!mbar_wait(&sm->sfready[slot], (j / kWStages) & 1, abort, p.wait_limit)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfa = smem_u32(base + slot * kWStageBytes) + 3 * kTile;
          const uint32_t sfb = sfa + (1 + (h & 1)) * kSfSlot;
          const uint32_t col = tmem + kWSfCol0 + slot * kSfCols;
          if (N256) {
            // activation atoms at columns 4 kk; the weight atoms of a K block
            // side by side (rows 0-127, then 128-255): 16 + 8 kk + 4 h
            if (h == 2) {
#pragma unroll
              for (int kk = 0; kk < kAtoms; ++kk)
                tc_cp_32x128b_warpx4(col + kk * 4, smem_desc(sfa + kk * 512, 16, 128, kSwizzleNone));
            } else {
#pragma unroll
              for (int kk = 0; kk < kAtoms; ++kk)
                tc_cp_32x128b_warpx4(col + 16 + 8 * kk + 4 * h, smem_desc(sfb + kk * 512, 16, 128, kSwizzleNone));
            }
          } else {
#pragma unroll
            for (int kk = h; kk < kAtoms; kk += 2)
              tc_cp_32x128b_warpx4(col + kk * 4, smem_desc(sfa + kk * 512, 16, 128, kSwizzleNone));
#pragma unroll
            for (int kk = 0; kk < kAtoms; ++kk)
              tc_cp_32x128b_warpx4(col + 16 + 16 * h + kk * 4, smem_desc(sfb + kk * 512, 16, 128, kSwizzleNone));
          }
          tc_commit(&sm->sf_full[slot]);
        }
        if (!ok) break;
      }
      tc_commit(&sm->drain_sf);
      drain_wait(&sm->drain_sf, 0);
    }
    __syncwarp();
  } else if (warp == kMmaWarp0 || warp == kMmaWarp0 + 1) {
    // ------------------------------------------------- MMA issuer of half h
    const int h = warp - kMmaWarp0;   // N256: only half 0's thread issues (N = 256)
    if (lane == 0 && !(N256 && h == 1)) {
      int j = 0, itc = 0;
      for (int item = blockIdx.x; item < total && !*abort; item += gridDim.x, ++itc) {
        if (!mbar_wait(&sm->tempty[h], (itc & 1) ^ 1, abort, p.wait_limit)) break;   // h = 0 with N256
        const uint32_t d = tmem + 128 * h;
        tc_fence_after();
        constexpr int kN = N256 ? 2 * kM : kM;
        const uint32_t idesc = idesc_nvf4(kM, kN);
        const uint32_t idesc_mx0 = idesc_mxf4(kM, kN, 0), idesc_mx2 = idesc_mxf4(kM, kN, 2);
        bool ok = true;
        for (int ks = 0; ks < KS; ++ks, ++j) {
          const int slot = j % kWStages;
          if (!mbar_wait(&sm->sf_full[slot], (j / kWStages) & 1, abort, p.wait_limit) ||
              !mbar_wait(&sm->aready[slot], (j / kWStages) & 1, abort, p.wait_limit) ||
              !mbar_wait(&sm->bready[slot], (j / kWStages) & 1, abort, p.wait_limit)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t as = smem_u32(base + slot * kWStageBytes);
          const uint32_t bs = as + (1 + h) * kTile;
          const uint32_t sfa_col = tmem + kWSfCol0 + slot * kSfCols;
          const uint32_t sfb_col = sfa_col + 16 + (N256 ? 0 : 16 * h);
          constexpr int kSfbStep = N256 ? 8 : 4;   // columns per weight atom index
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = smem_desc(as + kk * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(bs + kk * 32, 16, 1024, kSwizzle128B);
            if (MX)  // atom kk / 2, byte pair 2 * (kk % 2)
              mma_mxf4(d, ad, bd, (kk & 1) ? idesc_mx2 : idesc_mx0, sfa_col + (kk >> 1) * 4,
                       sfb_col + (kk >> 1) * kSfbStep, (ks | kk) != 0);
            else
              mma_nvf4(d, ad, bd, idesc, sfa_col + kk * 4, sfb_col + kk * kSfbStep, (ks | kk) != 0);
          }
          tc_commit(&sm->empty[slot]);
        }
        if (!ok) break;
        tc_commit(&sm->tfull[h]);
      }
      tc_commit(&sm->drain);
      drain_wait(&sm->drain, 0);
    }
    __syncwarp();
  } else {
    // --------------------------------------------- epilogue (warps 0..7)
    const int q = warp & 3, h = warp >> 2;
    const int rho = q * 32 + lane;   // TMEM lane = row of the item's tile
    const float inv_gs_b = MX ? 1.0f : 1.0f / *p.b_gs;
    const int row_last0 = p.out_last_f32 != nullptr ? p.group_offsets[G - 1] : 0;   // first shared row
    float amax = 0.0f;
    int itc = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++itc) {
      const Item it = decode_item(item, pref, tb, G, MT2, p.group_offsets);
      const PrepHeader* hdr = reinterpret_cast<const PrepHeader*>(weight_block(p, it.g));
      const float a0 = hdr->alpha[0] * inv_gs_b, a1 = hdr->alpha[1] * inv_gs_b;
      const bool last_f32 = !GATE_UP && p.out_last_f32 != nullptr && it.g == G - 1;  // shared expert: fp32
      // down: y = acc * (alpha * routing weight)
      const float fac =
          (!GATE_UP && p.row_scale && rho < it.rows) ? a0 * __ldg(p.row_scale + it.row0 + rho) : a0;
      if (!mbar_wait(&sm->tfull[N256 ? 0 : h], itc & 1, abort, p.wait_limit)) break;
      tc_fence_after();
      const uint32_t tacc = tmem + ((uint32_t)(q * 32) << 16) + 128 * h;
      uint64_t* tempty = &sm->tempty[N256 ? 0 : h];
      if (last_f32) {
        drain_rows<GATE_UP>(p, tacc, it, 2 * it.mt + h, rho, N, a0, a1, fac, true, row_last0, amax);
        tc_fence_before();
        mbar_arrive(tempty);
      } else {
        drain_rows_release<GATE_UP>(p, tacc, it, 2 * it.mt + h, rho, N, a0, a1, fac, amax, [&] {
          tc_fence_before();
          mbar_arrive(tempty);
        });
      }
    }
    if (GATE_UP && p.out_amax != nullptr) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (lane == 0) atomic_max_nonneg(p.out_amax, amax);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp0) tmem_dealloc(tmem, kWTmemCols);
  if (tid == 0 && sm->abort) set_status(p.status, MOE_ERR_TIMEOUT);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

}  // namespace

static size_t fp4_smem_bytes(int G, int stages) {
  return 1024 + (size_t)stages * kStageBytes + sizeof(Smem) + (size_t)(G + 1) * 8;
}

moe_status launch_gemm_tc_fp4(const GemmPlan& pl, cudaStream_t s) {
  if (pl.num_groups <= 0) return MOE_OK;
  if (pl.K % kBK || pl.N % kM) return MOE_ERR_UNSUPPORTED;
  const bool mx = pl.mode == MOE_MXFP4;
  if (pl.a == nullptr || pl.a_sf == nullptr || (!mx && pl.a_gs == nullptr) || pl.a_rows <= 0)
    return MOE_ERR_INVALID_ARG;
  auto encode = encode_tiled();
  if (encode == nullptr) return MOE_ERR_CUDA;
  // the FP4 activation codes [a_rows, K/2] in group order: boxes of 16..128 rows x 128 bytes, 128-byte swizzle
  BoxMaps maps;
  for (int q = 0; q < 4; ++q) {
    const cuuint64_t dims[2] = {(cuuint64_t)pl.K / 2, (cuuint64_t)pl.a_rows};
    const cuuint64_t strides[1] = {(cuuint64_t)pl.K / 2};
    const cuuint32_t box[2] = {(cuuint32_t)kRowBytes, (cuuint32_t)(16 << q)};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&maps.m[q], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(pl.a), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MOE_ERR_INVALID_ARG;
  }
  Args a;
  a.weights = pl.weights;
  a.stride = pl.weight_stride;
  a.last_weights = pl.last_weights;
  a.G = pl.num_groups;
  a.N = pl.N;
  a.K = pl.K;
  a.group_offsets = pl.group_offsets;
  a.b_sf_tiles = pl.a_sf;
  a.b_gs = pl.a_gs;
  a.row_scale = pl.row_scale;
  a.out = pl.out;
  a.out_last_f32 = pl.out_last_f32;
  a.out_amax = pl.out_amax;
  a.a_rows = pl.a_rows;
  a.status = pl.status;
  a.wait_limit = debug_wait_limit();
  // tile shape: 1 = one CTA per SM, weight rows on M; 2 = two CTAs per SM,
  // weight rows on M; 3 = two CTAs per SM, the group's rows on M; 4 = one CTA
  // per SM, the group's rows on M, 256 weight rows per tile (N a multiple of 256)
  const int forced = debug_fp4_tile(pl.gate_up != 0);
  int shape = forced != 0 ? forced : pl.ctas_per_sm == 1 ? 1 : 5;
  if (shape >= 4 && pl.N % (2 * kM) != 0) shape = 3;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  using KernelFn = void (*)(const BoxMaps, Args);
  const size_t wide_smem = 1024 + (size_t)wide::kWStages * wide::kWStageBytes + sizeof(wide::WSmem) +
                           (size_t)(pl.num_groups + 1) * 8;
  if ((shape == 4 || shape == 5) && wide_smem > 227 * 1024) shape = 3;
  if (shape == 4 || shape == 5) {
    const size_t smem = wide_smem;
    // [n256][mx][gate_up]
    static const KernelFn wtable[2][2][2] = {
        {{gemm_tc_fp4_wide_kernel<false, false, false>, gemm_tc_fp4_wide_kernel<true, false, false>},
         {gemm_tc_fp4_wide_kernel<false, true, false>, gemm_tc_fp4_wide_kernel<true, true, false>}},
        {{gemm_tc_fp4_wide_kernel<false, false, true>, gemm_tc_fp4_wide_kernel<true, false, true>},
         {gemm_tc_fp4_wide_kernel<false, true, true>, gemm_tc_fp4_wide_kernel<true, true, true>}}};
    const KernelFn k = wtable[shape == 5 ? 1 : 0][mx ? 1 : 0][pl.gate_up ? 1 : 0];
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    int fit = 0;   // one CTA of this kernel must fit an SM (registers and shared memory)
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, k, wide::kWThreads, smem) != cudaSuccess || fit < 1)
      return MOE_ERR_UNSUPPORTED;
    cudaError_t e = launch_ex(pl.pdl, k, dim3(sms), dim3(wide::kWThreads), smem, s, maps, a);
    if (e != cudaSuccess) return cuda_ok(e);
    count_launches(1);
    return MOE_OK;
  }
  const int ctas = shape == 1 ? 1 : 2;
  const size_t smem = fp4_smem_bytes(pl.num_groups, ctas == 2 ? Shape<2>::kStages : Shape<1>::kStages);
  if (smem > (ctas == 2 ? 113 : 227) * 1024) return MOE_ERR_UNSUPPORTED;
  // [mx][gate_up][shape - 1]
  static const KernelFn table[2][2][3] = {
      {{gemm_tc_fp4_kernel<false, 1, false, false>, gemm_tc_fp4_kernel<false, 2, false, false>,
        gemm_tc_fp4_kernel<false, 2, false, true>},
       {gemm_tc_fp4_kernel<true, 1, false, false>, gemm_tc_fp4_kernel<true, 2, false, false>,
        gemm_tc_fp4_kernel<true, 2, false, true>}},
      {{gemm_tc_fp4_kernel<false, 1, true, false>, gemm_tc_fp4_kernel<false, 2, true, false>,
        gemm_tc_fp4_kernel<false, 2, true, true>},
       {gemm_tc_fp4_kernel<true, 1, true, false>, gemm_tc_fp4_kernel<true, 2, true, false>,
        gemm_tc_fp4_kernel<true, 2, true, true>}}};
  const KernelFn k = table[mx ? 1 : 0][pl.gate_up ? 1 : 0][shape - 1];
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaError_t e = launch_ex(pl.pdl, k, dim3(sms * ctas), dim3(kThreads), smem, s, maps, a);
  if (e != cudaSuccess) return cuda_ok(e);
  count_launches(1);
  return MOE_OK;
}

}  // namespace moe
