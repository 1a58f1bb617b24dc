// Grouped NVFP4 GEMM for large groups, weight-only path (W4A16), with the
// dequantised weights in tensor memory.
//
// "vLLM on the NVIDIA DGX Spark: A Complete Technical Guide", section 4.3
// (the fused MoE's two expert GEMMs, SwiGLU and the top-k weight in the
// epilogues), section 5 (weight-only NVFP4: 4-bit weights dequantised to
// 16-bit inside the GEMM) and section 6.1 (alpha = 1/gs).
//
// Swap-AB tile: 128 weight rows are the MMA's M side, up to 128 rows of one
// expert group its N side, K in stages of 128 (two 64-wide halves).
//
// * Two loader warps move each stage with the tensor-memory-access engine:
//   one copies the stage's two 4608-byte chunks of raw e2m1 codes and E4M3
//   scales (one bulk copy) into a ring of four raw slots; the other loads the
//   group's activation rows, one box per K half (16, 32, 64 or 128 rows, the
//   smallest that covers the tile, through tensor maps over the f16
//   activation matrix, whose rows are in group order; 128-byte swizzle). Box
//   rows past the end of the matrix read as zero; rows of the next group that
//   fill a box are computed and not stored. A TMA or bulk instruction costs
//   its issuing thread tens of cycles and an mbarrier wait more than a
//   hundred, so a stage is few large copies and a 128-wide K step.
// * Eight dequant warps (two sets of four that take alternate stages; warp q
//   of a set owns TMEM lanes 32q..32q+31) rebuild their weight row from the
//   m16n8k16 fragment layout with one register exchange with the partner row
//   (lane ^ 8), convert with the hardware e2m1x2 conversion, multiply by the
//   block scale (exact in f16) and write the stage's 64 columns into TMEM
//   with tcgen05.st.
// * One thread issues tcgen05.mma (kind::f16, A from TMEM, B from shared
//   memory, fp32 accumulators in TMEM): one wait, eight MMAs and one commit
//   per stage.
// * Four epilogue warps read the accumulators (tcgen05.ld), multiply by the
//   activation row's 2^-s (the f16 copy's power-of-two scale), alpha and the
//   routing weight (GEMM 2) or apply SwiGLU (GEMM 1), and store bf16.
//
// Two tile shapes (F16Shape below): 128 token rows, two CTAs per SM, or 256
// token rows, one CTA per SM. Every wait is bounded; on a timeout the kernel records
// MOE_ERR_TIMEOUT, lets its copies and MMAs drain, frees TMEM and exits.
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
constexpr int kBK = 128;                     // K per stage
constexpr int kHalf = 64;                    // K per box / per 128-byte swizzled row
constexpr int kRowBytes = 128;
// Two tile shapes.
// Narrow (groups of up to 128 rows): up to 128 token rows per tile, two CTAs
//   per SM, two stages of activation tiles and TMEM A columns, four raw weight
//   slots. One thread issues a CTA's MMAs and each stage costs that thread a
//   few hundred cycles of barrier and commit latency in which its tensor core
//   would idle; two independent issuers keep it fed, and while one CTA drains
//   its accumulator in the epilogue the other one's MMAs run.
// Wide (groups of more than 128 rows): up to 256 token rows per tile (one
//   N = 256 MMA per K step, so each dequantised weight tile serves twice the
//   tokens), one CTA per SM, three stages, two raw weight slots (one per
//   dequant set).
// TMEM: the accumulator in columns [0, kBN), the A stages of 64 columns after it.
template <bool WIDE>
struct F16Shape {
  static constexpr int kBN = WIDE ? 256 : 128;
  static constexpr int kCtas = WIDE ? 1 : 2;
  static constexpr int kTmemCols = WIDE ? 512 : 256;
  static constexpr uint32_t kAcol0 = kBN;
  static constexpr int kBHalf = kBN * 128;   // one 64-wide K half of the activation tile (128-byte rows)
  static constexpr int kBStage = 2 * kBHalf;
  static constexpr int kStages = WIDE ? 3 : 2;
  static constexpr int kRawSlots = WIDE ? 2 : 4;
  static_assert(kAcol0 + 64 * kStages <= kTmemCols, "TMEM columns");
  static_assert(kRawSlots % 2 == 0, "each dequant set owns whole raw slots");
};
constexpr int kStagesMax = 3, kRawSlotsMax = 4;
// Warp roles. The epilogue warps are the oldest: the schedulers favour them
// over the ALU-heavy dequant warps, so an accumulator drains quickly.
constexpr int kEpiWarp0 = 0;                 // warps 0..3
constexpr int kMmaWarp = 4;
constexpr int kWLoadWarp = 5;
constexpr int kBLoadWarp = 6;
constexpr int kDeqWarp0 = 7;                 // warps 7..14: two dequant sets
constexpr int kThreads = (kDeqWarp0 + 8) * 32;
constexpr int kRawStage = 2 * kW16Chunk;     // two (128-row, 64-K) chunks
constexpr long long kWaitLimit = 4ll * 1000 * 1000 * 1000;

// Tensor maps over the f16 activation matrix with boxes of 16, 32, 64 and
// 128 rows (64 columns each).
struct BoxMaps {
  CUtensorMap m[4];
};

struct Args {
  const uint8_t* weights;
  size_t stride;
  const uint8_t* last_weights;
  int G, N, K;
  const int32_t* group_offsets;
  const float* a_mul;      // per A row multiplier (2^-s), group order
  const float* row_scale;
  uint16_t* out;
  float* out_last_f32;
  int rows_min, rows_max;   // the groups this launch computes: rows_min < rows <= rows_max
  int a_rows;               // rows of the f16 copy and of a_mul
  int* status;
  long long wait_limit;      // cycles per bounded wait (a timeout aborts the kernel)
};

template <int BN>
struct Smem {
  uint64_t w_full[kRawSlotsMax];   // raw weights of the stage landed
  uint64_t w_empty[kRawSlotsMax];  // the dequant set is done reading them
  uint64_t bfull[kStagesMax];      // activation rows of the stage landed
  uint64_t ready[kStagesMax];      // the four dequant warps wrote the stage's A columns
  uint64_t empty[kStagesMax];      // the stage's MMAs completed (activation tile and TMEM A free)
  uint64_t tfull;
  uint64_t tempty;
  // epilogue: per-row factors of the tile, one copy per epilogue warp, read
  // as float4 (gate/up: 2^-s * alpha_gate; down: 2^-s * routing weight * alpha)
  alignas(16) float rowmul[4][BN];
  alignas(16) float rowmul_up[4][BN];   // gate/up: 2^-s * alpha_up
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

struct Item {
  int g, row0, rows, bn, mt;
};

__device__ __forceinline__ Item decode_item(int idx, const int* pref, int G, int MT, const int32_t* off, int BN) {
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
  it.row0 = off[lo] + nt * BN;
  it.rows = min(BN, grows - nt * BN);
  it.bn = (it.rows + 15) & ~15;
  return it;
}

__device__ __forceinline__ const uint8_t* weight_block(const Args& p, int g) {
  return (g == p.G - 1 && p.last_weights != nullptr) ? p.last_weights : p.weights + (size_t)g * p.stride;
}

// Bounded wait that ignores the abort flag (draining after a timeout).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity) && clock64() - t0 < kWaitLimit) {
  }
}

template <bool GATE_UP, bool WIDE>
__global__ void __launch_bounds__(kThreads, F16Shape<WIDE>::kCtas)
    gemm_tc_f16_kernel(const __grid_constant__ BoxMaps maps, Args p) {
  using Sh = F16Shape<WIDE>;
  constexpr int kBN = Sh::kBN, kBHalf = Sh::kBHalf, kBStage = Sh::kBStage, kTmemCols = Sh::kTmemCols;
  constexpr int kStages = Sh::kStages, kRawSlots = Sh::kRawSlots;
  constexpr uint32_t kAcol0 = Sh::kAcol0;
  using Smem = ::moe::Smem<kBN>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* b_tiles = base;                               // kStages x 32 KB
  uint8_t* raw = b_tiles + kStages * kBStage;            // kRawSlots x 9 KB
  Smem* sm = reinterpret_cast<Smem*>(raw + kRawSlots * kRawStage);
  int* pref = reinterpret_cast<int*>(sm + 1);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.G, K = p.K, N = p.N;
  const int MT = N / kM;
  const int KS = (K + kBK - 1) / kBK;     // the last stage has one half when K % 128 == 64
  const int KB64 = K / kHalf;
  pdl_wait();
  if (p.group_offsets[G] > p.a_rows) {   // the copied rows do not cover the groups: compute nothing
    if (tid == 0) set_status(p.status, MOE_ERR_DEVICE);
    return;
  }

  for (int g = tid; g < G; g += kThreads) {
    const int rows = p.group_offsets[g + 1] - p.group_offsets[g];
    pref[g + 1] = rows > p.rows_min && rows <= p.rows_max ? ((rows + kBN - 1) / kBN) * MT : 0;
  }
  if (tid == 0) {
    pref[0] = 0;
    for (int i = 0; i < kRawSlots; ++i) {
      mbar_init(&sm->w_full[i], 1);
      mbar_init(&sm->w_empty[i], 4);
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm->bfull[i], 1);
      mbar_init(&sm->ready[i], 4);
      mbar_init(&sm->empty[i], 1);
    }
    mbar_init(&sm->tfull, 1);
    mbar_init(&sm->tempty, 128);
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
  if (warp == kMmaWarp) tmem_alloc(&sm->tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  const int total = pref[G];
  volatile int* abort = &sm->abort;

  if (warp == kWLoadWarp) {
    // --------------------------------------------------------- weight loader
    if (lane == 0) {
      int j = 0;
      for (int item = blockIdx.x; item < total && !*abort; item += gridDim.x) {
        const Item it = decode_item(item, pref, G, MT, p.group_offsets, kBN);
        const uint8_t* wdata = weight_block(p, it.g) + sizeof(PrepHeader);
        bool ok = true;
        for (int ks = 0; ks < KS; ++ks, ++j) {
          const int rs = j % kRawSlots;
          if (!mbar_wait(&sm->w_empty[rs], ((j / kRawSlots) & 1) ^ 1, abort, p.wait_limit)) { ok = false; break; }
          const uint32_t bytes = (uint32_t)(min(2, KB64 - 2 * ks) * kW16Chunk);
          mbar_arrive_expect_tx(&sm->w_full[rs], bytes);
          bulk_g2s(smem_u32(raw + rs * kRawStage), wdata + w4a16_chunk(it.mt, 2 * ks, KB64), bytes, &sm->w_full[rs]);
        }
        if (!ok) break;
      }
      if (*abort)  // let copies in flight land before the shared memory is released
        for (int i = max(0, j - kRawSlots); i < j; ++i) drain_wait(&sm->w_full[i % kRawSlots], (i / kRawSlots) & 1);
    }
    __syncwarp();
  } else if (warp == kBLoadWarp) {
    // ----------------------------------------------------- activation loader
    if (lane < 4) tma_prefetch_map(&maps.m[lane]);
    if (lane == 0) {
      int j = 0;
      for (int item = blockIdx.x; item < total && !*abort; item += gridDim.x) {
        const Item it = decode_item(item, pref, G, MT, p.group_offsets, kBN);
        // one box of 16 << q >= bn rows, or two boxes of 128 rows for bn > 128
        const int nbox = it.bn > 128 ? 2 : 1;
        const int q = nbox == 2 ? 3 : 32 - __clz((it.bn >> 4) - 1);
        const uint32_t half_bytes = (uint32_t)(nbox * (16 << q) * kRowBytes);
        bool ok = true;
        for (int ks = 0; ks < KS; ++ks, ++j) {
          const int slot = j % kStages;
          if (!mbar_wait(&sm->empty[slot], ((j / kStages) & 1) ^ 1, abort, p.wait_limit)) { ok = false; break; }
          const int nh = min(2, KB64 - 2 * ks);
          mbar_arrive_expect_tx(&sm->bfull[slot], nh * half_bytes);
          const uint32_t dst = smem_u32(b_tiles + slot * kBStage);
          for (int h = 0; h < nh; ++h)
            for (int bx = 0; bx < nbox; ++bx)
              tma_load_2d(dst + h * kBHalf + bx * 128 * kRowBytes, &maps.m[q], (2 * ks + h) * kHalf,
                          it.row0 + 128 * bx, &sm->bfull[slot]);
        }
        if (!ok) break;
      }
      // the boxes this warp issued land before the shared memory is released
      for (int i = max(0, j - kStages); i < j; ++i) drain_wait(&sm->bfull[i % kStages], (i / kStages) & 1);
    }
    __syncwarp();
  } else if (warp >= kDeqWarp0) {
    // --------------------------------------------------------------- dequant
    const int set = (warp - kDeqWarp0) >> 2;     // takes the stages j with j % 2 == set
    const int q = warp & 3;                      // TMEM lane quarter of this warp
    const int tau = q * 32 + lane;               // weight row of the tile
    const int blk = tau >> 4, g8 = tau & 7, hi = (tau >> 3) & 1;
    const uint32_t lane_taddr = tmem + ((uint32_t)(q * 32) << 16);
    // the partner row needs bytes (1-hi) and (3-hi) of my two fragment words;
    // I keep bytes hi and 2+hi
    const uint32_t sel_send = (uint32_t)((1 - hi) | ((5 - hi) << 4) | ((3 - hi) << 8) | ((7 - hi) << 12));
    const uint32_t sel_keep = (uint32_t)(hi | ((4 + hi) << 4) | ((2 + hi) << 8) | ((6 + hi) << 12));
    int j = 0;
    for (int item = blockIdx.x; item < total && !*abort; item += gridDim.x) {
      bool ok = true;
      for (int ks = 0; ks < KS; ++ks, ++j) {
        if ((j & 1) != set) continue;
        const int slot = j % kStages, rslot = j % kRawSlots;
        if (!mbar_wait(&sm->w_full[rslot], (j / kRawSlots) & 1, abort, p.wait_limit) ||
            !mbar_wait(&sm->empty[slot], ((j / kStages) & 1) ^ 1, abort, p.wait_limit)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int nh = min(2, KB64 - 2 * ks);
        // Releasing the raw slot. Its refill is a bulk copy, an async-proxy
        // write, and the reads here are generic loads: a load still in flight
        // when the slot is released could see the refill's bytes. The narrow
        // shape (two slots per set) releases the slot after the TMEM stores
        // have consumed the loaded words, so no read is in flight. The
        // wide shape (one slot per set) reads both halves up front and
        // releases at once, so that the refill overlaps the conversion; the
        // proxy fence orders those reads before the refill. (Without it the
        // wide shape computed a few wrong weight rows in some launches.)
        uint4 pwa[2], pwb[2];
        uint2 psc[2];
        if (WIDE) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (h < nh) {
              const uint8_t* rs = raw + rslot * kRawStage + h * kW16Chunk;
              pwa[h] = *reinterpret_cast<const uint4*>(rs + blk * 512 + (4 * g8 + 2 * hi) * 16);
              pwb[h] = *reinterpret_cast<const uint4*>(rs + blk * 512 + (4 * g8 + 2 * hi) * 16 + 16);
              psc[h] = *reinterpret_cast<const uint2*>(rs + kW16SfOff + blk * 64 + g8 * 8);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm->w_empty[rslot]);
        }
        for (int h = 0; h < nh; ++h) {
          uint4 wa4, wb4;
          uint2 sc;
          if (WIDE) {
            wa4 = h ? pwa[1] : pwa[0];
            wb4 = h ? pwb[1] : pwb[0];
            sc = h ? psc[1] : psc[0];
          } else {
            const uint8_t* rs = raw + rslot * kRawStage + h * kW16Chunk;
            wa4 = *reinterpret_cast<const uint4*>(rs + blk * 512 + (4 * g8 + 2 * hi) * 16);
            wb4 = *reinterpret_cast<const uint4*>(rs + blk * 512 + (4 * g8 + 2 * hi) * 16 + 16);
            sc = *reinterpret_cast<const uint2*>(rs + kW16SfOff + blk * 64 + g8 * 8);
          }
          const uint32_t wa[4] = {wa4.x, wa4.y, wa4.z, wa4.w};
          const uint32_t wb[4] = {wb4.x, wb4.y, wb4.z, wb4.w};
          uint32_t col[32];
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const uint32_t keep = __byte_perm(wa[s], wb[s], sel_keep);
            const uint32_t recv = __shfl_xor_sync(0xffffffffu, __byte_perm(wa[s], wb[s], sel_send), 8);
            // bytes of fragment lanes t = 0..3 for k 16s + 2t (lo) and 16s + 8 + 2t (hh)
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
          tmem_st32(lane_taddr + kAcol0 + slot * 64 + h * 32, col);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          // narrow: the TMEM stores above (asm statements, kept in order with
          // the arrive) consumed every word loaded from the slot
          if (!WIDE) mbar_arrive(&sm->w_empty[rslot]);
          mbar_arrive(&sm->ready[slot]);
        }
      }
      if (!ok) break;
    }
  } else if (warp < kEpiWarp0 + 4) {
    // -------------------------------------------------------------- epilogue
    const int q = warp & 3;
    const int rho = q * 32 + lane;
    const int row_last0 = p.out_last_f32 != nullptr ? p.group_offsets[G - 1] : 0;   // first shared row
    int itc = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++itc) {
      const Item it = decode_item(item, pref, G, MT, p.group_offsets, kBN);
      // per-row factors of the tile, alpha folded in, into this warp's shared
      // copy (no cross-warp sync)
      const PrepHeader* hdr = reinterpret_cast<const PrepHeader*>(weight_block(p, it.g));
      const float a0 = hdr->alpha[0], a1 = hdr->alpha[1];
      float* rowmul = sm->rowmul[q];
      float* rowmul_up = sm->rowmul_up[q];
      __syncwarp();  // done reading the previous item's factors
#pragma unroll
      for (int i = 0; i < kBN / 32; ++i) {
        const int n = 32 * i + lane;
        float m = 0.0f;
        if (n < it.rows) {
          const int r = it.row0 + n;
          m = __ldg(p.a_mul + r);
          if (!GATE_UP && p.row_scale) m *= __ldg(p.row_scale + r);
        }
        rowmul[n] = m * a0;
        if (GATE_UP) rowmul_up[n] = m * a1;
      }
      __syncwarp();
      if (!mbar_wait(&sm->tfull, itc & 1, abort, p.wait_limit)) break;
      tc_fence_after();
      const bool gate_lane = (rho & 8) == 0;   // rows 16j..16j+7 gate, 16j+8..16j+15 up (interleave by 8)
      const int f = 64 * it.mt + 8 * (rho >> 4) + (rho & 7);
      for (int c0 = 0; c0 < it.bn; c0 += 32) {  // columns past bn are read (within the buffer) and not stored
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + c0, r);
        tmem_ld_wait();
        if (GATE_UP) {
          // the gate lane finishes columns c0..c0+15 and its up partner (lane ^ 8)
          // columns c0+16..c0+31: one exchange of 16 raw values, 16 SiLUs each
          const int cb = gate_lane ? 0 : 16;  // first column this lane finishes
          float other[16];
#pragma unroll
          for (int c = 0; c < 16; ++c)
            other[c] = __shfl_xor_sync(0xffffffffu, __uint_as_float(gate_lane ? r[16 + c] : r[c]), 8);
#pragma unroll
          for (int c4 = 0; c4 < 16; c4 += 4) {
            const float4 g4 = *reinterpret_cast<const float4*>(rowmul + c0 + cb + c4);     // broadcast reads
            const float4 u4 = *reinterpret_cast<const float4*>(rowmul_up + c0 + cb + c4);
            const float gv[4] = {g4.x, g4.y, g4.z, g4.w}, uv[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
            for (int t = 0; t < 4; t += 2) {  // two tokens per bf16 conversion
              float h2[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int c = c4 + t + e;
                const float own = __uint_as_float(gate_lane ? r[c] : r[16 + c]);
                const float g = (gate_lane ? own : other[c]) * gv[t + e];
                const float u = (gate_lane ? other[c] : own) * uv[t + e];
                h2[e] = silu(g) * u;
              }
              const uint32_t hb = float2_to_bf16x2_bits(h2[0], h2[1]);
              const int n = c0 + cb + c4 + t;
              uint16_t* o = p.out + (size_t)(it.row0 + n) * (N / 2) + f;
              if (n < it.rows) o[0] = (uint16_t)(hb & 0xffffu);
              if (n + 1 < it.rows) o[N / 2] = (uint16_t)(hb >> 16);
            }
          }
        } else if (p.out_last_f32 != nullptr && it.g == G - 1) {
          // shared expert: kept fp32 for the combine
          float* o32 = p.out_last_f32 + (size_t)(it.row0 - row_last0) * N + it.mt * kM + rho;
#pragma unroll
          for (int c4 = 0; c4 < 32; c4 += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(rowmul + c0 + c4);  // broadcast read
            const float mv[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int n = c0 + c4 + t;
              if (n < it.rows) o32[(size_t)n * N] = __uint_as_float(r[c4 + t]) * mv[t];
            }
          }
        } else {
#pragma unroll
          for (int c4 = 0; c4 < 32; c4 += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(rowmul + c0 + c4);  // broadcast read
            const float mv[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int t = 0; t < 4; t += 2) {  // two tokens per bf16 conversion
              const uint32_t yb = float2_to_bf16x2_bits(__uint_as_float(r[c4 + t]) * mv[t],
                                                        __uint_as_float(r[c4 + t + 1]) * mv[t + 1]);
              const int n = c0 + c4 + t;
              uint16_t* o = p.out + (size_t)(it.row0 + n) * N + it.mt * kM + rho;
              if (n < it.rows) o[0] = (uint16_t)(yb & 0xffffu);
              if (n + 1 < it.rows) o[N] = (uint16_t)(yb >> 16);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm->tempty);
    }
  } else {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      const uint64_t bdesc0 = smem_desc(smem_u32(b_tiles), 16, 1024, kSwizzle128B);  // + 2 per 32-byte K step
      int j = 0, itc = 0;
      for (int item = blockIdx.x; item < total && !*abort; item += gridDim.x, ++itc) {
        const Item it = decode_item(item, pref, G, MT, p.group_offsets, kBN);
        if (!mbar_wait(&sm->tempty, (itc & 1) ^ 1, abort, p.wait_limit)) break;
        tc_fence_after();
        const uint32_t idesc = idesc_f16(kM, it.bn, 0);
        const uint32_t d = tmem;
        bool ok = true;
        for (int ks = 0; ks < KS; ++ks, ++j) {
          const int slot = j % kStages;
          if (!mbar_wait(&sm->bfull[slot], (j / kStages) & 1, abort, p.wait_limit) ||
              !mbar_wait(&sm->ready[slot], (j / kStages) & 1, abort, p.wait_limit)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t bd = bdesc0 + (uint64_t)((slot * kBStage) >> 4);
          const uint32_t a_t = tmem + kAcol0 + slot * 64;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_f16_tmem_a(d, a_t + kk * 8, bd + 2 * kk, idesc, (ks | kk) != 0);
          if (2 * ks + 1 < KB64) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_tmem_a(d, a_t + 32 + kk * 8, bd + (kBHalf >> 4) + 2 * kk, idesc, 1);
          }
          tc_commit(&sm->empty[slot]);
        }
        if (!ok) break;
        tc_commit(&sm->tfull);
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

template <bool WIDE>
static size_t smem_bytes(int G) {
  using Sh = F16Shape<WIDE>;
  return 1024 + (size_t)Sh::kStages * Sh::kBStage + (size_t)Sh::kRawSlots * kRawStage +
         sizeof(Smem<Sh::kBN>) + (size_t)(G + 1) * 4;
}

bool gemm_tc_f16_wide_fits(int num_groups) { return smem_bytes<true>(num_groups) <= 227 * 1024; }

moe_status launch_gemm_tc_f16(const GemmPlan& pl, int rows_min, int rows_max, bool wide, cudaStream_t s) {
  if (pl.num_groups <= 0) return MOE_OK;
  if (pl.a_f16 == nullptr || pl.a_mul == nullptr || pl.a_rows <= 0) return MOE_ERR_INVALID_ARG;
  auto encode = encode_tiled();
  if (encode == nullptr) return MOE_ERR_CUDA;
  // the f16 activation matrix [a_rows, K] in group order: boxes of 16..128 rows x 64 elements, 128-byte swizzle
  BoxMaps maps;
  for (int q = 0; q < 4; ++q) {
    const cuuint64_t dims[2] = {(cuuint64_t)pl.K, (cuuint64_t)pl.a_rows};
    const cuuint64_t strides[1] = {(cuuint64_t)pl.K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kHalf, (cuuint32_t)(16 << q)};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&maps.m[q], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(pl.a_f16), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
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
  a.a_mul = pl.a_mul;
  a.row_scale = pl.row_scale;
  a.out = pl.out;
  a.out_last_f32 = pl.out_last_f32;
  a.rows_min = rows_min;
  a.rows_max = rows_max;
  a.a_rows = pl.a_rows;
  a.status = pl.status;
  a.wait_limit = debug_wait_limit();
  const size_t smem = wide ? smem_bytes<true>(pl.num_groups) : smem_bytes<false>(pl.num_groups);
  const int ctas = wide ? F16Shape<true>::kCtas : F16Shape<false>::kCtas;
  if (smem > 227 * 1024) return MOE_ERR_UNSUPPORTED;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  auto k = wide ? (pl.gate_up ? gemm_tc_f16_kernel<true, true> : gemm_tc_f16_kernel<false, true>)
                : (pl.gate_up ? gemm_tc_f16_kernel<true, false> : gemm_tc_f16_kernel<false, false>);
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaError_t e = launch_ex(pl.pdl, k, dim3(sms * ctas), dim3(kThreads), smem, s, maps, a);
  if (e != cudaSuccess) return cuda_ok(e);
  count_launches(1);
  return MOE_OK;
}

}  // namespace moe
