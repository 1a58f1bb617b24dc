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
// active weights). Each weight byte is read from HBM once. One producer warp
// streams the weight tiles with bulk copies (cp.async.bulk, one copy per
// stage of up to 8 K blocks (36 KB), completion on mbarriers) into a ring of
// shared-memory stages. Sixteen MMA warps: warp b of part h owns the 16-row
// block b of a 128-row item and, in every stage, the K blocks h, h + 2, ...
// (more warps per scheduler hide the conversion -> multiply -> MMA latency
// chains, and with both parts on every stage a slot is freed for the next
// copy as soon as the stage is done); at the end of an item the part that
// finishes second adds the other's partial sums and runs the epilogue, while
// the first goes on. A warp loads its 16-byte A fragment per 64-wide K block
// from shared memory, turns the e2m1 codes into f16 with the hardware e2m1x2
// conversion, multiplies in the E4M3 block scales (e2m1 * e4m3 is exact in
// f16) and feeds mma.sync m16n8k16 with the group's rows (up to 8) as N.
//
// Activations enter as f16: each row is scaled by a power of two 2^s so that
// its largest magnitude lands in [2^14, 2^15); bf16 values are then exact in
// f16 (apart from magnitudes below 2^-24 of the row's maximum, which flush),
// and the epilogue multiplies by 2^-s again. The gate/up tile holds the gate
// and up rows of the same 8 features (prepared interleave), so SwiGLU is
// applied in registers.
//
// Work item = (group, chunk of 8 rows, 128 weight rows). CTAs are persistent
// (one per SM) and take contiguous item ranges. Every wait is bounded; on a
// timeout the kernel records MOE_ERR_TIMEOUT, lets its copies land and
// returns.
#include <algorithm>

#include "common.cuh"
#include "decode_mma.cuh"
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using namespace tc;

using decode::kBlockWarps;   // one per 16-row block of a 128-row item
// K split: part h takes the K blocks h, h + 2, ... of every ring stage. Every
// MMA warp consumes every stage in order, so it has consumed a slot's previous
// stage (j - S) before it waits for stage j: the slot's barrier is never a
// phase behind (an mbarrier parity wait cannot tell phase n from n - 2).
using decode::kHalves;
constexpr int kMmaWarps = kBlockWarps * kHalves;
constexpr int kThreads = (kMmaWarps + 1) * 32;  // + one producer warp
constexpr int kRowsPerPass = 8;
constexpr int kTileRows = 128;                   // weight rows per item
constexpr int kMaxGroups = 1025;
constexpr int kMaxSlots = 16;                    // ring slots of stage_kb K blocks (stage_kb * 4608 bytes)
constexpr long long kWaitLimit = 4ll * 1000 * 1000 * 1000;

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
  float* out_last_f32;
  int rows_limit;
  int stages;
  int stage_kb;       // max 64-wide K blocks per ring stage (1..8)
  int early_weights;  // stream weights before the dependency wait (offsets already final)
  int* status;
  long long wait_limit;  // cycles per bounded wait (a timeout aborts the kernel)
};

struct SmallSmem {
  uint64_t full[kMaxSlots];
  uint64_t empty[kMaxSlots];
  uint64_t xsync;                  // the MMA warps' barrier around x staging (one arrival per warp)
  int abort;
  float row_mul[kRowsPerPass];
  int row_out[kRowsPerPass];
  decode::HalfJoin join;           // the two parts' partial sums of an item
};

__device__ __forceinline__ int group_items(const int32_t* off, int g, int mt_count, int limit) {
  const int rows = off[g + 1] - off[g];
  if (rows <= 0 || rows > limit) return 0;
  return ((rows + kRowsPerPass - 1) / kRowsPerPass) * mt_count;
}

__device__ __forceinline__ int find_group(const int* pref, int G, int item) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pref[mid] <= item) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Barrier over the MMA warps (the producer never joins) on an mbarrier, with
// a bounded wait: every warp arrives once per use and waits for the phase.
__device__ __forceinline__ bool mma_warps_sync(uint64_t* bar, uint32_t& phase, volatile int* abort,
                                               long long limit) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
  const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, phase, abort, limit));   // the warp decides as one
  phase ^= 1u;
  __syncwarp();
  return ok;
}

template <bool GATE_UP>
__global__ void __launch_bounds__(kThreads, 1) gemm_small_kernel(SmallArgs p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int K = p.K, N = p.N;
  const int S = p.stages;
  const size_t kStageBytes = (size_t)p.stage_kb * kW16Chunk;
  const int xs_stride = K + 8;  // f16 elements per staged row (16-byte pad: conflict-free ldmatrix)
  uint8_t* stages = smem_raw;                                                   // S x kStageBytes
  uint16_t* xs = reinterpret_cast<uint16_t*>(stages + (size_t)S * kStageBytes);  // [8][K+8]
  SmallSmem* sm = reinterpret_cast<SmallSmem*>(xs + (size_t)kRowsPerPass * xs_stride);
  int* pref = reinterpret_cast<int*>(sm + 1);                                   // [G+1]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int mt_count = N / kTileRows;
  const int G = p.G;
  const int kblocks = K / 64;
  const int kBlocksPerStage = w16_stage_kb(kblocks, p.stage_kb);
  const int nstage = (kblocks + kBlocksPerStage - 1) / kBlocksPerStage;
  if (!p.early_weights) pdl_wait();

  for (int g = tid; g < G; g += kThreads) pref[g + 1] = group_items(p.group_offsets, g, mt_count, p.rows_limit);
  if (tid == 0) {
    pref[0] = 0;
    for (int i = 0; i < S; ++i) {
      mbar_init(&sm->full[i], 1);
      mbar_init(&sm->empty[i], kMmaWarps);  // both parts read every stage
    }
    mbar_init(&sm->xsync, kMmaWarps);
    decode::half_join_init(&sm->join, 0, 1);
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
  __syncthreads();
  const int total = pref[G];
  const int i0 = (int)((long long)total * blockIdx.x / gridDim.x);
  const int i1 = (int)((long long)total * (blockIdx.x + 1) / gridDim.x);
  volatile int* abort = &sm->abort;

  if (warp == kMmaWarps) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      int j = 0;
      for (int item = i0; item < i1 && !*abort; ++item) {
        const int g = find_group(pref, G, item);
        const int mt = (item - pref[g]) % mt_count;
        const uint8_t* blk = (g == G - 1 && p.last_weights != nullptr) ? p.last_weights
                                                                      : p.weights + (size_t)g * p.stride;
        const uint8_t* data = blk + sizeof(PrepHeader);
        for (int st = 0; st < nstage; ++st, ++j) {
          const int slot = j % S;
          if (!mbar_wait(&sm->empty[slot], ((j / S) & 1) ^ 1, abort, p.wait_limit)) break;
          const int kb0 = st * kBlocksPerStage;
          const int nkb = min(kBlocksPerStage, kblocks - kb0);
          const uint32_t bytes = (uint32_t)(nkb * kW16Chunk);
          mbar_arrive_expect_tx(&sm->full[slot], bytes);
          bulk_g2s(smem_u32(stages + (size_t)slot * kStageBytes), data + w4a16_chunk(mt, kb0, kblocks), bytes,
                   &sm->full[slot]);
        }
      }
      // the copies still in flight land before the CTA's shared memory is
      // released (after a timeout the MMA warps may already have left)
      for (int i = max(0, j - S); i < j; ++i) {
        const long long t0 = clock64();
        while (!mbar_try_wait(&sm->full[i % S], (i / S) & 1) && clock64() - t0 < kWaitLimit) {
        }
      }
    }
    return;
  }

  // ------------------------------------------------------------- MMA warps
  if (p.early_weights) pdl_wait();  // the activation rows come from the predecessor
  const int row_last0 = p.group_offsets[G - 1];   // first row of the last group
  const int blk = warp % kBlockWarps, half = warp / kBlockWarps;
  const int g8 = lane >> 2, t4 = lane & 3;
  int cur_g = -1, cur_c = -1;
  int j = 0, tile = 0;
  uint32_t xphase = 0;
  // ldmatrix row address of this lane: matrix q = lane / 8 covers the 8
  // staged rows at k offset 8 * q (two k16 steps per ldmatrix.x4)
  const int lrow = lane & 7, lq = lane >> 3;
  for (int item = i0; item < i1; ++item) {
    const int g = find_group(pref, G, item);
    const int local = item - pref[g];
    const int c = local / mt_count, mt = local % mt_count;
    const int row0 = p.group_offsets[g] + c * kRowsPerPass;
    const int nrows = min(kRowsPerPass, p.group_offsets[g + 1] - row0);

    if (g != cur_g || c != cur_c) {
      if (!mma_warps_sync(&sm->xsync, xphase, abort, p.wait_limit)) break;  // everyone is done with the previous rows
      if (warp < kRowsPerPass) {
        const int r = warp;  // warp w stages row w
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
            for (int q = 0; q < 4; ++q) m = max(m, max(finite_mag(w[q] & 0x7fffu), finite_mag((w[q] >> 16) & 0x7fffu)));
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
          // m = bf16 bits of the row max; its exponent e puts the max in [2^(e-127), 2^(e-126))
          const int e = (int)(m >> 7);
          int sh = (m == 0) ? 0 : 141 - max(e, 1);  // 2^(e-127+sh) = 2^14
          sh = max(-113, min(sh, 126));             // 2^sh and 2^-sh stay normal floats
          const float up = __int_as_float((127 + sh) << 23);
          for (int i = lane; i < K / 8; i += 32) {
            const uint4 v = __ldg(src + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const __half2 h = __floats2half2_rn(__uint_as_float(w[q] << 16) * up,
                                                  __uint_as_float(w[q] & 0xffff0000u) * up);
              o[q] = *reinterpret_cast<const uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(dst + i * 8) = make_uint4(o[0], o[1], o[2], o[3]);
          }
          if (lane == 0) {
            sm->row_mul[r] = __int_as_float((127 - sh) << 23);
            sm->row_out[r] = orow;
          }
        } else {
          for (int i = lane; i < K / 8; i += 32) *reinterpret_cast<uint4*>(dst + i * 8) = make_uint4(0, 0, 0, 0);
          if (lane == 0) {
            sm->row_mul[r] = 0.0f;
            sm->row_out[r] = -1;
          }
        }
      }
      cur_g = g;
      cur_c = c;
      if (!mma_warps_sync(&sm->xsync, xphase, abort, p.wait_limit)) break;
    }

    // the epilogue's alpha and routing weights, loaded now so that they
    // arrive during the stage loop
    const uint8_t* wb = (g == G - 1 && p.last_weights != nullptr) ? p.last_weights
                                                                 : p.weights + (size_t)g * p.stride;
    const PrepHeader* hdr = reinterpret_cast<const PrepHeader*>(wb);
    const float al0 = __ldg(&hdr->alpha[0]), al1 = __ldg(&hdr->alpha[1]);
    float rs2[2] = {1.0f, 1.0f};
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if (!GATE_UP && p.row_scale != nullptr && 2 * t4 + q < nrows) rs2[q] = __ldg(p.row_scale + row0 + 2 * t4 + q);
    // one accumulator per k16 step of a block: four independent MMA chains
    float acc4[4][4];
#pragma unroll
    for (int s = 0; s < 4; ++s) acc4[s][0] = acc4[s][1] = acc4[s][2] = acc4[s][3] = 0.f;
    const uint32_t xbase = smem_u32(xs) + (uint32_t)(lrow * xs_stride + 8 * lq) * 2;
    bool ok = true;
    for (int st = 0; st < nstage; ++st, ++j) {
      const int slot = j % S;
      if (!__all_sync(0xffffffffu, mbar_wait(&sm->full[slot], (j / S) & 1, abort, p.wait_limit))) {
        ok = false;
        break;
      }
      const int kb0 = st * kBlocksPerStage;
      decode::mma_stage(stages + (size_t)slot * kStageBytes, min(kBlocksPerStage, kblocks - kb0), half, kHalves,
                        blk, lane, xbase + (uint32_t)(kb0 * 64) * 2, acc4);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->empty[slot]);
    }
    if (!ok) break;
    float acc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = (acc4[0][q] + acc4[1][q]) + (acc4[2][q] + acc4[3][q]);

    // split-K join: the part that comes second sums and runs the epilogue
    bool second = false;
    if (!decode::half_join(&sm->join, blk, lane, tile++, acc, second, abort, p.wait_limit)) break;
    if (!second) continue;

    // Epilogue: c0,c1 = row g (tokens 2t, 2t+1); c2,c3 = row g+8.
    const int mb = mt * 8 + blk;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int n = 2 * t4 + q;
      if (n >= nrows) continue;
      const int orow = row0 + n;
      if (sm->row_out[n] != orow) {  // the staged rows must be this item's (a desync would be a bug)
        set_status(p.status, MOE_ERR_DEVICE);
        continue;
      }
      const float rm = sm->row_mul[n];
      if (GATE_UP) {
        const float gv = acc[q] * rm * al0;
        const float uv = acc[2 + q] * rm * al1;
        p.out[(size_t)orow * (N / 2) + 8 * mb + g8] = float_to_bf16_bits(silu(gv) * uv);
      } else {
        const float rs = rs2[q];
        const int hr = 16 * mb + g8;
        const float v0 = acc[q] * rm * al0 * rs, v1 = acc[2 + q] * rm * al0 * rs;
        if (p.out_last_f32 != nullptr && g == G - 1) {  // shared expert: kept fp32 for the combine
          float* o = p.out_last_f32 + (size_t)(orow - row_last0) * N;
          o[hr] = v0;
          o[hr + 8] = v1;
        } else {
          p.out[(size_t)orow * N + hr] = float_to_bf16_bits(v0);
          p.out[(size_t)orow * N + hr + 8] = float_to_bf16_bits(v1);
        }
      }
    }
  }
  if (lane == 0 && sm->abort) set_status(p.status, MOE_ERR_TIMEOUT);
}

}  // namespace

static size_t small_smem_bytes(int K, int G, int S, int stage_kb) {
  return (size_t)S * stage_kb * kW16Chunk + (size_t)kRowsPerPass * (K + 8) * 2 + sizeof(SmallSmem) +
         (size_t)(G + 1) * 4;
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
  a.out_last_f32 = pl.out_last_f32;
  a.rows_limit = rows_limit;
  a.status = pl.status;
  a.wait_limit = debug_wait_limit();
  a.early_weights = pl.pdl && pl.early_weights ? 1 : 0;
  const size_t limit = 227 * 1024;
  // ring slots of one stage of this K; as many as fit, up to 216 KB of ring
  // (eight 27 KB stages, or six 36 KB ones)
  const int skb = w16_stage_kb(pl.K / 64, decode_stage_kb());
  a.stage_kb = skb;
  int S = std::min(kMaxSlots, (int)((216 * 1024) / ((size_t)skb * kW16Chunk)));
  while (S > 2 && small_smem_bytes(pl.K, pl.num_groups, S, skb) > limit) --S;
  const size_t smem = small_smem_bytes(pl.K, pl.num_groups, S, skb);
  if (smem > limit) return MOE_ERR_UNSUPPORTED;  // K too large for the staged rows and two slots
  a.stages = S;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // upper bound on items: every row its own chunk
  const long long max_items = (long long)((pl.max_rows + kRowsPerPass - 1) / kRowsPerPass + pl.num_groups) *
                              (pl.N / kTileRows);
  const int grid = (int)std::max<long long>(1, std::min<long long>((long long)sms, max_items));
  auto k = pl.gate_up ? gemm_small_kernel<true> : gemm_small_kernel<false>;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaError_t e = launch_ex(pl.pdl, k, dim3(grid), dim3(kThreads), smem, s, a);
  if (e != cudaSuccess) return cuda_ok(e);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

}  // namespace moe
