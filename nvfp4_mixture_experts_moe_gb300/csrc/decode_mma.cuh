// The MMA loop of the small-group (decode) W4A16 GEMMs, shared by the
// multi-kernel decode GEMM (gemm_small.cu) and the single-kernel decode path
// (decode_fused.cu), so that the two sum in exactly the same order.
//
// "vLLM on the NVIDIA DGX Spark: A Complete Technical Guide", section 5
// (weight-only NVFP4: 4-bit weights dequantised to 16-bit inside the GEMM)
// and section 6.1 (e2m1 values, one E4M3 scale per 16).
#pragma once

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace decode {

constexpr int kBlockWarps = 8;   // one per 16-row block of a 128-row weight tile
constexpr int kHalves = 2;       // two halves of the MMA warps: alternate K blocks of every stage

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// One stage of one 128-row tile: this warp's 16-row block over the stage's
// K blocks kb_first, kb_first + kb_step, ... < nkb (half h of the MMA warps
// takes h, h + 2, ...), with four accumulator
// chains (one per k16 step of a block). The stage holds the tile's prepared
// chunks (4608 bytes per 64-wide K block: eight 512-byte blocks of codes in
// m16n8k16 A-fragment order, then eight 64-byte blocks of E4M3 scales); xa0
// is this lane's ldmatrix address of the staged f16 activation rows at the
// stage's first K column.
__device__ __forceinline__ void mma_stage(const uint8_t* sd, int nkb, int kb_first, int kb_step, int blk, int lane,
                                          uint32_t xa0, float (&acc4)[4][4]) {
  const int g8 = lane >> 2;
  const uint8_t* my_data = sd + blk * 512 + lane * 16;
  const uint8_t* my_sf = sd + kW16SfOff + blk * 64 + g8 * 8;
#pragma unroll 2
  for (int kb = kb_first; kb < nkb; kb += kb_step) {
    const uint4 wq = *reinterpret_cast<const uint4*>(my_data + kb * kW16Chunk);
    const uint2 sq = *reinterpret_cast<const uint2*>(my_sf + kb * kW16Chunk);
    const uint32_t wv[4] = {wq.x, wq.y, wq.z, wq.w};
    uint32_t bf[8];
    const uint32_t xa = xa0 + (uint32_t)(kb * 64) * 2;
    ldsm_x4(xa, bf[0], bf[1], bf[2], bf[3]);
    ldsm_x4(xa + 64, bf[4], bf[5], bf[6], bf[7]);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      uint32_t a[4];
      cvt_e2m1x8_f16(wv[s], a);
      // (scale of row g, scale of row g+8) for step s; e2m1 * e4m3 is exact in f16
      const uint32_t pr = cvt_e4m3x2_f16x2(((s < 2 ? sq.x : sq.y) >> (16 * (s & 1))) & 0xffffu);
      const __half2 sp = *reinterpret_cast<const __half2*>(&pr);
      const __half2 sg = __low2half2(sp), s8 = __high2half2(sp);
      __half2* ah = reinterpret_cast<__half2*>(a);
      ah[0] = __hmul2(ah[0], sg);
      ah[1] = __hmul2(ah[1], s8);
      ah[2] = __hmul2(ah[2], sg);
      ah[3] = __hmul2(ah[3], s8);
      mma_f16_16816(acc4[s], a, bf[2 * s], bf[2 * s + 1]);
    }
  }
}

// The two halves' partial sums of a tile meet here, without making the half
// that finishes first wait for the other: both count themselves in; the
// first writes its partial into the block's buffer and goes straight on to
// the next tile, the second adds that partial to its own and runs the tile's
// epilogue. IEEE addition is commutative, so the sum does not depend on which
// half comes first. The buffer is reused only once the previous tile of the
// block is joined (a half arrives at tile t + 1 only after tile t is joined),
// so the two arrivals of a tile are always the 2t-th and (2t+1)-th.
struct HalfJoin {
  float4 part[kBlockWarps][32];
  int arrivals[kBlockWarps];
  int ready[kBlockWarps];    // t + 1 once the first half's partial of tile t is written
  int joined[kBlockWarps];   // t + 1 once tile t's partial has been read
};

__device__ __forceinline__ void half_join_init(HalfJoin* hj, int tid, int nthreads) {
  for (int i = tid; i < kBlockWarps; i += nthreads) {
    hj->arrivals[i] = 0;
    hj->ready[i] = 0;
    hj->joined[i] = 0;
  }
}

// Bounded spin of lane 0 until *v >= target (shared memory, same CTA).
__device__ __forceinline__ bool spin_ge(const volatile int* v, int target, volatile int* abort, long long limit) {
  if (*v >= target) return true;
  const long long t0 = clock64();
  while (*v < target) {
    if (*abort) return false;
    if (clock64() - t0 > limit) {
      *abort = 1;
      return false;
    }
  }
  return true;
}

// Tile t (counted per warp; both halves count the same tiles). Returns false
// if a bounded wait gave up (abort set); otherwise `second` says whether this
// warp now holds the tile's total in acc and owns the epilogue.
__device__ __forceinline__ bool half_join(HalfJoin* hj, int blk, int lane, int t, float (&acc)[4], bool& second,
                                          volatile int* abort, long long limit) {
  int order = 0, ok = 1;
  if (lane == 0) {
    ok = spin_ge(&hj->joined[blk], t, abort, limit);
    if (ok) order = atomicAdd(&hj->arrivals[blk], 1) & 1;
  }
  if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
  second = __shfl_sync(0xffffffffu, order, 0) != 0;
  if (!second) {
    hj->part[blk][lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      *reinterpret_cast<volatile int*>(&hj->ready[blk]) = t + 1;
    }
    return true;
  }
  if (lane == 0) ok = spin_ge(&hj->ready[blk], t + 1, abort, limit);
  if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
  if (lane == 0) __threadfence_block();
  __syncwarp();   // lane 0 saw the partial published; the warp reads it after this
  const float4 o = hj->part[blk][lane];
  acc[0] += o.x;
  acc[1] += o.y;
  acc[2] += o.z;
  acc[3] += o.w;
  __syncwarp();
  if (lane == 0) {
    __threadfence_block();
    *reinterpret_cast<volatile int*>(&hj->joined[blk]) = t + 1;
  }
  return true;
}

}  // namespace decode
}  // namespace moe
