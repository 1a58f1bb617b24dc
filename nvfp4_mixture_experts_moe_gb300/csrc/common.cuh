// Shared device/host helpers of the CUDA path (sm_103a only).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "moe_nvfp4.h"  // from include/, on the compiler include path

namespace moe {

// ---------------------------------------------------------------------------
// Workspace header: every workspace starts with this 256-byte block. The
// first word is the device status (0 = OK, otherwise a moe_status code).
struct WsHeader {
  int status;
  int pad0;
  float amax[4];     // atomic-max slots for dynamic global scales
  // the single-kernel decode path's counters (two sets in the fused region
  // after this header): 1 once both sets are known to be zero; launch ticket
  // (one per CTA; launch n = ticket / grid uses set n % 2 and zeroes the
  // other); first-use grid barrier (counts up, never reset)
  int fused_clean;
  int pad1;
  unsigned long long fused_ticket;
  unsigned long long fused_gbar;
  int pad[52];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");
// A forward workspace keeps this many ints right after the header for the
// single-kernel decode path's two counter sets (kFusedSetInts each),
// whatever the call's shape, so no other buffer ever overlaps them.
constexpr size_t kFusedSetInts = 2048;
constexpr size_t kFusedRegionInts = 2 * kFusedSetInts;

constexpr size_t kAlign = 256;
__host__ __device__ inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------------------
// Prepared weight block header (first 256 bytes of every prepared matrix).
constexpr uint32_t kPrepMagic = 0x3446564Eu;  // "NVF4"
struct PrepHeader {
  uint32_t magic;
  int mode;      // moe_mode
  int gate_up;   // 1: [gate; up] pair, rows interleaved by 8
  int N, K;
  float alpha[2];  // 1/gs (gate, up) or (w, unused)
  int pad[57];
};
static_assert(sizeof(PrepHeader) == 256, "prepared header is 256 bytes");

// W4A16 layout after the header: one chunk of 4608 bytes per (128-row tile
// mt, 64-wide K block kb), at ((mt * K/64) + kb) * 4608, so that a tile's K
// blocks follow one another: eight 512-byte blocks of fragment-ordered codes
// (16-row blocks b = 0..7 of the tile, at 512 b), then their eight 64-byte
// blocks of E4M3 scales (at 4096 + 64 b). Within a data block, lane L = 4*g + t of a warp owns bytes
// [16L, 16L+16): word s (k16 step s of the block) holds, byte by byte, the
// code pairs of (row g, k 16s+2t..+1), (row g+8, same k), (row g, k+8..+9),
// (row g+8, k+8..+9) -- the A-fragment order of an m16n8k16 MMA. Within a
// scale block, group g owns bytes [8g, 8g+8): for k16 step s = 0..3 the pair
// (scale of row g, scale of row g+8), so one e4m3x2 conversion yields both
// rows' scales of a step.
constexpr int kW16Chunk = 4608;   // bytes of one (128-row tile, 64-wide K block) chunk
constexpr int kW16SfOff = 4096;   // scale blocks within a chunk
__host__ __device__ inline size_t w4a16_bytes(int N, int K) { return (size_t)N * K / 2 + (size_t)N * K / 16; }
__host__ __device__ inline size_t w4a16_chunk(int mt, int kb, int KB) { return ((size_t)mt * KB + kb) * kW16Chunk; }

// 64-wide K blocks per streamed stage of the small-group (decode) GEMMs
// (KB = K / 64 blocks per 128-row tile): the largest count <= kmax (at most
// 8) that divides KB into equal stages, else kmax itself (a short last
// stage). Both halves of the MMA warps read every stage, half h taking the
// stage's blocks h, h + 2, ...; every kernel that runs this loop with the
// same kmax therefore sums in the same order.
constexpr int kW16MaxStageKb = 8;
__host__ __device__ inline int w16_stage_kb(int KB, int kmax) {
  for (int kb = kmax; kb > 1; --kb)
    if (KB % kb == 0) return kb;
  return kmax < KB ? kmax : (KB > 0 ? KB : 1);
}

// ---------------------------------------------------------------------------
// Small device helpers.
__device__ __forceinline__ uint32_t cvt_e2m1x2_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n .reg .b8 b;\n cvt.u8.u32 b, %1;\n cvt.rn.f16x2.e2m1x2 %0, b;\n}" : "=r"(r) : "r"(byte));
  return r;
}

// Four e2m1 pairs (the four bytes of w) to four f16x2 words.
__device__ __forceinline__ void cvt_e2m1x8_f16(uint32_t w, uint32_t (&o)[4]) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]) : "r"(w));
}

// Two E4M3 bytes (low byte -> low half) to f16x2; exact.
__device__ __forceinline__ uint32_t cvt_e4m3x2_f16x2(uint32_t two_bytes) {
  uint32_t r;
  uint16_t h = (uint16_t)two_bytes;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(h));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ void mma_f16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ uint2 ldg_stream2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}

// A bf16 magnitude bit pattern with the NaN patterns (above 0x7f80, the
// infinity) mapped to 0. NaN activations are outside the contract; this keeps
// them from becoming a tensor's or a row's maximum (an infinite amax would
// make a global scale 0 and zero every code).
// One 32-byte global store (p 32-byte aligned): one L2 sector per thread.
__device__ __forceinline__ void stg_v8(void* p, const uint32_t (&v)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v[0]), "r"(v[1]), "r"(v[2]),
               "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

__device__ __forceinline__ uint32_t finite_mag(uint32_t mag_bits) { return mag_bits > 0x7f80u ? 0u : mag_bits; }

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

// fp32 -> bf16 bits, round to nearest even (the hardware conversion).
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

// Two floats -> two bf16 (round to nearest even) in one conversion: `lo` in
// bits 0-15, `hi` in bits 16-31.
__device__ __forceinline__ uint32_t float2_to_bf16x2_bits(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// atomic max of a non-negative float via its integer bit pattern (exact and
// order-independent).
__device__ __forceinline__ void atomic_max_nonneg(float* addr, float v) {
  atomicMax(reinterpret_cast<int*>(addr), __float_as_int(v));
}

__device__ __forceinline__ void set_status(int* status, int code) { atomicCAS(status, 0, code); }

// SiLU z * sigmoid(z) with the hardware exp2 approximation and the fast
// division (relative error a few ulp of fp32, far below the bf16 rounding of
// the result). The IEEE reciprocal or division costs tens of instructions per
// element and dominated the GEMM epilogues. Large negative z gives exp -> inf
// and a result of -0.
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

}  // namespace moe
