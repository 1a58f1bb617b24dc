// One-time weight preparation: linear NVFP4 matrices -> the tile layouts the
// GEMM kernels read. "Serving Solar Open 2 on DGX Spark", "Supporting real
// NVFP4 checkpoints" (pre-quantised checkpoint weights are converted once
// into the kernel's MMA tile layout, including the fused gate/up ordering).
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

// Source row of output row o. For a gate/up pair the N rows arrive as
// [gate (N/2); up (N/2)] and leave interleaved by 8: output rows 16j..16j+7
// are gate rows 8j..8j+7 and 16j+8..16j+15 are up rows 8j..8j+7, so one
// 16-row MMA tile holds the gate and up rows of the same 8 features.
__device__ __forceinline__ int src_row(int o, int N, int gate_up) {
  if (!gate_up) return o;
  const int j = o >> 4, w = o & 15;
  return w < 8 ? 8 * j + w : N / 2 + 8 * j + (w - 8);
}

__device__ __forceinline__ void check_sf(uint8_t v, int* flag) {
  if ((v & 0x80u) || v == 0x7fu) atomicOr(flag, 1);
}

// One thread per byte of fragment-ordered codes (block mb = 16 rows, kb).
__global__ void prepare_w4a16_data_kernel(const uint8_t* __restrict__ codes, int N, int K, int gate_up,
                                          uint8_t* __restrict__ out) {
  const size_t total = (size_t)N * K / 2;
  const int kblocks = K / 64;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t blk = i / 512;
    const int within = (int)(i % 512);
    const int mb = (int)(blk / kblocks), kb = (int)(blk % kblocks);
    const int lane = within / 16, s = (within / 4) % 4, b = within % 4;
    const int g = lane >> 2, t = lane & 3;
    const int r = 16 * mb + g + ((b & 1) ? 8 : 0);
    const int k = 64 * kb + 16 * s + 2 * t + ((b & 2) ? 8 : 0);
    out[w4a16_chunk(mb >> 3, kb, kblocks) + (mb & 7) * 512 + within] =
        codes[(size_t)src_row(r, N, gate_up) * (K / 2) + k / 2];
  }
}

__global__ void prepare_w4a16_sf_kernel(const uint8_t* __restrict__ sf, int N, int K, int gate_up,
                                        uint8_t* __restrict__ out, int* flag) {
  const size_t total = (size_t)N * K / 16;
  const int kblocks = K / 64;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t blk = i / 64;
    const int within = (int)(i % 64);
    const int mb = (int)(blk / kblocks), kb = (int)(blk % kblocks);
    // group g owns 8 bytes: (row g, row g+8) pairs for k16 steps 0..3
    const int g = within / 8, j = (within / 2) & 3, half = within & 1;
    const int r = 16 * mb + g + 8 * half;
    const uint8_t v = sf[(size_t)src_row(r, N, gate_up) * (K / 16) + 4 * kb + j];
    check_sf(v, flag);
    out[w4a16_chunk(mb >> 3, kb, kblocks) + kW16SfOff + (mb & 7) * 64 + within] = v;
  }
}

moe_status launch_prepare_w4a16(const uint8_t* codes, const uint8_t* sf, int N, int K, int gate_up,
                                uint8_t* out, int* flag, cudaStream_t s) {
  prepare_w4a16_data_kernel<<<1024, 256, 0, s>>>(codes, N, K, gate_up, out);
  count_launches(1);
  prepare_w4a16_sf_kernel<<<512, 256, 0, s>>>(sf, N, K, gate_up, out, flag);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

}  // namespace moe

namespace moe {

// W4A4 layout after the header: for every (128-row tile mt, 256-wide K stage
// ks) the 16 KB shared-memory image the block-scaled MMA reads (row r of the
// tile at r * 128 bytes, its 16-byte chunks XOR-swizzled by r % 8), then, in
// a second region, for every (mt, ks) four 512-byte scale-factor atoms (one
// per 64-wide K step; byte m0 * 16 + m1 * 4 + j holds scale j of row
// 32 * m1 + m0).
size_t prepare_w4a4_sf_bytes(int N, int K) { return (size_t)N * K / 16; }

__global__ void prepare_w4a4_data_kernel(const uint8_t* __restrict__ codes, int N, int K, int gate_up,
                                         uint8_t* __restrict__ out) {
  const size_t total = (size_t)N * K / 2;
  const int KS = K / 256;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t tile = i / 16384;
    const int within = (int)(i % 16384);
    const int mt = (int)(tile / KS), ks = (int)(tile % KS);
    const int r = within / 128;
    const int phys_chunk = (within % 128) / 16;
    const int c = ((phys_chunk ^ (r & 7)) << 4) + (within % 16);  // logical byte column
    const int o = mt * 128 + r;
    out[i] = codes[(size_t)src_row(o, N, gate_up) * (K / 2) + ks * 128 + c];
  }
}

__global__ void prepare_w4a4_sf_kernel(const uint8_t* __restrict__ sf, int N, int K, int gate_up,
                                       uint8_t* __restrict__ out, int* flag) {
  const size_t total = (size_t)N * K / 16;
  const int KS = K / 256;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t tile = i / 2048;
    const int within = (int)(i % 2048);
    const int mt = (int)(tile / KS), ks = (int)(tile % KS);
    const int kk = within / 512, a = within % 512;
    const int m0 = a / 16, m1 = (a % 16) / 4, jj = a % 4;
    const int r = 32 * m1 + m0;
    const int o = mt * 128 + r;
    const uint8_t v = sf[(size_t)src_row(o, N, gate_up) * (K / 16) + ks * 16 + kk * 4 + jj];
    check_sf(v, flag);
    out[i] = v;
  }
}

// MXFP4 ("vLLM on the NVIDIA DGX Spark", section 6.4): the same tile images;
// E8M0 scales, one per 32 along K, in 512-byte atoms that each hold four
// consecutive scales of the tile's 128 rows (K 128: two K=64 MMAs, the
// kind::mxf4 .scale_vec::2X layout, which picks bytes 0-1 or 2-3 of a row's
// word per MMA). Per (tile mt, 256-wide K stage ks): two atoms. Code 0xFF
// (NaN) is refused.
__global__ void prepare_mx_sf_kernel(const uint8_t* __restrict__ sf, int N, int K, int gate_up,
                                     uint8_t* __restrict__ out, int* flag) {
  const size_t total = (size_t)N * K / 32;
  const int KS = K / 256;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t tile = i / 1024;
    const int within = (int)(i % 1024);
    const int mt = (int)(tile / KS), ks = (int)(tile % KS);
    const int c = within / 512, a = within % 512;
    const int m0 = a / 16, m1 = (a % 16) / 4, jj = a % 4;
    const int o = mt * 128 + 32 * m1 + m0;
    const uint8_t v = sf[(size_t)src_row(o, N, gate_up) * (K / 32) + ks * 8 + c * 4 + jj];
    if (v == 0xffu) atomicOr(flag, 1);
    out[i] = v;
  }
}

moe_status launch_prepare_w4a4(const uint8_t* codes, const uint8_t* sf, int N, int K, int gate_up,
                               uint8_t* out_data, uint8_t* out_sf, int* flag, cudaStream_t s, bool mx) {
  if (K % 256) return MOE_ERR_INVALID_ARG;
  prepare_w4a4_data_kernel<<<1024, 256, 0, s>>>(codes, N, K, gate_up, out_data);
  count_launches(1);
  if (mx)
    prepare_mx_sf_kernel<<<512, 256, 0, s>>>(sf, N, K, gate_up, out_sf, flag);
  else
    prepare_w4a4_sf_kernel<<<512, 256, 0, s>>>(sf, N, K, gate_up, out_sf, flag);
  count_launches(1);
  return cuda_ok(cudaGetLastError());
}

}  // namespace moe
