// moe_permute_noalloc: the expert permutation for callers that cannot
// allocate device memory at call time. Its scratch lives in a fixed
// file-scope device array instead of a caller workspace.
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {
namespace {

// Scratch of the no-allocation permutation: a 256-byte status header, then
// the per-chunk expert histogram of the multi-CTA sort. Every device that
// loads this library holds these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = 64 * 1024;
static __device__ __align__(256) unsigned char g_permute_scratch[kNoAllocScratchBytes];

// Device address of g_permute_scratch per device. In host code the symbol is
// only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress with that device current.
std::mutex g_mu;
void* g_addr[64] = {nullptr};

moe_status scratch_address(void** out) {
  int dev = 0;
  moe_status st = cuda_ok(cudaGetDevice(&dev));
  if (st != MOE_OK) return st;
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    st = cuda_ok(cudaGetSymbolAddress(&p, g_permute_scratch));
    if (st != MOE_OK) return st;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_permute_noalloc(const int32_t* topk_ids, int T, int k, int E, int32_t* counts,
                                          int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                                          int32_t* device_status, moe_stream_t stream) {
  if (T < 0 || E < 1 || k < 1) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || (long long)T * k > (1LL << 30)) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_ids || !perm || !inv_perm)) return MOE_ERR_INVALID_ARG;
  // the scratch this call needs must fit the fixed array
  if (sizeof(WsHeader) + permute_scratch_bytes(T, k, E) > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;
  int dev = 0, major = 0, minor = 0;
  moe_status st = cuda_ok(cudaGetDevice(&dev));
  if (st != MOE_OK) return st;
  st = cuda_ok(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
  if (st != MOE_OK) return st;
  st = cuda_ok(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
  if (st != MOE_OK) return st;
  if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  auto* hdr = static_cast<WsHeader*>(scratch);
  // the array keeps the previous call's contents: the status word must start
  // at zero; the histogram is fully rewritten by every multi-CTA sort
  st = cuda_ok(cudaMemsetAsync(&hdr->status, 0, sizeof(int), s));
  if (st != MOE_OK) return st;
  st = launch_permute(topk_ids, T, k, E, counts, offsets, perm, inv_perm, &hdr->status,
                      static_cast<uint8_t*>(scratch) + sizeof(WsHeader), nullptr, nullptr, nullptr, nullptr, s);
  if (st != MOE_OK) return st;
  if (device_status != nullptr)
    st = cuda_ok(cudaMemcpyAsync(device_status, &hdr->status, sizeof(int), cudaMemcpyDeviceToDevice, s));
  return st;
}
