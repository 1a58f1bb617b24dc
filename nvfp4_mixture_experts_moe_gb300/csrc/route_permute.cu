// Router top-k and the stable expert permutation.
//
// Router: "Serving Solar Open 2 on DGX Spark", "Solar Open 2 in brief"
// (320 routed experts + 1 shared, top-8); "vLLM on the NVIDIA DGX Spark: A
// Complete Technical Guide", section 7.1 ([Router] stage).
// Permutation: same guide, section 4.3 (token dispatch) and section 7.1
// ([Permute-Experts-Unpermute]).
#include "common.cuh"
#include "kernels.cuh"
#include "route.cuh"

namespace moe {

template <int PER_LANE>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E,
                                                         int k, int32_t* __restrict__ ids,
                                                         float* __restrict__ w) {
  const int token = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (token >= T) return;
  route_token<PER_LANE>(logits, token, E, k, ids, w);
}

moe_status launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                             cudaStream_t s) {
  if (T == 0) return MOE_OK;
  const int threads = 256;
  const int blocks = (int)(((size_t)T * 32 + threads - 1) / threads);
  const int per = (E + 31) / 32;
#define MOE_ROUTE_CASE(P)                                                             \
  if (per <= P) {                                                                     \
    route_topk_kernel<P><<<blocks, threads, 0, s>>>(logits, T, E, k, ids, w);         \
    count_launches(1);                                                                \
    return cuda_ok(cudaGetLastError());                                               \
  }
  MOE_ROUTE_CASE(1)
  MOE_ROUTE_CASE(2)
  MOE_ROUTE_CASE(4)
  MOE_ROUTE_CASE(8)
  MOE_ROUTE_CASE(16)
  MOE_ROUTE_CASE(32)
#undef MOE_ROUTE_CASE
  return MOE_ERR_UNSUPPORTED;
}

// ---------------------------------------------------------------------------
// Stable counting sort of the P = T*k pairs by expert.
//
// Phase 1 (count): per chunk of pairs, a shared-memory histogram.
// Phase 2 (scan):  offsets[e] = sum of counts below e; the base of chunk b
//                  inside expert e's group = offsets[e] + counts of e in
//                  chunks before b.
// Phase 3 (scatter): per chunk, one warp walks its pairs in order, 32 at a
//                  time; lanes holding the same expert (match_any) take
//                  consecutive slots in lane order, so a pair's slot grows
//                  with its index p (stability).
// Small problems run all three phases in one CTA (one launch); large ones use
// three launches with one CTA per chunk.

constexpr int kPermChunk = 4096;  // pairs per chunk in the multi-CTA path

// Expert parallelism ("Serving Solar Open 2 on DGX Spark", "Adding Expert
// Parallelism to b12x": each node holds a contiguous shard of the experts,
// global ids are remapped to shard-local ones and out-of-shard pairs are
// filtered out). A global id in [lo, lo + n) maps to local group id - lo; a
// valid id of another shard gives -1 (the pair is dropped without an error:
// another shard computes it); an id outside [0, E_global) gives -2 (an error).
// Without sharding lo = 0 and n = E_global.
__device__ __forceinline__ int shard_local(int id, int lo, int n, int E_global) {
  if (id < 0 || id >= E_global) return -2;
  const int e = id - lo;
  return (e >= 0 && e < n) ? e : -1;
}

__device__ __forceinline__ void scatter_warp(const int32_t* __restrict__ ids, int p0, int p1, int E,
                                             int* cursor /* smem [E] */, int32_t* perm,
                                             int32_t* inv_perm, int* status, int lo, int E_global,
                                             const int32_t* lids = nullptr, int32_t* lperm = nullptr) {
  const int lane = threadIdx.x & 31;
  for (int base = p0; base < p1; base += 32) {
    const int p = base + lane;
    const bool in = p < p1;
    // ids written earlier in the same kernel: the shared copy, else an L2 load
    const int e = in ? shard_local(lids ? lids[p] : __ldcg(ids + p), lo, E, E_global) : -1;
    const bool valid = in && e >= 0;
    if (in && e == -2) set_status(status, MOE_ERR_DEVICE);
    const int key = valid ? e : -1 - lane;  // invalid lanes never match each other
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const unsigned lt = (1u << lane) - 1u;
    const int rank = __popc(peers & lt);
    int slot = 0;
    if (valid) slot = cursor[e] + rank;
    __syncwarp();
    if (valid) {
      perm[slot] = p;
      inv_perm[p] = slot;
      if (lperm) lperm[slot] = p;
      // highest lane of the peer group advances the cursor
      if ((peers >> lane) == 1u) cursor[e] += __popc(peers);
    } else if (in) {
      inv_perm[p] = -1;
    }
    __syncwarp();
  }
}

// Extra per-row outputs for the fused forward: the A-row (token) of each
// sorted row and its routing weight. The Pu routed rows that were kept (all
// P = T*k of them unless a shard or bad ids dropped some) come first, then
// the T shared rows at [Pu, Pu + T); rows past Pu + T are unused.
struct RowInfoOut {
  int32_t* row_token;    // [P + T] or nullptr
  float* row_weight;     // [P + T] or nullptr
  const float* topk_w;   // [P]
  int k, T;
  int32_t* gofs;         // [E+2] or nullptr: offsets[0..E] (offsets[E] = Pu), then Pu + T
};

__device__ __forceinline__ void row_info_one(const RowInfoOut& ri, int r, int Pu, int p, float wp) {
  if (r < Pu) {
    const bool ok = p >= 0;
    ri.row_token[r] = ok ? p / ri.k : 0;
    ri.row_weight[r] = ok ? wp : 0.0f;
  } else if (r < Pu + ri.T) {
    ri.row_token[r] = r - Pu;
    ri.row_weight[r] = 1.0f;
  } else {
    ri.row_token[r] = 0;
    ri.row_weight[r] = 0.0f;
  }
}

__device__ void write_row_info(const RowInfoOut& ri, const int32_t* perm, int P, int Pu,
                               const int32_t* lperm = nullptr, const float* lw = nullptr) {
  if (ri.row_token == nullptr) return;
  for (int r = threadIdx.x; r < P + ri.T; r += blockDim.x) {
    int p = -1;
    if (r < Pu) {
      p = lperm ? lperm[r] : perm[r];
      if (p < 0 || p >= P) p = -1;
    }
    row_info_one(ri, r, Pu, p, p >= 0 ? (lw ? lw[p] : ri.topk_w[p]) : 0.0f);
  }
}

// Block-wide exclusive scan of n <= blockDim.x * 4 ints in shared memory.
__device__ void block_exclusive_scan(int* data, int n, int* tmp /* smem [32] */) {
  const int tid = threadIdx.x;
  const int per = (n + blockDim.x - 1) / blockDim.x;
  int local = 0;
  for (int i = 0; i < per; ++i) {
    const int idx = tid * per + i;
    if (idx < n) local += data[idx];
  }
  int incl = local;
  const int lane = tid & 31, wid = tid >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) tmp[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int nw = (blockDim.x + 31) / 32;
    int v = lane < nw ? tmp[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += o;
    }
    if (lane < nw) tmp[lane] = v;
  }
  __syncthreads();
  int run = incl - local + (wid > 0 ? tmp[wid - 1] : 0);
  for (int i = 0; i < per; ++i) {
    const int idx = tid * per + i;
    if (idx < n) {
      const int d = data[idx];
      data[idx] = run;
      run += d;
    }
  }
  __syncthreads();
}

__device__ void permute_single_body(const int32_t* __restrict__ ids, int P, int E, int32_t* counts,
                                    int32_t* offsets, int32_t* perm, int32_t* inv_perm, int* status,
                                    const RowInfoOut& ri, int lo, int E_global, const int32_t* lids = nullptr,
                                    const float* lw = nullptr, int32_t* lperm = nullptr) {
  extern __shared__ int smem[];
  int* cnt = smem;            // [E]
  int* cursor = smem + E;     // [E]
  int* tmp = smem + 2 * E;    // [32]
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    perm[p] = -1;
    if (lperm) lperm[p] = -1;
  }
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    // ids written earlier in the same kernel: the shared copy, else an L2 load
    const int e = shard_local(lids ? lids[p] : __ldcg(ids + p), lo, E, E_global);
    if (e >= 0) atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    counts[e] = cnt[e];
    cursor[e] = cnt[e];
  }
  __syncthreads();
  block_exclusive_scan(cursor, E, tmp);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    offsets[e] = cursor[e];
    if (ri.gofs) ri.gofs[e] = cursor[e];
  }
  const int Pu = cursor[E - 1] + cnt[E - 1];  // routed pairs kept (this shard's, valid ids)
  if (threadIdx.x == 0) {
    offsets[E] = Pu;
    if (ri.gofs) {
      ri.gofs[E] = Pu;
      ri.gofs[E + 1] = Pu + ri.T;
    }
  }
  __syncthreads();
  if (threadIdx.x < 32) scatter_warp(ids, 0, P, E, cursor, perm, inv_perm, status, lo, E_global, lids, lperm);
  __syncthreads();
  __threadfence_block();
  write_row_info(ri, perm, P, Pu, lperm, lw);
}

__global__ void __launch_bounds__(1024) permute_single_kernel(const int32_t* __restrict__ ids, int P,
                                                              int E, int32_t* counts, int32_t* offsets,
                                                              int32_t* perm, int32_t* inv_perm,
                                                              int* status, RowInfoOut ri, int lo, int E_global) {
  pdl_wait();
  permute_single_body(ids, P, E, counts, offsets, perm, inv_perm, status, ri, lo, E_global);
}

// Small batches: route and permute in one CTA (one launch). Warp w routes
// tokens w, w + 32, ...; the permutation starts once every id is written.
// E_global experts are routed; the permutation groups the pairs of the E
// experts [lo, lo + E) of this shard (E = E_global, lo = 0 without sharding).
template <int PER_LANE>
__global__ void __launch_bounds__(1024) route_permute_small_kernel(const float* __restrict__ logits, int T,
                                                                   int E_global, int k, int32_t* ids, float* w,
                                                                   int32_t* counts, int32_t* offsets,
                                                                   int32_t* perm, int32_t* inv_perm,
                                                                   int* status, RowInfoOut ri, int lo, int E) {
  extern __shared__ int smem_rp[];
  const int P = T * k;
  // after the permutation's own shared arrays ([2E + 32] ints): ids, weights, perm of the pairs
  int32_t* sids = smem_rp + 2 * E + 32;
  float* sw = reinterpret_cast<float*>(sids + P);
  int32_t* sperm = reinterpret_cast<int32_t*>(sw + P);
  for (int t = threadIdx.x >> 5; t < T; t += blockDim.x >> 5)
    route_token<PER_LANE>(logits, t, E_global, k, ids, w, sids, sw);
  __syncthreads();
  permute_single_body(ids, P, E, counts, offsets, perm, inv_perm, status, ri, lo, E_global, sids, sw, sperm);
}

moe_status launch_route_permute_small(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                                      int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv_perm,
                                      int* status, int32_t* row_token, float* row_weight, int32_t* gofs,
                                      cudaStream_t s, int shard_lo, int shard_n) {
  RowInfoOut ri{row_token, row_weight, w, k, T, gofs};
  const size_t smem = (2 * (size_t)shard_n + 32 + 3 * (size_t)T * k) * sizeof(int);
  if (smem > 48 * 1024) return MOE_ERR_UNSUPPORTED;
  const int per = (E + 31) / 32;
#define MOE_RP_CASE(PL)                                                                                  \
  if (per <= PL) {                                                                                       \
    route_permute_small_kernel<PL><<<1, 1024, smem, s>>>(logits, T, E, k, ids, w, counts, offsets, perm, \
                                                         inv_perm, status, ri, shard_lo, shard_n);       \
    count_launches(1);                                                                                   \
    return cuda_ok(cudaGetLastError());                                                                  \
  }
  MOE_RP_CASE(1)
  MOE_RP_CASE(2)
  MOE_RP_CASE(4)
  MOE_RP_CASE(8)
  MOE_RP_CASE(10)
  MOE_RP_CASE(16)
  MOE_RP_CASE(32)
#undef MOE_RP_CASE
  return MOE_ERR_UNSUPPORTED;
}

__global__ void __launch_bounds__(1024) permute_count_kernel(const int32_t* __restrict__ ids, int P, int E,
                                                             int32_t* chunk_hist /* [nchunks][E] */,
                                                             int32_t* perm, int lo, int E_global) {
  pdl_wait();
  extern __shared__ int cnt[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * kPermChunk;
  const int p1 = min(P, p0 + kPermChunk);
  for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    const int e = shard_local(__ldg(ids + p), lo, E, E_global);
    perm[p] = -1;
    if (e >= 0) atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_hist[(size_t)blockIdx.x * E + e] = cnt[e];
}

__global__ void __launch_bounds__(1024) permute_scan_kernel(int32_t* chunk_hist, int nchunks, int E, int P,
                                                            int32_t* counts, int32_t* offsets,
                                                            int32_t* gofs, int T) {
  pdl_wait();
  extern __shared__ int smem[];
  int* tot = smem;         // [E]
  int* tmp = smem + E;     // [32]
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int b = 0; b < nchunks; ++b) {
      const int c = chunk_hist[(size_t)b * E + e];
      chunk_hist[(size_t)b * E + e] = run;  // becomes the base within the group
      run += c;
    }
    tot[e] = run;
    counts[e] = run;
  }
  __syncthreads();
  int last = 0;
  if (threadIdx.x == 0) last = tot[E - 1];
  block_exclusive_scan(tot, E, tmp);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    offsets[e] = tot[e];
    if (gofs) gofs[e] = tot[e];
    for (int b = 0; b < nchunks; ++b) chunk_hist[(size_t)b * E + e] += tot[e];
  }
  if (threadIdx.x == 0) {
    const int Pu = tot[E - 1] + last;   // routed pairs kept; the shared rows follow them
    offsets[E] = Pu;
    if (gofs) {
      gofs[E] = Pu;
      gofs[E + 1] = Pu + T;
    }
  }
}

// Phase 3 inside a chunk: kScatterWarps warps take consecutive sub-chunks;
// each counts its own pairs per expert, the counts are scanned across the
// warps on top of the chunk's base, and every warp then scatters its
// sub-chunk in order (stable: earlier sub-chunks get the lower slots).
constexpr int kScatterWarps = 8;

__global__ void __launch_bounds__(kScatterWarps * 32) permute_scatter_kernel(const int32_t* __restrict__ ids, int P,
                                                                            int E, const int32_t* chunk_base,
                                                                            int32_t* perm, int32_t* inv_perm,
                                                                            int* status, int lo, int E_global) {
  pdl_wait();
  extern __shared__ int cursor[];  // [kScatterWarps][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kScatterWarps * E; i += blockDim.x) cursor[i] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * kPermChunk;
  const int p1 = min(P, p0 + kPermChunk);
  constexpr int kSub = kPermChunk / kScatterWarps;
  const int q0 = min(p1, p0 + warp * kSub), q1 = min(p1, q0 + kSub);
  for (int p = q0 + lane; p < q1; p += 32) {
    const int e = shard_local(__ldg(ids + p), lo, E, E_global);
    if (e >= 0) atomicAdd(&cursor[warp * E + e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = chunk_base[(size_t)blockIdx.x * E + e];
    for (int w = 0; w < kScatterWarps; ++w) {
      const int c = cursor[w * E + e];
      cursor[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  if (q0 < q1) scatter_warp(ids, q0, q1, E, cursor + warp * E, perm, inv_perm, status, lo, E_global);
}

__global__ void row_info_kernel(const int32_t* perm, int P, const int32_t* offsets_end, RowInfoOut ri) {
  pdl_wait();
  // grid-stride version of write_row_info; the kept routed rows end at offsets[E]
  const int Pu = __ldcg(offsets_end);
  const int n = P + ri.T;
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < n; r += gridDim.x * blockDim.x) {
    int p = r < Pu ? perm[r] : -1;
    if (p >= P) p = -1;
    row_info_one(ri, r, Pu, p, p >= 0 ? ri.topk_w[p] : 0.0f);
  }
}

size_t permute_scratch_bytes(int T, int k, int E) {
  const size_t P = (size_t)T * k;
  if (P <= (size_t)kPermSingleMax) return 0;
  const size_t nchunks = (P + kPermChunk - 1) / kPermChunk;
  return align_up(nchunks * (size_t)E * sizeof(int32_t));
}

moe_status launch_permute(const int32_t* ids, int T, int k, int E, int32_t* counts, int32_t* offsets,
                          int32_t* perm, int32_t* inv_perm, int* status, void* scratch,
                          int32_t* row_token, float* row_weight, const float* topk_w, int32_t* gofs,
                          cudaStream_t s, bool pdl, int shard_lo, int E_global) {
  const int P = T * k;
  if (E_global <= 0) E_global = E;
  RowInfoOut ri{row_token, row_weight, topk_w, k, T, gofs};
  if (P <= kPermSingleMax) {
    const size_t smem = (2 * (size_t)E + 32) * sizeof(int);
    cudaError_t e = launch_ex(pdl, permute_single_kernel, dim3(1), dim3(1024), smem, s, ids, P, E, counts,
                              offsets, perm, inv_perm, status, ri, shard_lo, E_global);
    if (e != cudaSuccess) return cuda_ok(e);
    count_launches(1);
    return cuda_ok(cudaGetLastError());
  }
  const int nchunks = (P + kPermChunk - 1) / kPermChunk;
  int32_t* hist = static_cast<int32_t*>(scratch);
  cudaError_t e = launch_ex(pdl, permute_count_kernel, dim3(nchunks), dim3(1024), (size_t)E * sizeof(int), s,
                            ids, P, E, hist, perm, shard_lo, E_global);
  if (e != cudaSuccess) return cuda_ok(e);
  count_launches(1);
  e = launch_ex(pdl, permute_scan_kernel, dim3(1), dim3(1024), ((size_t)E + 32) * sizeof(int), s, hist,
                nchunks, E, P, counts, offsets, gofs, T);
  if (e != cudaSuccess) return cuda_ok(e);
  count_launches(1);
  e = launch_ex(pdl, permute_scatter_kernel, dim3(nchunks), dim3(kScatterWarps * 32),
                (size_t)kScatterWarps * E * sizeof(int), s, ids, P, E, (const int32_t*)hist, perm, inv_perm, status,
                shard_lo, E_global);
  if (e != cudaSuccess) return cuda_ok(e);
  count_launches(1);
  if (row_token != nullptr) {
    const int n = P + T;
    e = launch_ex(pdl, row_info_kernel, dim3((n + 255) / 256), dim3(256), 0, s, (const int32_t*)perm, P,
                  (const int32_t*)(offsets + E), ri);
    if (e != cudaSuccess) return cuda_ok(e);
    count_launches(1);
  }
  return cuda_ok(cudaGetLastError());
}

}  // namespace moe
