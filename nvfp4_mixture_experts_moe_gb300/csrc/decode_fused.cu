// The whole layer in one kernel for decode batches (W4A16, up to 8 tokens):
// route, permute, gate/up GEMM + SwiGLU, down GEMM + routing weight and the
// combine, in one persistent launch ("micro path").
//
// "Serving Solar Open 2 on DGX Spark", "The fix" (a separate micro path for
// small decode batches); "vLLM on the NVIDIA DGX Spark: A Complete Technical
// Guide", section 4.3 (dispatch, both expert GEMMs, SwiGLU and the top-k
// weight reduction fused into one kernel), section 5 (weight-only NVFP4:
// 4-bit weights dequantised to 16-bit inside the GEMM) and section 6.1
// (alpha = 1/gs).
//
// At a few tokens the layer is bound by the bytes of the touched experts'
// weights; everything else is latency. One CTA per SM (cooperative launch, so
// all CTAs are resident and may wait on one another with bounded spins):
//
// * Routing and the permutation are computed by every CTA in shared memory
//   (a few hundred logits per token); meanwhile the x rows arrive by bulk
//   copy and are converted in place to f16 with a power-of-two row scale;
//   they stay resident for the gate/up phase.
// * Work items are (active expert group, 128-row weight tile): gate/up items
//   0..N1-1, then down items. Each CTA's producer takes the next item from a
//   grid-wide counter when it is about to stream the last stage of its
//   current one, so CTAs that stream faster take more items and all finish
//   within about one item of each other. A CTA's items increase, so a down
//   item's group has had all its gate/up items taken before (long before, in
//   all but the last groups). The producer publishes each item in a small
//   per-CTA queue that the other warps read in order.
// * The producer streams every item's weight tiles (stages of up to 8
//   64-wide K blocks, 36 KB, in a ring of as many as fit) with bulk copies
//   from the gate/up phase straight into the down phase, so the down weights
//   are already in flight when the gate/up items end.
// * Sixteen MMA warps (8 row blocks x 2 halves; in every stage half h takes
//   the K blocks h, h + 2, ...)
//   turn the e2m1 codes into f16 with the hardware conversion, multiply in
//   the E4M3 block scales and run mma.sync m16n8k16 with the group's rows as
//   N; at the end of an item the half that finishes second adds the other's
//   partial sums and runs the epilogue, while the first goes on to the next
//   item. The stage sizes and the split are those of the multi-kernel
//   path's decode GEMM, so the arithmetic (and the result, bit for bit) is
//   the same (the same stage loop and join, decode_mma.cuh).
// * Gate/up epilogue: SwiGLU, h stored bf16 in the workspace with a running
//   per-row max |h|. Down epilogue: y = h W2^T * alpha * routing weight,
//   stored bf16 (the shared expert's rows fp32). Neither waits on a global
//   fence: the MMA warps hand each finished item to a signal warp through an
//   mbarrier.
// * The signal warp counts a gate/up item in gu_done[group] (one release at
//   gpu scope, cumulative over the MMA warps' stores); a helper warp stages
//   a down item's h rows (as f16 with a row scale) once all gate/up tiles of
//   the group are counted (acquire). For a down item the signal warp counts
//   each (token, 128 output columns) contribution; the one that completes the
//   k + 1 of a token sums the token's rows in the fixed order j = 0..k-1,
//   then the shared row, in fp32 and writes the bf16 output. The sum order
//   never depends on which CTA does it: the result is deterministic.
//
// Every wait (mbarriers, the gate/up counters) is bounded; on a timeout the
// kernel records MOE_ERR_TIMEOUT, lets its bulk copies land and exits.
#include <algorithm>

#include "common.cuh"
#include "decode_mma.cuh"
#include "kernels.cuh"
#include "route.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kMaxT = kDecodeFusedMaxT;           // tokens (each group has at most this many rows)
constexpr int kMaxK = 32;
using decode::kBlockWarps;                         // one per 16-row block of a 128-row tile
using decode::kHalves;                             // halves: alternate K blocks of every stage
constexpr int kMmaWarps = kBlockWarps * kHalves;
constexpr int kProducerWarp = kMmaWarps;
constexpr int kHelperWarp = kMmaWarps + 1;
constexpr int kSignalWarp = kMmaWarps + 2;
constexpr int kThreads = (kMmaWarps + 3) * 32;
constexpr int kTile = 128;
constexpr int kMaxSlots = 16;                      // ring slots of stage_kb K blocks (stage_kb * 4608 bytes)
constexpr int kHSlots = 2;                         // staged h row sets (down items)
constexpr int kMaxRows = kMaxT * kMaxK + kMaxT;    // routed pairs + shared rows
constexpr int kMaxGroups = kMaxT * kMaxK + 1;      // active groups: at most one per pair, + shared
constexpr int kQueue = 8;
constexpr int kDoneSlots = 4;                      // finished items the signal warp may lag behind                          // the CTA's published items not yet taken over
constexpr long long kDrainLimit = 4ll * 1000 * 1000 * 1000;  // cycles for in-flight copies to land

struct Args {
  const float* logits;
  const uint16_t* x;
  const uint8_t* w13;
  size_t s13;
  const uint8_t* w13_shared;
  const uint8_t* w2;
  size_t s2;
  const uint8_t* w2_shared;
  int T, H, I, E, k, has_shared;
  uint16_t* out;
  int32_t* topk_ids_out;
  uint16_t* h;          // [rows, I] bf16
  uint16_t* y;          // [T*k, H] routed rows, bf16
  float* y_shared;      // [T, H] the shared expert's rows, fp32
  // two counter sets (set 1 set_ints ints after set 0), each: gu_done
  // [groups], cmb_cnt [T][H/128], hmax [rows] (bf16 magnitude bits of max
  // |h|), the grid's item counter
  int* counters;
  int set_ints;
  int counter_ints;
  int* clean;                    // header: 1 = both sets were zeroed once
  unsigned long long* ticket;    // header: one per CTA per launch
  unsigned long long* gbar;      // header: first-use grid barrier (counts up)
  int* status;
  int slots;
  int stage_kb;         // K blocks per ring slot (the larger of the two phases' stages)
  int kmax;             // max 64-wide K blocks per stage (1..8)
  long long wait_limit;
  int extra_arrivals;   // test hook: arrivals expected per gate/up tile beyond the real ones
};

struct Smem {
  uint64_t full[kMaxSlots];
  uint64_t empty[kMaxSlots];
  uint64_t hfull[kHSlots];
  uint64_t hland[kHSlots];       // the helper's bulk copies of a slot's h rows have landed
  uint64_t hempty[kHSlots];
  uint64_t xfull;                // the x rows (bf16) have landed in shared memory
  uint64_t xfree;                // every MMA warp is done with the resident x rows
  uint64_t done[kDoneSlots];     // an item's epilogue stores are issued (one warp per row block)
  int released;                  // items the signal warp has taken over (counts up; no parity aliasing)
  int q_item[kQueue];            // the CTA's c-th item (its descriptor) at c % kQueue (-1: no more items)
  int q_count;                   // items published
  int first_down;                // index c of the CTA's first down item (or of the end)
  int* ctr;                      // this launch's counter set
  int abort;
  int A;                         // active groups
  int32_t ids[kMaxT * kMaxK];
  float w[kMaxT * kMaxK];
  int32_t inv[kMaxT * kMaxK];    // pair -> grouped row
  int32_t row_tok[kMaxRows];
  int32_t row_e[kMaxT * kMaxK];  // expert of grouped row r (routed rows)
  float row_w[kMaxRows];
  int32_t grp_e[kMaxGroups];     // expert of active group a (E = shared)
  int32_t grp_r0[kMaxGroups];
  int32_t grp_n[kMaxGroups];
  float xmul[kMaxT];
  float hmul[kHSlots][kMaxT];
  decode::HalfJoin join;         // the two halves' partial sums of an item
};

// This launch's counters inside its set.
struct Ctr {
  int* gu_done;
  int* cmb_cnt;
  unsigned* hmax;
  int* next_item;
};
__device__ __forceinline__ Ctr ctr_of(int* base, const Args& p) {
  Ctr c;
  const int rows = p.T * p.k + (p.has_shared ? p.T : 0);
  c.gu_done = base;
  c.cmb_cnt = base + p.E + 1;
  c.hmax = reinterpret_cast<unsigned*>(c.cmb_cnt + p.T * (p.H / 128));
  c.next_item = reinterpret_cast<int*>(c.hmax + rows);
  return c;
}

// Power-of-two row scale from a row's largest bf16 magnitude (bit pattern m):
// 2^sh brings the maximum into [2^14, 2^15), where every bf16 value down to
// 2^-24 of the maximum is exact in f16. Returns sh.
__device__ __forceinline__ int row_shift(uint32_t m) {
  const int e = (int)(m >> 7);
  int sh = (m == 0) ? 0 : 141 - max(e, 1);
  return max(-113, min(sh, 126));
}

// A queue entry describes an item by its phase (bit 30: down), its group a
// (bits 12..29) and its 128-row weight tile mt (bits 0..11), so that no warp
// divides to decode it; -1 is the end of the CTA's items.
__device__ __forceinline__ int item_desc(int ph, int a, int mt) { return (ph << 30) | (a << 12) | mt; }
__device__ __forceinline__ int desc_ph(int d) { return (d >> 30) & 1; }
__device__ __forceinline__ int desc_a(int d) { return (d >> 12) & 0x3ffff; }
__device__ __forceinline__ int desc_mt(int d) { return d & 0xfff; }

// Barrier over the first n threads of the CTA (named barrier id, not 0).
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// The CTA's c-th item from its queue (lane 0 waits, bounded; broadcast):
// >= 0 an item, -1 no more items, -2 the wait gave up.
__device__ __forceinline__ int queue_get(Smem* sm, int c, volatile int* abort, long long limit, int lane) {
  int v = -2;
  if (lane == 0 && decode::spin_ge(&sm->q_count, c + 1, abort, limit)) {
    __threadfence_block();
    v = *reinterpret_cast<volatile int*>(&sm->q_item[c % kQueue]);
  }
  return __shfl_sync(0xffffffffu, v, 0);
}

// The c-th item if it is published already, else -3 (no wait).
__device__ __forceinline__ int queue_peek(Smem* sm, int c, int lane) {
  int v = -3;
  if (lane == 0 && *reinterpret_cast<volatile int*>(&sm->q_count) > c) {
    __threadfence_block();
    v = *reinterpret_cast<volatile int*>(&sm->q_item[c % kQueue]);
  }
  return __shfl_sync(0xffffffffu, v, 0);
}

// Bounded wait for *ctr >= target (another CTA's release increments), or abort.
__device__ __forceinline__ bool wait_counter(const int* ctr, int target, volatile int* abort, long long limit) {
  const long long t0 = clock64();
  while (true) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) return true;
    if (*abort) return false;
    if (clock64() - t0 > limit) {
      *abort = 1;
      return false;
    }
    __nanosleep(64);
  }
}

__device__ __forceinline__ bool wait_counter64(const unsigned long long* ctr, unsigned long long target,
                                               volatile int* abort, long long limit) {
  const long long t0 = clock64();
  while (true) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(ctr) : "memory");
    if (v >= target) return true;
    if (*abort) return false;
    if (clock64() - t0 > limit) {
      *abort = 1;
      return false;
    }
    __nanosleep(64);
  }
}

__device__ __forceinline__ void release_add(int* ctr, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(ctr), "r"(v) : "memory");
}


// out[t, col .. col+8) = sum_j y[inv[t, j]] (j = 0..k-1 in order) + y_shared[t]
// in fp32, rounded once to bf16: the same sum, in the same order, as the
// multi-kernel path's combine. All of the token's row loads are issued
// before the first add (no chain of dependent loads).
__device__ __forceinline__ void combine_cols8(const Args& p, const int32_t* inv, int t, int k, int H, int col) {
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  for (int j0 = 0; j0 < k; j0 += 8) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      v[u] = j0 + u < k ? __ldcg(reinterpret_cast<const uint4*>(p.y + (size_t)inv[t * k + j0 + u] * H + col))
                        : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (j0 + u >= k) break;
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] += __uint_as_float(w[i] << 16);
        acc[2 * i + 1] += __uint_as_float(w[i] & 0xffff0000u);
      }
    }
  }
  if (p.has_shared) {
    const float4* ys = reinterpret_cast<const float4*>(p.y_shared + (size_t)t * H + col);
    const float4 a = __ldcg(ys), b = __ldcg(ys + 1);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += v[i];
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = (uint32_t)float_to_bf16_bits(acc[2 * i]) | ((uint32_t)float_to_bf16_bits(acc[2 * i + 1]) << 16);
  *reinterpret_cast<uint4*>(p.out + (size_t)t * H + col) = make_uint4(o[0], o[1], o[2], o[3]);
}

__global__ void __launch_bounds__(kThreads, 1) decode_fused_kernel(Args p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int T = p.T, H = p.H, I = p.I, E = p.E, k = p.k;
  const int S = p.slots;
  const int P = T * k;
  const int KB1 = H / 64, KB2 = I / 64;
  const int MT1 = (2 * I) / kTile, MT2 = H / kTile;
  const size_t kStageBytes = (size_t)p.stage_kb * kW16Chunk;   // ring slot: the larger phase's stage
  const int KBS1 = w16_stage_kb(KB1, p.kmax), KBS2 = w16_stage_kb(KB2, p.kmax);   // K blocks per stage
  const int NST1 = (KB1 + KBS1 - 1) / KBS1, NST2 = (KB2 + KBS2 - 1) / KBS2;
  const int xs_stride = H + 8;    // f16 per resident x row (16-byte pad: conflict-free ldmatrix)
  const int hs_stride = I + 8;
  uint8_t* ring = smem_raw;
  uint16_t* act = reinterpret_cast<uint16_t*>(ring + (size_t)S * kStageBytes);
  const size_t act_elems = max((size_t)T * xs_stride, (size_t)kHSlots * kMaxT * hs_stride);
  Smem* sm = reinterpret_cast<Smem*>(act + act_elems);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  volatile int* abort = &sm->abort;
  const long long limit = p.wait_limit;

  // ------------------------------------------------------------ phase 0
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&sm->full[i], 1);
      mbar_init(&sm->empty[i], kMmaWarps);  // both halves read every stage
    }
    for (int i = 0; i < kHSlots; ++i) {
      mbar_init(&sm->hland[i], 1);
      mbar_init(&sm->hfull[i], 1);
      mbar_init(&sm->hempty[i], kMmaWarps);
    }
    decode::half_join_init(&sm->join, 0, 1);
    mbar_init(&sm->xfree, kMmaWarps);
    mbar_init(&sm->xfull, 1);
    for (int i = 0; i < kDoneSlots; ++i) {
      mbar_init(&sm->done[i], kBlockWarps);
    }
    sm->abort = 0;
    sm->released = 0;
    sm->q_count = 0;
    sm->first_down = 0;
    fence_barrier_init();
  }
  __syncthreads();   // barriers initialised
  int first_item = 0;
  if (warp == kProducerWarp && lane == 0) {
    // Launch n (tickets n*grid .. n*grid + grid-1, one per CTA) counts in set
    // n % 2, which launch n-1's helper zeroed. The first launch that finds
    // the sets not known to be zero has CTA 0 zero both while the grid waits
    // at a barrier (all CTAs are co-resident: cooperative launch).
    const unsigned long long tk = atomicAdd(p.ticket, 1ull);
    int clean;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(clean) : "l"(p.clean) : "memory");
    if (clean == 0) {
      if (b == 0) {
        for (int i = 0; i < 2 * p.set_ints; i += 4) *reinterpret_cast<int4*>(p.counters + i) = make_int4(0, 0, 0, 0);
        __threadfence();
      }
      const unsigned long long g = gridDim.x, arrived = atomicAdd(p.gbar, 1ull);
      wait_counter64(p.gbar, (arrived / g + 1) * g, abort, limit);   // a timeout sets abort
      __threadfence();
      if (b == 0) atomicExch(p.clean, 1);   // every CTA has read the flag (it reached the barrier)
    }
    int* ctr = p.counters + (size_t)((tk / gridDim.x) & 1) * p.set_ints;
    sm->ctr = ctr;
    first_item = atomicAdd(ctr_of(ctr, p).next_item, 1);   // latency hidden by phase 0
  }
  if (warp == kProducerWarp && lane == 0) {
    // the T x rows (bf16) into the activation area, one bulk copy per row
    mbar_arrive_expect_tx(&sm->xfull, (uint32_t)(T * H * 2));
    for (int t = 0; t < T; ++t)
      bulk_g2s(smem_u32(act + (size_t)t * xs_stride), p.x + (size_t)t * H, (uint32_t)(H * 2), &sm->xfull);
    // The shared expert's gate/up tiles are the first items; while the CTAs
    // route (HBM otherwise idle), each brings its slice of them into L2.
    if (p.has_shared) {
      const size_t tot = (size_t)MT1 * KB1 * kW16Chunk;   // the prepared tiles after the header
      const size_t per = ((tot + gridDim.x - 1) / gridDim.x + 15) & ~(size_t)15;
      const size_t off = per * blockIdx.x;
      if (off < tot) {
        const uint32_t n = (uint32_t)min(per, tot - off);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.w13_shared + sizeof(PrepHeader) + off),
                     "r"(n)
                     : "memory");
      }
    }
  }
  if (warp < T) {
    // registers per lane sized to E (E <= 32, 128, 320, 1024)
    if (E <= 32)
      route_token<1>(p.logits, warp, E, k, nullptr, nullptr, sm->ids, sm->w);
    else if (E <= 128)
      route_token<4>(p.logits, warp, E, k, nullptr, nullptr, sm->ids, sm->w);
    else if (E <= 320)
      route_token<10>(p.logits, warp, E, k, nullptr, nullptr, sm->ids, sm->w);
    else
      route_token<32>(p.logits, warp, E, k, nullptr, nullptr, sm->ids, sm->w);
  } else if (warp >= kBlockWarps && warp < kBlockWarps + T) {
    // x row t -> f16 in place with its row scale, resident for the gate/up items
    const int t = warp - kBlockWarps;
    // (the warp decides as one: the conversion below uses warp shuffles)
    if (__all_sync(0xffffffffu, mbar_wait(&sm->xfull, 0, abort, limit))) {
      uint4* row = reinterpret_cast<uint4*>(act + (size_t)t * xs_stride);
      uint32_t m = 0;
      for (int i = lane; i < H / 8; i += 32) {
        const uint4 v = row[i];
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
          m = max(m, max(finite_mag(wv[q] & 0x7fffu), finite_mag((wv[q] >> 16) & 0x7fffu)));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
      const int sh = row_shift(m);
      const float up = __int_as_float((127 + sh) << 23);
      for (int i = lane; i < H / 8; i += 32) {
        const uint4 v = row[i];
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const __half2 hh = __floats2half2_rn(__uint_as_float(wv[q] << 16) * up,
                                               __uint_as_float(wv[q] & 0xffff0000u) * up);
          o[q] = *reinterpret_cast<const uint32_t*>(&hh);
        }
        row[i] = make_uint4(o[0], o[1], o[2], o[3]);
      }
      if (lane == 0) sm->xmul[t] = __int_as_float((127 - sh) << 23);
    }
  }
  // The permutation needs only the routing: warps 0..7 (which route, and hold
  // the P <= 256 pairs) sort among themselves on a named barrier while warps
  // 8.. still convert x.
  if (warp < kBlockWarps) named_sync(1, kBlockWarps * 32);
  if (tid < P) {
    // rank of pair q in the order (expert, pair index): its grouped row, so
    // the rows of an expert keep the pairs' order (a stable sort, the same
    // permutation as the multi-kernel path's)
    const int q = tid, e = sm->ids[q];
    int r = 0;
    for (int q2 = 0; q2 < P; ++q2) {
      const int e2 = sm->ids[q2];
      r += (e2 < e || (e2 == e && q2 < q)) ? 1 : 0;
    }
    sm->inv[q] = r;
    sm->row_tok[r] = q / k;
    sm->row_w[r] = sm->w[q];
    sm->row_e[r] = e;
  }
  if (warp < kBlockWarps) named_sync(1, kBlockWarps * 32);
  if (warp == 0) {
    // active groups in expert order: a group starts where the expert changes
    int na = 0;
    for (int r0 = 0; r0 < P; r0 += 32) {
      const int r = r0 + lane;
      const bool start = r < P && (r == 0 || sm->row_e[r] != sm->row_e[r - 1]);
      const unsigned starts = __ballot_sync(0xffffffffu, start);
      if (start) {
        const int a = na + __popc(starts & ((1u << lane) - 1u));
        sm->grp_e[a] = sm->row_e[r];
        sm->grp_r0[a] = r;
      }
      na += __popc(starts);
    }
    __syncwarp();
    // top-k picks distinct experts, so a group holds at most one row per
    // token (<= kMaxT); the clamp keeps any input inside the staging buffers
    for (int a = lane; a < na; a += 32) sm->grp_n[a] = min((a + 1 < na ? sm->grp_r0[a + 1] : P) - sm->grp_r0[a], kMaxT);
    __syncwarp();
    if (p.has_shared) {
      if (lane == 0) {
        sm->grp_e[na] = E;
        sm->grp_r0[na] = P;
        sm->grp_n[na] = T;
      }
      for (int t = lane; t < T; t += 32) {
        sm->row_tok[P + t] = t;
        sm->row_w[P + t] = 1.0f;
      }
      ++na;
    }
    if (lane == 0) sm->A = na;
    if (b == 0 && p.topk_ids_out != nullptr)
      for (int q = lane; q < P; q += 32) p.topk_ids_out[q] = sm->ids[q];
  }
  __syncthreads();
  const int A = sm->A;
  const Ctr cc = ctr_of(sm->ctr, p);
  const int N1 = A * MT1, N2 = A * MT2;   // items: gate/up 0..N1-1, then down N1..N1+N2-1
  // Items take the groups in the order shared expert first, then the routed
  // groups by expert: the shared expert's rows are the contributions every
  // token waits for, and taking them first leaves the last items of the
  // kernel (whose signal warps sum the finished tokens) few rows each.
  const int rot = p.has_shared ? A - 1 : 0;

  if (warp == kProducerWarp) {
    // --------------------------------------------------------------- producer
    // Takes the CTA's items one at a time from the grid-wide counter (the
    // first was taken at entry), publishes each in the CTA's queue for the
    // other warps, then streams its stages; the next item is taken while
    // the last stage of the current one streams.
    if (lane == 0) {
      int j = 0, slot = 0, par = 0, item = first_item, c = 0;
      for (;; ++c) {
        // a queue entry is reused once the signal warp has taken over the
        // item kQueue places before it (every warp is past that item)
        if (!decode::spin_ge(&sm->released, c - kQueue + 1, abort, limit)) break;
        const int ph = item < N1 ? 0 : 1, i = ph ? item - N1 : item;
        const int MT = ph == 0 ? MT1 : MT2, KB = ph == 0 ? KB1 : KB2, NST = ph == 0 ? NST1 : NST2;
        const int KBS = ph == 0 ? KBS1 : KBS2;
        const int a = (i / MT + rot) % A, mt = i % MT;
        const int pub = item < N1 + N2 ? item_desc(ph, a, mt) : -1;
        *reinterpret_cast<volatile int*>(&sm->q_item[c % kQueue]) = pub;
        __threadfence_block();
        *reinterpret_cast<volatile int*>(&sm->q_count) = c + 1;
        if (pub < 0) break;
        const int e = sm->grp_e[a];
        const uint8_t* blk = ph == 0 ? (e == E ? p.w13_shared : p.w13 + (size_t)e * p.s13)
                                     : (e == E ? p.w2_shared : p.w2 + (size_t)e * p.s2);
        const uint8_t* data = blk + sizeof(PrepHeader);
        bool ok = true;
        int next = N1 + N2;
        for (int st = 0; st < NST; ++st, ++j) {
          if (!mbar_wait(&sm->empty[slot], par ^ 1, abort, limit)) { ok = false; break; }
          const int kb0 = st * KBS;
          const uint32_t bytes = (uint32_t)(min(KBS, KB - kb0) * kW16Chunk);
          mbar_arrive_expect_tx(&sm->full[slot], bytes);
          bulk_g2s(smem_u32(ring + (size_t)slot * kStageBytes), data + w4a16_chunk(mt, kb0, KB), bytes,
                   &sm->full[slot]);
          if (st == NST - 1) next = atomicAdd(cc.next_item, 1);
          if (++slot == S) {
            slot = 0;
            par ^= 1;
          }
        }
        if (!ok) break;
        item = next;
      }
      // copies still in flight land before the CTA's shared memory is released
      // (a fixed limit: the test hook's short wait limit must not cut this short)
      for (int i = max(0, j - S); i < j; ++i) {
        const long long t0 = clock64();
        while (!mbar_try_wait(&sm->full[i % S], (i / S) & 1) && clock64() - t0 < kDrainLimit) {
        }
      }
      const long long t0 = clock64();   // and the x rows (their wait may have given up)
      while (!mbar_try_wait(&sm->xfull, 0) && clock64() - t0 < kDrainLimit) {
      }
    }
    return;
  }

  if (warp == kHelperWarp) {
    // ------------------------------------- h rows of the down items -> f16
    // (the h slots reuse the x rows' shared memory: wait until no MMA warp
    // reads x any more)
    // The group's h rows (bf16, written by other CTAs and published by the
    // gu_done release) arrive by bulk copy into the slot and are converted
    // there in place, as the x rows are.
    // The CTA takes its items in increasing order, so every item from its
    // first down item on is a down item.
    if (b == (int)gridDim.x - 1) {
      // the other counter set, which the previous launch used, zeroed for the next
      int* other = sm->ctr == p.counters ? p.counters + p.set_ints : p.counters;
      for (int i = 4 * lane; i < p.set_ints; i += 128) *reinterpret_cast<int4*>(other + i) = make_int4(0, 0, 0, 0);
    }
    int m = 0, issued = 0;
    const bool xok = __all_sync(0xffffffffu, mbar_wait(&sm->xfree, 0, abort, limit));
    for (int c = xok ? sm->first_down : 0; xok; ++c, ++m) {
      const int item = queue_get(sm, c, abort, limit, lane);
      if (item < 0) break;   // no more items (-1) or a timeout (-2)
      const int slot = m % kHSlots;
      if (!__all_sync(0xffffffffu, mbar_wait(&sm->hempty[slot], ((m / kHSlots) & 1) ^ 1, abort, limit))) break;
      const int a = desc_a(item);
      if (!wait_counter(cc.gu_done + a, MT1 * (1 + p.extra_arrivals), abort, limit)) break;
      const int r0 = sm->grp_r0[a], n = sm->grp_n[a];
      uint16_t* dst = act + (size_t)slot * kMaxT * hs_stride;
      if (lane == 0) {
        // the other CTAs' generic stores of h, acquired above, before the copy engine reads them
        asm volatile("fence.proxy.async.global;" ::: "memory");
        mbar_arrive_expect_tx(&sm->hland[slot], (uint32_t)(n * I * 2));
        for (int q = 0; q < n; ++q)
          bulk_g2s(smem_u32(dst + (size_t)q * hs_stride), p.h + (size_t)(r0 + q) * I, (uint32_t)(I * 2),
                   &sm->hland[slot]);
      }
      ++issued;
      const unsigned mx = lane < n ? __ldcg(cc.hmax + r0 + lane) : 0u;
      if (!__all_sync(0xffffffffu, mbar_wait(&sm->hland[slot], (m / kHSlots) & 1, abort, limit))) break;
      for (int q = 0; q < n; ++q) {
        const int sh = row_shift(__shfl_sync(0xffffffffu, mx, q));
        const float up = __int_as_float((127 + sh) << 23);
        uint4* row = reinterpret_cast<uint4*>(dst + (size_t)q * hs_stride);
        for (int c = lane; c < I / 8; c += 32) {
          const uint4 v = row[c];
          const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __half2 hh = __floats2half2_rn(__uint_as_float(wv[e] << 16) * up,
                                                 __uint_as_float(wv[e] & 0xffff0000u) * up);
            o[e] = *reinterpret_cast<const uint32_t*>(&hh);
          }
          row[c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if (lane == 0) sm->hmul[slot][q] = __int_as_float((127 - sh) << 23);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->hfull[slot]);
    }
    if (lane == 0 && issued > 0) {
      // the last slot's copies land before the shared memory is released (its
      // wait may have given up); earlier slots were waited for before reuse
      const int lm = issued - 1;
      const long long t0 = clock64();
      while (!mbar_try_wait(&sm->hland[lm % kHSlots], (lm / kHSlots) & 1) && clock64() - t0 < kDrainLimit) {
      }
    }
    if (lane == 0 && *abort) set_status(p.status, MOE_ERR_TIMEOUT);
    return;
  }

  if (warp == kSignalWarp) {
    // ------------------------------------------------------------ signal
    // Takes each finished item over from the MMA warps, so that no MMA warp
    // ever waits on a global fence: gate/up items are counted in
    // gu_done[group] (release, gpu scope; cumulative over the MMA warps'
    // stores of h, which the done barrier ordered before it); down items
    // count their (token, 128-column tile) contributions, and the
    // contribution that completes one sums the token's rows in the fixed
    // order j = 0..k-1, then the shared row, and writes the bf16 output.
    const int need = k + (p.has_shared ? 1 : 0);
    for (int cnt_items = 0;; ++cnt_items) {
      {
        const int item = queue_get(sm, cnt_items, abort, limit, lane);
        if (item < 0) break;
        const int ph = desc_ph(item);
        const int ds = cnt_items % kDoneSlots;
        if (!__all_sync(0xffffffffu, mbar_wait(&sm->done[ds], (cnt_items / kDoneSlots) & 1, abort, limit))) break;
        const int a = desc_a(item), mt = desc_mt(item);
        if (ph == 0) {
          if (lane == 0) release_add(cc.gu_done + a, 1);
        } else {
          const int r0 = sm->grp_r0[a], n = sm->grp_n[a];
          // count the item's rows: one per (token, 128-column tile). The fence
          // publishes the MMA warps' y stores (ordered before by the done
          // barrier) ahead of the counts; the count that completes a token's
          // tile (k routed rows + the shared row) is followed by a fence
          // before the rows are read back.
          __threadfence();
          int last = 0, tok = 0;
          if (lane < n) {
            tok = sm->row_tok[r0 + lane];
            last = atomicAdd(cc.cmb_cnt + (size_t)tok * MT2 + mt, 1) == need - 1;
          }
          unsigned todo = __ballot_sync(0xffffffffu, last);
          if (todo) {
            __threadfence();
            while (todo) {  // two finished (token, tile) at a time, 16 lanes of 8 columns each
              const int s0 = __ffs(todo) - 1;
              todo &= todo - 1;
              const int s1 = todo ? __ffs(todo) - 1 : -1;
              if (s1 >= 0) todo &= todo - 1;
              const int src = lane < 16 ? s0 : s1;
              const int t = __shfl_sync(0xffffffffu, tok, src < 0 ? 0 : src);
              if (src >= 0) combine_cols8(p, sm->inv, t, k, H, mt * kTile + (lane & 15) * 8);
            }
          }
        }
        __syncwarp();
        if (lane == 0) {
          __threadfence_block();
          *reinterpret_cast<volatile int*>(&sm->released) = cnt_items + 1;
        }
      }
    }
    if (lane == 0 && *abort) set_status(p.status, MOE_ERR_TIMEOUT);
    return;
  }

  // -------------------------------------------------------------- MMA warps
  const int blk = warp % kBlockWarps, half = warp / kBlockWarps;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int lrow = lane & 7, lq = lane >> 3;
  int slot = 0, par = 0, m = 0;   // ring slot and phase parity of the next stage
  bool ok = true;
  bool x_released = false;
  // x (and the slot of the first down item's h rows, which reuses its shared
  // memory) is released at the CTA's first down item, or earlier: after the
  // stage loop of a gate/up item whose successor in the queue is already
  // known to be a down item (or the end)
  auto release_x = [&](int c) {
    if (x_released) return;
    if (warp == 0 && lane == 0) sm->first_down = c;
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm->xfree);
    x_released = true;
  };
  for (int cnt_items = 0; ok; ++cnt_items) {
    {
      const int item = queue_get(sm, cnt_items, abort, limit, lane);
      if (item == -2) { ok = false; break; }
      if (item < 0 || desc_ph(item) == 1) release_x(cnt_items);
      if (item < 0) break;
      const int ph = desc_ph(item);
      const int KB = ph == 0 ? KB1 : KB2, NST = ph == 0 ? NST1 : NST2;
      const int KBS = ph == 0 ? KBS1 : KBS2;
      const int a = desc_a(item), mt = desc_mt(item);
      const int e = sm->grp_e[a], r0 = sm->grp_r0[a], n = sm->grp_n[a];
      const int hslot = m % kHSlots;
      // ldmatrix row of this lane: the group's row lrow (rows past the group
      // repeat row 0; their columns are computed and dropped)
      const int rsel = lrow < n ? lrow : 0;
      uint32_t xa0;
      if (ph == 0) {
        xa0 = smem_u32(act + (size_t)sm->row_tok[r0 + rsel] * xs_stride + 8 * lq);
      } else {
        if (!__all_sync(0xffffffffu, mbar_wait(&sm->hfull[hslot], (m / kHSlots) & 1, abort, limit))) {
          ok = false;
          break;
        }
        xa0 = smem_u32(act + (size_t)hslot * kMaxT * hs_stride + (size_t)rsel * hs_stride + 8 * lq);
      }
      // the epilogue's alpha, loaded now so that it arrives during the stage loop
      const uint8_t* wb = ph == 0 ? (e == E ? p.w13_shared : p.w13 + (size_t)e * p.s13)
                                  : (e == E ? p.w2_shared : p.w2 + (size_t)e * p.s2);
      const PrepHeader* hdr = reinterpret_cast<const PrepHeader*>(wb);
      const float al0 = __ldg(&hdr->alpha[0]), al1 = __ldg(&hdr->alpha[1]);
      float acc4[4][4];
#pragma unroll
      for (int s = 0; s < 4; ++s) acc4[s][0] = acc4[s][1] = acc4[s][2] = acc4[s][3] = 0.f;
      // both halves read every stage: half h sums its K blocks h, h + 2, ...
      // (j counts every stage of this CTA)
      for (int st = 0; st < NST; ++st) {
        if (!__all_sync(0xffffffffu, mbar_wait(&sm->full[slot], par, abort, limit))) { ok = false; break; }
        const int kb0 = st * KBS;
        decode::mma_stage(ring + (size_t)slot * kStageBytes, min(KBS, KB - kb0), half, kHalves, blk, lane,
                          xa0 + (uint32_t)(kb0 * 64) * 2, acc4);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->empty[slot]);
        if (++slot == S) {
          slot = 0;
          par ^= 1;
        }
      }
      if (!ok) break;
      float hm[2] = {1.0f, 1.0f};   // row multipliers of this lane's two token columns
      if (ph == 0) {
        const int nx = queue_peek(sm, cnt_items + 1, lane);   // -3: not published yet
        if (nx == -1 || (nx >= 0 && desc_ph(nx) == 1)) release_x(cnt_items + 1);
      } else {  // the staged h rows (and their multipliers) are no longer read
#pragma unroll
        for (int q = 0; q < 2; ++q) hm[q] = sm->hmul[hslot][min(2 * t4 + q, kMaxT - 1)];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm->hempty[hslot]);
        ++m;
      }
      float acc[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[q] = (acc4[0][q] + acc4[1][q]) + (acc4[2][q] + acc4[3][q]);
      // the half that comes second sums and runs the epilogue
      bool second = false;
      if (!decode::half_join(&sm->join, blk, lane, cnt_items, acc, second, abort, limit)) { ok = false; break; }
      if (!second) continue;

      const int mb = mt * kBlockWarps + blk;
      if (ph == 0) {
        // SwiGLU: lane pair (row g8 gate, row g8 + 8 up) of feature 8 * mb + g8
        const int f = 8 * mb + g8;
        uint32_t hb2[2] = {0u, 0u};
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int c = 2 * t4 + q;
          if (c < n) {
            const float rm = sm->xmul[sm->row_tok[r0 + c]];
            const float hv = silu(acc[q] * rm * al0) * (acc[2 + q] * rm * al1);
            const uint16_t bits = float_to_bf16_bits(hv);
            p.h[(size_t)(r0 + c) * I + f] = bits;
            hb2[q] = bits & 0x7fffu;
          }
        }
        // per-row max |h| over this warp's 8 features, then one atomic per row
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t v = finite_mag(hb2[q]);
          v = max(v, __shfl_xor_sync(0xffffffffu, v, 4));
          v = max(v, __shfl_xor_sync(0xffffffffu, v, 8));
          v = max(v, __shfl_xor_sync(0xffffffffu, v, 16));
          const int c = 2 * t4 + q;
          if (g8 == 0 && c < n) atomicMax(cc.hmax + r0 + c, v);
        }
      } else {
        // y = acc * 2^-s * alpha * routing weight
        const int col = mt * kTile + 16 * blk;   // this warp's 16 output columns
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int c = 2 * t4 + q;
          if (c < n) {
            const int r = r0 + c;
            // the multi-kernel path's order of operations, so the two paths agree bit for bit
            const float rw = sm->row_w[r];
            const float v0 = acc[q] * hm[q] * al0 * rw, v1 = acc[2 + q] * hm[q] * al0 * rw;
            if (e == E) {  // shared expert: kept fp32 for the combine
              p.y_shared[(size_t)(r - P) * H + col + g8] = v0;
              p.y_shared[(size_t)(r - P) * H + col + g8 + 8] = v1;
            } else {
              p.y[(size_t)r * H + col + g8] = float_to_bf16_bits(v0);
              p.y[(size_t)r * H + col + g8 + 8] = float_to_bf16_bits(v1);
            }
          }
        }
      }
      // hand the item to the signal warp (its slot must be free: the item
      // kDoneSlots before it taken over)
      const int ds = cnt_items % kDoneSlots;
      int freed = 1;
      if (lane == 0) freed = decode::spin_ge(&sm->released, cnt_items - kDoneSlots + 1, abort, limit);
      if (!__shfl_sync(0xffffffffu, freed, 0)) { ok = false; break; }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm->done[ds]);
    }
  }
  if (lane == 0 && *abort) set_status(p.status, MOE_ERR_TIMEOUT);
}

}  // namespace

static size_t fused_smem_bytes(int T, int H, int I, int E, int slots, int stage_kb) {
  const size_t act = std::max((size_t)T * (H + 8), (size_t)kHSlots * kMaxT * (I + 8)) * 2;
  return (size_t)slots * stage_kb * kW16Chunk + act + sizeof(Smem);
}

// Ring slots for a stage size: as many as fit, at most 144 KB of ring (four
// 36 KB stages, eight 18 KB ones), never fewer than 4. Every MMA warp reads
// every stage in order, so a slot's previous stage was consumed by each
// waiter before it waits on the slot again.
static int fused_slots(int T, int H, int I, int E, int stage_kb) {
  int slots = std::min(kMaxSlots, (int)((144 * 1024) / ((size_t)stage_kb * kW16Chunk)));
  while (slots > 4 && fused_smem_bytes(T, H, I, E, slots, stage_kb) > 227 * 1024) --slots;
  return slots;
}

// Ring slot size in K blocks: the larger stage of the two phases.
static int fused_stage_kb(int H, int I) {
  return std::max(w16_stage_kb(H / 64, decode_stage_kb()), w16_stage_kb(I / 64, decode_stage_kb()));
}

bool decode_fused_supported(int T, int H, int I, int E, int k) {
  if (T < 1 || T > kMaxT || k > kMaxK || E > 1024) return false;
  if (H % kTile || (2 * I) % kTile || I % 64) return false;
  const int skb = fused_stage_kb(H, I);
  return fused_smem_bytes(T, H, I, E, fused_slots(T, H, I, E, skb), skb) <= 227 * 1024;
}

moe_status launch_decode_fused(const DecodeFusedPlan& q, cudaStream_t s) {
  if (!decode_fused_supported(q.T, q.H, q.I, q.E, q.k)) return MOE_ERR_UNSUPPORTED;
  Args a;
  a.logits = q.logits;
  a.x = q.x;
  a.w13 = q.w13;
  a.s13 = q.s13;
  a.w13_shared = q.w13_shared;
  a.w2 = q.w2;
  a.s2 = q.s2;
  a.w2_shared = q.w2_shared;
  a.T = q.T;
  a.H = q.H;
  a.I = q.I;
  a.E = q.E;
  a.k = q.k;
  a.has_shared = q.w13_shared != nullptr ? 1 : 0;
  a.out = q.out;
  a.topk_ids_out = q.topk_ids_out;
  a.h = q.h;
  a.y = q.y;
  a.y_shared = q.y_shared;
  a.counters = q.counters;
  a.set_ints = q.set_ints;
  a.counter_ints = q.counter_ints;
  a.clean = q.clean;
  a.ticket = q.ticket;
  a.gbar = q.gbar;
  a.status = q.status;
  a.wait_limit = q.wait_limit;
  a.extra_arrivals = q.extra_arrivals;
  const int skb = fused_stage_kb(q.H, q.I);
  const int slots = fused_slots(q.T, q.H, q.I, q.E, skb);
  if (fused_smem_bytes(q.T, q.H, q.I, q.E, slots, skb) > 227 * 1024) return MOE_ERR_UNSUPPORTED;
  a.slots = slots;
  a.stage_kb = skb;
  a.kmax = decode_stage_kb();
  const size_t smem = fused_smem_bytes(q.T, q.H, q.I, q.E, slots, skb);
  int dev = 0, sms = 0;
  moe_status st = cuda_ok(cudaGetDevice(&dev));
  if (st != MOE_OK) return st;
  st = cuda_ok(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  if (st != MOE_OK) return st;
  st = cuda_ok(cudaFuncSetAttribute(decode_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  if (st != MOE_OK) return st;
  // every CTA must be resident (they wait on one another): one per SM, launched cooperatively
  int per_sm = 0;
  st = cuda_ok(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_fused_kernel, kThreads, smem));
  if (st != MOE_OK) return st;
  if (per_sm < 1) return MOE_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  st = cuda_ok(cudaLaunchKernelEx(&cfg, decode_fused_kernel, a));
  if (st != MOE_OK) return st;
  count_launches(1);
  return MOE_OK;
}

}  // namespace moe
