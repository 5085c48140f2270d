// Grouping token rows by expert: count, exclusive scan, stable scatter.
//
// AFN-019 "Hide SSD misses before the router knows they exist", section "Why
// overlap alone cannot defeat the byte roofline": grouping token rows by
// expert is one of the byte owners.  Rows of one expert are kept in ascending
// flat route order r = t*k + j, which makes the grouping deterministic and
// comparable bit for bit.
//
// One CTA of up to 32 route-owning warps.  Warp w owns a contiguous run of routes.  Pass 1: each
// warp counts its routes per expert with __match_any_sync (one shared-memory
// add per distinct expert per 32 routes, no atomics).  Pass 2: per expert, an
// exclusive prefix over the 32 warps, then one exclusive scan over experts
// gives the segment offsets.  Pass 3: each warp replays its run and places
// every route at offsets[e] + (routes of e in earlier warps) + (earlier routes
// of e in this warp), which is the stable order.  Integer work only, a few
// microseconds even at 40,960 routes, so one CTA is enough.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

constexpr int kWarps = 32;

__global__ void __launch_bounds__(kWarps * 32, 1)
    permute_kernel(const int32_t* __restrict__ ids, int R, int E, int32_t* __restrict__ counts,
                   int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                   int32_t* status) {
  extern __shared__ int32_t sh[];
  // Only as many warps own routes as there are 32-route steps (a decode
  // block of 160 routes uses 5), which keeps the per-warp tables small.
  const int W = min(kWarps, max(1, (R + 31) / 32));
  int32_t* hist = sh;          // [W][E]
  int32_t* base = sh + W * E;  // [E]
  __shared__ int bad;
  __shared__ int warp_tot[kWarps];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  for (int i = tid; i < W * E; i += blockDim.x) hist[i] = 0;
  if (tid == 0) bad = 0;
  pdl_wait();
  pdl_trigger();
  __syncthreads();

  const int per = (R + W - 1) / W;
  const int r0 = (warp < W) ? min(R, warp * per) : R;
  const int r1 = (warp < W) ? min(R, r0 + per) : R;
  int32_t* my_hist = hist + min(warp, W - 1) * E;

  // pass 1: per-warp histogram
  for (int b = r0; b < r1; b += 32) {
    const int r = b + lane;
    const bool act = r < r1;
    int e = act ? ids[r] : -1;
    if (act && (e < 0 || e >= E)) {
      bad = 1;
      e = -1;
    }
    // inactive or invalid lanes get a key no valid route can share
    const int key = (act && e >= 0) ? e : -(lane + 2);
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    if (key >= 0 && lane == __ffs(peers) - 1) my_hist[key] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  if (bad) {
    if (tid == 0) set_status(status, MOE_DEV_BAD_EXPERT);
    return;
  }

  // pass 2: per-expert prefix over warps, then an exclusive scan over experts
  for (int e = tid; e < E; e += blockDim.x) {
    int s = 0;
    for (int w = 0; w < W; ++w) {
      const int c = hist[w * E + e];
      hist[w * E + e] = s;
      s += c;
    }
    base[e] = s;
  }
  __syncthreads();
  // E <= 1024 = blockDim.x: one expert per thread
  const int c = (tid < E) ? base[tid] : 0;
  int incl = c;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int wt = warp_tot[lane];
    int wi = wt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, d);
      if (lane >= d) wi += y;
    }
    warp_tot[lane] = wi - wt;  // exclusive prefix of warp totals
  }
  __syncthreads();
  const int excl = warp_tot[warp] + incl - c;
  if (tid < E) {
    counts[tid] = c;
    offsets[tid] = excl;
    base[tid] = excl;
  }
  if (tid == 0) offsets[E] = R;
  __syncthreads();

  // pass 3: stable scatter
  for (int b = r0; b < r1; b += 32) {
    const int r = b + lane;
    const bool act = r < r1;
    const int key = act ? ids[r] : -(lane + 2);
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    int slot = 0;
    if (act) {
      const unsigned lower = peers & ((1u << lane) - 1u);
      slot = base[key] + my_hist[key] + __popc(lower);
      perm[slot] = r;
      inv[r] = slot;
    }
    __syncwarp();
    if (act && lane == __ffs(peers) - 1) my_hist[key] += __popc(peers);
    __syncwarp();
  }
}

__global__ void gather_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm, int R, int k,
                                   int T, int H, uint16_t* __restrict__ xp) {
  pdl_wait();
  pdl_trigger();
  const int vpr = H / 8;
  const size_t n = static_cast<size_t>(R) * vpr;
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int s = static_cast<int>(idx / vpr);
    const int c = static_cast<int>(idx - static_cast<size_t>(s) * vpr);
    const int r = perm[s];
    if (r < 0 || r >= R) continue;  // routing rejected upstream: leave the row alone
    const int t = r / k;
    if (t >= T) continue;
    reinterpret_cast<uint4*>(xp)[idx] = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H)[c];
  }
}

}  // namespace

cudaError_t launch_permute(const int32_t* ids, int R, int k, int E, int32_t* counts, int32_t* offsets, int32_t* perm,
                           int32_t* inv, int32_t* st_word, cudaStream_t st) {
  (void)k;
  const int W = std::min(kWarps, std::max(1, (R + 31) / 32));
  const size_t smem = static_cast<size_t>(W + 1) * E * sizeof(int32_t);
  cudaError_t e = ensure_smem(permute_kernel, static_cast<int>((kWarps + 1) * kMaxE * sizeof(int32_t)));
  if (e != cudaSuccess) return e;
  return launch_pdl(permute_kernel, dim3(1), dim3(kWarps * 32), smem, st, ids, R, E, counts, offsets, perm, inv,
                    st_word);
}

cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* perm, int R, int k, int T, int H, uint16_t* x_perm,
                               cudaStream_t st) {
  const size_t n = static_cast<size_t>(R) * (H / 8);
  const int threads = 256;
  size_t blocks = (n + threads - 1) / threads;
  const size_t cap = static_cast<size_t>(sm_count() > 0 ? sm_count() : 148) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks == 0) blocks = 1;
  return launch_pdl(gather_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, st, x, perm, R, k, T,
                    H, x_perm);
}

}  // namespace moe
