// Grouping token rows by expert: count, exclusive scan, stable scatter.
//
// AFN-019 "Hide SSD misses before the router knows they exist", section "Why
// overlap alone cannot defeat the byte roofline": grouping token rows by
// expert is one of the byte owners.  Rows of one expert are kept in ascending
// flat route order r = t*k + j, which makes the grouping deterministic and
// comparable bit for bit.
//
// One CTA of up to 32 route-owning warps.  Warp w owns a contiguous run of
// routes.  Pass 1: each warp counts its routes per expert in its own table
// (shared-memory atomic adds: order does not matter for a count).  Pass 2:
// per expert, an exclusive prefix over the warps, then one exclusive scan
// over experts gives the segment offsets.  Pass 3: each warp replays its run
// 32 routes at a time and places every route at offsets[e] + (routes of e in
// earlier warps) + (earlier routes of e in this warp), which is the stable
// order; within a 32-route batch the lanes holding the same expert find one
// another through a per-warp table of lane masks (each lane ORs its bit into
// the word of its expert, reads the word back, and the lowest lane clears
// it), which costs a few instructions whatever the number of distinct
// experts in the batch.  Each warp loads kUnroll batches of its run before
// it processes them, so a pass waits for global-load latency once per
// kUnroll batches.  Integer work only.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

constexpr int kWarps = 32;
constexpr int kUnroll = 8;                // 32-route batches loaded ahead per warp
constexpr int kPermuteSmem = 200 * 1024;  // per-warp count and mask tables

// Route-owning warps: one per 32 routes up to 32, fewer when E is so large
// that two [W][E] tables would not fit in shared memory.
int permute_warps(int R, int E) {
  const int w_rows = std::max(1, (R + 31) / 32);
  const int w_smem = std::max(1, (kPermuteSmem / (4 * E) - 1) / 2);
  return std::min(kWarps, std::min(w_rows, w_smem));
}

__global__ void __launch_bounds__(kWarps * 32, 1)
    permute_kernel(const int32_t* __restrict__ ids, int R, int E, int W, int32_t* __restrict__ counts,
                   int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                   int32_t* status) {
  extern __shared__ int32_t sh[];
  int32_t* hist = sh;                                            // [W][E]
  int32_t* base = sh + W * E;                                    // [E]
  unsigned* lmask = reinterpret_cast<unsigned*>(base + E);       // [W][E]
  __shared__ int bad;
  __shared__ int warp_tot[kWarps];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  for (int i = tid; i < W * E; i += blockDim.x) {
    hist[i] = 0;
    lmask[i] = 0u;
  }
  if (tid == 0) bad = 0;
  pdl_wait();
  pdl_trigger();
  __syncthreads();

  const int per = (R + W - 1) / W;
  const int r0 = (warp < W) ? min(R, warp * per) : R;
  const int r1 = (warp < W) ? min(R, r0 + per) : R;
  int32_t* my_hist = hist + min(warp, W - 1) * E;
  unsigned* my_mask = lmask + min(warp, W - 1) * E;

  // pass 1: per-warp histogram
  for (int b = r0; b < r1; b += 32 * kUnroll) {
    int ev[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int r = b + u * 32 + lane;
      ev[u] = r < r1 ? ids[r] : 0;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (b + u * 32 + lane < r1) {
        const int e = ev[u];
        if (e < 0 || e >= E) {
          bad = 1;
        } else {
          atomicAdd(&my_hist[e], 1);
        }
      }
    }
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

  // pass 3: stable scatter (every ID is valid here)
  for (int b = r0; b < r1; b += 32 * kUnroll) {
    int ev[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int r = b + u * 32 + lane;
      ev[u] = r < r1 ? ids[r] : 0;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int r = b + u * 32 + lane;
      const bool act = r < r1;
      const int key = ev[u];
      if (act) atomicOr(&my_mask[key], 1u << lane);
      __syncwarp();
      // lanes of this batch routed to the same expert as this lane
      const unsigned peers = act ? my_mask[key] : 0u;
      if (act) {
        const unsigned lower = peers & ((1u << lane) - 1u);
        const int slot = base[key] + my_hist[key] + __popc(lower);
        perm[slot] = r;
        inv[r] = slot;
      }
      __syncwarp();
      if (act && lane == __ffs(peers) - 1) {
        my_hist[key] += __popc(peers);
        my_mask[key] = 0u;
      }
      __syncwarp();
    }
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
  const int W = permute_warps(R, E);
  const size_t smem = static_cast<size_t>(2 * W + 1) * E * sizeof(int32_t);
  cudaError_t e = ensure_smem(permute_kernel, kPermuteSmem + 4 * kMaxE);
  if (e != cudaSuccess) return e;
  return launch_pdl(permute_kernel, dim3(1), dim3(kWarps * 32), smem, st, ids, R, E, W, counts, offsets, perm, inv,
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
