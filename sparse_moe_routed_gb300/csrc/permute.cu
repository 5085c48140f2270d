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

// Groups routes [rb, re) of ids in one CTA of up to kWarps warps.  ext ==
// nullptr: the CTA owns all R routes (rb = 0, re = R) and writes counts and
// offsets.  ext != nullptr: a chunk of a larger grouping; ext[e] is where
// this chunk's routes of expert e start (the counts of earlier chunks added
// to offsets[e]), and counts / offsets are left to the chunk scan.
__device__ __forceinline__ void group_range(const int32_t* __restrict__ ids, int rb, int re, int R, int E, int W,
                                            int32_t* sh, const int32_t* ext, int32_t* __restrict__ counts,
                                            int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                                            int32_t* __restrict__ inv, int32_t* status) {
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
  __syncthreads();

  const int n = re - rb;
  const int per = (n + W - 1) / W;
  const int r0 = (warp < W) ? min(re, rb + warp * per) : re;
  const int r1 = (warp < W) ? min(re, r0 + per) : re;
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
  // (or, for a chunk, the chunk's given starts)
  for (int e = tid; e < E; e += blockDim.x) {
    int s = 0;
    for (int w = 0; w < W; ++w) {
      const int c = hist[w * E + e];
      hist[w * E + e] = s;
      s += c;
    }
    base[e] = ext != nullptr ? ext[e] : s;
  }
  __syncthreads();
  if (ext == nullptr) {
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
  }

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

__global__ void __launch_bounds__(kWarps * 32, 1)
    permute_kernel(const int32_t* __restrict__ ids, int R, int E, int W, int32_t* __restrict__ counts,
                   int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                   int32_t* status) {
  extern __shared__ int32_t sh[];
  pdl_wait();
  pdl_trigger();
  group_range(ids, 0, R, R, E, W, sh, nullptr, counts, offsets, perm, inv, status);
}

// Large route counts: chunks of kChunk routes on C CTAs.  Workspace: [C][E]
// int32 (each chunk's counts, then where its routes of each expert start),
// [C] bad-ID flags, then one word that tells the scatter to write nothing.
constexpr int kChunk = 2048;

__global__ void __launch_bounds__(1024) chunk_count_kernel(const int32_t* __restrict__ ids, int R, int E,
                                                           int32_t* __restrict__ ws) {
  __shared__ int32_t hist[kMaxE];
  __shared__ int bad;
  const int c = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  if (threadIdx.x == 0) bad = 0;
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  const int rb = c * kChunk, re = min(R, rb + kChunk);
  for (int r = rb + threadIdx.x; r < re; r += blockDim.x) {
    const int e = ids[r];
    if (e < 0 || e >= E) {
      bad = 1;
    } else {
      atomicAdd(&hist[e], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) ws[static_cast<size_t>(c) * E + e] = hist[e];
  if (threadIdx.x == 0) ws[static_cast<size_t>(gridDim.x) * E + c] = bad;
}

// One CTA: counts, offsets (exclusive scan over experts) and, per chunk and
// expert, where the chunk's routes start; a bad ID anywhere writes nothing.
__global__ void __launch_bounds__(1024) chunk_scan_kernel(int R, int E, int C, int32_t* __restrict__ ws,
                                                          int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                          int32_t* status) {
  __shared__ int warp_tot[32];
  __shared__ int anybad;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) anybad = 0;
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  for (int c = tid; c < C; c += blockDim.x)
    if (ws[static_cast<size_t>(C) * E + c]) anybad = 1;
  __syncthreads();
  if (anybad) {
    if (tid == 0) {
      set_status(status, MOE_DEV_BAD_EXPERT);
      ws[static_cast<size_t>(C) * E + C] = 1;
    }
    return;
  }
  int tot = 0;
  if (tid < E)
    for (int c = 0; c < C; ++c) tot += ws[static_cast<size_t>(c) * E + tid];
  int incl = tot;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int wt = warp_tot[lane];
    int wi = wt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, d);
      if (lane >= d) wi += y;
    }
    warp_tot[lane] = wi - wt;
  }
  __syncthreads();
  if (tid < E) {
    int run = warp_tot[warp] + incl - tot;  // offsets[e]
    counts[tid] = tot;
    offsets[tid] = run;
    for (int c = 0; c < C; ++c) {
      const size_t i = static_cast<size_t>(c) * E + tid;
      const int v = ws[i];
      ws[i] = run;
      run += v;
    }
  }
  if (tid == 0) {
    offsets[E] = R;
    ws[static_cast<size_t>(C) * E + C] = 0;
  }
}

__global__ void __launch_bounds__(kWarps * 32, 1)
    chunk_scatter_kernel(const int32_t* __restrict__ ids, int R, int E, int W, const int32_t* __restrict__ ws,
                         int32_t* __restrict__ perm, int32_t* __restrict__ inv, int32_t* status) {
  extern __shared__ int32_t sh[];
  pdl_wait();
  pdl_trigger();
  const int C = gridDim.x;
  if (ws[static_cast<size_t>(C) * E + C]) return;  // a bad ID: nothing is written
  const int c = blockIdx.x;
  group_range(ids, c * kChunk, min(R, (c + 1) * kChunk), R, E, W, sh, ws + static_cast<size_t>(c) * E, nullptr,
              nullptr, perm, inv, status);
}

// Rows of x into slot order, one warp per token: the warp reads the token's
// k slots (inv), then moves the row in pieces of 32 x kGatherVec 16-byte
// vectors, each piece loaded once and stored to all k slots.  x is read once
// in token order, and every x_perm row is written once.  After a grouping
// that met a bad expert ID inv was not written, so nothing is gathered.
constexpr int kGatherThreads = 256;
constexpr int kGatherVec = 8;  // 16-byte vectors in flight per lane

__global__ void __launch_bounds__(kGatherThreads)
    gather_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ inv, int R, int k, int T, int H,
                       uint16_t* __restrict__ xp, const int32_t* st_word) {
  pdl_wait();
  pdl_trigger();
  if (*reinterpret_cast<const volatile int32_t*>(st_word) & MOE_DEV_BAD_EXPERT) return;
  const int lane = threadIdx.x & 31;
  const int wpb = kGatherThreads / 32;
  const int stride = gridDim.x * wpb;
  const int vpr = H / 8;  // 16-byte vectors per row
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += stride) {
    // lane j < k holds the slot of route (t, j); out of range: left alone
    int my = lane < k ? inv[static_cast<size_t>(t) * k + lane] : -1;
    if (my < 0 || my >= R) my = -1;
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
    for (int c0 = 0; c0 < vpr; c0 += 32 * kGatherVec) {
      uint4 v[kGatherVec];
#pragma unroll
      for (int u = 0; u < kGatherVec; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < vpr) v[u] = src[c];
      }
      for (int j = 0; j < k; ++j) {
        const int s = __shfl_sync(0xffffffffu, my, j);
        if (s < 0) continue;
        uint4* dst = reinterpret_cast<uint4*>(xp + static_cast<size_t>(s) * H);
#pragma unroll
        for (int u = 0; u < kGatherVec; ++u) {
          const int c = c0 + u * 32 + lane;
          if (c < vpr) dst[c] = v[u];
        }
      }
    }
  }
}

// The same rows for small launches (a decode block has too few tokens to
// keep a warp per token busy): one thread per 16-byte vector of x_perm, the
// slot's route read from perm.
__global__ void gather_rows_by_slot_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm, int R,
                                           int k, int T, int H, uint16_t* __restrict__ xp, const int32_t* st_word) {
  pdl_wait();
  pdl_trigger();
  if (*reinterpret_cast<const volatile int32_t*>(st_word) & MOE_DEV_BAD_EXPERT) return;
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

// Below this many tokens the gather runs one thread per vector of x_perm.
constexpr int kGatherPerTokenMinT = 1024;

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

size_t permute_chunked_ws_bytes(int R, int E) {
  const size_t C = (static_cast<size_t>(R) + kChunk - 1) / kChunk;
  return ((C * E + C + 1) * sizeof(int32_t) + 255) / 256 * 256;
}

cudaError_t launch_permute_chunked(const int32_t* ids, int R, int E, int32_t* counts, int32_t* offsets, int32_t* perm,
                                   int32_t* inv, int32_t* ws, int32_t* st_word, cudaStream_t st) {
  const int C = (R + kChunk - 1) / kChunk;
  cudaError_t e = launch_pdl(chunk_count_kernel, dim3(C), dim3(1024), 0, st, ids, R, E, ws);
  if (e != cudaSuccess) return e;
  e = launch_pdl(chunk_scan_kernel, dim3(1), dim3(1024), 0, st, R, E, C, ws, counts, offsets, st_word);
  if (e != cudaSuccess) return e;
  const int W = permute_warps(kChunk, E);
  const size_t smem = static_cast<size_t>(2 * W + 1) * E * sizeof(int32_t);
  e = ensure_smem(chunk_scatter_kernel, kPermuteSmem + 4 * kMaxE);
  if (e != cudaSuccess) return e;
  return launch_pdl(chunk_scatter_kernel, dim3(C), dim3(kWarps * 32), smem, st, ids, R, E, W, ws, perm, inv,
                    st_word);
}

cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* perm, const int32_t* inv, int R, int k, int T, int H,
                               uint16_t* x_perm, const int32_t* st_word, cudaStream_t st) {
  if (T < kGatherPerTokenMinT) {
    const size_t n = static_cast<size_t>(R) * (H / 8);
    const int threads = 256;
    size_t blocks = (n + threads - 1) / threads;
    const size_t cap = static_cast<size_t>(sm_count() > 0 ? sm_count() : 148) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    return launch_pdl(gather_rows_by_slot_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, st, x, perm,
                      R, k, T, H, x_perm, st_word);
  }
  if (k > 32) return cudaErrorInvalidValue;  // one lane per route of a token
  const int wpb = kGatherThreads / 32;
  size_t blocks = (static_cast<size_t>(T) + wpb - 1) / wpb;
  const size_t cap = static_cast<size_t>(sm_count() > 0 ? sm_count() : 148) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks == 0) blocks = 1;
  return launch_pdl(gather_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kGatherThreads), 0, st, x, inv,
                    R, k, T, H, x_perm, st_word);
}

}  // namespace moe
