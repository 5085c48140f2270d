// Expert records resident in host memory, served through an HBM slot cache.
//
// AFN-019 "Hide SSD misses before the router knows they exist", sections
// "Why overlap alone cannot defeat the byte roofline" and "Hypothesis H4":
// the routed records a token needs are fetched from a slower tier and the
// bytes fetched are the first-order cost.  On GB300 the slower tier is the
// Grace LPDDR5X behind NVLink-C2C: the tile-packed records of every expert
// live in pinned host memory, which the GPU reads directly; S slots of HBM
// hold recently used experts.
//
// cache_plan_kernel (one CTA, one thread per expert and per slot):
//   routed experts already resident are hits; the others are misses, ordered
//   by expert ID.  Slots whose expert is routed in this call are pinned; the
//   others are eligible victims, taken in the policy's order and given to the
//   misses in turn:
//     FIFO  rotation order from the hand (the oldest fill first);
//     LRU   empty slots first, then least recent use (the control);
//     SCORE empty slots first, then lowest score(record) (AFN-019, section
//           "Two storage workloads, not one": P(use before eviction) x
//           expected exposed latency avoided / resident bytes).  Records are
//           whole and of one size, so the score orders as P(use), estimated
//           per expert by an exponentially weighted use rate
//           f <- decay * f + [routed] (one fused multiply-add in fp32);
//   ties go to the lower slot.  The plan is written as (miss_list,
//   miss_slot, counters of this call, running totals) and the slot table is
//   updated in place; if the misses do not fit in the slots not pinned by
//   this call's routes, MOE_DEV_CACHE_FULL is set and the slots stay as they
//   were (the call counter and the use rates still advance).
// cache_fetch_kernel (grid-stride, 16-byte loads from host memory, eight in
//   flight per thread): copies each missing expert's gate/up and down records
//   into its slot.
#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

constexpr int kPlanThreads = 1024;

__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  __syncthreads();  // warp_sums free for reuse
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += warp_sums[w];
  return before + incl - v;
}

__global__ void __launch_bounds__(kPlanThreads) cache_plan_kernel(const int32_t* __restrict__ counts, int E,
                                                                  int32_t* slot_of, int32_t* expert_of, int S,
                                                                  int32_t* hand, int policy, float decay,
                                                                  float* score, int32_t* last_use,
                                                                  int32_t* __restrict__ miss_list,
                                                                  int32_t* __restrict__ miss_slot,
                                                                  int32_t* __restrict__ stats, int32_t* status) {
  __shared__ int warp_sums[32];
  __shared__ int s_missexp[kMaxE];
  __shared__ unsigned long long s_key[kPlanThreads];
  __shared__ int s_nmiss;
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x;
  const int h0 = ((hand[0] % S) + S) % S;
  const int step = hand[1];
  // experts: hit / miss; use rates
  bool miss = false, hit = false;
  if (tid < E) {
    const bool routed = counts[tid] > 0;
    hit = routed && slot_of[tid] >= 0;
    miss = routed && !hit;
    if (policy == MOE_CACHE_SCORE) score[tid] = __fmaf_rn(decay, score[tid], routed ? 1.0f : 0.0f);
  }
  const int midx = block_exclusive_scan(miss ? 1 : 0, warp_sums);
  if (miss) s_missexp[midx] = tid;
  if (tid == E - 1) s_nmiss = midx + (miss ? 1 : 0);
  const int nhit = __syncthreads_count(hit);  // also publishes the use rates
  // eligible slots and their order keys: (primary << 32) | slot
  bool elig = false;
  unsigned long long key = ~0ull;
  if (tid < S) {
    const int ex = expert_of[tid];
    const bool occupied = ex >= 0 && ex < E;
    elig = !(occupied && counts[ex] > 0);
    if (elig) {
      uint32_t primary;
      if (policy == MOE_CACHE_FIFO) {
        primary = 1u + static_cast<uint32_t>((tid - h0 + S) % S);
      } else if (!occupied) {
        primary = 0u;
      } else if (policy == MOE_CACHE_LRU) {
        primary = 1u + static_cast<uint32_t>(max(last_use[tid], 0));
      } else {
        primary = 1u + __float_as_uint(score[ex]);
      }
      key = (static_cast<unsigned long long>(primary) << 32) | static_cast<unsigned>(tid);
    }
  }
  s_key[tid] = key;
  const int nelig = __syncthreads_count(elig);
  const int nmiss = s_nmiss;
  if (nmiss > nelig) {  // cannot hold this call's experts: no slot changes
    if (tid == 0) {
      set_status(status, MOE_DEV_CACHE_FULL);
      stats[0] = nhit;
      stats[1] = 0;
      stats[2] += nhit;
      hand[1] = step + 1;
    }
    return;
  }
  // bitonic sort of the keys, ascending (ineligible slots sort last)
  int n2 = 1;
  while (n2 < S) n2 <<= 1;
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      if (tid < n2) {
        const int other = tid ^ stride;
        if (other > tid) {
          const unsigned long long a = s_key[tid], b = s_key[other];
          const bool up = (tid & size) == 0;
          if ((a > b) == up) {
            s_key[tid] = b;
            s_key[other] = a;
          }
        }
      }
    }
  }
  __syncthreads();
  // miss m takes the m-th victim; evict the victims' experts first (none of
  // them is routed in this call, so no miss is touched)
  for (int m = tid; m < nmiss; m += kPlanThreads) {
    const int v = static_cast<int>(s_key[m] & 0xffffffffu);
    const int old = expert_of[v];
    if (old >= 0 && old < E) slot_of[old] = -1;
    miss_list[m] = s_missexp[m];
    miss_slot[m] = v;
  }
  __syncthreads();
  for (int m = tid; m < nmiss; m += kPlanThreads) {
    const int e = s_missexp[m], v = static_cast<int>(s_key[m] & 0xffffffffu);
    slot_of[e] = v;
    expert_of[v] = e;
    if (policy == MOE_CACHE_LRU) last_use[v] = step;
  }
  if (policy == MOE_CACHE_LRU && hit) last_use[slot_of[tid]] = step;
  if (tid == 0) {
    if (policy == MOE_CACHE_FIFO && nmiss > 0) *hand = (static_cast<int>(s_key[nmiss - 1] & 0xffffffffu) + 1) % S;
    hand[1] = step + 1;
    stats[0] = nhit;
    stats[1] = nmiss;
    stats[2] += nhit;
    stats[3] += nmiss;
  }
}

__global__ void cache_fetch_kernel(const uint8_t* __restrict__ host_gu, const uint8_t* __restrict__ host_dn,
                                   size_t rec_gu, size_t rec_dn, const int32_t* __restrict__ miss_list,
                                   const int32_t* __restrict__ miss_slot, const int32_t* __restrict__ stats,
                                   uint8_t* __restrict__ pool_gu, uint8_t* __restrict__ pool_dn) {
  pdl_wait();
  pdl_trigger();
  const int nmiss = stats[1];
  const size_t ugu = rec_gu / 16, udn = rec_dn / 16, urec = ugu + udn;
  const size_t total = static_cast<size_t>(nmiss) * urec;
  constexpr int U = 8;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i0 = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i0 < total; i0 += U * stride) {
    uint4 v[U];
    uint4* dst[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const size_t i = i0 + u * stride;
      dst[u] = nullptr;
      if (i < total) {
        const size_t m = i / urec, w = i - m * urec;
        const size_t e = static_cast<size_t>(miss_list[m]), sl = static_cast<size_t>(miss_slot[m]);
        if (w < ugu) {
          v[u] = reinterpret_cast<const uint4*>(host_gu + e * rec_gu)[w];
          dst[u] = reinterpret_cast<uint4*>(pool_gu + sl * rec_gu) + w;
        } else {
          v[u] = reinterpret_cast<const uint4*>(host_dn + e * rec_dn)[w - ugu];
          dst[u] = reinterpret_cast<uint4*>(pool_dn + sl * rec_dn) + (w - ugu);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (dst[u]) *dst[u] = v[u];
  }
}

}  // namespace

cudaError_t launch_cache_plan(const int32_t* counts, int E, int32_t* slot_of, int32_t* expert_of, int S,
                              int32_t* hand, int policy, float decay, float* score, int32_t* last_use,
                              int32_t* miss_list, int32_t* miss_slot, int32_t* stats, int32_t* st_word,
                              cudaStream_t st) {
  return launch_pdl(cache_plan_kernel, dim3(1), dim3(kPlanThreads), 0, st, counts, E, slot_of, expert_of, S, hand,
                    policy, decay, score, last_use, miss_list, miss_slot, stats, st_word);
}

cudaError_t launch_cache_fetch(const void* host_gu, const void* host_dn, size_t rec_gu, size_t rec_dn,
                               const int32_t* miss_list, const int32_t* miss_slot, const int32_t* stats,
                               void* pool_gu, void* pool_dn, cudaStream_t st) {
  const int grid = sm_count() > 0 ? sm_count() * 4 : 512;
  return launch_pdl(cache_fetch_kernel, dim3(grid), dim3(256), 0, st, static_cast<const uint8_t*>(host_gu),
                    static_cast<const uint8_t*>(host_dn), rec_gu, rec_dn, miss_list, miss_slot, stats,
                    static_cast<uint8_t*>(pool_gu), static_cast<uint8_t*>(pool_dn));
}

}  // namespace moe
