// Deduplication of repeated routes across a verifier block, with the exact
// routed bytes the block needs.
//
// AFN-019 "Hide SSD misses before the router knows they exist", section "Why
// overlap alone cannot defeat the byte roofline": deduplicating repeated
// routes across a verifier block is a byte owner; ideal payload is
// parameters x bits / 8 per record.  Section "Hypothesis H7: DFlash block size
// must follow I/O cost": a block costs 48 * U_B * record bytes, break-even
// U_B < 10 * tau(B).
//
// One CTA per block of tokens walks every layer: a shared-memory expert
// bitmask (atomicOr per route), popcount in one warp, the per-layer mask and
// U written out, and the byte totals accumulated in the CTA (integers, so the
// result is exact).  IDs of the whole block are validated first so a bad
// block writes nothing.
#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

constexpr int kDedupThreads = 256;

__global__ void __launch_bounds__(kDedupThreads)
    dedup_kernel(const int32_t* __restrict__ ids, int L, int Ttot, int k, int E, int B, long long P,
                 uint32_t* __restrict__ mask, int32_t* __restrict__ U, int64_t* __restrict__ bytes2,
                 int64_t* __restrict__ bytes4, int32_t* status) {
  __shared__ uint32_t m[kMaxE / 32];
  __shared__ int bad;
  const int b = blockIdx.x;
  const int nb = gridDim.x;
  const int W = (E + 31) / 32;
  const int t0 = b * B;
  const int t1 = min(Ttot, t0 + B);
  const int n = (t1 - t0) * k;
  if (threadIdx.x == 0) bad = 0;
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  for (int l = 0; l < L; ++l) {
    const int32_t* src = ids + (static_cast<size_t>(l) * Ttot + t0) * k;
    for (int i = threadIdx.x; i < n; i += kDedupThreads) {
      const int e = src[i];
      if (e < 0 || e >= E) bad = 1;
    }
  }
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) set_status(status, MOE_DEV_BAD_EXPERT);
    return;
  }
  long long usum = 0;
  for (int l = 0; l < L; ++l) {
    for (int i = threadIdx.x; i < W; i += kDedupThreads) m[i] = 0u;
    __syncthreads();
    const int32_t* src = ids + (static_cast<size_t>(l) * Ttot + t0) * k;
    for (int i = threadIdx.x; i < n; i += kDedupThreads) {
      const int e = src[i];
      atomicOr(&m[e >> 5], 1u << (e & 31));
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      int u = 0;
      for (int i = threadIdx.x; i < W; i += 32) {
        const uint32_t word = m[i];
        mask[(static_cast<size_t>(l) * nb + b) * W + i] = word;
        u += __popc(word);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) u += __shfl_xor_sync(0xffffffffu, u, off);
      if (threadIdx.x == 0) U[static_cast<size_t>(l) * nb + b] = u;
      usum += u;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    bytes2[b] = static_cast<int64_t>(usum * P * 2 / 8);
    bytes4[b] = static_cast<int64_t>(usum * P * 4 / 8);
  }
}

}  // namespace

cudaError_t launch_dedup(const int32_t* ids, int L, int Ttot, int k, int E, int B, long long P, uint32_t* mask,
                         int32_t* U, int64_t* bytes2, int64_t* bytes4, int32_t* st_word, cudaStream_t st) {
  const int nb = (Ttot + B - 1) / B;
  return launch_pdl(dedup_kernel, dim3(nb), dim3(kDedupThreads), 0, st, ids, L, Ttot, k, E, B, P, mask, U, bytes2,
                    bytes4, st_word);
}

}  // namespace moe
