// Router: logits, top-k in rank order, renormalised softmax weights.
//
// AFN-001 "Porting Qwen3.8-Flash-Next to Hebrus: evidence before execution",
// section "Phase 1: separate math from acceleration": float32 router softmax
// and normalized top-10 selection.  AFN-021 "Replay decode as prefill", section
// "The key equivalence -- and where it breaks": expert IDs and their rank
// order are the label, so selection is exact on the fp32 logits with a fixed
// tie rule (lower expert ID first), not on rounded probabilities.
//
// Small token counts (decode blocks) use warp-level MMA on the tensor cores
// with a K split over the warps of a CTA; large token counts use the tcgen05
// grouped kernel in its dense router mode (gemm.cu).  Selection is one warp
// per token: each lane keeps ceil(E/32) logits in registers, sorted once, and
// k+1 rounds of warp-wide reductions pick the route and the next logit (for
// the decision gap).
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace moe {

namespace {

// Small-T logits on the tensor cores with warp-level MMA (m16n8k16, bf16 in,
// fp32 accumulate).  A cluster of four CTAs covers 16 tokens x 8 experts;
// CTA r of the cluster takes the r-th quarter of K and divides it among its
// 8 warps, each of which chains its MMAs in ascending K.  The CTA sums its
// warps' tiles in warp order in shared memory, and CTA 0 of the cluster adds
// the four CTA tiles in rank order over distributed shared memory, so every
// logit is summed in one fixed order on every call.  The router rows are
// constant: their fragments are loaded before the wait on the upstream
// kernel; the token fragments come straight from global memory.  At decode
// sizes the contraction is ~42 MFLOP over 256 CTAs: the latency of a global
// round trip, not MMA throughput, sets its time.
constexpr int kLogitThreads = 256;
constexpr int kLogitWarps = kLogitThreads / 32;
constexpr int kLogitTok = 16;    // tokens per CTA (MMA M)
constexpr int kLogitExp = 8;     // experts per CTA (MMA N)
constexpr int kLogitSplit = 4;   // CTAs per cluster, one K quarter each
constexpr int kLogitChunk = 8;   // k16 steps per register batch

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Load of the same shared-memory word in CTA `rank` of the cluster (volatile
// so that it stays between the cluster barriers; loads issued back to back
// are still in flight together).
__device__ __forceinline__ float ld_cluster_f32(const float* local, uint32_t rank) {
  uint32_t remote;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(ptx::smem_u32(local)), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

__global__ void __launch_bounds__(kLogitThreads) router_logits_mma_kernel(const uint16_t* __restrict__ x,
                                                                          const uint16_t* __restrict__ wr, int T,
                                                                          int H, int E, float* __restrict__ logits) {
  __shared__ float red[kLogitWarps][kLogitTok][kLogitExp];
  __shared__ float tile[kLogitTok][kLogitExp];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;  // fragment row group
  const int q = lane & 3;   // thread in group
  const uint32_t rank = cluster_ctarank();
  const int e0 = blockIdx.x * kLogitExp;
  const int t0 = blockIdx.y * kLogitTok;
  // k16 steps of this warp: worker rank * 8 + warp of 32
  const int steps_all = H / 16;
  constexpr int kWorkers = kLogitSplit * kLogitWarps;
  const int per = (steps_all + kWorkers - 1) / kWorkers;
  const int s_begin = min(steps_all, (static_cast<int>(rank) * kLogitWarps + warp) * per);
  const int steps = min(steps_all, s_begin + per) - s_begin;
  const int kbase = s_begin * 16;
  // B fragment: expert e0 + g, K pairs (q*2, q*2+1) and (q*2+8, q*2+9)
  const bool e_ok = e0 + g < E;
  const uint32_t* wrow = reinterpret_cast<const uint32_t*>(wr + static_cast<size_t>(e_ok ? e0 + g : 0) * H + kbase);
  // A fragment rows: tokens t0 + g and t0 + g + 8
  const bool ta = t0 + g < T, tb = t0 + g + 8 < T;
  const uint32_t* xa = reinterpret_cast<const uint32_t*>(x + static_cast<size_t>(ta ? t0 + g : 0) * H + kbase);
  const uint32_t* xb = reinterpret_cast<const uint32_t*>(x + static_cast<size_t>(tb ? t0 + g + 8 : 0) * H + kbase);

  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  uint32_t bw[kLogitChunk][2];
#pragma unroll
  for (int s = 0; s < kLogitChunk; ++s) {
    const bool in = e_ok && s < steps;
    bw[s][0] = in ? __ldg(wrow + s * 8 + q) : 0u;
    bw[s][1] = in ? __ldg(wrow + s * 8 + 4 + q) : 0u;
  }
  pdl_wait();
  pdl_trigger();
  for (int c0 = 0; c0 < steps; c0 += kLogitChunk) {
    if (c0 > 0) {
#pragma unroll
      for (int s = 0; s < kLogitChunk; ++s) {
        const bool in = e_ok && c0 + s < steps;
        bw[s][0] = in ? __ldg(wrow + (c0 + s) * 8 + q) : 0u;
        bw[s][1] = in ? __ldg(wrow + (c0 + s) * 8 + 4 + q) : 0u;
      }
    }
    uint32_t af[kLogitChunk][4];
#pragma unroll
    for (int s = 0; s < kLogitChunk; ++s) {
      const bool in = c0 + s < steps;
      const int o = (c0 + s) * 8 + q;
      af[s][0] = (in && ta) ? xa[o] : 0u;
      af[s][1] = (in && tb) ? xb[o] : 0u;
      af[s][2] = (in && ta) ? xa[o + 4] : 0u;
      af[s][3] = (in && tb) ? xb[o + 4] : 0u;
    }
#pragma unroll
    for (int s = 0; s < kLogitChunk; ++s)
      if (c0 + s < steps) mma_bf16_16816(acc, af[s], bw[s]);
  }
  red[warp][g][2 * q] = acc[0];
  red[warp][g][2 * q + 1] = acc[1];
  red[warp][g + 8][2 * q] = acc[2];
  red[warp][g + 8][2 * q + 1] = acc[3];
  __syncthreads();
  const int t = threadIdx.x / kLogitExp;
  const int e = threadIdx.x % kLogitExp;
  if (threadIdx.x < kLogitTok * kLogitExp) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kLogitWarps; ++w) sum += red[w][t][e];
    tile[t][e] = sum;
  }
  cluster_sync_all();  // every CTA's tile is complete and visible to the cluster
  if (rank == 0 && threadIdx.x < kLogitTok * kLogitExp) {
    float part[kLogitSplit];
    part[0] = tile[t][e];
#pragma unroll
    for (int r = 1; r < kLogitSplit; ++r) part[r] = ld_cluster_f32(&tile[t][e], r);
    float sum = part[0];
#pragma unroll
    for (int r = 1; r < kLogitSplit; ++r) sum += part[r];
    if (t0 + t < T && e0 + e < E) logits[static_cast<size_t>(t0 + t) * E + e0 + e] = sum;
  }
  cluster_sync_all();  // keep every tile alive until CTA 0 has read it
}

// Order-preserving map of a float to an unsigned key (NaN mapped to -inf by
// the caller, -0 to +0), so that warp-wide unsigned max/min reductions select
// the largest logit and, among equal logits, the lowest expert ID.
__device__ __forceinline__ uint32_t f2key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key2f(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Descending bitonic sort of N (a power of two) values held in registers.
template <int N>
__device__ __forceinline__ void sort_desc(uint64_t (&v)[N]) {
#pragma unroll
  for (int k = 2; k <= N; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
      for (int i = 0; i < N; ++i) {
        const int l = i ^ j;
        if (l > i) {
          const uint64_t a = v[i], b = v[l];
          const bool swap = ((i & k) == 0) ? (a < b) : (a > b);
          v[i] = swap ? b : a;
          v[l] = swap ? a : b;
        }
      }
    }
  }
}

// Descending bitonic sort of one value per lane across the warp (lane r ends
// with the r-th largest).
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xffffffffu, v, j);
      const bool keep_max = ((lane & k) == 0) == ((lane & j) == 0);
      v = keep_max ? (v > o ? v : o) : (v < o ? v : o);
    }
  }
  return v;
}

// One warp per token.  Lane l holds the logits of experts l, l+32, ... as
// 64-bit keys (order key of the logit, then the bitwise complement of the
// expert ID), so the largest key is the largest logit and, among equal
// logits, the lowest expert ID; every key is distinct.  Let n = min(k+1, E)
// (the k routes and the next logit, for the decision gap).  The n-th largest
// of the 32 lane maxima is a threshold that at least n keys reach (those
// lanes' maxima), so the n largest keys are all at or above it.  The keys at
// or above it -- rarely more than a few beyond n -- are compacted and sorted
// across the warp in one bitonic pass, and lane r then holds rank r.  If
// more than 32 keys reach the threshold (or n > 32), each lane sorts its own
// keys and n rounds of warp-wide max reductions take the largest head.
template <int EPL>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                                                   int T, int E, int k, int32_t* __restrict__ ids,
                                                   float* __restrict__ w, float* __restrict__ gap) {
  __shared__ uint64_t cand[8][32];
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  // all loads first, then the keys
  float lv[EPL], bv[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = j * 32 + lane;
    lv[j] = e < E ? logits[static_cast<size_t>(t) * E + e] : 0.f;
    bv[j] = (bias && e < E) ? bias[e] : 0.f;
  }
  uint64_t v[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = j * 32 + lane;
    v[j] = 0;  // below every valid key (f2key(-inf) > 0)
    if (e < E) {
      float l = lv[j];
      if (bias) l += bv[j];
      if (isnan(l)) l = -INFINITY;
      if (l == 0.0f) l = 0.0f;
      v[j] = (static_cast<uint64_t>(f2key(l)) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(e));
    }
  }
  const int n = min(k + 1, E);
  uint64_t mine = 0;  // lane r: the key of rank r (r < n)
  bool done = false;
  if (n <= 32) {
    uint64_t m = v[0];
#pragma unroll
    for (int j = 1; j < EPL; ++j) m = v[j] > m ? v[j] : m;
    const uint64_t thr = __shfl_sync(0xffffffffu, warp_sort_desc(m, lane), n - 1);
    int c = 0;
#pragma unroll
    for (int j = 0; j < EPL; ++j) c += v[j] >= thr ? 1 : 0;
    int incl = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (total <= 32) {
      int pos = incl - c;
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        if (v[j] >= thr) cand[warp][pos++] = v[j];
      __syncwarp();
      mine = warp_sort_desc(lane < total ? cand[warp][lane] : 0, lane);
      done = true;
    }
  }
  if (!done) {
    sort_desc<EPL>(v);
    for (int r = 0; r < n; ++r) {
      const uint32_t hi = static_cast<uint32_t>(v[0] >> 32);
      const uint32_t lo = static_cast<uint32_t>(v[0]);
      const uint32_t m_hi = __reduce_max_sync(0xffffffffu, hi);
      const uint32_t m_lo = __reduce_max_sync(0xffffffffu, hi == m_hi ? lo : 0u);
      if (hi == m_hi && lo == m_lo) {
#pragma unroll
        for (int j = 0; j + 1 < EPL; ++j) v[j] = v[j + 1];
        v[EPL - 1] = 0;
      }
      if (lane == r) mine = (static_cast<uint64_t>(m_hi) << 32) | m_lo;
    }
  }
  const uint32_t my_key = static_cast<uint32_t>(mine >> 32);
  const int my_e = static_cast<int>(~static_cast<uint32_t>(mine));
  const uint32_t next_key = static_cast<uint32_t>(__shfl_sync(0xffffffffu, mine, k & 31) >> 32);
  const float my_v = key2f(my_key);
  const float v0 = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = (lane < k) ? expf(my_v - v0) : 0.f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  const float vk1 = __shfl_sync(0xffffffffu, my_v, k - 1);
  if (lane < k) {
    ids[static_cast<size_t>(t) * k + lane] = my_e;
    w[static_cast<size_t>(t) * k + lane] = ex / sum;
  }
  if (gap && lane == 0) gap[t] = (k < E) ? (vk1 - key2f(next_key)) : INFINITY;
}

template <int EPL>
cudaError_t run_topk(const float* logits, const float* bias, int T, int E, int k, int32_t* ids, float* w, float* gap,
                     cudaStream_t st) {
  const int blocks = (T + 7) / 8;
  return launch_pdl(topk_kernel<EPL>, dim3(blocks), dim3(256), 0, st, logits, bias, T, E, k, ids, w, gap);
}

}  // namespace

cudaError_t launch_router_logits_small(const uint16_t* x, const uint16_t* wr, int T, int H, int E, float* logits,
                                       cudaStream_t st) {
  const dim3 grid((E + kLogitExp - 1) / kLogitExp, (T + kLogitTok - 1) / kLogitTok, kLogitSplit);
  return launch_pdl_cluster(router_logits_mma_kernel, grid, dim3(kLogitThreads), dim3(1, 1, kLogitSplit), 0, st, x,
                            wr, T, H, E, logits);
}

cudaError_t launch_topk(const float* logits, const float* bias, int T, int E, int k, int32_t* ids, float* w,
                        float* gap, cudaStream_t st) {
  const int epl = (E + 31) / 32;
  if (epl <= 1) return run_topk<1>(logits, bias, T, E, k, ids, w, gap, st);
  if (epl <= 2) return run_topk<2>(logits, bias, T, E, k, ids, w, gap, st);
  if (epl <= 4) return run_topk<4>(logits, bias, T, E, k, ids, w, gap, st);
  if (epl <= 8) return run_topk<8>(logits, bias, T, E, k, ids, w, gap, st);
  if (epl <= 16) return run_topk<16>(logits, bias, T, E, k, ids, w, gap, st);
  return run_topk<32>(logits, bias, T, E, k, ids, w, gap, st);
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Allocation-free router entry point.
//
// Some callers cannot allocate device memory when they call the router: a
// host framework that owns every device buffer and hands a plugin only its
// inputs and outputs, or code that must not allocate while it runs (for
// example on a path where an allocator call could block or is forbidden).
// For them, moe_route_noalloc() keeps its scratch (the [T, E] fp32 logits)
// in the fixed array below instead of in a caller-provided workspace.
//
//  * Limit: T <= 64 tokens and E <= 1024 experts (64 x 1024 fp32 = 256 KB).
//    Every GPU that loads the library holds this array until the process
//    exits.  Larger calls are rejected with MOE_EWORKSPACE.
//  * The host-side name g_route_scratch is not a device address; the first
//    call on a device looks the device address up with
//    cudaGetSymbolAddress() (with that device current) and remembers it, so
//    that first call should come before any stream capture.
//  * All calls share the array and it keeps the last call's contents.
//    Nothing in it needs to start at zero: the logits kernel overwrites the
//    whole [T, E] region before the selection kernel reads it.  Calls that
//    overlap on the GPU (for instance on two streams at once) race on it.
//  * No cudaMalloc, cudaFree or allocating library routine is called.
// ---------------------------------------------------------------------------
namespace {

constexpr int kNoAllocMaxT = 64;
constexpr int kNoAllocMaxE = 1024;
static __device__ __align__(256) float g_route_scratch[kNoAllocMaxT * kNoAllocMaxE];

// Device address of g_route_scratch on the current device (nullptr on error).
float* noalloc_scratch_for_current_device() {
  static std::mutex mu;
  static float* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<float*>(p);
  }
  return addr[dev];
}

}  // namespace

extern "C" moe_status moe_route_noalloc(const uint16_t* x, const uint16_t* w_router, const float* bias, int T, int H,
                                        int E, int k, int32_t* topk_ids, float* topk_w, float* gap, void* stream) {
  if (T < 0 || H <= 0 || E <= 0 || k <= 0) return MOE_ESHAPE;
  if (k > moe::kMaxK || k > E || E > moe::kMaxE || H % 128 != 0 || H > 16384) return MOE_ENOTSUP;
  if (!x || !w_router || !topk_ids || !topk_w) return MOE_EINVAL;
  auto aligned = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
  if (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(topk_ids, 4) || !aligned(topk_w, 4)) return MOE_EINVAL;
  if ((bias && !aligned(bias, 4)) || (gap && !aligned(gap, 4))) return MOE_EINVAL;
  if (T > kNoAllocMaxT || E > kNoAllocMaxE) return MOE_EWORKSPACE;
  if (T == 0) return MOE_OK;
  float* logits = noalloc_scratch_for_current_device();
  if (!logits) return MOE_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (moe::launch_router_logits_small(x, w_router, T, H, E, logits, st) != cudaSuccess) return MOE_ECUDA;
  if (moe::launch_topk(logits, bias, T, E, k, topk_ids, topk_w, gap, st) != cudaSuccess) return MOE_ECUDA;
  return MOE_OK;
}
