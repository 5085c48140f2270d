// Router: logits, top-k in rank order, renormalised softmax weights.
//
// AFN-001 "Porting Qwen3.8-Flash-Next to Hebrus: evidence before execution",
// section "Phase 1: separate math from acceleration": float32 router softmax
// and normalized top-10 selection.  AFN-021 "Replay decode as prefill", section
// "The key equivalence -- and where it breaks": expert IDs and their rank
// order are the label, so selection is exact on the fp32 logits with a fixed
// tie rule (lower expert ID first), not on rounded probabilities.
//
// Small token counts (decode blocks) use CUDA cores: two warps per expert row,
// all router-row loads in flight at once, the block's token rows staged once
// in shared memory.  Large token counts use the tcgen05 grouped kernel in its
// dense router mode (gemm.cu).  Selection is one warp per token: each lane
// keeps ceil(E/32) logits in registers and k+1 rounds of warp-wide max/min
// reductions pick the route and the next logit (for the decision gap).
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// One CTA = 8 warps = 4 experts x 2 halves of K.  The router rows are
// constant, so each lane issues all of its (up to 8 x 16-byte) weight loads
// before waiting on the upstream kernel; the token tile is then staged once
// in shared memory and every lane runs TT dot products over its K range.
constexpr int kLogitThreads = 256;
constexpr int kLogitExperts = 4;
constexpr int kWChunk = 8;  // 16-byte weight vectors a lane keeps in flight

template <int TT>
__global__ void __launch_bounds__(kLogitThreads) router_logits_simt_kernel(const uint16_t* __restrict__ x,
                                                                           const uint16_t* __restrict__ wr,
                                                                           int T, int H, int E,
                                                                           float* __restrict__ logits) {
  extern __shared__ uint4 xs[];  // [TT][H/8]
  __shared__ float part[kLogitExperts][TT];
  const int vpr = H / 8;
  const int hv = vpr / 2;  // 16-byte vectors per K half
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * kLogitExperts + (warp >> 1);
  const int half = warp & 1;
  const int t0 = blockIdx.y * TT;
  const int nt = min(TT, T - t0);
  const bool active = e < E;
  const uint4* wrow = reinterpret_cast<const uint4*>(wr + static_cast<size_t>(active ? e : 0) * H) + half * hv;

  uint4 wv[kWChunk];
#pragma unroll
  for (int j = 0; j < kWChunk; ++j) {
    const int c = lane + 32 * j;
    wv[j] = (active && c < hv) ? __ldg(wrow + c) : make_uint4(0, 0, 0, 0);
  }

  pdl_wait();
  pdl_trigger();
  for (int idx = threadIdx.x; idx < TT * vpr; idx += kLogitThreads) {
    const int r = idx / vpr;
    const int c = idx - r * vpr;
    xs[idx] = (r < nt) ? reinterpret_cast<const uint4*>(x + static_cast<size_t>(t0 + r) * H)[c]
                       : make_uint4(0, 0, 0, 0);
  }
  __syncthreads();

  float acc[TT];
#pragma unroll
  for (int t = 0; t < TT; ++t) acc[t] = 0.f;
  for (int c0 = 0; c0 < hv; c0 += 32 * kWChunk) {
    if (c0 > 0) {
#pragma unroll
      for (int j = 0; j < kWChunk; ++j) {
        const int c = c0 + lane + 32 * j;
        wv[j] = (active && c < hv) ? __ldg(wrow + c) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int j = 0; j < kWChunk; ++j) {
      const int c = c0 + lane + 32 * j;
      if (c < hv) {
        float wf[8];
        unpack8(wv[j], wf);
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          float xf[8];
          unpack8(xs[t * vpr + half * hv + c], xf);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[t] = fmaf(wf[i], xf[i], acc[t]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TT; ++t) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
  }
  float mine = 0.f;
#pragma unroll
  for (int t = 0; t < TT; ++t)
    if (lane == t) mine = acc[t];
  if (half == 1 && lane < TT) part[warp >> 1][lane] = mine;
  __syncthreads();
  if (half == 0 && active && lane < nt)
    logits[static_cast<size_t>(t0 + lane) * E + e] = mine + part[warp >> 1][lane];
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

// One warp per token.  Lane l holds the logits of experts l, l+32, ...; each
// round one __reduce_max_sync finds the largest remaining logit and one
// __reduce_min_sync the lowest expert ID holding it; only the winning lane
// rescans its own EPL values.
template <int EPL>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                                                   int T, int E, int k, int32_t* __restrict__ ids,
                                                   float* __restrict__ w, float* __restrict__ gap) {
  pdl_wait();
  pdl_trigger();
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  uint32_t key[EPL];
  uint32_t taken = 0;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = j * 32 + lane;
    if (e < E) {
      float l = logits[static_cast<size_t>(t) * E + e];
      if (bias) l += bias[e];
      if (isnan(l)) l = -INFINITY;
      if (l == 0.0f) l = 0.0f;
      key[j] = f2key(l);
    } else {
      key[j] = 0u;
      taken |= 1u << j;
    }
  }
  auto local_best = [&](uint32_t& bk, int& be) {
    bk = 0u;
    be = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      if (!((taken >> j) & 1u) && (be == 0x7fffffff || key[j] > bk)) {
        bk = key[j];
        be = j * 32 + lane;
      }
    }
  };
  uint32_t bk;
  int be;
  local_best(bk, be);
  uint32_t my_key = 0u, next_key = 0u;
  int my_e = 0;
  const int rounds = min(k + 1, E);
  for (int r = 0; r < rounds; ++r) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
    const int cand = (be != 0x7fffffff && bk == m) ? be : 0x7fffffff;
    const int emin = __reduce_min_sync(0xffffffffu, cand);
    if ((emin & 31) == lane) {
      taken |= 1u << (emin >> 5);
      local_best(bk, be);
    }
    if (r < k && lane == r) {
      my_key = m;
      my_e = emin;
    }
    if (r == k) next_key = m;
  }
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

cudaError_t launch_router_logits_simt(const uint16_t* x, const uint16_t* wr, int T, int H, int E, float* logits,
                                      cudaStream_t st) {
  const dim3 grid((E + kLogitExperts - 1) / kLogitExperts, 1);
  if (H <= 6144) {
    constexpr int TT = 16;
    const size_t smem = static_cast<size_t>(TT) * H * 2;
    cudaError_t e = ensure_smem(router_logits_simt_kernel<TT>, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_pdl(router_logits_simt_kernel<TT>, dim3(grid.x, (T + TT - 1) / TT), dim3(kLogitThreads), smem,
                      st, x, wr, T, H, E, logits);
  }
  constexpr int TT = 8;
  const size_t smem = static_cast<size_t>(TT) * H * 2;
  cudaError_t e = ensure_smem(router_logits_simt_kernel<TT>, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(router_logits_simt_kernel<TT>, dim3(grid.x, (T + TT - 1) / TT), dim3(kLogitThreads), smem, st,
                    x, wr, T, H, E, logits);
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
  if (moe::launch_router_logits_simt(x, w_router, T, H, E, logits, st) != cudaSuccess) return MOE_ECUDA;
  if (moe::launch_topk(logits, bias, T, E, k, topk_ids, topk_w, gap, st) != cudaSuccess) return MOE_ECUDA;
  return MOE_OK;
}
