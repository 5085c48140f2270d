// Router: logits, top-k in rank order, renormalised softmax weights.
//
// AFN-001 "Porting Qwen3.8-Flash-Next to Hebrus: evidence before execution",
// section "Phase 1: separate math from acceleration": float32 router softmax
// and normalized top-10 selection.  AFN-021 "Replay decode as prefill", section
// "The key equivalence -- and where it breaks": expert IDs and their rank
// order are the label, so selection is exact on the fp32 logits with a fixed
// tie rule (lower expert ID first), not on rounded probabilities.
//
// Small token counts (decode blocks) use CUDA cores: one warp per expert row,
// the block's token rows staged once in shared memory, 16-byte loads of the
// router row.  Large token counts use the tcgen05 grouped kernel in its dense
// router mode (gemm.cu).  Selection is one warp per token: each lane keeps
// ceil(E/32) logits in registers and k+1 rounds of warp arg-max pick the
// route and the next logit (for the decision gap).
#include <math.h>

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

template <int TT>
__global__ void __launch_bounds__(256) router_logits_simt_kernel(const uint16_t* __restrict__ x,
                                                                 const uint16_t* __restrict__ wr, int T, int H,
                                                                 int E, float* __restrict__ logits) {
  extern __shared__ uint4 xs[];  // [TT][H/8]
  const int vpr = H / 8;
  const int t0 = blockIdx.y * TT;
  const int nt = min(TT, T - t0);
  for (int idx = threadIdx.x; idx < TT * vpr; idx += blockDim.x) {
    const int r = idx / vpr;
    const int c = idx - r * vpr;
    xs[idx] = (r < nt) ? reinterpret_cast<const uint4*>(x + static_cast<size_t>(t0 + r) * H)[c]
                       : make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp;
  if (e >= E) return;
  float acc[TT];
#pragma unroll
  for (int t = 0; t < TT; ++t) acc[t] = 0.f;
  const uint4* wrow = reinterpret_cast<const uint4*>(wr + static_cast<size_t>(e) * H);
  for (int c = lane; c < vpr; c += 32) {
    float wf[8];
    unpack8(__ldg(wrow + c), wf);
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      float xf[8];
      unpack8(xs[t * vpr + c], xf);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[t] = fmaf(wf[i], xf[i], acc[t]);
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
  if (lane < nt) logits[static_cast<size_t>(t0 + lane) * E + e] = mine;
}

// better(a, b): larger logit, ties to the lower expert ID
__device__ __forceinline__ bool better(float va, int ea, float vb, int eb) {
  return va > vb || (va == vb && ea < eb);
}

template <int EPL>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                                                   int T, int E, int k, int32_t* __restrict__ ids,
                                                   float* __restrict__ w, float* __restrict__ gap) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  float v[EPL];
  uint32_t taken = 0;
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = j * 32 + lane;
    if (e < E) {
      float l = logits[static_cast<size_t>(t) * E + e];
      if (bias) l += bias[e];
      v[j] = isnan(l) ? -INFINITY : l;
    } else {
      v[j] = -INFINITY;
      taken |= 1u << j;
    }
  }
  float my_v = -INFINITY, next_v = -INFINITY;
  int my_e = 0;
  const int rounds = min(k + 1, E);
  for (int r = 0; r < rounds; ++r) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      if (!((taken >> j) & 1u) && better(v[j], j * 32 + lane, bv, be)) {
        bv = v[j];
        be = j * 32 + lane;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (better(ov, oe, bv, be)) {
        bv = ov;
        be = oe;
      }
    }
    if (be != 0x7fffffff && (be & 31) == lane) taken |= 1u << (be >> 5);
    if (r < k && lane == r) {
      my_v = bv;
      my_e = be;
    }
    if (r == k) next_v = bv;
  }
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
  if (gap && lane == 0) gap[t] = (k < E) ? (vk1 - next_v) : INFINITY;
}

template <int EPL>
cudaError_t run_topk(const float* logits, const float* bias, int T, int E, int k, int32_t* ids, float* w, float* gap,
                     cudaStream_t st) {
  const int blocks = (T + 7) / 8;
  topk_kernel<EPL><<<blocks, 256, 0, st>>>(logits, bias, T, E, k, ids, w, gap);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_logits_simt(const uint16_t* x, const uint16_t* wr, int T, int H, int E, float* logits,
                                      cudaStream_t st) {
  const dim3 block(256);
  if (H <= 6144) {
    constexpr int TT = 16;
    const size_t smem = static_cast<size_t>(TT) * H * 2;
    cudaError_t e = cudaFuncSetAttribute(router_logits_simt_kernel<TT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const dim3 grid((E + 7) / 8, (T + TT - 1) / TT);
    router_logits_simt_kernel<TT><<<grid, block, smem, st>>>(x, wr, T, H, E, logits);
  } else {
    constexpr int TT = 8;
    const size_t smem = static_cast<size_t>(TT) * H * 2;
    cudaError_t e = cudaFuncSetAttribute(router_logits_simt_kernel<TT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const dim3 grid((E + 7) / 8, (T + TT - 1) / TT);
    router_logits_simt_kernel<TT><<<grid, block, smem, st>>>(x, wr, T, H, E, logits);
  }
  return cudaGetLastError();
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
