// Weighted combine in route-rank order, and the zero-centred RMSNorm that
// feeds a residual stack layer.
//
// AFN-019 "Hide SSD misses before the router knows they exist", section
// "Hypothesis H4: ExpertMajor should stream as a wavefront, not a barrier":
// expert results may be produced in any order into separate slots, but the
// final weighted sum follows a deterministic route-rank order.  Here every
// output element is summed by one thread over j = 0..k-1 in order, so the
// result is bit-identical from run to run whatever order the experts ran in.
//
// AFN-001 "Porting Qwen3.8-Flash-Next to Hebrus", section "Phase 1: separate
// math from acceleration": zero-centred RMS normalisation (gain 1 + gamma).
//
// Both kernels are HBM/L2-bound gathers: 16-byte loads, one CTA per
// (token, 512 columns) for the combine, one CTA per token row for RMSNorm.
//
// The recall kernel scores a predicted route against the native one (AFN-019,
// section "Hypothesis H2: predict expert routes before attention, not after
// it": a predictor may move bytes but never chooses experts; it is judged by
// how many of the exact top-k it names).
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

constexpr int kCombineThreads = 128;  // x 4 floats = 512 columns per CTA (fp32 rows)
constexpr int kCombineBatch = 16;     // fp32 rows whose loads a thread has in flight (k <= 16: one round trip)
constexpr int kCombineBatchW = 8;     // bf16 rows (prefill-sized launches: 16 measured slower)

__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const float* __restrict__ y, const int32_t* __restrict__ inv, const float* __restrict__ w, int T,
                   int k, int H, int R, const float* residual, uint16_t* __restrict__ out_bf16, float* out_f32,
                   int32_t* status) {
  // residual and out_f32 may be the same buffer (an in-place residual
  // stream): each element is read and then written by the same thread.
  __shared__ int slot[kMaxK];
  __shared__ float wt[kMaxK];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.y;
  if (threadIdx.x < k) {
    int s = inv[static_cast<size_t>(t) * k + threadIdx.x];
    if (s < 0 || s >= R) s = -1;
    slot[threadIdx.x] = s;
    wt[threadIdx.x] = w[static_cast<size_t>(t) * k + threadIdx.x];
  }
  __syncthreads();
  const int c4 = blockIdx.x * kCombineThreads + threadIdx.x;
  if (c4 * 4 >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  bool bad = false;
  // kCombineBatch rows' loads in flight, then their terms in j order
  for (int j0 = 0; j0 < k; j0 += kCombineBatch) {
    float4 v[kCombineBatch];
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) {
      const int s = j0 + u < k ? slot[j0 + u] : -1;
      v[u] = s >= 0 ? reinterpret_cast<const float4*>(y + static_cast<size_t>(s) * H)[c4]
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) {
      const int j = j0 + u;
      if (j < k) {
        if (slot[j] < 0) {
          bad = true;
        } else {
          const float wj = wt[j];
          acc.x = fmaf(wj, v[u].x, acc.x);
          acc.y = fmaf(wj, v[u].y, acc.y);
          acc.z = fmaf(wj, v[u].z, acc.z);
          acc.w = fmaf(wj, v[u].w, acc.w);
        }
      }
    }
  }
  if (residual) {
    const float4 r = reinterpret_cast<const float4*>(residual + static_cast<size_t>(t) * H)[c4];
    acc.x += r.x;
    acc.y += r.y;
    acc.z += r.z;
    acc.w += r.w;
  }
  if (status && (bad || !isfinite(acc.x) || !isfinite(acc.y) || !isfinite(acc.z) || !isfinite(acc.w)))
    set_status(status, bad ? MOE_DEV_BAD_EXPERT : MOE_DEV_NONFINITE);
  if (out_f32) reinterpret_cast<float4*>(out_f32 + static_cast<size_t>(t) * H)[c4] = acc;
  if (out_bf16) {
    uint2 pk;
    pk.x = static_cast<uint32_t>(f32_to_bf16(acc.x)) | (static_cast<uint32_t>(f32_to_bf16(acc.y)) << 16);
    pk.y = static_cast<uint32_t>(f32_to_bf16(acc.z)) | (static_cast<uint32_t>(f32_to_bf16(acc.w)) << 16);
    reinterpret_cast<uint2*>(out_bf16 + static_cast<size_t>(t) * H)[c4] = pk;
  }
}

// The same sum over expert outputs that the down epilogue already multiplied
// by their route weights and stored in bf16 (yw [R, H]): acc = sum_j
// yw[inv[t*k + j]] in j order, fp32.  Eight columns per thread (one 16-byte
// load per row, kCombineBatchW rows in flight), 1,024 columns per CTA.
__global__ void __launch_bounds__(kCombineThreads)
    combine_weighted_kernel(const uint16_t* __restrict__ yw, const int32_t* __restrict__ inv, int T, int k, int H,
                            int R, const float* residual, uint16_t* __restrict__ out_bf16, float* out_f32,
                            int32_t* status) {
  __shared__ int slot[kMaxK];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.y;
  if (threadIdx.x < k) {
    int s = inv[static_cast<size_t>(t) * k + threadIdx.x];
    if (s < 0 || s >= R) s = -1;
    slot[threadIdx.x] = s;
  }
  __syncthreads();
  const int c8 = blockIdx.x * kCombineThreads + threadIdx.x;
  if (c8 * 8 >= H) return;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  bool bad = false;
  for (int j0 = 0; j0 < k; j0 += kCombineBatchW) {
    uint4 v[kCombineBatchW];
#pragma unroll
    for (int u = 0; u < kCombineBatchW; ++u) {
      const int s = j0 + u < k ? slot[j0 + u] : -1;
      v[u] = s >= 0 ? reinterpret_cast<const uint4*>(yw + static_cast<size_t>(s) * H)[c8] : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kCombineBatchW; ++u) {
      const int j = j0 + u;
      if (j < k) {
        if (slot[j] < 0) {
          bad = true;
        } else {
          const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[2 * i] += bf16_to_f32(static_cast<uint16_t>(w4[i] & 0xffffu));
            acc[2 * i + 1] += bf16_to_f32(static_cast<uint16_t>(w4[i] >> 16));
          }
        }
      }
    }
  }
  if (residual) {
    const float4* rr = reinterpret_cast<const float4*>(residual + static_cast<size_t>(t) * H) + 2 * c8;
    const float4 r0 = rr[0], r1 = rr[1];
    acc[0] += r0.x;
    acc[1] += r0.y;
    acc[2] += r0.z;
    acc[3] += r0.w;
    acc[4] += r1.x;
    acc[5] += r1.y;
    acc[6] += r1.z;
    acc[7] += r1.w;
  }
  bool fin = true;
#pragma unroll
  for (int i = 0; i < 8; ++i) fin = fin && isfinite(acc[i]);
  if (status && (bad || !fin)) set_status(status, bad ? MOE_DEV_BAD_EXPERT : MOE_DEV_NONFINITE);
  if (out_f32) {
    float4* o = reinterpret_cast<float4*>(out_f32 + static_cast<size_t>(t) * H) + 2 * c8;
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
  if (out_bf16) {
    uint4 pk;
    pk.x = static_cast<uint32_t>(f32_to_bf16(acc[0])) | (static_cast<uint32_t>(f32_to_bf16(acc[1])) << 16);
    pk.y = static_cast<uint32_t>(f32_to_bf16(acc[2])) | (static_cast<uint32_t>(f32_to_bf16(acc[3])) << 16);
    pk.z = static_cast<uint32_t>(f32_to_bf16(acc[4])) | (static_cast<uint32_t>(f32_to_bf16(acc[5])) << 16);
    pk.w = static_cast<uint32_t>(f32_to_bf16(acc[6])) | (static_cast<uint32_t>(f32_to_bf16(acc[7])) << 16);
    reinterpret_cast<uint4*>(out_bf16 + static_cast<size_t>(t) * H)[c8] = pk;
  }
}

constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads)
    rmsnorm_kernel(const float* __restrict__ x, const float* __restrict__ gamma, float eps, int H,
                   uint16_t* __restrict__ out, uint16_t* __restrict__ raw) {
  __shared__ float part[kNormThreads / 32];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const float4* xr = reinterpret_cast<const float4*>(x + static_cast<size_t>(t) * H);
  const int n4 = H / 4;
  float ss = 0.f;
  for (int c = threadIdx.x; c < n4; c += kNormThreads) {
    const float4 v = xr[c];
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kNormThreads / 32; ++i) tot += part[i];
  const float r = 1.0f / sqrtf(tot / static_cast<float>(H) + eps);
  for (int c = threadIdx.x; c < n4; c += kNormThreads) {
    const float4 v = xr[c];
    float g[4] = {0.f, 0.f, 0.f, 0.f};
    if (gamma) {
      const float4 gv = reinterpret_cast<const float4*>(gamma)[c];
      g[0] = gv.x; g[1] = gv.y; g[2] = gv.z; g[3] = gv.w;
    }
    uint2 pk;
    pk.x = static_cast<uint32_t>(f32_to_bf16(v.x * r * (1.f + g[0]))) |
           (static_cast<uint32_t>(f32_to_bf16(v.y * r * (1.f + g[1]))) << 16);
    pk.y = static_cast<uint32_t>(f32_to_bf16(v.z * r * (1.f + g[2]))) |
           (static_cast<uint32_t>(f32_to_bf16(v.w * r * (1.f + g[3]))) << 16);
    reinterpret_cast<uint2*>(out + static_cast<size_t>(t) * H)[c] = pk;
    if (raw) {
      uint2 rk;
      rk.x = static_cast<uint32_t>(f32_to_bf16(v.x)) | (static_cast<uint32_t>(f32_to_bf16(v.y)) << 16);
      rk.y = static_cast<uint32_t>(f32_to_bf16(v.z)) | (static_cast<uint32_t>(f32_to_bf16(v.w)) << 16);
      reinterpret_cast<uint2*>(raw + static_cast<size_t>(t) * H)[c] = rk;
    }
  }
}

// Recall of a predicted route against the native one: one warp per token;
// lane j < k holds the j-th native expert and tests it against the k
// predicted experts (both routes hold k distinct IDs).
__global__ void __launch_bounds__(256) recall_kernel(const int32_t* __restrict__ pred,
                                                     const int32_t* __restrict__ ref, int T, int k,
                                                     int32_t* __restrict__ hits) {
  pdl_wait();
  pdl_trigger();
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int mine = (lane < k) ? ref[static_cast<size_t>(t) * k + lane] : -1;
  const int p = (lane < k) ? pred[static_cast<size_t>(t) * k + lane] : -2;
  bool found = false;
  for (int i = 0; i < k; ++i) found |= (__shfl_sync(0xffffffffu, p, i) == mine);
  const unsigned m = __ballot_sync(0xffffffffu, found && lane < k);
  if (lane == 0) hits[t] = __popc(m);
}

}  // namespace

cudaError_t launch_combine(const float* y, const int32_t* inv, const float* w, int T, int k, int H, int R,
                           const float* residual, uint16_t* out_bf16, float* out_f32, int32_t* st_word,
                           cudaStream_t st) {
  const dim3 grid((H / 4 + kCombineThreads - 1) / kCombineThreads, T);
  return launch_pdl(combine_kernel, grid, dim3(kCombineThreads), 0, st, y, inv, w, T, k, H, R, residual, out_bf16,
                    out_f32, st_word);
}

cudaError_t launch_combine_weighted(const uint16_t* yw, const int32_t* inv, int T, int k, int H, int R,
                                    const float* residual, uint16_t* out_bf16, float* out_f32, int32_t* st_word,
                                    cudaStream_t st) {
  const dim3 grid((H / 8 + kCombineThreads - 1) / kCombineThreads, T);
  return launch_pdl(combine_weighted_kernel, grid, dim3(kCombineThreads), 0, st, yw, inv, T, k, H, R, residual,
                    out_bf16, out_f32, st_word);
}

cudaError_t launch_rmsnorm(const float* x, const float* gamma, float eps, int T, int H, uint16_t* out,
                           uint16_t* raw, cudaStream_t st) {
  return launch_pdl(rmsnorm_kernel, dim3(T), dim3(kNormThreads), 0, st, x, gamma, eps, H, out, raw);
}

cudaError_t launch_recall(const int32_t* pred, const int32_t* ref, int T, int k, int32_t* hits, cudaStream_t st) {
  return launch_pdl(recall_kernel, dim3((T + 7) / 8), dim3(256), 0, st, pred, ref, T, k, hits);
}

}  // namespace moe
