// Internal launchers of libmoe (host side).  Each returns the CUDA error of
// its launch; the extern "C" layer in api.cu validates arguments first.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

int sm_count();

// Raise a kernel's dynamic shared memory limit once per (kernel, device):
// the attribute call is not free, and the limit only ever needs to grow.
cudaError_t ensure_smem_fn(const void* kern, int bytes);
template <typename... KArgs>
cudaError_t ensure_smem(void (*kern)(KArgs...), int bytes) {
  return ensure_smem_fn(reinterpret_cast<const void*>(kern), bytes);
}

// A launch may leave a token on its stream: the address of a buffer it read
// only after its grid-dependency wait and did not write.  Every launch of
// this library clears its stream's token first, so a token seen before a
// launch names the launch right before it.  (Launches outside the library
// do not clear it, but they do not let a later launch start early either.)
void stream_token_set(cudaStream_t st, const void* token);
const void* stream_token_get(cudaStream_t st);
void stream_token_clear(cudaStream_t st);

// Launch with programmatic stream serialization (see pdl_wait in common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  stream_token_clear(st);
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// launch_pdl for a grid of thread-block clusters of the given shape.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, dim3 cluster, size_t smem,
                               cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster.x;
  attr[1].val.clusterDim.y = cluster.y;
  attr[1].val.clusterDim.z = cluster.z;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  stream_token_clear(st);
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// route.cu
cudaError_t launch_router_logits_small(const uint16_t* x, const uint16_t* wr, int T, int H, int E, float* logits,
                                       cudaStream_t st);
cudaError_t launch_topk(const float* logits, const float* bias, int T, int E, int k, int32_t* ids, float* w,
                        float* gap, cudaStream_t st);
cudaError_t launch_route_permute(const uint16_t* x, const uint16_t* wr, const float* bias, int T, int H, int E, int k,
                                 int32_t* ids, float* w, float* gap, int32_t* counts, int32_t* offsets, int32_t* perm,
                                 int32_t* inv, int32_t* st_word, cudaStream_t st);

// route.cu: route sidecar
cudaError_t launch_sidecar_prepare(const uint16_t* w_head, const uint16_t* emb, int E, int r, int L, float* c,
                                   cudaStream_t st);
cudaError_t launch_sidecar_forward(const uint16_t* feat, const uint16_t* w_trunk, const uint16_t* w_head,
                                   const float* c, int T, int F, int r, int E, int L, int N, float* z, int32_t* cand,
                                   float* score, int32_t* st_word, cudaStream_t st);

// cache.cu
cudaError_t launch_cache_plan(const int32_t* counts, int E, int32_t* slot_of, int32_t* expert_of, int S,
                              int32_t* hand, int policy, float decay, float* score, int32_t* last_use,
                              int32_t* miss_list, int32_t* miss_slot, int32_t* stats, int32_t* st_word,
                              cudaStream_t st);
cudaError_t launch_cache_fetch(const void* host_gu, const void* host_dn, size_t rec_gu, size_t rec_dn,
                               const int32_t* miss_list, const int32_t* miss_slot, const int32_t* stats,
                               void* pool_gu, void* pool_dn, cudaStream_t st);

// permute.cu
cudaError_t launch_permute(const int32_t* ids, int R, int k, int E, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* st_word,
                           cudaStream_t st);
size_t permute_chunked_ws_bytes(int R, int E);
cudaError_t launch_permute_chunked(const int32_t* ids, int R, int E, int32_t* counts, int32_t* offsets,
                                   int32_t* perm, int32_t* inv, int32_t* ws, int32_t* st_word,
                                   cudaStream_t st);
cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* perm, const int32_t* inv, int R, int k, int T,
                               int H, uint16_t* x_perm, const int32_t* st_word, cudaStream_t st);

// gemm.cu (tcgen05 grouped GEMM)
enum class GemmKind { kGateUp = 0, kDown = 1, kRouter = 2 };

// gemm.cu: the int4 GEMV (decode-sized launches only) over a pool of S
// tile-packed int4 records, expert e read from record slot_of[e];
// cudaErrorNotSupported for launches the GEMV does not take
namespace gk {
cudaError_t launch_int4_slots(int kind, const uint16_t* rows, const int32_t* offsets, int E, int R, int H, int I,
                              const void* pool, int S, const int32_t* slot_of, void* out, int32_t* st_word,
                              cudaStream_t st);
// ... its gate/up launch fetching the planned misses' records (both
// components) from host memory while the resident experts compute
cudaError_t launch_int4_fetch(const uint16_t* rows, const int32_t* offsets, int E, int R, int H, int I, void* pool_gu,
                              void* pool_dn, int S, const int32_t* slot_of, const void* host_gu, const void* host_dn,
                              const int32_t* miss_list, const int32_t* miss_slot, const int32_t* stats, uint16_t* h,
                              int32_t* fsync, int32_t* st_word, cudaStream_t st);
}
// Grouped weight-stationary GEMM: for every (segment e, 128-row weight block,
// chunk of token rows) tile, D = W_e[rows] . B[rows of segment]^T on the
// tensor cores; epilogue per kind.  Returns cudaErrorInvalidValue when a
// tensor map cannot be encoded.
cudaError_t launch_grouped_gemm(GemmKind kind, int fmt, const void* w, const uint16_t* scales,
                                const uint16_t* b_rows, const int32_t* offsets, int E, int R, int H, int I,
                                int router_E, void* out, int32_t* st_word, cudaStream_t st);

// pack.cu
size_t packed_component_bytes(int fmt_tiled, int E, int H, int I, int which);
cudaError_t launch_pack(int fmt_in, const void* w, const uint16_t* s, int E, int H, int I, int which, void* out,
                        cudaStream_t st);

// Gate/up + SwiGLU + down in one persistent launch (tile-packed bf16).
// With x set, the launch first gathers x_perm[s] = x[perm[s] / k] itself.
// With cache set, w_gateup / w_down are slot pools read through slot_of;
// with cache->host_gu also set, the launch fetches the planned misses itself.
struct FusedCache {
  const int32_t* slot_of;
  int S;
  const void* host_gu;
  const void* host_dn;
  const int32_t* miss_list;
  const int32_t* miss_slot;
  const int32_t* stats;
  int wave;
};
cudaError_t launch_swiglu_fused(const uint16_t* x, int k, const int32_t* perm, uint16_t* x_perm,
                                const int32_t* offsets, int E, int R, int H, int I, const void* w_gateup,
                                const void* w_down, const FusedCache* cache, uint16_t* h, float* y,
                                const float* topk_w, uint16_t* yw, int32_t* ready, int32_t* st_word,
                                cudaStream_t st);

// combine.cu
cudaError_t launch_combine(const float* y, const int32_t* inv, const float* w, int T, int k, int H,
                           int R, const float* residual, uint16_t* out_bf16, float* out_f32,
                           int32_t* st_word, cudaStream_t st);
cudaError_t launch_combine_weighted(const uint16_t* yw, const int32_t* inv, int T, int k, int H, int R,
                                    const float* residual, uint16_t* out_bf16, float* out_f32, int32_t* st_word,
                                    cudaStream_t st);
cudaError_t launch_rmsnorm(const float* x, const float* gamma, float eps, int T, int H,
                           uint16_t* out, uint16_t* raw, cudaStream_t st);
cudaError_t launch_recall(const int32_t* pred, const int32_t* ref, int T, int k, int32_t* hits,
                          cudaStream_t st);

// dedup.cu
cudaError_t launch_dedup(const int32_t* ids, int L, int Ttot, int k, int E, int B, long long P,
                         uint32_t* mask, int32_t* U, int64_t* bytes2, int64_t* bytes4,
                         int32_t* st_word, cudaStream_t st);

}  // namespace moe
