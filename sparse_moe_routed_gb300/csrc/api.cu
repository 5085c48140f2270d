// extern "C" boundary of libmoe: host-side admission of every argument, then
// the kernel launches on the caller's stream.  Nothing is enqueued and nothing
// is written unless every check passes (AFN-010 "One bank flip is enough:
// make the whole inference chunk transactional", section "The publication
// model": output stays caller-private while work is fallible; AFN-001, section
// "Phase 3: reject before the GPU exists": admission happens before any GPU
// work).  Declarations and argument contracts: include/moe.h.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/moe.h"
#include "common.cuh"
#include "launch.h"

namespace moe {

int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (dev < 0 || dev >= 64) return -1;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

cudaError_t ensure_smem_fn(const void* kern, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  int& have = done[std::make_pair(kern, dev)];
  if (have >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}

// The token each stream's last launch left (see launch.h), per device.
namespace {
std::mutex g_token_mu;
std::map<std::pair<int, cudaStream_t>, const void*> g_token;
std::pair<int, cudaStream_t> token_key(cudaStream_t st) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  return std::make_pair(dev, st);
}
}  // namespace

void stream_token_set(cudaStream_t st, const void* token) {
  std::lock_guard<std::mutex> lock(g_token_mu);
  g_token[token_key(st)] = token;
}

const void* stream_token_get(cudaStream_t st) {
  std::lock_guard<std::mutex> lock(g_token_mu);
  const auto it = g_token.find(token_key(st));
  return it == g_token.end() ? nullptr : it->second;
}

void stream_token_clear(cudaStream_t st) {
  std::lock_guard<std::mutex> lock(g_token_mu);
  const auto it = g_token.find(token_key(st));
  if (it != g_token.end()) it->second = nullptr;
}

}  // namespace moe

namespace {

inline bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool a4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline bool a8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

inline moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ECUDA; }

// Geometry envelope shared by the layer calls.
inline moe_status check_geometry(int H, int E, int k, int I_or_zero) {
  if (H <= 0 || E <= 0 || k <= 0 || I_or_zero < 0) return MOE_ESHAPE;
  if (k > moe::kMaxK || k > E || E > moe::kMaxE) return MOE_ENOTSUP;
  if (H % 128 != 0 || H > 16384) return MOE_ENOTSUP;
  if (I_or_zero > 0 && (I_or_zero % 64 != 0 || I_or_zero > 16384)) return MOE_ENOTSUP;
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_abi_version(void) { return 104; }

const char* moe_status_str(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_EINVAL: return "MOE_EINVAL: null or misaligned pointer, or bad enum";
    case MOE_ESHAPE: return "MOE_ESHAPE: inconsistent or non-positive sizes";
    case MOE_ERANGE: return "MOE_ERANGE: value out of range";
    case MOE_ECUDA: return "MOE_ECUDA: a CUDA call failed";
    case MOE_ENOTSUP: return "MOE_ENOTSUP: geometry outside the supported envelope";
    case MOE_EDEVICE_TIMEOUT: return "MOE_EDEVICE_TIMEOUT: a bounded device wait ran out";
    case MOE_EWORKSPACE: return "MOE_EWORKSPACE: workspace missing or too small";
  }
  return "MOE_UNKNOWN";
}

int moe_device_sm_count(void) { return moe::sm_count(); }

size_t moe_route_workspace_size(int T, int E) {
  if (T <= 0 || E <= 0) return 0;
  const size_t logits = static_cast<size_t>(T) * static_cast<size_t>(E) * sizeof(float);
  return (logits + 255) & ~static_cast<size_t>(255);
}

moe_status moe_route(const uint16_t* x, const uint16_t* w_router, const float* bias, int T, int H, int E, int k,
                     int32_t* topk_ids, float* topk_w, float* gap, void* workspace, size_t workspace_bytes,
                     void* stream) {
  if (T < 0) return MOE_ESHAPE;
  moe_status g = check_geometry(H, E, k, 0);
  if (g != MOE_OK) return g;
  if (static_cast<long long>(T) * k >= (1LL << 31)) return MOE_ENOTSUP;
  if (!x || !w_router || !topk_ids || !topk_w) return MOE_EINVAL;
  if (!a16(x) || !a16(w_router) || !a4(topk_ids) || !a4(topk_w)) return MOE_EINVAL;
  if ((bias && !a4(bias)) || (gap && !a4(gap))) return MOE_EINVAL;
  if (T == 0) return MOE_OK;
  if (!workspace || !a16(workspace)) return workspace ? MOE_EINVAL : MOE_EWORKSPACE;
  if (workspace_bytes < moe_route_workspace_size(T, E)) return MOE_EWORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* logits = static_cast<float*>(workspace);
  cudaError_t e;
  if (T > 64 && E % 128 == 0)
    e = moe::launch_grouped_gemm(moe::GemmKind::kRouter, MOE_W_BF16, w_router, nullptr, x, nullptr, 1, T, H, 0, E,
                                 logits, nullptr, st);
  else
    e = moe::launch_router_logits_small(x, w_router, T, H, E, logits, st);
  if (e != cudaSuccess) return MOE_ECUDA;
  return cuda_status(moe::launch_topk(logits, bias, T, E, k, topk_ids, topk_w, gap, st));
}

moe_status moe_route_permute(const uint16_t* x, const uint16_t* w_router, const float* bias, int T, int H, int E,
                             int k, int32_t* topk_ids, float* topk_w, float* gap, int32_t* counts, int32_t* offsets,
                             int32_t* perm, int32_t* inv_perm, int32_t* dev_status, void* stream) {
  if (T < 0) return MOE_ESHAPE;
  moe_status g = check_geometry(H, E, k, 0);
  if (g != MOE_OK) return g;
  if (T > 16) return MOE_ENOTSUP;
  if (!x || !w_router || !topk_ids || !topk_w || !counts || !offsets || !perm || !inv_perm || !dev_status)
    return MOE_EINVAL;
  if (!a16(x) || !a16(w_router) || !a4(topk_ids) || !a4(topk_w) || !a4(counts) || !a4(offsets) || !a4(perm) ||
      !a4(inv_perm) || !a4(dev_status))
    return MOE_EINVAL;
  if ((bias && !a4(bias)) || (gap && !a4(gap))) return MOE_EINVAL;
  if (T == 0) return MOE_OK;
  const cudaError_t e = moe::launch_route_permute(x, w_router, bias, T, H, E, k, topk_ids, topk_w, gap, counts,
                                                  offsets, perm, inv_perm, dev_status,
                                                  static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return MOE_ENOTSUP;
  return cuda_status(e);
}

moe_status moe_permute(const int32_t* topk_ids, int T, int k, int E, const uint16_t* x, int H, int32_t* counts,
                       int32_t* offsets, int32_t* perm, int32_t* inv_perm, uint16_t* x_perm, int32_t* dev_status,
                       void* stream) {
  if (T < 0 || k <= 0 || E <= 0) return MOE_ESHAPE;
  if (k > moe::kMaxK || k > E || E > moe::kMaxE) return MOE_ENOTSUP;
  if (static_cast<long long>(T) * k >= (1LL << 31)) return MOE_ENOTSUP;
  if (!topk_ids || !counts || !offsets || !perm || !inv_perm || !dev_status) return MOE_EINVAL;
  if (!a4(topk_ids) || !a4(counts) || !a4(offsets) || !a4(perm) || !a4(inv_perm) || !a4(dev_status))
    return MOE_EINVAL;
  if (x_perm) {
    if (!x) return MOE_EINVAL;
    if (H <= 0) return MOE_ESHAPE;
    if (H % 128 != 0 || H > 16384) return MOE_ENOTSUP;
    if (!a16(x) || !a16(x_perm)) return MOE_EINVAL;
  }
  if (T == 0) return MOE_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int R = T * k;
  cudaError_t e = moe::launch_permute(topk_ids, R, k, E, counts, offsets, perm, inv_perm, dev_status, st);
  if (e != cudaSuccess) return MOE_ECUDA;
  if (x_perm) {
    e = moe::launch_gather_rows(x, perm, inv_perm, R, k, T, H, x_perm, dev_status, st);
    if (e != cudaSuccess) return MOE_ECUDA;
    // the row gather neither writes the offsets nor starts before they are
    // complete: the contraction after it may read them at its start
    moe::stream_token_set(st, offsets);
  }
  return MOE_OK;
}

size_t moe_permute_workspace_size(int T, int k, int E) {
  if (T <= 0 || k <= 0 || E <= 0) return 0;
  return moe::permute_chunked_ws_bytes(T * k, E);
}

moe_status moe_permute_ws(const int32_t* topk_ids, int T, int k, int E, const uint16_t* x, int H, int32_t* counts,
                          int32_t* offsets, int32_t* perm, int32_t* inv_perm, uint16_t* x_perm, void* workspace,
                          size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (T < 0 || k <= 0 || E <= 0) return MOE_ESHAPE;
  if (k > moe::kMaxK || k > E || E > moe::kMaxE) return MOE_ENOTSUP;
  if (static_cast<long long>(T) * k >= (1LL << 31)) return MOE_ENOTSUP;
  if (!topk_ids || !counts || !offsets || !perm || !inv_perm || !dev_status) return MOE_EINVAL;
  if (!a4(topk_ids) || !a4(counts) || !a4(offsets) || !a4(perm) || !a4(inv_perm) || !a4(dev_status))
    return MOE_EINVAL;
  if (x_perm) {
    if (!x) return MOE_EINVAL;
    if (H <= 0) return MOE_ESHAPE;
    if (H % 128 != 0 || H > 16384) return MOE_ENOTSUP;
    if (!a16(x) || !a16(x_perm)) return MOE_EINVAL;
  }
  if (T == 0) return MOE_OK;
  if (!workspace || !a16(workspace)) return workspace ? MOE_EINVAL : MOE_EWORKSPACE;
  if (workspace_bytes < moe_permute_workspace_size(T, k, E)) return MOE_EWORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int R = T * k;
  cudaError_t e = moe::launch_permute_chunked(topk_ids, R, E, counts, offsets, perm, inv_perm,
                                              static_cast<int32_t*>(workspace), dev_status, st);
  if (e != cudaSuccess) return MOE_ECUDA;
  if (x_perm) {
    e = moe::launch_gather_rows(x, perm, inv_perm, R, k, T, H, x_perm, dev_status, st);
    if (e != cudaSuccess) return MOE_ECUDA;
    // the row gather neither writes the offsets nor starts before they are
    // complete: the contraction after it may read them at its start
    moe::stream_token_set(st, offsets);
  }
  return MOE_OK;
}

static moe_status check_expert_args(int R, int E, int H, int I, int fmt) {
  if (R < 0 || E <= 0 || H <= 0 || I <= 0) return MOE_ESHAPE;
  if (fmt != MOE_W_BF16 && fmt != MOE_W_INT4_G64 && fmt != MOE_W_BF16_TILED && fmt != MOE_W_INT4_G64_TILED)
    return MOE_EINVAL;
  if (fmt == MOE_W_INT4_G64) return MOE_ENOTSUP;  // plain int4 records are packed first
  if (E > moe::kMaxE) return MOE_ENOTSUP;
  if (H % 128 != 0 || H > 16384 || I % 64 != 0 || I > 16384) return MOE_ENOTSUP;
  if (static_cast<long long>(E) * H >= (1LL << 31)) return MOE_ENOTSUP;
  return MOE_OK;
}

// The contraction takes weights only: every format carries its scales
// inside the (packed) record.
static bool scales_ok(int fmt, const uint16_t* s) {
  (void)fmt;
  return s == nullptr;
}

moe_status moe_expert_gateup(const uint16_t* x_perm, const int32_t* offsets, int R, int E, int H, int I, int fmt,
                             const void* w_gateup, const uint16_t* s_gateup, uint16_t* h, int32_t* dev_status,
                             void* stream) {
  moe_status c = check_expert_args(R, E, H, I, fmt);
  if (c != MOE_OK) return c;
  if (!x_perm || !offsets || !w_gateup || !h || !dev_status) return MOE_EINVAL;
  if (!scales_ok(fmt, s_gateup)) return MOE_EINVAL;
  if (!a16(x_perm) || !a16(w_gateup) || !a16(h) || !a4(offsets) || !a4(dev_status)) return MOE_EINVAL;
  if (R == 0) return MOE_OK;
  cudaError_t e = moe::launch_grouped_gemm(moe::GemmKind::kGateUp, fmt, w_gateup, s_gateup, x_perm, offsets, E, R, H,
                                           I, 0, h, dev_status, static_cast<cudaStream_t>(stream));
  return cuda_status(e);
}

moe_status moe_expert_down(const uint16_t* h, const int32_t* offsets, int R, int E, int H, int I, int fmt,
                           const void* w_down, const uint16_t* s_down, float* y_perm, int32_t* dev_status,
                           void* stream) {
  moe_status c = check_expert_args(R, E, H, I, fmt);
  if (c != MOE_OK) return c;
  if (!h || !offsets || !w_down || !y_perm || !dev_status) return MOE_EINVAL;
  if (!scales_ok(fmt, s_down)) return MOE_EINVAL;
  if (!a16(h) || !a16(w_down) || !a16(y_perm) || !a4(offsets) || !a4(dev_status)) return MOE_EINVAL;
  if (R == 0) return MOE_OK;
  cudaError_t e = moe::launch_grouped_gemm(moe::GemmKind::kDown, fmt, w_down, s_down, h, offsets, E, R, H, I, 0,
                                           y_perm, dev_status, static_cast<cudaStream_t>(stream));
  return cuda_status(e);
}

moe_status moe_expert_int4_slots(int kind, const uint16_t* rows, const int32_t* offsets, int R, int E, int H, int I,
                                 const void* pool, int S, const int32_t* slot_of, void* out, int32_t* dev_status,
                                 void* stream) {
  if (kind != 0 && kind != 1) return MOE_EINVAL;
  moe_status c = check_expert_args(R, E, H, I, MOE_W_INT4_G64_TILED);
  if (c != MOE_OK) return c;
  if (S <= 0) return MOE_ESHAPE;
  if (S > moe::kMaxE) return MOE_ENOTSUP;
  if (!rows || !offsets || !pool || !slot_of || !out || !dev_status) return MOE_EINVAL;
  if (!a16(rows) || !a16(pool) || !a16(out) || !a4(offsets) || !a4(slot_of) || !a4(dev_status)) return MOE_EINVAL;
  if (R == 0) return MOE_OK;
  const cudaError_t e = moe::gk::launch_int4_slots(kind, rows, offsets, E, R, H, I, pool, S, slot_of, out, dev_status,
                                                   static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return MOE_ENOTSUP;
  return cuda_status(e);
}

moe_status moe_expert_int4_fetch(const uint16_t* x_perm, const int32_t* offsets, int R, int E, int H, int I,
                                 void* pool_gateup, void* pool_down, int S, const int32_t* slot_of,
                                 const void* host_gateup, const void* host_down, const int32_t* miss_list,
                                 const int32_t* miss_slot, const int32_t* stats, uint16_t* h, int32_t* sync_ws,
                                 int32_t* dev_status, void* stream) {
  moe_status c = check_expert_args(R, E, H, I, MOE_W_INT4_G64_TILED);
  if (c != MOE_OK) return c;
  if (S <= 0) return MOE_ESHAPE;
  if (S > moe::kMaxE) return MOE_ENOTSUP;
  if (!x_perm || !offsets || !pool_gateup || !pool_down || !slot_of || !host_gateup || !host_down || !miss_list ||
      !miss_slot || !stats || !h || !dev_status)
    return MOE_EINVAL;
  if (!sync_ws) return MOE_EWORKSPACE;
  if (!a16(x_perm) || !a16(pool_gateup) || !a16(pool_down) || !a16(host_gateup) || !a16(host_down) || !a16(h) ||
      !a4(offsets) || !a4(slot_of) || !a4(miss_list) || !a4(miss_slot) || !a4(stats) || !a4(sync_ws) ||
      !a4(dev_status))
    return MOE_EINVAL;
  if (R == 0) return MOE_OK;
  const cudaError_t e = moe::gk::launch_int4_fetch(x_perm, offsets, E, R, H, I, pool_gateup, pool_down, S, slot_of,
                                                   host_gateup, host_down, miss_list, miss_slot, stats, h, sync_ws,
                                                   dev_status, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return MOE_ENOTSUP;
  return cuda_status(e);
}

moe_status moe_grouped_swiglu(const uint16_t* x_perm, const int32_t* offsets, int R, int E, int H, int I, int fmt,
                              const void* w_gateup, const uint16_t* s_gateup, const void* w_down,
                              const uint16_t* s_down, uint16_t* h, float* y_perm, int32_t* dev_status,
                              void* stream) {
  moe_status c = check_expert_args(R, E, H, I, fmt);
  if (c != MOE_OK) return c;
  if (!x_perm || !offsets || !w_gateup || !w_down || !h || !y_perm || !dev_status) return MOE_EINVAL;
  if (!scales_ok(fmt, s_gateup) || !scales_ok(fmt, s_down)) return MOE_EINVAL;
  if (!a16(x_perm) || !a16(w_gateup) || !a16(w_down) || !a16(h) || !a16(y_perm) || !a4(offsets) ||
      !a4(dev_status))
    return MOE_EINVAL;
  if (R == 0) return MOE_OK;
  c = moe_expert_gateup(x_perm, offsets, R, E, H, I, fmt, w_gateup, s_gateup, h, dev_status, stream);
  if (c != MOE_OK) return c;
  return moe_expert_down(h, offsets, R, E, H, I, fmt, w_down, s_down, y_perm, dev_status, stream);
}

static moe_status check_fused(const uint16_t* x, int k, const int32_t* perm, uint16_t* x_perm,
                              const int32_t* offsets, int R, int E, int H, int I, int fmt, const void* w_gateup,
                              const void* w_down, uint16_t* h, float* y_perm, int32_t* sync_ws,
                              int32_t* dev_status) {
  moe_status c = check_expert_args(R, E, H, I, fmt);
  if (c != MOE_OK) return c;
  if (fmt != MOE_W_BF16_TILED) return MOE_ENOTSUP;
  if (!x_perm || !offsets || !w_gateup || !w_down || !h || !y_perm || !dev_status) return MOE_EINVAL;
  if (!sync_ws) return MOE_EWORKSPACE;
  if (!a16(x_perm) || !a16(w_gateup) || !a16(w_down) || !a16(h) || !a16(y_perm) || !a4(offsets) ||
      !a4(dev_status) || !a4(sync_ws))
    return MOE_EINVAL;
  if (x) {  // gather in the same launch
    if (k <= 0 || R % k != 0) return MOE_ESHAPE;
    if (k > moe::kMaxK) return MOE_ENOTSUP;
    if (!perm || !a16(x) || !a4(perm)) return MOE_EINVAL;
  }
  return MOE_OK;
}

moe_status moe_expert_swiglu_fused(const uint16_t* x, int k, const int32_t* perm, uint16_t* x_perm,
                                   const int32_t* offsets, int R, int E, int H, int I, int fmt, const void* w_gateup,
                                   const void* w_down, uint16_t* h, float* y_perm, int32_t* sync_ws,
                                   int32_t* dev_status, void* stream) {
  const moe_status c =
      check_fused(x, k, perm, x_perm, offsets, R, E, H, I, fmt, w_gateup, w_down, h, y_perm, sync_ws, dev_status);
  if (c != MOE_OK) return c;
  if (R == 0) return MOE_OK;
  return cuda_status(moe::launch_swiglu_fused(x, k, perm, x_perm, offsets, E, R, H, I, w_gateup, w_down, nullptr, h,
                                              y_perm, nullptr, nullptr, sync_ws, dev_status,
                                              static_cast<cudaStream_t>(stream)));
}

moe_status moe_expert_swiglu_fused_weighted(const uint16_t* x, int k, const int32_t* perm, uint16_t* x_perm,
                                            const int32_t* offsets, int R, int E, int H, int I, int fmt,
                                            const void* w_gateup, const void* w_down, const float* topk_w,
                                            uint16_t* h, uint16_t* yw_perm, int32_t* sync_ws, int32_t* dev_status,
                                            void* stream) {
  // yw_perm stands in for y_perm in the shared checks (same alignment rule)
  const moe_status c = check_fused(x, k, perm, x_perm, offsets, R, E, H, I, fmt, w_gateup, w_down, h,
                                   reinterpret_cast<float*>(yw_perm), sync_ws, dev_status);
  if (c != MOE_OK) return c;
  if (k <= 0 || R % k != 0) return MOE_ESHAPE;
  if (k > moe::kMaxK) return MOE_ENOTSUP;
  if (!perm || !topk_w || !a4(perm) || !a4(topk_w)) return MOE_EINVAL;
  if (R == 0) return MOE_OK;
  return cuda_status(moe::launch_swiglu_fused(x, k, perm, x_perm, offsets, E, R, H, I, w_gateup, w_down, nullptr, h,
                                              nullptr, topk_w, yw_perm, sync_ws, dev_status,
                                              static_cast<cudaStream_t>(stream)));
}

moe_status moe_expert_swiglu_cached(const uint16_t* x, int k, const int32_t* perm, uint16_t* x_perm,
                                    const int32_t* offsets, int R, int E, int H, int I, int fmt, void* pool_gateup,
                                    void* pool_down, int S, const int32_t* slot_of, const void* host_gateup,
                                    const void* host_down, const int32_t* miss_list, const int32_t* miss_slot,
                                    const int32_t* stats, int wave, uint16_t* h, float* y_perm, int32_t* sync_ws,
                                    int32_t* dev_status, void* stream) {
  const moe_status c = check_fused(x, k, perm, x_perm, offsets, R, E, H, I, fmt, pool_gateup, pool_down, h, y_perm,
                                   sync_ws, dev_status);
  if (c != MOE_OK) return c;
  if (S <= 0) return MOE_ESHAPE;
  if (S > 1024) return MOE_ENOTSUP;
  if (!slot_of || !a4(slot_of)) return MOE_EINVAL;
  if ((H / 64) % 2 != 0 || (I / 64) % 2 != 0) return MOE_ENOTSUP;
  const bool fetch = host_gateup != nullptr;
  if (fetch) {
    if (wave <= 0) return MOE_ESHAPE;
    if (!host_down || !miss_list || !miss_slot || !stats) return MOE_EINVAL;
    if (!a16(host_gateup) || !a16(host_down) || !a4(miss_list) || !a4(miss_slot) || !a4(stats)) return MOE_EINVAL;
  }
  if (R == 0) return MOE_OK;
  moe::FusedCache fc{};
  fc.slot_of = slot_of;
  fc.S = S;
  if (fetch) {
    fc.host_gu = host_gateup;
    fc.host_dn = host_down;
    fc.miss_list = miss_list;
    fc.miss_slot = miss_slot;
    fc.stats = stats;
    fc.wave = wave;
  }
  return cuda_status(moe::launch_swiglu_fused(x, k, perm, x_perm, offsets, E, R, H, I, pool_gateup, pool_down, &fc,
                                              h, y_perm, nullptr, nullptr, sync_ws, dev_status,
                                              static_cast<cudaStream_t>(stream)));
}

moe_status moe_cache_plan(const int32_t* counts, int E, int32_t* slot_of, int32_t* expert_of, int S, int32_t* hand,
                          int policy, float decay, float* score, int32_t* last_use, int32_t* miss_list,
                          int32_t* miss_slot, int32_t* stats, int32_t* dev_status, void* stream) {
  if (E <= 0 || S <= 0) return MOE_ESHAPE;
  if (E > moe::kMaxE || S > 1024) return MOE_ENOTSUP;
  if (policy != MOE_CACHE_FIFO && policy != MOE_CACHE_LRU && policy != MOE_CACHE_SCORE) return MOE_EINVAL;
  if (!counts || !slot_of || !expert_of || !hand || !miss_list || !miss_slot || !stats || !dev_status)
    return MOE_EINVAL;
  if (!a4(counts) || !a4(slot_of) || !a4(expert_of) || !a4(hand) || !a4(miss_list) || !a4(miss_slot) || !a4(stats) ||
      !a4(dev_status))
    return MOE_EINVAL;
  if (policy == MOE_CACHE_LRU && (!last_use || !a4(last_use))) return MOE_EINVAL;
  if (policy == MOE_CACHE_SCORE) {
    if (!score || !a4(score)) return MOE_EINVAL;
    if (!(decay >= 0.0f && decay < 1.0f)) return MOE_ERANGE;
  }
  return cuda_status(moe::launch_cache_plan(counts, E, slot_of, expert_of, S, hand, policy, decay, score, last_use,
                                            miss_list, miss_slot, stats, dev_status,
                                            static_cast<cudaStream_t>(stream)));
}

moe_status moe_cache_fetch(const void* host_gateup, const void* host_down, size_t rec_gateup, size_t rec_down,
                           const int32_t* miss_list, const int32_t* miss_slot, const int32_t* stats, void* pool_gateup,
                           void* pool_down, void* stream) {
  if (rec_gateup == 0 || rec_down == 0 || rec_gateup % 16 != 0 || rec_down % 16 != 0) return MOE_ESHAPE;
  if (!host_gateup || !host_down || !miss_list || !miss_slot || !stats || !pool_gateup || !pool_down)
    return MOE_EINVAL;
  if (!a16(host_gateup) || !a16(host_down) || !a16(pool_gateup) || !a16(pool_down) || !a4(miss_list) ||
      !a4(miss_slot) || !a4(stats))
    return MOE_EINVAL;
  return cuda_status(moe::launch_cache_fetch(host_gateup, host_down, rec_gateup, rec_down, miss_list, miss_slot,
                                             stats, pool_gateup, pool_down, static_cast<cudaStream_t>(stream)));
}

moe_status moe_layer_stream(const void* host_gateup, const void* host_down, size_t bytes_gateup, size_t bytes_down,
                            void* dev_gateup, void* dev_down, void* stream) {
  if (bytes_gateup == 0 && bytes_down == 0) return MOE_OK;
  if (bytes_gateup % 16 != 0 || bytes_down % 16 != 0) return MOE_ESHAPE;
  if ((bytes_gateup && (!host_gateup || !dev_gateup)) || (bytes_down && (!host_down || !dev_down))) return MOE_EINVAL;
  if (!a16(host_gateup) || !a16(host_down) || !a16(dev_gateup) || !a16(dev_down)) return MOE_EINVAL;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // one copy per component, on the copy engines: no SM time taken from the
  // contraction that runs meanwhile
  if (bytes_gateup) {
    const cudaError_t e = cudaMemcpyAsync(dev_gateup, host_gateup, bytes_gateup, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return MOE_ECUDA;
  }
  if (bytes_down) {
    const cudaError_t e = cudaMemcpyAsync(dev_down, host_down, bytes_down, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return MOE_ECUDA;
  }
  return MOE_OK;
}

int moe_stream_mode(int U, int E, double record_bytes, double selected_gbs, double layer_gbs,
                    double selected_overhead_us, double* t_selected_us, double* t_layer_us) {
  if (U < 0 || E <= 0 || U > E || !(record_bytes > 0.0) || !(selected_gbs > 0.0) || !(layer_gbs > 0.0) ||
      !(selected_overhead_us >= 0.0))
    return -1;
  const double ts = U > 0 ? selected_overhead_us + U * record_bytes / (selected_gbs * 1e3) : 0.0;
  const double tl = E * record_bytes / (layer_gbs * 1e3);
  if (t_selected_us) *t_selected_us = ts;
  if (t_layer_us) *t_layer_us = tl;
  return tl < ts ? MOE_STREAM_LAYER : MOE_STREAM_SELECTED;
}

moe_status moe_sidecar_prepare(const uint16_t* w_head, const uint16_t* layer_emb, int E, int r, int L,
                               float* head_bias, void* stream) {
  if (E <= 0 || r <= 0 || L <= 0) return MOE_ESHAPE;
  if (E > 1024 || r > 1024 || r % 8 != 0 || L > 65535) return MOE_ENOTSUP;
  if (!w_head || !layer_emb || !head_bias) return MOE_EINVAL;
  if (!a16(w_head) || !a4(head_bias) || (reinterpret_cast<uintptr_t>(layer_emb) & 1u)) return MOE_EINVAL;
  return cuda_status(moe::launch_sidecar_prepare(w_head, layer_emb, E, r, L, head_bias,
                                                 static_cast<cudaStream_t>(stream)));
}

moe_status moe_sidecar_forward(const uint16_t* feat, const uint16_t* w_trunk, const uint16_t* w_head,
                               const float* head_bias, int T, int F, int r, int E, int L, int N, float* z,
                               int32_t* cand, float* cand_score, int32_t* dev_status, void* stream) {
  if (T < 0 || F <= 0 || r <= 0 || E <= 0 || L <= 0 || N <= 0) return MOE_ESHAPE;
  if (F % 128 != 0 || F > 16384 || r % 8 != 0 || r > 1024 || E > 1024 || L > 65535 || N > 32 || N > E)
    return MOE_ENOTSUP;
  if (!feat || !w_trunk || !w_head || !head_bias || !z || !cand || !cand_score || !dev_status) return MOE_EINVAL;
  if (!a16(feat) || !a16(w_trunk) || !a16(w_head) || !a4(head_bias) || !a4(z) || !a4(cand) || !a4(cand_score) ||
      !a4(dev_status))
    return MOE_EINVAL;
  if (T == 0) return MOE_OK;
  return cuda_status(moe::launch_sidecar_forward(feat, w_trunk, w_head, head_bias, T, F, r, E, L, N, z, cand,
                                                 cand_score, dev_status, static_cast<cudaStream_t>(stream)));
}

size_t moe_pack_size(int fmt_in, int E, int H, int I, int which) {
  if (E <= 0 || H <= 0 || I <= 0 || (which != 0 && which != 1)) return 0;
  if (H % 128 != 0 || I % 64 != 0) return 0;
  if (fmt_in == MOE_W_BF16) return moe::packed_component_bytes(MOE_W_BF16_TILED, E, H, I, which);
  if (fmt_in == MOE_W_INT4_G64) return moe::packed_component_bytes(MOE_W_INT4_G64_TILED, E, H, I, which);
  return 0;
}

moe_status moe_pack_experts(int fmt_in, const void* w, const uint16_t* s, int E, int H, int I, int which, void* out,
                            size_t out_bytes, void* stream) {
  if (E <= 0 || H <= 0 || I <= 0) return MOE_ESHAPE;
  if (which != 0 && which != 1) return MOE_EINVAL;
  if (fmt_in != MOE_W_BF16 && fmt_in != MOE_W_INT4_G64) return MOE_EINVAL;
  if (E > moe::kMaxE || H % 128 != 0 || H > 16384 || I % 64 != 0 || I > 16384) return MOE_ENOTSUP;
  if (!w || !out || !a16(w) || !a16(out)) return MOE_EINVAL;
  if (fmt_in == MOE_W_INT4_G64 ? (!s || !a4(s)) : (s != nullptr)) return MOE_EINVAL;
  const size_t need = moe_pack_size(fmt_in, E, H, I, which);
  if (out_bytes < need) return MOE_EWORKSPACE;
  return cuda_status(moe::launch_pack(fmt_in, w, s, E, H, I, which, out, static_cast<cudaStream_t>(stream)));
}

moe_status moe_combine(const float* y_perm, const int32_t* inv_perm, const float* topk_w, int T, int k, int H,
                       const float* residual, uint16_t* out_bf16, float* out_f32, int32_t* dev_status,
                       void* stream) {
  if (T < 0 || k <= 0 || H <= 0) return MOE_ESHAPE;
  if (k > moe::kMaxK || H % 128 != 0 || H > 16384) return MOE_ENOTSUP;
  if (static_cast<long long>(T) * k >= (1LL << 31)) return MOE_ENOTSUP;
  if (!y_perm || !inv_perm || !topk_w || (!out_bf16 && !out_f32)) return MOE_EINVAL;
  if (!a16(y_perm) || !a4(inv_perm) || !a4(topk_w)) return MOE_EINVAL;
  if ((residual && !a16(residual)) || (out_bf16 && !a16(out_bf16)) || (out_f32 && !a16(out_f32)) ||
      (dev_status && !a4(dev_status)))
    return MOE_EINVAL;
  if (T == 0) return MOE_OK;
  return cuda_status(moe::launch_combine(y_perm, inv_perm, topk_w, T, k, H, T * k, residual, out_bf16, out_f32,
                                         dev_status, static_cast<cudaStream_t>(stream)));
}

moe_status moe_combine_weighted(const uint16_t* yw_perm, const int32_t* inv_perm, int T, int k, int H,
                                const float* residual, uint16_t* out_bf16, float* out_f32, int32_t* dev_status,
                                void* stream) {
  if (T < 0 || k <= 0 || H <= 0) return MOE_ESHAPE;
  if (k > moe::kMaxK || H % 128 != 0 || H > 16384) return MOE_ENOTSUP;
  if (static_cast<long long>(T) * k >= (1LL << 31)) return MOE_ENOTSUP;
  if (!yw_perm || !inv_perm || (!out_bf16 && !out_f32)) return MOE_EINVAL;
  if (!a16(yw_perm) || !a4(inv_perm)) return MOE_EINVAL;
  if ((residual && !a16(residual)) || (out_bf16 && !a16(out_bf16)) || (out_f32 && !a16(out_f32)) ||
      (dev_status && !a4(dev_status)))
    return MOE_EINVAL;
  if (T == 0) return MOE_OK;
  return cuda_status(moe::launch_combine_weighted(yw_perm, inv_perm, T, k, H, T * k, residual, out_bf16, out_f32,
                                                  dev_status, static_cast<cudaStream_t>(stream)));
}

moe_status route_block_dedup(const int32_t* ids, int L, int T_tot, int k, int E, int block, int H, int I,
                             uint32_t* mask, int32_t* U, int64_t* bytes2, int64_t* bytes4, int32_t* dev_status,
                             void* stream) {
  if (L <= 0 || T_tot < 0 || k <= 0 || E <= 0 || block <= 0 || H <= 0 || I <= 0) return MOE_ESHAPE;
  if (k > moe::kMaxK || E > moe::kMaxE) return MOE_ENOTSUP;
  if (static_cast<long long>(L) * T_tot * k >= (1LL << 31)) return MOE_ENOTSUP;
  if (!ids || !mask || !U || !bytes2 || !bytes4 || !dev_status) return MOE_EINVAL;
  if (!a4(ids) || !a4(mask) || !a4(U) || !a8(bytes2) || !a8(bytes4) || !a4(dev_status)) return MOE_EINVAL;
  if (T_tot == 0) return MOE_OK;
  const long long P = 3LL * H * I;
  return cuda_status(moe::launch_dedup(ids, L, T_tot, k, E, block, P, mask, U, bytes2, bytes4, dev_status,
                                       static_cast<cudaStream_t>(stream)));
}

moe_status moe_rmsnorm(const float* x, const float* gamma, float eps, int T, int H, uint16_t* out,
                       uint16_t* raw_bf16, void* stream) {
  if (T < 0 || H <= 0) return MOE_ESHAPE;
  if (H % 128 != 0 || H > 16384) return MOE_ENOTSUP;
  if (!(eps >= 0.0f)) return MOE_EINVAL;
  if (!x || !out) return MOE_EINVAL;
  if (!a16(x) || !a16(out) || (gamma && !a16(gamma)) || (raw_bf16 && !a16(raw_bf16))) return MOE_EINVAL;
  if (T == 0) return MOE_OK;
  return cuda_status(moe::launch_rmsnorm(x, gamma, eps, T, H, out, raw_bf16, static_cast<cudaStream_t>(stream)));
}

moe_status moe_route_recall(const int32_t* pred_ids, const int32_t* ref_ids, int T, int k, int32_t* hits,
                            void* stream) {
  if (T < 0 || k <= 0) return MOE_ESHAPE;
  if (k > moe::kMaxK) return MOE_ENOTSUP;
  if (!pred_ids || !ref_ids || !hits) return MOE_EINVAL;
  if (!a4(pred_ids) || !a4(ref_ids) || !a4(hits)) return MOE_EINVAL;
  if (T == 0) return MOE_OK;
  return cuda_status(moe::launch_recall(pred_ids, ref_ids, T, k, hits, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
