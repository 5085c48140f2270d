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

// Store to the same shared-memory word in CTA `rank` of the cluster.
__device__ __forceinline__ void st_cluster_f32(float* local, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(ptx::smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

__device__ __forceinline__ void st_cluster_s32(int* local, uint32_t rank, int v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(ptx::smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}

__global__ void __launch_bounds__(kLogitThreads) router_logits_mma_kernel(const uint16_t* __restrict__ x,
                                                                          const uint16_t* __restrict__ wr, int T,
                                                                          int H, int E, float* __restrict__ logits) {
  __shared__ float red[kLogitWarps][kLogitTok][kLogitExp];
  __shared__ float tile[kLogitSplit][kLogitTok][kLogitExp];  // CTA 0: every CTA's K-quarter sums
  // arrive now, wait before the first store into CTA 0's shared memory: by
  // then every CTA of the cluster has started
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
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
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  if (threadIdx.x < kLogitTok * kLogitExp) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kLogitWarps; ++w) sum += red[w][t][e];
    st_cluster_f32(&tile[rank][t][e], 0, sum);  // into CTA 0's slot for this CTA
  }
  // every CTA's sums are in CTA 0's shared memory (release / acquire); the
  // other CTAs are done, and nothing reads their shared memory afterwards
  cluster_sync_all();
  if (rank == 0 && threadIdx.x < kLogitTok * kLogitExp) {
    float sum = tile[0][t][e];
#pragma unroll
    for (int r = 1; r < kLogitSplit; ++r) sum += tile[r][t][e];
    if (t0 + t < T && e0 + e < E) logits[static_cast<size_t>(t0 + t) * E + e0 + e] = sum;
  }
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
// Top-k of one token by one warp: lv/bv hold the logits and bias of experts
// lane, lane + 32, ... (bias ignored if has_bias is false).  Writes the
// token's ids/w row and gap; returns on lane r < k the expert of rank r.
template <int EPL>
__device__ __forceinline__ int select_topk(const float (&lv)[EPL], const float (&bv)[EPL], bool has_bias, int E,
                                           int k, int lane, uint64_t* cand, int32_t* ids_row, float* w_row,
                                           float* gap_t) {
  uint64_t v[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    const int e = j * 32 + lane;
    v[j] = 0;  // below every valid key (f2key(-inf) > 0)
    if (e < E) {
      float l = lv[j];
      if (has_bias) l += bv[j];
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
        if (v[j] >= thr) cand[pos++] = v[j];
      __syncwarp();
      mine = warp_sort_desc(lane < total ? cand[lane] : 0, lane);
      done = true;
    }
  }
  uint32_t rank32_key = 0;  // with k = 32 the next logit (rank 32) has no lane of its own
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
      if (r == 32) rank32_key = m_hi;
    }
  }
  const uint32_t my_key = static_cast<uint32_t>(mine >> 32);
  const int my_e = static_cast<int>(~static_cast<uint32_t>(mine));
  const uint32_t next_key =
      k < 32 ? static_cast<uint32_t>(__shfl_sync(0xffffffffu, mine, k & 31) >> 32) : rank32_key;
  const float my_v = key2f(my_key);
  const float v0 = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = (lane < k) ? expf(my_v - v0) : 0.f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  const float vk1 = __shfl_sync(0xffffffffu, my_v, k - 1);
  if (lane < k) {
    ids_row[lane] = my_e;
    w_row[lane] = ex / sum;
  }
  if (gap_t && lane == 0) *gap_t = (k < E) ? (vk1 - key2f(next_key)) : INFINITY;
  return my_e;
}

// One warp per token; see select_topk.
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
  select_topk<EPL>(lv, bv, bias != nullptr, E, k, lane, cand[warp], ids + static_cast<size_t>(t) * k,
                   w + static_cast<size_t>(t) * k, gap ? gap + t : nullptr);
}

// ---------------------------------------------------------------------------
// Decode block (T <= 16): router logits, top-k and the expert grouping in one
// launch of one 16-CTA thread-block cluster, so the three steps meet at no
// kernel boundary.  CTA c computes the logits of experts [c*epc, c*epc + epc)
// for the block's tokens with warp-level MMA (the 8 warps split K and are
// summed in warp order), keeping its [16][epc] tile in shared memory.  After a
// cluster barrier, CTA t < T selects token t's route: lane l reads the logits
// of experts l, l + 32, ... from their owner CTAs over distributed shared
// memory, then select_topk; each route is also written into CTA 0's shared
// memory.  After a second barrier CTA 0 groups the T*k routes by expert:
// counts, exclusive offsets, and the stable slot order (ascending flat route
// index inside each expert), exactly what permute_kernel writes.
constexpr int kRpCtas = 16;
constexpr int kRpThreads = 256;
constexpr int kRpWarps = kRpThreads / 32;
constexpr int kRpChunk = 8;   // k16 steps per register batch
constexpr int kRpMaxNt = 8;   // n8 tiles per CTA (epc <= 64: E <= 1024)

template <int NT, int EPL>
__global__ void __launch_bounds__(kRpThreads) route_permute_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr, const float* __restrict__ bias, int T, int H,
    int E, int k, int32_t* __restrict__ ids, float* __restrict__ w, float* __restrict__ gap,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
    int32_t* __restrict__ inv, int32_t* status) {
  constexpr int epc = 8 * NT;  // experts per CTA
  __shared__ float red[kRpWarps][kLogitTok][epc];
  __shared__ float tile[kLogitTok][epc];
  __shared__ uint64_t cand[32];
  __shared__ int s_ids[kLogitTok * kMaxK];  // CTA 0: the block's routes
  __shared__ int s_cnt[kMaxE + 1];
  __shared__ int s_bad;
  __shared__ int s_wsum[kRpWarps];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const uint32_t rank = cluster_ctarank();
  const int e_base = static_cast<int>(rank) * epc;
  // ------------------------------------------------------------ logits
  const int kw = H / kRpWarps;  // K per warp (a multiple of 16: H % 128 == 0)
  const int steps = kw / 16;
  const int kbase = warp * kw;
  const bool ta = g < T, tb = g + 8 < T;
  const uint32_t* xa = reinterpret_cast<const uint32_t*>(x + static_cast<size_t>(ta ? g : 0) * H + kbase);
  const uint32_t* xb = reinterpret_cast<const uint32_t*>(x + static_cast<size_t>(tb ? g + 8 : 0) * H + kbase);
  const uint32_t* wrow[NT];
  bool e_ok[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int e = e_base + nt * 8 + g;
    e_ok[nt] = e < E;
    wrow[nt] = reinterpret_cast<const uint32_t*>(wr + static_cast<size_t>(e_ok[nt] ? e : 0) * H + kbase);
  }
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  if (threadIdx.x == 0) s_bad = 0;
  pdl_wait();
  pdl_trigger();
  for (int c0 = 0; c0 < steps; c0 += kRpChunk) {
    uint32_t af[kRpChunk][4];
    uint32_t bw[kRpChunk][NT][2];
#pragma unroll
    for (int s2 = 0; s2 < kRpChunk; ++s2) {
      const bool in = c0 + s2 < steps;
      const int o = (c0 + s2) * 8 + q;
      af[s2][0] = (in && ta) ? xa[o] : 0u;
      af[s2][1] = (in && tb) ? xb[o] : 0u;
      af[s2][2] = (in && ta) ? xa[o + 4] : 0u;
      af[s2][3] = (in && tb) ? xb[o + 4] : 0u;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        bw[s2][nt][0] = (in && e_ok[nt]) ? __ldg(wrow[nt] + o) : 0u;
        bw[s2][nt][1] = (in && e_ok[nt]) ? __ldg(wrow[nt] + o + 4) : 0u;
      }
    }
#pragma unroll
    for (int s2 = 0; s2 < kRpChunk; ++s2)
      if (c0 + s2 < steps) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(acc[nt], af[s2], bw[s2][nt]);
      }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    red[warp][g][nt * 8 + 2 * q] = acc[nt][0];
    red[warp][g][nt * 8 + 2 * q + 1] = acc[nt][1];
    red[warp][g + 8][nt * 8 + 2 * q] = acc[nt][2];
    red[warp][g + 8][nt * 8 + 2 * q + 1] = acc[nt][3];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kLogitTok * epc; i += kRpThreads) {
    const int t = i / epc, e = i % epc;
    float sum = 0.f;
#pragma unroll
    for (int ww = 0; ww < kRpWarps; ++ww) sum += red[ww][t][e];
    tile[t][e] = sum;
  }
  cluster_sync_all();  // every CTA's logit tile is complete
  // ------------------------------------------------------------ top-k
  if (static_cast<int>(rank) < T && warp == 0) {
    const int t = static_cast<int>(rank);
    float lv[EPL], bv[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const int e = j * 32 + lane;
      lv[j] = e < E ? ld_cluster_f32(&tile[t][e % epc], static_cast<uint32_t>(e / epc)) : 0.f;
      bv[j] = (bias && e < E) ? bias[e] : 0.f;
    }
    const int my_e = select_topk<EPL>(lv, bv, bias != nullptr, E, k, lane, cand, ids + static_cast<size_t>(t) * k,
                                      w + static_cast<size_t>(t) * k, gap ? gap + t : nullptr);
    if (lane < k) st_cluster_s32(&s_ids[t * k + lane], 0u, my_e);
  }
  cluster_sync_all();  // every route is in CTA 0
  if (rank != 0) return;
  // ------------------------------------------------------------ grouping
  const int R = T * k;
  for (int e = threadIdx.x; e <= E; e += kRpThreads) s_cnt[e] = 0;
  __syncthreads();
  for (int r = threadIdx.x; r < R; r += kRpThreads) {
    const int e = s_ids[r];
    if (e < 0 || e >= E) s_bad = 1;
    else atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) set_status(status, MOE_DEV_BAD_EXPERT);
    return;
  }
  // exclusive scan of s_cnt over E experts: each thread a contiguous run
  const int per = (E + kRpThreads - 1) / kRpThreads;
  const int e0 = min(E, threadIdx.x * per), e1 = min(E, e0 + per);
  int run = 0;
  for (int e = e0; e < e1; ++e) run += s_cnt[e];
  int incl = run;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int ww = 0; ww < warp; ++ww) before += s_wsum[ww];
  int off = before + incl - run;
  for (int e = e0; e < e1; ++e) {
    const int c = s_cnt[e];
    counts[e] = c;
    offsets[e] = off;
    s_cnt[e] = off;  // now the segment start
    off += c;
  }
  if (threadIdx.x == 0) offsets[E] = R;
  __syncthreads();
  for (int r = threadIdx.x; r < R; r += kRpThreads) {
    const int e = s_ids[r];
    int before_r = 0;  // earlier routes of the same expert: stable order
    for (int r2 = 0; r2 < r; ++r2) before_r += (s_ids[r2] == e) ? 1 : 0;
    const int slot = s_cnt[e] + before_r;
    perm[slot] = r;
    inv[r] = slot;
  }
}

// ---------------------------------------------------------------------------
// Route sidecar forward pass (AFN-021 "Replay decode as prefill: a training
// flywheel for predictive MoE I/O", section "What feature should the sidecar
// see?"): a feature vector f -> shared low-rank trunk z = Wt f -> plus the
// target layer's embedding e_l -> scores against the shared expert-head
// embeddings, s_l = Wh (z + e_l) -> the N highest-scoring experts of every
// layer, ranked (ties to the lower expert ID).  s_l is computed as
// Wh z + Wh e_l: the [L, E] table Wh e_l depends on the weights only and is
// prepared once (sidecar_prepare_kernel); per call the trunk runs on the
// router's small-T logits kernel (trunk rows in place of router rows) and
// sidecar_head_kernel forms Wh z once per position and selects every layer's
// candidates from Wh z + Wh e_l.
constexpr int kSideThreads = 512;
constexpr int kSideWarps = kSideThreads / 32;
constexpr int kSideMaxR = 1024;

// One warp: dots of kSideBatch bf16 rows w[e0 + b][0, r) (rows of r inputs,
// rows past E read as zero) with the fp32 vector v[0, r) in shared memory;
// lane l takes inputs 8l .. 8l+7 of every 256-wide chunk, one 16-byte load
// per row in flight at once, then a butterfly sum per row.  r % 8 == 0, w
// 16-byte aligned.  Every lane returns the kSideBatch dots.
constexpr int kSideBatch = 16;

__device__ __forceinline__ void warp_dots_bf16(const uint16_t* __restrict__ w, int e0, int E, int r, const float* v,
                                               int lane, float (&out)[kSideBatch]) {
  float acc[kSideBatch];
#pragma unroll
  for (int b = 0; b < kSideBatch; ++b) acc[b] = 0.f;
  for (int j0 = lane * 8; j0 < r; j0 += 256) {
    uint4 q[kSideBatch];
#pragma unroll
    for (int b = 0; b < kSideBatch; ++b)
      q[b] = e0 + b < E ? __ldg(reinterpret_cast<const uint4*>(w + static_cast<size_t>(e0 + b) * r + j0))
                        : make_uint4(0u, 0u, 0u, 0u);
    const float4 va = *reinterpret_cast<const float4*>(v + j0);
    const float4 vb = *reinterpret_cast<const float4*>(v + j0 + 4);
    const float vv[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
#pragma unroll
    for (int b = 0; b < kSideBatch; ++b) {
      const uint32_t u[4] = {q[b].x, q[b].y, q[b].z, q[b].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[b] = fmaf(__uint_as_float(u[i] << 16), vv[2 * i], acc[b]);
        acc[b] = fmaf(__uint_as_float(u[i] & 0xffff0000u), vv[2 * i + 1], acc[b]);
      }
    }
  }
#pragma unroll
  for (int b = 0; b < kSideBatch; ++b) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], off);
    out[b] = acc[b];
  }
}

// c[l, e] = Wh[e, :] . emb[l, :]; one CTA per layer.
__global__ void __launch_bounds__(kSideThreads) sidecar_prepare_kernel(const uint16_t* __restrict__ w_head,
                                                                       const uint16_t* __restrict__ emb, int E,
                                                                       int r, float* __restrict__ c) {
  __shared__ __align__(16) float v[kSideMaxR];
  const int l = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  for (int j = threadIdx.x; j < r; j += kSideThreads)
    v[j] = __uint_as_float(static_cast<uint32_t>(emb[static_cast<size_t>(l) * r + j]) << 16);
  __syncthreads();
  for (int e0 = warp * kSideBatch; e0 < E; e0 += kSideWarps * kSideBatch) {
    float d[kSideBatch];
    warp_dots_bf16(w_head, e0, E, r, v, lane, d);
#pragma unroll
    for (int b = 0; b < kSideBatch; ++b)
      if (lane == b && e0 + b < E) c[static_cast<size_t>(l) * E + e0 + b] = d[b];
  }
}

// CTA (t, y): u = Wh z[t] into shared memory, then the warps rank the
// layers [y per, (y + 1) per), per = ceil(L / gridDim.y), layer y per + w,
// + 16, ... by warp w: scores u + c[l] through select_topk.  For a few
// positions the CTAs of one position each form u (W_h comes from L2) so that
// every warp ranks one layer; for many, one CTA per position ranks them all.
template <int EPL>
__global__ void __launch_bounds__(kSideThreads) sidecar_head_kernel(const float* __restrict__ z,
                                                                    const uint16_t* __restrict__ w_head,
                                                                    const float* __restrict__ c, int r, int E, int L,
                                                                    int N, int32_t* __restrict__ cand,
                                                                    float* __restrict__ score, int32_t* status) {
  __shared__ __align__(16) float zs[kSideMaxR];
  __shared__ float u[32 * EPL];
  __shared__ uint64_t keys[kSideWarps][32];
  __shared__ float wscr[kSideWarps][32];
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  const int per = (L + gridDim.y - 1) / gridDim.y;
  const int l0 = blockIdx.y * per, l1 = min(L, l0 + per);
  if (l0 >= l1) return;
  for (int j = threadIdx.x; j < r; j += kSideThreads) zs[j] = z[static_cast<size_t>(t) * r + j];
  __syncthreads();
  bool bad = false;
  for (int e0 = warp * kSideBatch; e0 < E; e0 += kSideWarps * kSideBatch) {
    float d[kSideBatch];
    warp_dots_bf16(w_head, e0, E, r, zs, lane, d);
#pragma unroll
    for (int b = 0; b < kSideBatch; ++b)
      if (lane == b && e0 + b < E) {
        u[e0 + b] = d[b];
        bad |= !isfinite(d[b]);
      }
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0 && blockIdx.y == 0) set_status(status, MOE_DEV_NONFINITE);
  for (int l = l0 + warp; l < l1; l += kSideWarps) {
    float lv[EPL], bv[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const int e = j * 32 + lane;
      lv[j] = e < E ? u[e] : 0.f;
      bv[j] = e < E ? c[static_cast<size_t>(l) * E + e] : 0.f;
    }
    const size_t row = (static_cast<size_t>(t) * L + l) * N;
    const int my_e = select_topk<EPL>(lv, bv, true, E, N, lane, keys[warp], cand + row, wscr[warp], nullptr);
    if (lane < N) {
      float sc = u[my_e];
      sc += c[static_cast<size_t>(l) * E + my_e];
      score[row + lane] = sc;
    }
    __syncwarp();
  }
}

template <int EPL>
cudaError_t run_sidecar_head(const float* z, const uint16_t* w_head, const float* c, int T, int r, int E, int L,
                             int N, int32_t* cand, float* score, int32_t* st_word, cudaStream_t st) {
  const int ysplit = T <= 32 ? (L + kSideWarps - 1) / kSideWarps : 1;
  return launch_pdl(sidecar_head_kernel<EPL>, dim3(T, ysplit), dim3(kSideThreads), 0, st, z, w_head, c, r, E, L, N,
                    cand, score, st_word);
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

template <int NT, int EPL>
cudaError_t run_route_permute(const uint16_t* x, const uint16_t* wr, const float* bias, int T, int H, int E, int k,
                              int32_t* ids, float* w, float* gap, int32_t* counts, int32_t* offsets, int32_t* perm,
                              int32_t* inv, int32_t* st_word, cudaStream_t st) {
  static_assert(NT <= kRpMaxNt, "n8 tiles per CTA");
  auto kern = route_permute_kernel<NT, EPL>;
  static std::mutex mu;
  static int ready[64] = {0};  // per device: 1 usable, -1 not
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (ready[dev] == 0) {
      ready[dev] = -1;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kRpCtas);
        cfg.blockDim = dim3(kRpThreads);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = kRpCtas;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) == cudaSuccess && clusters > 0) ready[dev] = 1;
      }
      cudaGetLastError();
    }
    if (ready[dev] < 0) return cudaErrorNotSupported;
  }
  return launch_pdl_cluster(kern, dim3(kRpCtas), dim3(kRpThreads), dim3(kRpCtas, 1, 1), 0, st, x, wr, bias, T, H, E,
                            k, ids, w, gap, counts, offsets, perm, inv, st_word);
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

cudaError_t launch_sidecar_prepare(const uint16_t* w_head, const uint16_t* emb, int E, int r, int L, float* c,
                                   cudaStream_t st) {
  return launch_pdl(sidecar_prepare_kernel, dim3(L), dim3(kSideThreads), 0, st, w_head, emb, E, r, c);
}

cudaError_t launch_sidecar_forward(const uint16_t* feat, const uint16_t* w_trunk, const uint16_t* w_head,
                                   const float* c, int T, int F, int r, int E, int L, int N, float* z, int32_t* cand,
                                   float* score, int32_t* st_word, cudaStream_t st) {
  if (r > kSideMaxR || E > 1024) return cudaErrorInvalidValue;
  cudaError_t e = launch_router_logits_small(feat, w_trunk, T, F, r, z, st);
  if (e != cudaSuccess) return e;
  const int epl = (E + 31) / 32;
  if (epl <= 1) return run_sidecar_head<1>(z, w_head, c, T, r, E, L, N, cand, score, st_word, st);
  if (epl <= 2) return run_sidecar_head<2>(z, w_head, c, T, r, E, L, N, cand, score, st_word, st);
  if (epl <= 4) return run_sidecar_head<4>(z, w_head, c, T, r, E, L, N, cand, score, st_word, st);
  if (epl <= 8) return run_sidecar_head<8>(z, w_head, c, T, r, E, L, N, cand, score, st_word, st);
  if (epl <= 16) return run_sidecar_head<16>(z, w_head, c, T, r, E, L, N, cand, score, st_word, st);
  return run_sidecar_head<32>(z, w_head, c, T, r, E, L, N, cand, score, st_word, st);
}

// One-launch route + grouping for a decode block (T <= 16); cudaErrorNotSupported
// if this device cannot run a 16-CTA cluster.
cudaError_t launch_route_permute(const uint16_t* x, const uint16_t* wr, const float* bias, int T, int H, int E, int k,
                                 int32_t* ids, float* w, float* gap, int32_t* counts, int32_t* offsets, int32_t* perm,
                                 int32_t* inv, int32_t* st_word, cudaStream_t st) {
  const int nt = ((E + kRpCtas - 1) / kRpCtas + 7) / 8;  // n8 tiles per CTA
  const int epl = (E + 31) / 32;
  if (nt <= 1 && epl <= 2)
    return run_route_permute<1, 2>(x, wr, bias, T, H, E, k, ids, w, gap, counts, offsets, perm, inv, st_word, st);
  if (nt <= 2 && epl <= 8)
    return run_route_permute<2, 8>(x, wr, bias, T, H, E, k, ids, w, gap, counts, offsets, perm, inv, st_word, st);
  if (nt <= 4 && epl <= 16)
    return run_route_permute<4, 16>(x, wr, bias, T, H, E, k, ids, w, gap, counts, offsets, perm, inv, st_word, st);
  return run_route_permute<8, 32>(x, wr, bias, T, H, E, k, ids, w, gap, counts, offsets, perm, inv, st_word, st);
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
//    exits.  T > 64 is rejected with MOE_EWORKSPACE; E > 1024 is beyond the
//    router's own limit and is rejected first, with MOE_ENOTSUP.
//  * The host-side name g_route_scratch is not a device address.  Every
//    call looks the device address up with cudaGetSymbolAddress() for the
//    device that is current (a host-side lookup, no allocation), so a call
//    after a device reset or a new context never uses an address from an
//    earlier one.  The first call on a device may load the library's device
//    code for that device, so it should come before any stream capture.
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

// Device address of g_route_scratch on the current device (nullptr on
// error).  Looked up on each call rather than cached: after cudaDeviceReset()
// or a new primary context the module is loaded again and the array can move.
float* noalloc_scratch_for_current_device() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess) return nullptr;
  return static_cast<float*>(p);
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
