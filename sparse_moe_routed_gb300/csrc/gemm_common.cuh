// Internal header of the expert-contraction translation units -- gemm.cu
// (grouped tcgen05 kernels: bf16 and int4, plus their host side), fused.cu
// (gate/up + SwiGLU + down in one persistent launch, with the expert cache's
// slot tables and fetch warps) and q4.cu (the int4 matrix-vector kernel of
// decode-sized launches): tile geometry, the argument block, bounded waits,
// the tile schedule and the TMEM epilogue they share.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace moe {
namespace gk {

constexpr int kBM = 128;                             // weight rows per tile (MMA M)
constexpr int kBK = 64;                              // K per stage: one 128-byte swizzled row of bf16
constexpr int kUK = 16;                              // K per MMA instruction
constexpr int kABytes = kBM * kBK * 2;               // 16 KB bf16 operand tile
constexpr int kBoxRows = 16;                         // token rows per B TMA box (tiles of up to 64 rows)
constexpr int kBBoxBytes = kBoxRows * kBK * 2;       // 2 KB
constexpr int kGUBoxBytes = 2 * kBoxRows * kBK * 2;  // 16 gate + 16 up rows: 4 KB
constexpr int kQBytes = kBM * kBK / 2;               // int4 codes of one stage: 4 KB
constexpr int kSBytes = kBM * 2;                     // one bf16 scale per row: 256 B
constexpr int kQChunk = kQBytes + kSBytes;           // one packed int4 stage chunk: 4,352 B
constexpr int kCoreThreads = 192;                    // producers, MMA, 4 epilogue warps
constexpr int kSmemTail = 16 + 2 * (kMaxE + 1) * 4;  // misc words + tile prefix + segment offsets
constexpr uint64_t kWaitNs = 2000000000ull;

// Token rows per B TMA box for tiles of nmax rows: decode-sized tiles hold a
// few rows per expert, so 16-row boxes; 128-row tiles take 64-row boxes, so
// that one producer thread issues two copies per K step rather than eight
// (rows past a tile's end belong to the next expert or are zero-filled past
// the last row, and are never stored).
constexpr int box_rows_for(int nmax) { return nmax >= 128 ? 64 : kBoxRows; }

// bf16 weights: one ring; a stage holds G consecutive K steps: A (G x 16 KB)
// + B (G x NMAX token rows).  Tile-packed weights take G = 2 (one 32 KB bulk
// copy per stage), halving the per-request and per-handoff costs.
template <int NMAX, int G>
struct CfgB {
  static constexpr int kThreads = kCoreThreads;
  static constexpr int kBBytes = NMAX * kBK * 2;
  static constexpr int kStageBytes = G * (kABytes + kBBytes);
  static constexpr int kBudget = 196 * 1024;
  static constexpr int kStages = kBudget / kStageBytes < 2 ? 2 : (kBudget / kStageBytes > 10 ? 10 : kBudget / kStageBytes);
  static constexpr int kTmemCols = 2 * NMAX < 32 ? 32 : 2 * NMAX;
  static constexpr int kNumBars = 2 * kStages + 5;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kNumBars * 8 + kSmemTail;
  static_assert(kBBytes % 1024 == 0, "B stage must keep 1024-byte alignment");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// int4 g64 weights: a deep ring of packed chunks, a ring of bf16 operand
// tiles with one slot per dequantiser warp (SA), a ring of token rows (SB).
// One bulk copy fills a ring slot with QG consecutive K steps' chunks (QG = 4
// for gate/up, 2 for down: runtime, kQRingBytes / (QG x 4,352) slots).
// Dequantiser warp w owns every SA-th K step, so SA steps are dequantised at
// once.
template <int NMAX>
struct CfgQ {
  // The dequantised operand never touches shared memory: dequantiser warps
  // write it to tensor memory (tcgen05.st) and the MMA reads A from there.
  // TMEM lane quarters bind warps to rows: warp w may access lanes
  // 32 (w % 4) .. +31, so dequantiser warps come in groups of four (one per
  // quarter) and the groups take turns over the K steps.  Shared memory
  // holds only the packed chunk ring (which covers HBM latency) and the
  // token-row ring.
  static constexpr int kDqGroups = 2;
  static constexpr int kDqWarps = 4 * kDqGroups;
  static constexpr int kDqWarp0 = 7;  // warp 6 produces token rows
  static constexpr int kThreads = 32 * (kDqWarp0 + kDqWarps);
  static constexpr int kBBytes = NMAX * kBK * 2;
  static constexpr int kTmemCols = 512;               // accumulators first, then the operand ring
  static constexpr int kTmemA = 2 * NMAX < 32 ? 32 : 2 * NMAX;
  static constexpr int SA = (kTmemCols - kTmemA) / 32 > 12 ? 12 : (kTmemCols - kTmemA) / 32;  // 32 columns each
  // token rows: one small stage per K step, so a deep ring for small NMAX
  static constexpr int SB = NMAX <= 16 ? 24 : (NMAX <= 32 ? 12 : (NMAX <= 64 ? 6 : 4));
  static constexpr int SQmax = NMAX <= 16 ? 32 : (NMAX <= 32 ? 24 : (NMAX <= 64 ? 24 : 16));  // chunks
  static constexpr int kQRingBytes = SQmax * kQChunk;
  static constexpr int kNumBars = 2 * (SQmax + SA + SB) + 5;
  static constexpr int kSmemBytes = 1024 + SB * kBBytes + kQRingBytes + kNumBars * 8 + kSmemTail;
  static_assert(kBBytes % 1024 == 0, "B stage must keep 1024-byte alignment");
  static_assert(2 * NMAX <= kTmemA, "accumulators below the operand ring");
  static_assert(kTmemA + SA * 32 <= kTmemCols, "operand ring inside the allocation");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct GemmArgs {
  const int32_t* offsets;  // [E+1] segment starts (null for one dense segment)
  int E;                   // segments
  int R;                   // rows of the B operand
  int ksteps;              // K / 64
  int mblocks;             // 128-row weight blocks per segment
  int seg_rows;            // weight rows per segment in the A map (down: H)
  const uint8_t* tiles;    // tile-packed weights (bulk-copy modes), chunk per (e, mb, ks)
  int qgroup;              // int4: K steps per bulk copy (divides ksteps)
  const uint16_t* brows;   // int4 GEMV: the token rows [R][K] bf16 (staged per tile by bulk copies)
  void* out;
  int ldo;                 // leading dimension of out (elements)
  int32_t* status;
  // int4 GEMV over an expert cache (slot_of != nullptr): tiles is a pool of
  // S records and expert e's record is record slot_of[e]
  const int32_t* slot_of;
  int S;
  // ... and, for a gate/up launch with host records (host_gu != nullptr),
  // the planned misses are fetched in the launch: fetch warps copy the
  // gate/up records (pieces of cpp chunks, counted per 128-row block in
  // fsync[2 + e * mblocks + block]) and then the down records (into pool_dn,
  // for the down launch that follows); fsync[0] is the piece queue, fsync[1]
  // the exit count.
  const uint8_t* host_gu;
  const uint8_t* host_dn;
  uint8_t* pool_dn;
  size_t rec_gu, rec_dn;
  int cpp;  // chunks per gate/up piece (divides ksteps)
  const int32_t* miss_list;
  const int32_t* miss_slot;
  const int32_t* stats;
  int32_t* fsync;
};

// Bounded mbarrier wait.  Polls back off with __nanosleep(kSleepNs) so that
// waiting warps leave issue slots to the warps doing work (0 for the
// single-thread producer and MMA roles, whose latency matters most).  The
// (slow) %globaltimer is read only every 1024 polls, starting the clock at
// the first read; after kWaitNs the wait flags MOE_DEV_TIMEOUT and gives up.
template <uint32_t kSleepNs>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                             int32_t* status) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (kSleepNs != 0 && it >= 2) __nanosleep(kSleepNs);
    if ((it & 1023u) == 1023u) {
      if (*abort_flag) return false;
      const uint64_t now = globaltimer_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > kWaitNs) {
        *abort_flag = 1;
        set_status(status, MOE_DEV_TIMEOUT);
        return false;
      }
    }
  }
}

// Acquire load of a device-wide counter, and the fence that orders generic
// stores before later bulk/TMA reads of the same bytes (in any CTA).
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

constexpr uint32_t kSpin = 0;         // producer / MMA threads
constexpr uint32_t kSleepEpi = 256;   // epilogue warps (one wait per tile)

// Drain wait used during teardown after an abort: ignores the abort flag.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    __nanosleep(256);
    if (globaltimer_ns() - t0 > kWaitNs) return;
  }
}


// One packed 32-bit word of eight int4 g64 codes -> eight bf16 (16 bytes).
// The packer stores each code offset by +8 and orders a word's nibbles as
// elements 0,2,4,6,1,3,5,7, so one mask-and-or per pair places two codes in
// the mantissas of 128 + (q + 8) (exact in bf16); subtracting 136 is exact and
// the product with the group scale is rounded once.
__device__ __forceinline__ uint4 dequant8(uint32_t word, __nv_bfloat162 scale2) {
  const __nv_bfloat162 off2 = __floats2bfloat162_rn(136.0f, 136.0f);
  uint32_t out[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint32_t bits = ((word >> (4 * p)) & 0x000F000Fu) | 0x43004300u;
    __nv_bfloat162 b;
    std::memcpy(&b, &bits, 4);
    const __nv_bfloat162 w = __hmul2(__hsub2(b, off2), scale2);
    std::memcpy(&out[p], &w, 4);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

struct Tile {
  int e, mb, row0, nrows;
};

// Shared per-CTA scheduling state: clamped segment offsets and the tile
// prefix over segments, both in shared memory.
struct Sched {
  const int* prefix;
  const int* soff;
  int E;
  int mblocks;
  int nmax;
  const int* order = nullptr;  // expert at each position of the tile order (null: ID order)

  __device__ __forceinline__ Tile tile(int t) const {
    int lo = 0, hi = E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= t) lo = mid; else hi = mid;
    }
    const int local = t - prefix[lo];
    const int chunk = local / mblocks;
    const int e = order != nullptr ? order[lo] : lo;
    const int start = soff[e];
    const int len = max(soff[e + 1] - start, 0);
    Tile tl;
    tl.e = e;
    tl.mb = local - chunk * mblocks;
    tl.row0 = start + chunk * nmax;
    tl.nrows = min(nmax, len - chunk * nmax);
    return tl;
  }
};

// Segment offsets into shared memory, clamped into [0, R] (a segment's length
// is never negative) so that corrupt offsets can never address rows outside
// the buffers; then the per-segment tile prefix (warp 0).  Ends with a
// CTA-wide barrier.  Returns the total number of tiles.
template <int NMAX>
__device__ __forceinline__ int build_schedule(const GemmArgs& p, bool dense, int E, int* prefix, int* soff) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i <= E; i += blockDim.x)
    soff[i] = dense ? (i == 0 ? 0 : p.R) : min(max(__ldcg(p.offsets + i), 0), p.R);
  __syncthreads();
  if (warp == 0) {
    int running = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      int n = 0;
      if (e < E) n = max(soff[e + 1] - soff[e], 0);
      const int tiles = ((n + NMAX - 1) / NMAX) * p.mblocks;
      int incl = tiles;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
      }
      if (e < E) prefix[e] = running + incl - tiles;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) prefix[E] = running;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  return prefix[E];
}

// Epilogue warps (2..5): drain finished accumulators from TMEM.  Gate/up
// (KIND 0): h = bf16(silu(g) * u); down (KIND 1) and router logits (KIND 2):
// fp32 rows, one 128-byte store per warp per token row.
template <int NMAX, int KIND>
__device__ __forceinline__ void epilogue_role(const GemmArgs& p, const Sched& sc, int total, uint32_t tmem_base,
                                              uint32_t accf0, uint32_t acce0, volatile uint32_t* abort_flag) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int q = warp & 3;  // TMEM lane quarter this warp may access
  const int row_in_tile = q * 32 + lane;
  int acc = 0;
  uint32_t aph = 0;
  for (int t = blockIdx.x; t < total; t += gridDim.x) {
    const Tile tl = sc.tile(t);
    const bool ok = wait_bounded<kSleepEpi>(accf0 + 8 * acc, aph, abort_flag, p.status);
    if (!__all_sync(0xffffffffu, ok)) break;
    ptx::tc_fence_after();
    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * NMAX);
    if (KIND == 0) {
      uint16_t* hout = static_cast<uint16_t*>(p.out);
      const bool up_lane = lane >= 16;
      const int i = tl.mb * 64 + q * 16 + (lane & 15);
      for (int c0 = 0; c0 < tl.nrows; c0 += 16) {
        float v[16];
        ptx::tmem_ld16(taddr + static_cast<uint32_t>(c0), v);
        float recv[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const float send = up_lane ? v[jj] : v[8 + jj];
          recv[jj] = __shfl_xor_sync(0xffffffffu, send, 16);
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int col = c0 + (up_lane ? 8 : 0) + jj;
          const float g = up_lane ? recv[jj] : v[jj];
          const float u = up_lane ? v[8 + jj] : recv[jj];
          if (col < tl.nrows) {
            const float hval = g / (1.0f + expf(-g)) * u;
            hout[static_cast<size_t>(tl.row0 + col) * p.ldo + i] = f32_to_bf16(hval);
          }
        }
      }
    } else {
      float* yout = static_cast<float*>(p.out);
      const int j = tl.mb * kBM + row_in_tile;
      for (int c0 = 0; c0 < tl.nrows; c0 += 16) {
        float v[16];
        ptx::tmem_ld16(taddr + static_cast<uint32_t>(c0), v);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int col = c0 + jj;
          if (col < tl.nrows) yout[static_cast<size_t>(tl.row0 + col) * p.ldo + j] = v[jj];
        }
      }
    }
    ptx::tc_fence_before();
    ptx::mbar_arrive(acce0 + 8 * acc);
    if (++acc == 2) {
      acc = 0;
      aph ^= 1u;
    }
  }
}

__device__ __forceinline__ void issue_k_step(uint32_t d_tmem, uint32_t a0, uint32_t b0, uint32_t idesc, int ks) {
#pragma unroll
  for (int kk = 0; kk < kBK / kUK; ++kk)
    ptx::umma_bf16(d_tmem, ptx::sdesc_k_sw128(a0 + kk * kUK * 2), ptx::sdesc_k_sw128(b0 + kk * kUK * 2), idesc,
                   (ks | kk) != 0 ? 1u : 0u);
}

// ---- host helpers (gemm.cu)
// Row-major [rows][K] bf16 tensor map with boxes of box_rows x 64.
bool make_rows_map(CUtensorMap* m, const void* ptr, int K, int rows, int box_rows);
// Token rows per tile for a launch of rows_hint rows.
int pick_nmax(int rows_hint);

// ---- int4 matrix-vector launches (q4.cu)
// Whether a launch of R rows over K inputs takes the int4 matrix-vector kernel.
bool use_gemv_q4(int fmt, int R, int K);
// Gate/up (kind 0) or down (kind 1) on the int4 matrix-vector kernel.
cudaError_t launch_gemv_q4(int kind, const GemmArgs& args, cudaStream_t st);

}  // namespace gk
}  // namespace moe
