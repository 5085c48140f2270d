// Grouped expert contraction on the 5th-generation tensor cores (sm_103a).
//
// The expert SwiGLU of AFN-019 "Hide SSD misses before the router knows they
// exist" (section "Why overlap alone cannot defeat the byte roofline": gate
// [I,H], up [I,H], down [H,I] per expert; section "Hypothesis H4": gate and up
// together, down once the SwiGLU intermediate exists), written for GB300:
//
//  * Weight-stationary, swap-AB tiles.  An expert sees few token rows (1-16 at
//    decode, ~80 at prefill) but owns 9.8 MB of weights, so the weight rows are
//    the MMA's M = 128 side and the expert's token rows are N (16..NMAX, padded
//    to 16).  D[128, N] = W[128, K] . X[N, K]^T accumulates in TMEM (fp32).
//  * A tile is (expert e, 128-row weight block, chunk of <= NMAX token rows);
//    tiles of one expert are consecutive so its token rows stay in L2 while its
//    weights stream once from HBM (L2 evict-first hint on weights).
//  * Persistent CTAs (one per SM) walk the tile list round-robin.  Tile
//    counts come from the device-side expert offsets, never from the host.
//  * Warp roles: warp 0 = producer (TMA / bulk copies), warp 1 = MMA issuer
//    (and TMEM owner), warps 2..5 = epilogue; for int4 weights warp 6 also
//    produces (token rows) and warps 7.. dequantise.  Shared-memory rings with mbarriers feed the tensor
//    core; two TMEM accumulators let the epilogue of one tile overlap the main
//    loop of the next.
//  * Gate/up tiles interleave 16 gate rows with the 16 matching up rows, so
//    each epilogue warp holds g in lanes 0..15 and u in lanes 16..31 of the
//    same intermediate index: SwiGLU needs one shuffle, no shared-memory
//    exchange.
//  * Weight tiles come either through TMA tensor maps from the plain bf16
//    record layout, or as one bulk copy per stage from a tile-packed record
//    (pack.cu): a 16 KB pre-swizzled bf16 tile, or a 4,352-byte int4 g64
//    chunk (128 rows x 64 codes + the rows' bf16 group scales).
//  * int4 g64 weights (AFN-001 "Porting Qwen3.8-Flash-Next to Hebrus", section
//    "Phase 2": affine4 with group size 64, read as symmetric codes with one
//    bf16 scale per group) move 4.25x fewer bytes per stage, so their packed
//    chunks get a deep ring of their own (~70 KB in flight per SM); dequantiser
//    warps turn each chunk into a 128-byte-swizzled bf16 operand tile in a
//    short second ring (w = bf16(code * scale)), fence the generic-proxy
//    writes for the async proxy and arrive on the tile's barrier; token rows
//    have a third ring fed by a second producer warp.
//  * Every mbarrier wait is bounded (2 s of globaltimer, read sparingly; waits
//    of the many-thread roles back off with __nanosleep); on expiry the CTA
//    flags MOE_DEV_TIMEOUT, waits (bounded) for its copies and MMAs in flight,
//    frees its TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <map>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kBM = 128;                             // weight rows per tile (MMA M)
constexpr int kBK = 64;                              // K per stage: one 128-byte swizzled row of bf16
constexpr int kUK = 16;                              // K per MMA instruction
constexpr int kABytes = kBM * kBK * 2;               // 16 KB bf16 operand tile
constexpr int kBoxRows = 16;                         // token rows per B TMA box
constexpr int kBBoxBytes = kBoxRows * kBK * 2;       // 2 KB
constexpr int kGUBoxBytes = 2 * kBoxRows * kBK * 2;  // 16 gate + 16 up rows: 4 KB
constexpr int kQBytes = kBM * kBK / 2;               // int4 codes of one stage: 4 KB
constexpr int kSBytes = kBM * 2;                     // one bf16 scale per row: 256 B
constexpr int kQChunk = kQBytes + kSBytes;           // one packed int4 stage chunk: 4,352 B
constexpr int kCoreThreads = 192;                    // producers, MMA, 4 epilogue warps
constexpr int kSmemTail = 16 + 2 * (kMaxE + 1) * 4;  // misc words + tile prefix + segment offsets
constexpr uint64_t kWaitNs = 2000000000ull;

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

  __device__ __forceinline__ Tile tile(int t) const {
    int lo = 0, hi = E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= t) lo = mid; else hi = mid;
    }
    const int local = t - prefix[lo];
    const int chunk = local / mblocks;
    const int start = soff[lo];
    const int len = max(soff[lo + 1] - start, 0);
    Tile tl;
    tl.e = lo;
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
    soff[i] = dense ? (i == 0 ? 0 : p.R) : min(max(p.offsets[i], 0), p.R);
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

// ============================================================== bf16 kernel
// AMODE 0: weight tiles through the TMA tensor map tmA (plain bf16 record);
// AMODE 1: one 16 KB bulk copy per stage (tile-packed bf16 record).
template <int NMAX, int KIND, int AMODE, int G>
__global__ void __launch_bounds__(kCoreThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        GemmArgs p) {
  using C = CfgB<NMAX, G>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;                  // [S][G][16 KB] bf16 operand tiles (swizzled)
  uint8_t* sB = sA + S * G * kABytes;  // [S][G][NMAX x 128 B] token rows (swizzled)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + S * G * C::kBBytes);
  const uint32_t full0 = ptx::smem_u32(bars);  // operand tiles landed
  const uint32_t empty0 = full0 + 8 * S;       // MMA finished with a stage
  const uint32_t accf0 = empty0 + 8 * S;
  const uint32_t acce0 = accf0 + 16;
  const uint32_t drain = acce0 + 16;
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(bars + C::kNumBars);
  int* prefix = const_cast<int*>(reinterpret_cast<volatile int*>(misc + 4));
  int* soff = prefix + (kMaxE + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool dense = (p.offsets == nullptr);
  const int E = dense ? 1 : p.E;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(full0 + 8 * s, 1);
      ptx::mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(accf0 + 8 * a, 1);
      ptx::mbar_init(acce0 + 8 * a, 128);
    }
    ptx::mbar_init(drain, 1);
    misc[1] = 0;
    ptx::fence_mbar_init();
    if (AMODE == 0) ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(const_cast<uint32_t*>(&misc[0])), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  // Everything above overlaps the previous kernel's tail; from here on the
  // kernel reads upstream data (offsets, activation rows) and writes outputs.
  pdl_wait();
  pdl_trigger();
  const int total = build_schedule<NMAX>(p, dense, E, prefix, soff);
  const uint32_t tmem_base = misc[0];
  const Sched sc{prefix, soff, E, p.mblocks, NMAX};

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = ptx::policy_evict_first();
    const uint64_t pol_x = ptx::policy_evict_last();
    int armed[S];
#pragma unroll
    for (int s = 0; s < S; ++s) armed[s] = -1;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile tl = sc.tile(t);
      const int nblk = (tl.nrows + kBoxRows - 1) / kBoxRows;
      for (int ks = 0; ks < p.ksteps; ks += G) {
        if (!wait_bounded<kSpin>(empty0 + 8 * s, ph ^ 1u, misc + 1, p.status)) {
          ok = false;
          break;
        }
        const uint32_t fb = full0 + 8 * s;
        ptx::mbar_arrive_expect_tx(fb, G * (kABytes + nblk * kBBoxBytes));
        armed[s] = static_cast<int>(ph);
        const uint32_t a_dst = ptx::smem_u32(sA + s * G * kABytes);
        const uint32_t b_dst = ptx::smem_u32(sB + s * G * C::kBBytes);
        if (AMODE == 1) {
          const size_t chunk = (static_cast<size_t>(tl.e) * p.mblocks + tl.mb) * p.ksteps + ks;
          ptx::bulk_load(a_dst, p.tiles + chunk * kABytes, G * kABytes, fb, pol_w);
        } else {
#pragma unroll
          for (int j = 0; j < G; ++j) {
            const uint32_t aj = a_dst + j * kABytes;
            if (KIND == 0) {
#pragma unroll
              for (int b = 0; b < 4; ++b)
                ptx::tma_load_4d(aj + b * kGUBoxBytes, &tmA, fb, (ks + j) * kBK, tl.mb * 64 + b * 16, 0, tl.e,
                                 pol_w);
            } else if (KIND == 1) {
              ptx::tma_load_2d(aj, &tmA, fb, (ks + j) * kBK, tl.e * p.seg_rows + tl.mb * kBM, pol_w);
            } else {
              ptx::tma_load_2d(aj, &tmA, fb, (ks + j) * kBK, tl.mb * kBM, pol_w);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < G; ++j)
          for (int b = 0; b < nblk; ++b)
            ptx::tma_load_2d(b_dst + j * C::kBBytes + b * kBBoxBytes, &tmB, fb, (ks + j) * kBK,
                             tl.row0 + b * kBoxRows, pol_x);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok || misc[1]) {
      // abort: let every copy already issued land before the CTA exits
#pragma unroll
      for (int q = 0; q < S; ++q)
        if (armed[q] >= 0) wait_drain(full0 + 8 * q, static_cast<uint32_t>(armed[q]));
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    int s = 0;
    uint32_t ph = 0;
    int acc = 0;
    uint32_t aph = 0;
    bool ok = true;
    bool issued = false;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile tl = sc.tile(t);
      const uint32_t idesc = ptx::idesc_bf16_f32(kBM, static_cast<uint32_t>((tl.nrows + 15) & ~15));
      if (!wait_bounded<kSpin>(acce0 + 8 * acc, aph ^ 1u, misc + 1, p.status)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * NMAX);
      for (int ks = 0; ks < p.ksteps; ks += G) {
        if (!wait_bounded<kSpin>(full0 + 8 * s, ph, misc + 1, p.status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
#pragma unroll
        for (int j = 0; j < G; ++j)
          issue_k_step(d_tmem, ptx::smem_u32(sA + (s * G + j) * kABytes), ptx::smem_u32(sB + (s * G + j) * C::kBBytes),
                       idesc, ks + j);
        issued = true;
        ptx::umma_commit(empty0 + 8 * s);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      ptx::umma_commit(accf0 + 8 * acc);
      if (++acc == 2) {
        acc = 0;
        aph ^= 1u;
      }
    }
    if ((!ok || misc[1]) && issued) {
      ptx::umma_commit(drain);
      wait_drain(drain, 0);
    }
  } else if (warp >= 2) {
    epilogue_role<NMAX, KIND>(p, sc, total, tmem_base, accf0, acce0, misc + 1);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ============================================================== fused SwiGLU
// Gate/up and down of every routed expert in one persistent launch (tile-
// packed bf16 records).  The tile list is all gate/up tiles (expert-major)
// followed by all down tiles (expert-major); each CTA's producer claims the
// next tile from a device-wide queue and hands its index to the CTA's MMA
// issuer and epilogue through a small ring in shared memory.  A down tile of
// expert e may start once the gate/up tiles of e have stored their h rows:
// each of their epilogue warps fences its generic stores for the async proxy
// and bumps ready[e]; the producer of a down tile polls ready[e] (acquire,
// bounded) before its TMA loads of h.  Down tiles thus fill the SMs the
// gate/up tail would leave idle, and there is no kernel boundary between the
// two contractions.  The last CTA to exit resets the sync words to zero for
// the next call.
struct FusedArgs {
  const int32_t* offsets;
  int E, R;
  const uint8_t* tiles_gu;  // packed gate/up records
  const uint8_t* tiles_dn;  // packed down records
  int ks_gu, ks_dn;         // K steps per tile: H/64, I/64
  int mb_gu, mb_dn;         // weight blocks per expert: I/64, H/128
  uint16_t* h;              // [R, I]
  float* y;                 // [R, H]
  int I, H;
  int* ready;               // sync words: [E] per-expert h readiness, then the exit and gather counters
                            // and the tile queue
  int32_t* status;
  // Row gather (x != nullptr): the epilogue warps of every CTA copy its share
  // of the rows x_perm[s] = x[perm[s] / k] at the start of the launch, while
  // the producer already streams weights; the producers start their
  // token-row loads once all CTAs have done so.
  const uint16_t* x;
  uint16_t* x_perm;
  const int32_t* perm;
  int k;
  // Expert cache (CACHED kernels): expert e's records are record slot_of[e]
  // of tiles_gu / tiles_dn, pools of S records in HBM.
  const int32_t* slot_of;
  int S;
  // In-launch fetch (CACHED kernels, stats != nullptr): four more warps per
  // CTA copy the planned misses' records from host memory (host_gu /
  // host_dn, reached over the CPU-GPU link) into their slots in kFetchChunk
  // pieces, in wave order, while the other warps compute; the producer of a
  // missing expert's tile waits until its weight block has landed.  Sync
  // words: ready[E + 3] is the fetch queue, ready[E + 4 + e * (mb_gu + mb_dn)
  // + b] counts the landed pieces of expert e's weight block b (gate/up
  // blocks first, then down blocks).
  const uint8_t* host_gu;
  const uint8_t* host_dn;
  uint8_t* pool_gu;
  uint8_t* pool_dn;
  size_t rec_gu, rec_dn;  // record bytes
  int nch_gu, nch_dn;     // pieces per record
  const int32_t* miss_list;
  const int32_t* miss_slot;
  const int32_t* stats;   // [1]: number of misses
  int wave;               // wave width in experts
};

constexpr int kFetchWarps = 4;
constexpr int kFusedDynamicRows = 4096;  // launches up to this many rows claim tiles dynamically
constexpr int kFetchChunk = 32768;

// The n-th piece of the fetch plan in wave order (wave width W experts, cg /
// cd pieces per gate/up / down record): the gate/up records of wave 0, then
// for each later wave w its gate/up records followed by the down records of
// wave w - 1, then the down records of the last wave.  Gate/up arrive first
// because down is needed only once the SwiGLU intermediate exists.
struct FetchItem {
  int m, comp, c;  // miss index, 0 gate/up or 1 down, piece
};

__device__ __forceinline__ FetchItem fetch_item(int q, int n, int W, int cg, int cd) {
  const int nw = (n + W - 1) / W;
  const int L = n - (nw - 1) * W;  // experts in the last wave
  if (nw == 1) {
    if (q < n * cg) return {q / cg, 0, q % cg};
    q -= n * cg;
    return {q / cd, 1, q % cd};
  }
  if (q < W * cg) return {q / cg, 0, q % cg};
  q -= W * cg;
  const int bf = W * (cg + cd), nf = nw - 2;  // full waves 1 .. nw-2
  if (q < nf * bf) {
    const int w = 1 + q / bf;
    int r = q - (w - 1) * bf;
    if (r < W * cg) return {w * W + r / cg, 0, r % cg};
    r -= W * cg;
    return {(w - 1) * W + r / cd, 1, r % cd};
  }
  q -= nf * bf;
  if (q < L * cg) return {(nw - 1) * W + q / cg, 0, q % cg};
  q -= L * cg;
  if (q < W * cd) return {(nw - 2) * W + q / cd, 1, q % cd};
  q -= W * cd;
  return {(nw - 1) * W + q / cd, 1, q % cd};
}

template <int NMAX, int GG, bool CACHED>
struct CfgF {
  static constexpr int G = GG;
  static constexpr int kBBytes = NMAX * kBK * 2;
  static constexpr int kStageBytes = G * (kABytes + kBBytes);
  static constexpr int kBudget = 196 * 1024;
  static constexpr int kStages = kBudget / kStageBytes < 2 ? 2 : (kBudget / kStageBytes > 10 ? 10 : kBudget / kStageBytes);
  static constexpr int kTmemCols = 2 * NMAX < 32 ? 32 : 2 * NMAX;
  static constexpr int kTileRing = 4;  // tile ids the producer publishes ahead
  static constexpr int kNumBars = 2 * kStages + 5 + 2 * kTileRing;
  // misc words and the tile-id ring; offsets and the two tile prefixes;
  // cached: also slots and the expert order
  static constexpr int kTail = 32 + (CACHED ? 5 : 3) * (kMaxE + 1) * 4;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kNumBars * 8 + kTail;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

struct FTile {
  int kind;  // 0 gate/up, 1 down
  int j, e;  // position in the expert order, expert
  int mb, row0, nrows;
};

// The tiles one CTA runs, in order: its round-robin share of the gate/up
// tiles, then down tiles.  A gate/up tile costs wg K steps and a down tile wd;
// the CTAs left one gate/up tile short first take wg / wd down tiles each
// (the earliest experts' down tiles), and the rest of the down tiles go round
// robin from the first such CTA.  This levels the CTAs' total K steps to
// within one down tile, where plain round robin over the whole list can leave
// a CTA a gate/up tile plus a down tile above the mean.  Every role of the
// CTA walks the same sequence, and every tile is in exactly one CTA's.
struct FSeq {
  int b, P, tgu, tdn, g_b, li, fill, nfill, F, rr0;
  __device__ FSeq(int b_, int P_, int tgu_, int tdn_, int wg, int wd) : b(b_), P(P_), tgu(tgu_), tdn(tdn_) {
    g_b = tgu > b ? (tgu - 1 - b) / P + 1 : 0;
    const int r = tgu % P;
    const bool low = r != 0 && b >= r;
    fill = (r != 0 && wd > 0) ? max(wg / wd, 1) : 0;
    F = min((r != 0 ? P - r : 0) * fill, tdn);
    li = b - r;
    nfill = low ? min(max(F - li * fill, 0), fill) : 0;
    rr0 = ((b - r) % P + P) % P;
  }
  // Index (gate/up tiles first, then down tiles) of the n-th tile, or -1.
  __device__ int tile(int n) const {
    if (n < g_b) return b + n * P;
    n -= g_b;
    if (n < nfill) return tgu + li * fill + n;
    n -= nfill;
    const int d = F + rr0 + n * P;
    return d < tdn ? tgu + d : -1;
  }
  __device__ int count() const {
    const int rest = tdn - F - rr0;
    return g_b + nfill + (rest > 0 ? (rest - 1) / P + 1 : 0);
  }
};

// With an expert cache: the tiles of the experts already resident (phase A:
// their gate/up, then their down tiles) come before those of the experts
// being fetched (phase B), so no CTA holds resident work behind a tile that
// waits for the link.  Phase A is levelled as FSeq levels the whole list;
// phase B, whose tiles wait for the link rather than for compute, gives the
// CTAs after its gate/up tiles one down tile each before any CTA gets two.
// Returns the index in the combined list (all gate/up tiles by position in
// the expert order, then all down tiles), or -1.
struct FOrder {
  FSeq a, b;
  int na, tguA, tdnA, tguB, total_gu;
  __device__ FOrder(int blk, int P, int tguA_, int tdnA_, int tguB_, int tdnB_, int wg, int wd)
      : a(blk, P, tguA_, tdnA_, wg, wd),
        b(blk, P, tguB_, tdnB_, 1, 1),
        na(a.count()),
        tguA(tguA_),
        tdnA(tdnA_),
        tguB(tguB_),
        total_gu(tguA_ + tguB_) {}
  __device__ int tile(int n) const {
    if (n < na) {
      const int t = a.tile(n);
      return t < tguA ? t : total_gu + (t - tguA);
    }
    const int t = b.tile(n - na);
    if (t < 0) return -1;
    return t < tguB ? tguA + t : total_gu + tdnA + (t - tguB);
  }
};

// Decode-sized launches instead claim tiles from a device-wide queue (one
// atomic per tile) in a global order: all gate/up tiles, then all down
// tiles.  A CTA that finishes early takes the next tile, so the CTAs end
// within about one tile of each other whatever bandwidth each one sees (the
// static order leaves a spread of several microseconds at the end of a
// decode launch); on large launches the static order measured faster.  A down tile waits for the gate/up
// tiles of its expert, which all come earlier in the queue and wait for
// nothing, so every wait ends.  With an expert cache the order is: the
// resident experts' gate/up tiles, their down tiles, then the fetched
// experts' gate/up and down tiles (which also wait for the link), so no
// resident work queues behind a tile that waits for the link.  Returns the
// index in the combined list (all gate/up tiles by position in the expert
// order, then all down tiles).
__device__ __forceinline__ int fused_tile_at(int g, int tguA, int tdnA, int tguB, int total_gu) {
  if (g < tguA) return g;
  g -= tguA;
  if (g < tdnA) return total_gu + g;
  g -= tdnA;
  if (g < tguB) return tguA + g;
  return total_gu + tdnA + (g - tguB);
}

// The fetch warps of a cached launch: each warp claims the next piece of the
// plan, copies it host -> slot with eight 16-byte loads in flight per lane,
// fences its stores for the TMA reads of other CTAs, and counts the piece as
// landed in its weight block's word.
__device__ __forceinline__ void fetch_records(const FusedArgs& p, int E, int n, int lane) {
  if (n <= 0) return;
  const int W = max(1, min(p.wave, n));
  const int total = n * (p.nch_gu + p.nch_dn);
  for (;;) {
    int q = 0;
    if (lane == 0) q = atomicAdd(p.ready + E + 3, 1);
    q = __shfl_sync(0xffffffffu, q, 0);
    if (q >= total) break;
    const FetchItem f = fetch_item(q, n, W, p.nch_gu, p.nch_dn);
    const int e = p.miss_list[f.m], sl = p.miss_slot[f.m];
    const bool valid = e >= 0 && e < E && sl >= 0 && sl < p.S;
    if (valid) {
      const size_t rec = f.comp ? p.rec_dn : p.rec_gu;
      const size_t off = static_cast<size_t>(f.c) * kFetchChunk;
      const int nv = static_cast<int>(min(rec - off, static_cast<size_t>(kFetchChunk)) / 16);
      const uint4* src = reinterpret_cast<const uint4*>((f.comp ? p.host_dn : p.host_gu) + e * rec + off);
      uint4* dst = reinterpret_cast<uint4*>((f.comp ? p.pool_dn : p.pool_gu) + sl * rec + off);
      constexpr int U = 8;
      for (int i0 = lane; i0 < nv; i0 += U * 32) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (i0 + u * 32 < nv) v[u] = src[i0 + u * 32];
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (i0 + u * 32 < nv) dst[i0 + u * 32] = v[u];
      }
      fence_proxy_async_global();
    } else if (lane == 0) {
      set_status(p.status, MOE_DEV_BAD_EXPERT);
    }
    __threadfence();
    __syncwarp();
    if (lane == 0 && valid) {
      // pieces never straddle a weight block: a block is ks / 2 pieces
      const int blk = f.comp ? p.mb_gu + f.c / (p.ks_dn / 2) : f.c / (p.ks_gu / 2);
      atomicAdd(p.ready + E + 4 + e * (p.mb_gu + p.mb_dn) + blk, 1);
    }
  }
}

template <int NMAX, int GG, bool CACHED>
__global__ void __launch_bounds__(kCoreThreads + (CACHED ? 32 * kFetchWarps : 0), 1)
    grouped_swiglu_fused_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmH,
                                FusedArgs p) {
  using C = CfgF<NMAX, GG, CACHED>;
  // the compute warps' barrier: all threads, or, with fetch warps that run
  // on their own, a named barrier of the first kCoreThreads
  auto compute_sync = [] {
    if constexpr (CACHED) {
      asm volatile("bar.sync 1, %0;" ::"n"(kCoreThreads) : "memory");
    } else {
      __syncthreads();
    }
  };
  constexpr int S = C::kStages;
  constexpr int G = C::G;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = sA + S * G * kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + S * G * C::kBBytes);
  const uint32_t full0 = ptx::smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * S;
  const uint32_t accf0 = empty0 + 8 * S;
  const uint32_t acce0 = accf0 + 16;
  const uint32_t drain = acce0 + 16;
  constexpr int QR = C::kTileRing;
  const uint32_t tqf0 = drain + 8;          // tile id published (QR slots)
  const uint32_t tqe0 = tqf0 + 8 * QR;      // tile id read by the MMA issuer and the 4 epilogue warps
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(bars + C::kNumBars);
  volatile int* tq = reinterpret_cast<volatile int*>(misc + 4);  // [QR] tile ids
  int* pre_gu = const_cast<int*>(reinterpret_cast<volatile int*>(misc + 8));
  int* pre_dn = pre_gu + (kMaxE + 1);
  int* soff = pre_dn + (kMaxE + 1);
  int* sslot = soff + (kMaxE + 1);  // cached: slot of each expert
  int* eord = sslot + (kMaxE + 1);  // cached: expert at each position of the tile order

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int E = p.E;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(full0 + 8 * s, 1);
      ptx::mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(accf0 + 8 * a, 1);
      ptx::mbar_init(acce0 + 8 * a, 128);
    }
    ptx::mbar_init(drain, 1);
    for (int q = 0; q < QR; ++q) {
      ptx::mbar_init(tqf0 + 8 * q, 1);
      ptx::mbar_init(tqe0 + 8 * q, 1 + 4);
    }
    misc[1] = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmX);
    ptx::prefetch_tmap(&tmH);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(const_cast<uint32_t*>(&misc[0])), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  pdl_wait();
  pdl_trigger();
  const int nmiss = (CACHED && p.stats != nullptr) ? min(max(p.stats[1], 0), min(E, p.S)) : 0;
  if (CACHED && warp >= 6) {
    // ------------------------------------------------------------ fetch
    // The fetch warps start at once; the compute warps' set-up below syncs
    // on a named barrier of their own.
    fetch_records(p, E, nmiss, lane);
  } else {
  for (int i = threadIdx.x; i <= E; i += kCoreThreads) soff[i] = min(max(p.offsets[i], 0), p.R);
  if constexpr (CACHED) {
    for (int i = threadIdx.x; i < E; i += kCoreThreads) {
      int rec = p.slot_of[i];
      // a routed expert without a slot (the cache could not hold the call):
      // flag it and read slot 0, so every access stays inside the pool
      if (rec < 0 || rec >= p.S) {
        if (p.offsets[i + 1] > p.offsets[i]) set_status(p.status, MOE_DEV_CACHE_FULL);
        rec = 0;
      }
      sslot[i] = rec;
      eord[i] = i;
      pre_dn[i] = -1;  // fetch-plan position of each expert until the prefix pass
    }
    if (nmiss > 0) {
      compute_sync();
      for (int m = threadIdx.x; m < nmiss; m += kCoreThreads) {
        const int e = p.miss_list[m];
        if (e >= 0 && e < E) pre_dn[e] = m;
      }
    }
  }
  compute_sync();
  if (warp == 0) {
    if (CACHED && nmiss > 0) {
      // tile order: the experts that are resident (ID order), then the ones
      // being fetched, in fetch-plan order, so resident experts compute while
      // the records of the others are in flight
      int run = 0;
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const int mp = e < E ? pre_dn[e] : 0;
        const bool keep = e < E && mp < 0;
        const unsigned bal = __ballot_sync(0xffffffffu, keep);
        if (keep) {
          eord[run + __popc(bal & ((1u << lane) - 1u))] = e;
        } else if (e < E) {
          eord[E - nmiss + mp] = e;
        }
        run += __popc(bal);
      }
      __syncwarp();
    }
    int run_gu = 0, run_dn = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int j = e0 + lane;
      int n = 0;
      if (j < E) {
        const int e = CACHED ? eord[j] : j;
        n = max(soff[e + 1] - soff[e], 0);
      }
      const int chunks = (n + NMAX - 1) / NMAX;
      int a = chunks * p.mb_gu, b = chunks * p.mb_dn;
      int ia = a, ib = b;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int ya = __shfl_up_sync(0xffffffffu, ia, d);
        const int yb = __shfl_up_sync(0xffffffffu, ib, d);
        if (lane >= d) {
          ia += ya;
          ib += yb;
        }
      }
      __syncwarp();
      if (j < E) {
        pre_gu[j] = run_gu + ia - a;
        pre_dn[j] = run_dn + ib - b;
      }
      run_gu += __shfl_sync(0xffffffffu, ia, 31);
      run_dn += __shfl_sync(0xffffffffu, ib, 31);
    }
    if (lane == 0) {
      pre_gu[E] = run_gu;
      pre_dn[E] = run_dn;
    }
  }
  ptx::tc_fence_before();
  compute_sync();
  ptx::tc_fence_after();
  const uint32_t tmem_base = misc[0];
  const int total_gu = pre_gu[E];
  const int total = total_gu + pre_dn[E];
  const int jB = E - nmiss;  // first position of a fetched expert
  const int tguA = pre_gu[jB], tdnA = pre_dn[jB], tguB = total_gu - tguA;
  int* const queue = p.ready + E + 2;  // device-wide tile queue
  const bool dynamic = p.R <= kFusedDynamicRows;
  const FSeq seq1(blockIdx.x, gridDim.x, total_gu, pre_dn[E], p.ks_gu, p.ks_dn);
  const FOrder seq2(blockIdx.x, gridDim.x, tguA, tdnA, tguB, pre_dn[E] - tdnA, p.ks_gu, p.ks_dn);
  // the MMA issuer and the epilogue warps follow the producer's tile ids
  auto read_tile = [&](int& qs, uint32_t& qph, int* t) -> bool {
    if (!wait_bounded<kSpin>(tqf0 + 8 * qs, qph, misc + 1, p.status)) return false;
    *t = tq[qs];
    return true;
  };

  auto tile_of = [&](int t) {
    FTile tl;
    tl.kind = t >= total_gu;
    const int* pre = tl.kind ? pre_dn : pre_gu;
    const int tt = tl.kind ? t - total_gu : t;
    const int mbk = tl.kind ? p.mb_dn : p.mb_gu;
    int lo = 0, hi = E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pre[mid] <= tt) lo = mid; else hi = mid;
    }
    const int local = tt - pre[lo];
    const int chunk = local / mbk;
    tl.j = lo;
    tl.e = CACHED ? eord[lo] : lo;
    const int start = soff[tl.e];
    const int len = max(soff[tl.e + 1] - start, 0);
    tl.mb = local - chunk * mbk;
    tl.row0 = start + chunk * NMAX;
    tl.nrows = min(NMAX, len - chunk * NMAX);
    return tl;
  };

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_w = ptx::policy_evict_first();
    const uint64_t pol_x = ptx::policy_evict_last();
    int armed[S];
#pragma unroll
    for (int s = 0; s < S; ++s) armed[s] = -1;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    int ready_e = -1;  // expert whose h rows are known to be complete
    // Until every CTA has gathered its token rows, stages get their weight
    // chunk at once and their token rows later (at most S stages deferred).
    bool gathered = p.x == nullptr;
    int npend = 0;
    uint32_t pend_dst[S], pend_bar[S];
    int pend_ks[S], pend_row[S], pend_nblk[S];
    auto flush_pending = [&]() -> bool {
      if (!gathered) {
        uint64_t t0 = 0;
        for (uint32_t it = 0; ld_acquire_gpu(p.ready + E + 1) < static_cast<int>(gridDim.x); ++it) {
          __nanosleep(32);
          if ((it & 1023u) == 1023u) {
            if (misc[1]) return false;
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) {
              t0 = now;
            } else if (now - t0 > kWaitNs) {
              misc[1] = 1;
              set_status(p.status, MOE_DEV_TIMEOUT);
              return false;
            }
          }
        }
        fence_proxy_async_global();
        gathered = true;
      }
      for (int q = 0; q < npend; ++q)
        for (int j = 0; j < G; ++j)
          for (int b = 0; b < pend_nblk[q]; ++b)
            ptx::tma_load_2d(pend_dst[q] + j * C::kBBytes + b * kBBoxBytes, &tmX, pend_bar[q], (pend_ks[q] + j) * kBK,
                             pend_row[q] + b * kBoxRows, pol_x);
      npend = 0;
      return true;
    };
    int qs = 0;
    uint32_t qph = 0;
    int next = dynamic ? atomicAdd(queue, 1) : 0;
    for (int n = 0; ok; ++n) {
      int t;
      if (dynamic) {
        const int g = next;
        t = g < total ? (CACHED ? fused_tile_at(g, tguA, tdnA, tguB, total_gu) : g) : -1;
        if (t >= 0) next = atomicAdd(queue, 1);  // the following claim, in flight while this tile's loads go out
      } else {
        t = CACHED ? seq2.tile(n) : seq1.tile(n);
      }
      // publish the tile id for the MMA issuer and the epilogue
      if (!wait_bounded<kSpin>(tqe0 + 8 * qs, qph ^ 1u, misc + 1, p.status)) {
        ok = false;
        break;
      }
      tq[qs] = t;
      ptx::mbar_arrive(tqf0 + 8 * qs);
      if (++qs == QR) {
        qs = 0;
        qph ^= 1u;
      }
      if (t < 0) break;
      const FTile tl = tile_of(t);
      const int nblk = (tl.nrows + kBoxRows - 1) / kBoxRows;
      const int KS = tl.kind ? p.ks_dn : p.ks_gu;
      const uint8_t* wt = tl.kind ? p.tiles_dn : p.tiles_gu;
      const CUtensorMap* tb = tl.kind ? &tmH : &tmX;
      if (tl.kind && (npend > 0 || !gathered) && !flush_pending()) {
        ok = false;
        break;
      }
      if (tl.kind && tl.e != ready_e) {
        // wait until every gate/up tile of expert e has stored its h rows
        // (each tile's four epilogue warps arrive once)
        const int target = 4 * (pre_gu[tl.j + 1] - pre_gu[tl.j]);
        uint64_t t0 = 0;
        for (uint32_t it = 0; ld_acquire_gpu(p.ready + tl.e) < target; ++it) {
          __nanosleep(64);
          if ((it & 1023u) == 1023u) {
            if (misc[1]) {
              ok = false;
              break;
            }
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) {
              t0 = now;
            } else if (now - t0 > kWaitNs) {
              misc[1] = 1;
              set_status(p.status, MOE_DEV_TIMEOUT);
              ok = false;
              break;
            }
          }
        }
        if (!ok) break;
        fence_proxy_async_global();
        ready_e = tl.e;
      }
      if (CACHED && tl.j >= jB) {
        // a fetched expert: wait until the pieces of this tile's weight block
        // have landed in its slot
        const int* word = p.ready + E + 4 + tl.e * (p.mb_gu + p.mb_dn) + (tl.kind ? p.mb_gu : 0) + tl.mb;
        const int target = (tl.kind ? p.ks_dn : p.ks_gu) / 2;
        uint64_t t0 = 0;
        for (uint32_t it = 0; ld_acquire_gpu(word) < target; ++it) {
          __nanosleep(64);
          if ((it & 1023u) == 1023u) {
            if (misc[1]) {
              ok = false;
              break;
            }
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) {
              t0 = now;
            } else if (now - t0 > kWaitNs) {
              misc[1] = 1;
              set_status(p.status, MOE_DEV_TIMEOUT);
              ok = false;
              break;
            }
          }
        }
        if (!ok) break;
        fence_proxy_async_global();
      }
      const int rec = CACHED ? sslot[tl.e] : tl.e;
      const size_t chunk0 = (static_cast<size_t>(rec) * (tl.kind ? p.mb_dn : p.mb_gu) + tl.mb) * KS;
      for (int ks = 0; ks < KS; ks += G) {
        if (!wait_bounded<kSpin>(empty0 + 8 * s, ph ^ 1u, misc + 1, p.status)) {
          ok = false;
          break;
        }
        const uint32_t fb = full0 + 8 * s;
        ptx::mbar_arrive_expect_tx(fb, G * (kABytes + nblk * kBBoxBytes));
        armed[s] = static_cast<int>(ph);
        const uint32_t a_dst = ptx::smem_u32(sA + s * G * kABytes);
        const uint32_t b_dst = ptx::smem_u32(sB + s * G * C::kBBytes);
        ptx::bulk_load(a_dst, wt + (chunk0 + ks) * kABytes, G * kABytes, fb, pol_w);
        if (!gathered) {
          pend_dst[npend] = b_dst;
          pend_bar[npend] = fb;
          pend_ks[npend] = ks;
          pend_row[npend] = tl.row0;
          pend_nblk[npend] = nblk;
          if (++npend == S && !flush_pending()) {
            ok = false;
            break;
          }
        } else {
#pragma unroll
          for (int j = 0; j < G; ++j)
            for (int b = 0; b < nblk; ++b)
              ptx::tma_load_2d(b_dst + j * C::kBBytes + b * kBBoxBytes, tb, fb, (ks + j) * kBK,
                               tl.row0 + b * kBoxRows, pol_x);
        }
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (ok && npend > 0 && !flush_pending()) ok = false;
    }
    if (!ok || misc[1]) {
#pragma unroll
      for (int q = 0; q < S; ++q)
        if (armed[q] >= 0) wait_drain(full0 + 8 * q, static_cast<uint32_t>(armed[q]));
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    int s = 0;
    uint32_t ph = 0;
    int acc = 0;
    uint32_t aph = 0;
    bool ok = true;
    bool issued = false;
    int qs = 0;
    uint32_t qph = 0;
    while (ok) {
      int t = -1;
      if (!read_tile(qs, qph, &t)) {
        ok = false;
        break;
      }
      ptx::mbar_arrive(tqe0 + 8 * qs);
      if (++qs == QR) {
        qs = 0;
        qph ^= 1u;
      }
      if (t < 0) break;
      const FTile tl = tile_of(t);
      const int KS = tl.kind ? p.ks_dn : p.ks_gu;
      const uint32_t idesc = ptx::idesc_bf16_f32(kBM, static_cast<uint32_t>((tl.nrows + 15) & ~15));
      if (!wait_bounded<kSpin>(acce0 + 8 * acc, aph ^ 1u, misc + 1, p.status)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * NMAX);
      for (int ks = 0; ks < KS; ks += G) {
        if (!wait_bounded<kSpin>(full0 + 8 * s, ph, misc + 1, p.status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
#pragma unroll
        for (int j = 0; j < G; ++j)
          issue_k_step(d_tmem, ptx::smem_u32(sA + (s * G + j) * kABytes), ptx::smem_u32(sB + (s * G + j) * C::kBBytes),
                       idesc, ks + j);
        issued = true;
        ptx::umma_commit(empty0 + 8 * s);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      ptx::umma_commit(accf0 + 8 * acc);
      if (++acc == 2) {
        acc = 0;
        aph ^= 1u;
      }
    }
    if ((!ok || misc[1]) && issued) {
      ptx::umma_commit(drain);
      wait_drain(drain, 0);
    }
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------------ epilogue
    if (p.x != nullptr) {
      // Row gather, done here so that it overlaps the first weight loads:
      // this CTA's contiguous share of the permuted token rows, eight 16-byte
      // loads in flight per thread.  The producers start their token-row
      // loads once every CTA has published its share.
      constexpr int kEpiThreads = 128;
      const int et = threadIdx.x - 64;
      const int s0 = static_cast<int>(static_cast<long long>(p.R) * blockIdx.x / gridDim.x);
      const int s1 = static_cast<int>(static_cast<long long>(p.R) * (blockIdx.x + 1) / gridDim.x);
      const int vpr = p.H / 8;
      const int n = (s1 - s0) * vpr;
      constexpr int U = 8;
      for (int i0 = et; i0 < n; i0 += U * kEpiThreads) {
        uint4 v[U];
        int dst[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = i0 + u * kEpiThreads;
          dst[u] = -1;
          if (i < n) {
            const int sl = s0 + i / vpr;
            const int c = i - (sl - s0) * vpr;
            const int r = p.perm[sl];
            if (r >= 0 && r < p.R) {
              v[u] = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(r / p.k) * p.H)[c];
              dst[u] = sl * vpr + c;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (dst[u] >= 0) reinterpret_cast<uint4*>(p.x_perm)[dst[u]] = v[u];
      }
      // publish to the TMA loads of every CTA: fence for the async proxy, then
      // one arrival per CTA
      fence_proxy_async_global();
      __threadfence();
      asm volatile("bar.sync 2, %0;" ::"n"(kEpiThreads) : "memory");
      if (et == 0) atomicAdd(p.ready + E + 1, 1);
    }
    const int q = warp & 3;
    const int row_in_tile = q * 32 + lane;
    int acc = 0;
    uint32_t aph = 0;
    int qs = 0;
    uint32_t qph = 0;
    for (;;) {
      int t = -1;
      if (!__all_sync(0xffffffffu, read_tile(qs, qph, &t))) break;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(tqe0 + 8 * qs);
      if (++qs == QR) {
        qs = 0;
        qph ^= 1u;
      }
      if (t < 0) break;
      const FTile tl = tile_of(t);
      const bool ok = wait_bounded<kSleepEpi>(accf0 + 8 * acc, aph, misc + 1, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      ptx::tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * NMAX);
      if (tl.kind == 0) {
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
            if (col < tl.nrows)
              p.h[static_cast<size_t>(tl.row0 + col) * p.I + i] = f32_to_bf16(g / (1.0f + expf(-g)) * u);
          }
        }
        // publish this warp's h rows to TMA loads in other CTAs: each lane
        // fences its own stores, then one arrival per warp (4 per tile)
        fence_proxy_async_global();
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(p.ready + tl.e, 1);
      } else {
        const int j = tl.mb * kBM + row_in_tile;
        for (int c0 = 0; c0 < tl.nrows; c0 += 16) {
          float v[16];
          ptx::tmem_ld16(taddr + static_cast<uint32_t>(c0), v);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int col = c0 + jj;
            if (col < tl.nrows) p.y[static_cast<size_t>(tl.row0 + col) * p.H + j] = v[jj];
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
  }  // compute warps

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(misc[0], C::kTmemCols);
  }
  // The last CTA out resets the sync words for the next call.
  if (threadIdx.x == 0) {
    __threadfence();
    misc[2] = atomicAdd(p.ready + E, 1) == static_cast<int>(gridDim.x) - 1;
  }
  __syncthreads();
  if (misc[2]) {
    __threadfence();
    for (int e = threadIdx.x; e < (CACHED ? E + 4 : E + 3); e += blockDim.x) p.ready[e] = 0;
    if (CACHED && nmiss > 0) {
      const int nb = p.mb_gu + p.mb_dn;
      for (int i = threadIdx.x; i < nmiss * nb; i += blockDim.x) {
        const int e = p.miss_list[i / nb];
        if (e >= 0 && e < E) p.ready[E + 4 + e * nb + i % nb] = 0;
      }
    }
    __threadfence();
  }
}

// ============================================================== int4 kernel
// QG (packed chunks per bulk copy) is a template parameter so that the ring
// positions of a K step are shifts and masks, not divisions: the per-step
// bookkeeping runs once per 4.3 KB of weights and must stay cheap.
template <int NMAX, int KIND, int QG>
__global__ void __launch_bounds__(CfgQ<NMAX>::kThreads, 1)
    grouped_gemm_q4_kernel(const __grid_constant__ CUtensorMap tmB, GemmArgs p) {
  using C = CfgQ<NMAX>;
  constexpr int SA = C::SA, SB = C::SB;
  constexpr int SQ = C::SQmax / QG;  // logical slots of QG chunks each
  static_assert(C::SQmax % QG == 0, "ring holds whole groups");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sB = base;                  // [SB][NMAX x 128 B] token rows (swizzled)
  uint8_t* sQ = sB + SB * C::kBBytes;  // [SQ][QG x 4,352 B] packed codes + scales
  uint64_t* bars = reinterpret_cast<uint64_t*>(sQ + C::kQRingBytes);
  const uint32_t qfull0 = ptx::smem_u32(bars);      // packed chunks landed
  const uint32_t qempty0 = qfull0 + 8 * C::SQmax;   // dequantisers done reading them
  const uint32_t afull0 = qempty0 + 8 * C::SQmax;   // operand slot written (TMEM)
  const uint32_t aempty0 = afull0 + 8 * SA;     // MMA done with the slot
  const uint32_t bfull0 = aempty0 + 8 * SA;     // token rows landed
  const uint32_t bempty0 = bfull0 + 8 * SB;     // MMA done with the rows
  const uint32_t accf0 = bempty0 + 8 * SB;
  const uint32_t acce0 = accf0 + 16;
  const uint32_t drain = acce0 + 16;
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(bars + C::kNumBars);
  int* prefix = const_cast<int*>(reinterpret_cast<volatile int*>(misc + 4));
  int* soff = prefix + (kMaxE + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int E = p.E;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SQ; ++s) {
      ptx::mbar_init(qfull0 + 8 * s, 1);
      ptx::mbar_init(qempty0 + 8 * s, QG * 4);  // each chunk is read by the four warps of one group
    }
    for (int s = 0; s < SA; ++s) {
      ptx::mbar_init(afull0 + 8 * s, 4);
      ptx::mbar_init(aempty0 + 8 * s, 1);
    }
    for (int s = 0; s < SB; ++s) {
      ptx::mbar_init(bfull0 + 8 * s, 1);
      ptx::mbar_init(bempty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(accf0 + 8 * a, 1);
      ptx::mbar_init(acce0 + 8 * a, 128);
    }
    ptx::mbar_init(drain, 1);
    misc[1] = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(const_cast<uint32_t*>(&misc[0])), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  pdl_wait();
  pdl_trigger();
  const int total = build_schedule<NMAX>(p, false, E, prefix, soff);
  const uint32_t tmem_base = misc[0];
  const Sched sc{prefix, soff, E, p.mblocks, NMAX};

  if ((warp == 0 || warp == 6) && lane == 0) {
    // ------------------------------------------------- producers: warp 0 moves
    // packed weight chunks (deep ring), warp 6 moves token rows (B ring); one
    // thread each, in separate warps so neither spin starves the other
    const bool weights = (warp == 0);
    const int S = weights ? SQ : SB;
    const uint32_t full0 = weights ? qfull0 : bfull0;
    const uint32_t empty0 = weights ? qempty0 : bempty0;
    const uint64_t pol = weights ? ptx::policy_evict_first() : ptx::policy_evict_last();
    uint32_t armed_mask = 0, armed_ph = 0;  // bit s: stage s armed / its parity
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile tl = sc.tile(t);
      const int nblk = (tl.nrows + kBoxRows - 1) / kBoxRows;
      for (int ks = 0; ks < p.ksteps; ks += (weights ? QG : 1)) {
        if (!wait_bounded<kSpin>(empty0 + 8 * s, ph ^ 1u, misc + 1, p.status)) {
          ok = false;
          break;
        }
        const uint32_t fb = full0 + 8 * s;
        armed_mask |= 1u << s;
        armed_ph = (armed_ph & ~(1u << s)) | (ph << s);
        if (weights) {
          ptx::mbar_arrive_expect_tx(fb, QG * kQChunk);
          const size_t chunk = (static_cast<size_t>(tl.e) * p.mblocks + tl.mb) * p.ksteps + ks;
          ptx::bulk_load(ptx::smem_u32(sQ + s * QG * kQChunk), p.tiles + chunk * kQChunk, QG * kQChunk, fb, pol);
        } else {
          ptx::mbar_arrive_expect_tx(fb, nblk * kBBoxBytes);
          const uint32_t b_dst = ptx::smem_u32(sB + s * C::kBBytes);
          for (int b = 0; b < nblk; ++b)
            ptx::tma_load_2d(b_dst + b * kBBoxBytes, &tmB, fb, ks * kBK, tl.row0 + b * kBoxRows, pol);
        }
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok || misc[1]) {
      for (int q = 0; q < S; ++q)
        if ((armed_mask >> q) & 1u) wait_drain(full0 + 8 * q, (armed_ph >> q) & 1u);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    int sa = 0, sb = 0;
    uint32_t pha = 0, phb = 0;
    int acc = 0;
    uint32_t aph = 0;
    bool ok = true;
    bool issued = false;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile tl = sc.tile(t);
      const uint32_t idesc = ptx::idesc_bf16_f32(kBM, static_cast<uint32_t>((tl.nrows + 15) & ~15));
      if (!wait_bounded<kSpin>(acce0 + 8 * acc, aph ^ 1u, misc + 1, p.status)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * NMAX);
      for (int ks = 0; ks < p.ksteps; ++ks) {
        if (!wait_bounded<kSpin>(afull0 + 8 * sa, pha, misc + 1, p.status) ||
            !wait_bounded<kSpin>(bfull0 + 8 * sb, phb, misc + 1, p.status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t a_tmem = tmem_base + static_cast<uint32_t>(C::kTmemA + sa * 32);
        const uint32_t b0 = ptx::smem_u32(sB + sb * C::kBBytes);
#pragma unroll
        for (int kk = 0; kk < kBK / kUK; ++kk)
          ptx::umma_bf16_ts(d_tmem, a_tmem + static_cast<uint32_t>(kk * kUK / 2), ptx::sdesc_k_sw128(b0 + kk * kUK * 2),
                            idesc, (ks | kk) != 0 ? 1u : 0u);
        issued = true;
        ptx::umma_commit(aempty0 + 8 * sa);
        ptx::umma_commit(bempty0 + 8 * sb);
        if (++sa == SA) {
          sa = 0;
          pha ^= 1u;
        }
        if (++sb == SB) {
          sb = 0;
          phb ^= 1u;
        }
      }
      if (!ok) break;
      ptx::umma_commit(accf0 + 8 * acc);
      if (++acc == 2) {
        acc = 0;
        aph ^= 1u;
      }
    }
    if ((!ok || misc[1]) && issued) {
      ptx::umma_commit(drain);
      wait_drain(drain, 0);
    }
  } else if (warp >= 2 && warp < 6) {
    epilogue_role<NMAX, KIND>(p, sc, total, tmem_base, accf0, acce0, misc + 1);
  } else if (warp >= C::kDqWarp0) {
    // ------------------------------------------------------------ dequantisers
    // Group j of four warps takes K steps g = j, j + kDqGroups, ... of this
    // CTA's stream; lane l of the group's warp for lane quarter q converts
    // row 32 q + l (64 inputs) into 32 TMEM columns of operand slot g % SA.
    // A warp's TMEM store of one step completes while it loads and converts
    // its next step; only then does it mark the slot full.  Each warp frees
    // the packed chunk as soon as its codes are read.
    const int dw = warp - C::kDqWarp0;
    const int grp = dw / 4;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                               static_cast<uint32_t>(C::kTmemA);
    uint32_t g = 0;  // this CTA's running K-step index
    bool ok = true;
    int pending = -1;  // slot whose store is in flight
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      for (int ks = 0; ks < p.ksteps; ++ks, ++g) {
        if (static_cast<int>(g % C::kDqGroups) != grp) continue;
        const uint32_t gg = g / QG;  // ring group (QG consecutive K steps)
        const uint32_t sq = gg % SQ;
        const uint32_t phq = (gg / SQ) & 1u;
        const uint32_t sa = g % SA;
        const uint32_t pha = (g / SA) & 1u;
        bool got = wait_bounded<kSpin>(qfull0 + 8 * sq, phq, misc + 1, p.status);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const uint8_t* chunk = sQ + (sq * QG + (g - gg * QG)) * kQChunk;
        const uint4 qa = reinterpret_cast<const uint4*>(chunk + row * 32)[0];
        const uint4 qb = reinterpret_cast<const uint4*>(chunk + row * 32)[1];
        const uint16_t sbits = reinterpret_cast<const uint16_t*>(chunk + kQBytes)[row];
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(qempty0 + 8 * sq);
        __nv_bfloat16 scv;
        std::memcpy(&scv, &sbits, 2);
        const __nv_bfloat162 sc2 = __halves2bfloat162(scv, scv);
        uint32_t cols[32];
        const uint32_t words[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const uint4 d = dequant8(words[w], sc2);  // inputs 8w .. 8w + 7 as four bf16 pairs
          cols[4 * w] = d.x;
          cols[4 * w + 1] = d.y;
          cols[4 * w + 2] = d.z;
          cols[4 * w + 3] = d.w;
        }
        if (pending >= 0) {  // the previous step's columns are in TMEM: publish them
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(afull0 + 8 * pending);
          pending = -1;
        }
        got = wait_bounded<kSpin>(aempty0 + 8 * sa, pha ^ 1u, misc + 1, p.status);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        ptx::tmem_st32(lane_base + sa * 32, cols);
        pending = static_cast<int>(sa);
      }
    }
    ptx::tmem_wait_st();
    if (pending >= 0 && ok) {
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(afull0 + 8 * pending);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ============================================================ int4 GEMV
// Decode-sized int4 tiles.  With about one token row per expert a tile is a
// matrix-vector product, and what limits it is instructions per weight, not
// MMA throughput: a tcgen05 MMA must read its operands from shared or tensor
// memory, so the codes of each K step would be expanded into a 16 KB bf16
// tile and read back (measured: ~0.35 us per 4.3 KB step), while a CUDA-core
// dot product spends ~6 instructions per weight.  Here the weights go from
// registers straight into warp-level MMAs (mma.sync m16n8k16, bf16 in, fp32
// accumulate): each code pair becomes an exact bf16 pair (code - 8) in three
// instructions, token values enter as bf16 with no conversion, and one MMA
// instruction consumes 256 weights against up to 8 token rows.
//
// Warps: 0 streams packed chunks (bulk copies, deep ring), 1 stages each
// tile's token rows (one bulk copy per row, double-buffered), the rest
// compute in kGvGroups groups of four.  The groups take K steps in turn, so
// each warp has several steps' time for the latency chain of one (wait,
// loads, dequantise, MMAs).  Warp w of a group owns tile rows 32w .. 32w + 31
// as two MMA row tiles that share the token fragments: per K step (one scale
// group of 64 inputs) it runs eight MMAs from zero and adds scale x partial
// to its fp32 accumulators.  In a gate/up record rows 32w .. 32w + 15 are gate
// and 32w + 16 .. 32w + 31 the up rows of the same h columns, so each lane
// ends a tile holding gate and up of the same outputs.  At the end of a tile
// groups 1.. hand their sums (valid token columns only) to group 0 through
// shared memory, which adds them in group order (a fixed order: same bits
// every call) and stores y, or h = silu(gate) * up.  Token columns past the
// tile's rows read stale staged rows and are never stored (an MMA column
// depends on its own B column only).
constexpr int kGvRows = 4;                     // token rows per tile
constexpr int kGvN = 8;                        // MMA N: token columns (those past kGvRows are never stored)
constexpr int kGvGroups = 4;
constexpr int kGvWpg = 4;                      // compute warps per group, 32 rows each
constexpr int kGvWarps = 2 + kGvWpg * kGvGroups;
constexpr int kGvThreads = 32 * kGvWarps;
constexpr int kGvMaxK = 2560;                  // inputs per row the token-row stage holds

struct CfgV {
  static constexpr int SQmax = 36;  // packed chunks in flight
  // one tile's token rows, each row padded by 16 bytes so that the four
  // rows' MMA fragment words fall in different shared-memory banks
  static constexpr int kXBytes = kGvRows * (kGvMaxK * 2 + 16);
  static constexpr int kUpFloats = 0;
  static constexpr int kRedFloats = (kGvGroups - 1) * kBM * kGvRows;  // other groups' sums: [G-1][128][4]
  static constexpr int kNumBars = 2 * SQmax + 12;
  static constexpr int kSmemBytes = 1024 + SQmax * kQChunk + 2 * kXBytes + 2 * kUpFloats * 4 +
                                    2 * kRedFloats * 4 + kNumBars * 8 + kSmemTail;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ void mma_16816_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Codes of inputs 2p, 2p+1 of a packed word -> bf16 pair (128 + stored code),
// exact; the stored code is the weight code + 8, so this is 136 + code.
__device__ __forceinline__ uint32_t code_pair_biased(uint32_t word, int p) {
  return ((word >> (4 * p)) & 0x000F000Fu) | 0x43004300u;
}

// Codes of inputs 2p, 2p+1 of a packed word -> bf16 pair (code - 8), exact.
__device__ __forceinline__ uint32_t code_pair_bf16x2(uint32_t word, int p) {
  const uint32_t bits = ((word >> (4 * p)) & 0x000F000Fu) | 0x43004300u;  // bf16 128 + code
  __nv_bfloat162 b;
  std::memcpy(&b, &bits, 4);
  const __nv_bfloat162 v = __hsub2(b, __floats2bfloat162_rn(136.0f, 136.0f));
  uint32_t u;
  std::memcpy(&u, &v, 4);
  return u;
}

template <int KIND, int QG>
__global__ void __launch_bounds__(kGvThreads, 1) gemv_q4_kernel(GemmArgs p) {
  using C = CfgV;
  constexpr int SQ = C::SQmax / QG;  // ring slots of QG chunks each
  static_assert(C::SQmax % QG == 0, "ring holds whole groups");
  const int K = p.ksteps * kBK;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;                                  // [SQ][QG x 4,352 B] packed codes + scales
  uint8_t* sX = sQ + C::SQmax * kQChunk;               // [2][8 rows][K] bf16 token rows of a tile
  float* sRed = reinterpret_cast<float*>(sX + 2 * C::kXBytes);  // [2][G-1][128][4] other groups' sums
  uint64_t* bars = reinterpret_cast<uint64_t*>(sRed + 2 * C::kRedFloats);
  const uint32_t qfull0 = ptx::smem_u32(bars);
  const uint32_t qempty0 = qfull0 + 8 * C::SQmax;
  const uint32_t xfull0 = qempty0 + 8 * C::SQmax;  // token rows of a tile staged (2 buffers)
  const uint32_t xempty0 = xfull0 + 16;            // every compute warp done with them
  const uint32_t redf0 = xempty0 + 16;             // other groups' sums written (2 buffers)
  const uint32_t rede0 = redf0 + 16;               // group 0 done with them (2 buffers)
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(bars + C::kNumBars);
  int* prefix = const_cast<int*>(reinterpret_cast<volatile int*>(misc + 4));
  int* soff = prefix + (kMaxE + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int E = p.E;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SQ; ++s) {
      ptx::mbar_init(qfull0 + 8 * s, 1);
      ptx::mbar_init(qempty0 + 8 * s, QG * kGvWpg);  // every chunk is read by the warps of one group
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(xfull0 + 8 * b, 1);
      ptx::mbar_init(xempty0 + 8 * b, kGvWpg * kGvGroups);
      ptx::mbar_init(redf0 + 8 * b, kGvWpg * (kGvGroups - 1));
      ptx::mbar_init(rede0 + 8 * b, kGvWpg);
    }
    misc[1] = 0;
    ptx::fence_mbar_init();
  }
  pdl_wait();
  pdl_trigger();
  const int total = build_schedule<kGvRows>(p, false, E, prefix, soff);
  const Sched sc{prefix, soff, E, p.mblocks, kGvRows};

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ packed chunk producer
    const uint64_t pol = ptx::policy_evict_first();
    uint32_t armed_mask = 0, armed_ph = 0;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile tl = sc.tile(t);
      for (int ks = 0; ks < p.ksteps; ks += QG) {
        if (!wait_bounded<kSpin>(qempty0 + 8 * s, ph ^ 1u, misc + 1, p.status)) {
          ok = false;
          break;
        }
        const uint32_t fb = qfull0 + 8 * s;
        armed_mask |= 1u << s;
        armed_ph = (armed_ph & ~(1u << s)) | (ph << s);
        ptx::mbar_arrive_expect_tx(fb, QG * kQChunk);
        const size_t chunk = (static_cast<size_t>(tl.e) * p.mblocks + tl.mb) * p.ksteps + ks;
        ptx::bulk_load(ptx::smem_u32(sQ + s * QG * kQChunk), p.tiles + chunk * kQChunk, QG * kQChunk, fb, pol);
        if (++s == SQ) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok || misc[1]) {
      for (int q = 0; q < SQ; ++q)
        if ((armed_mask >> q) & 1u) wait_drain(qfull0 + 8 * q, (armed_ph >> q) & 1u);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------ token-row producer
    const uint64_t pol = ptx::policy_evict_last();
    uint32_t armed_mask = 0, armed_ph = 0;
    bool ok = true;
    int ntile = 0;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++ntile) {
      const Tile tl = sc.tile(t);
      const int b = ntile & 1;
      const uint32_t use = static_cast<uint32_t>(ntile >> 1) & 1u;
      if (!wait_bounded<kSpin>(xempty0 + 8 * b, use ^ 1u, misc + 1, p.status)) {
        ok = false;
        break;
      }
      const int n = min(tl.nrows, kGvRows);
      const uint32_t fb = xfull0 + 8 * b;
      armed_mask |= 1u << b;
      armed_ph = (armed_ph & ~(1u << b)) | (use << b);
      ptx::mbar_arrive_expect_tx(fb, static_cast<uint32_t>(n * K * 2));
      for (int j = 0; j < n; ++j)
        ptx::bulk_load(ptx::smem_u32(sX + b * C::kXBytes + j * (K * 2 + 16)), p.brows + static_cast<size_t>(tl.row0 + j) * K,
                       static_cast<uint32_t>(K * 2), fb, pol);
    }
    if (!ok || misc[1]) {
      for (int q = 0; q < 2; ++q)
        if ((armed_mask >> q) & 1u) wait_drain(xfull0 + 8 * q, (armed_ph >> q) & 1u);
    }
  } else if (warp >= 2) {
    // ---------------------------------------------------------- compute
    const int grp = (warp - 2) / kGvWpg;  // takes the K steps gk with gk % kGvGroups == grp
    const int cw = (warp - 2) % kGvWpg;   // owns tile rows 32 cw .. 32 cw + 31
    const int g = lane >> 2;              // MMA fragment row group / token column
    const int q = lane & 3;               // thread in group
    const int r0 = 32 * cw + g;           // rows r0, r0 + 8 (tile 0), r0 + 16, r0 + 24 (tile 1)
    uint32_t gbase = 0;  // running K step of this CTA at the start of the tile
    int ntile = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++ntile) {
      const Tile tl = sc.tile(t);
      const int b = ntile & 1;
      const uint32_t use = static_cast<uint32_t>(ntile >> 1) & 1u;
      bool got = wait_bounded<kSpin>(xfull0 + 8 * b, use, misc + 1, p.status);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      // B fragments read token row g of the stage; columns g >= the tile's
      // rows read a stale row and are never stored
      const uint32_t* xrow =
          reinterpret_cast<const uint32_t*>(sX + b * C::kXBytes + (g & (kGvRows - 1)) * (K * 2 + 16));
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      const int ks0 = static_cast<int>((static_cast<uint32_t>(grp) + kGvGroups - gbase % kGvGroups) % kGvGroups);
      for (int ks = ks0; ks < p.ksteps; ks += kGvGroups) {
        const uint32_t gk = gbase + ks;
        const uint32_t gg = gk / QG;
        const uint32_t sq = gg % SQ;
        const uint32_t phq = (gg / SQ) & 1u;
        got = wait_bounded<kSpin>(qfull0 + 8 * sq, phq, misc + 1, p.status);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const uint8_t* chunk = sQ + (sq * QG + (gk - gg * QG)) * kQChunk;
        uint32_t w[4][8];  // codes of rows r0, r0 + 8, r0 + 16, r0 + 24
        float sc4[4];
        const uint16_t* scl = reinterpret_cast<const uint16_t*>(chunk + kQBytes);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 c0 = reinterpret_cast<const uint4*>(chunk + (r0 + 8 * i) * 32)[0];
          const uint4 c1 = reinterpret_cast<const uint4*>(chunk + (r0 + 8 * i) * 32)[1];
          w[i][0] = c0.x;
          w[i][1] = c0.y;
          w[i][2] = c0.z;
          w[i][3] = c0.w;
          w[i][4] = c1.x;
          w[i][5] = c1.y;
          w[i][6] = c1.z;
          w[i][7] = c1.w;
          sc4[i] = bf16_to_f32(scl[r0 + 8 * i]);
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(qempty0 + 8 * sq);
        const uint32_t* xk = xrow + ks * (kBK / 2) + q;  // token row words of this K step
        // The MMAs take the codes as exact bf16 (136 + code) pairs, two
        // instructions a pair; a ninth MMA with all-ones A sums each token's
        // 64 inputs, and sum((136 + c) x) - 136 sum(x) = sum(c x).
        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f}, dx[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t ones[4] = {0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u};
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // k16 block j: inputs 16 j .. 16 j + 15 of the step
          const uint32_t b0 = xk[8 * j], b1 = xk[8 * j + 4];
          uint32_t a[4];
          a[0] = code_pair_biased(w[0][2 * j], q);      // row r0, inputs 16j + 2q, +1
          a[1] = code_pair_biased(w[1][2 * j], q);      // row r0 + 8
          a[2] = code_pair_biased(w[0][2 * j + 1], q);  // row r0, inputs 16j + 8 + 2q, +1
          a[3] = code_pair_biased(w[1][2 * j + 1], q);  // row r0 + 8
          mma_16816_bf16(d0, a, b0, b1);
          a[0] = code_pair_biased(w[2][2 * j], q);      // row r0 + 16
          a[1] = code_pair_biased(w[3][2 * j], q);      // row r0 + 24
          a[2] = code_pair_biased(w[2][2 * j + 1], q);
          a[3] = code_pair_biased(w[3][2 * j + 1], q);
          mma_16816_bf16(d1, a, b0, b1);
          mma_16816_bf16(dx, ones, b0, b1);
        }
        acc[0] = fmaf(sc4[0], fmaf(-136.0f, dx[0], d0[0]), acc[0]);  // row r0, token 2q
        acc[1] = fmaf(sc4[0], fmaf(-136.0f, dx[1], d0[1]), acc[1]);  // row r0, token 2q + 1
        acc[2] = fmaf(sc4[1], fmaf(-136.0f, dx[0], d0[2]), acc[2]);  // row r0 + 8
        acc[3] = fmaf(sc4[1], fmaf(-136.0f, dx[1], d0[3]), acc[3]);
        acc[4] = fmaf(sc4[2], fmaf(-136.0f, dx[0], d1[0]), acc[4]);  // row r0 + 16
        acc[5] = fmaf(sc4[2], fmaf(-136.0f, dx[1], d1[1]), acc[5]);
        acc[6] = fmaf(sc4[3], fmaf(-136.0f, dx[0], d1[2]), acc[6]);  // row r0 + 24
        acc[7] = fmaf(sc4[3], fmaf(-136.0f, dx[1], d1[3]), acc[7]);
      }
      if (!ok) break;
      gbase += static_cast<uint32_t>(p.ksteps);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(xempty0 + 8 * b);
      // groups 1.. hand their sums of the valid token columns (lanes q < 2)
      // to group 0
      if (grp > 0) {
        got = wait_bounded<kSleepEpi>(rede0 + 8 * b, use ^ 1u, misc + 1, p.status);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        if (q < kGvRows / 2) {
          float* red = sRed + b * C::kRedFloats + (grp - 1) * (kBM * kGvRows);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            red[(r0 + 8 * i) * kGvRows + 2 * q] = acc[2 * i];
            red[(r0 + 8 * i) * kGvRows + 2 * q + 1] = acc[2 * i + 1];
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(redf0 + 8 * b);
        continue;
      }
      got = wait_bounded<kSpin>(redf0 + 8 * b, use, misc + 1, p.status);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      if (q < kGvRows / 2) {
#pragma unroll
        for (int gi = 0; gi < kGvGroups - 1; ++gi) {
          const float* red = sRed + b * C::kRedFloats + gi * (kBM * kGvRows);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[2 * i] += red[(r0 + 8 * i) * kGvRows + 2 * q];
            acc[2 * i + 1] += red[(r0 + 8 * i) * kGvRows + 2 * q + 1];
          }
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(rede0 + 8 * b);
      const int t0 = 2 * q, t1 = 2 * q + 1;
      if (KIND == 1) {
        float* y = reinterpret_cast<float*>(p.out);
        const int col = tl.mb * kBM;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (t0 < tl.nrows) y[static_cast<size_t>(tl.row0 + t0) * p.ldo + col + r0 + 8 * i] = acc[2 * i];
          if (t1 < tl.nrows) y[static_cast<size_t>(tl.row0 + t1) * p.ldo + col + r0 + 8 * i] = acc[2 * i + 1];
        }
        continue;
      }
      // gate/up tile: gate row 32 cw + r (r = g or g + 8) pairs with up row
      // 32 cw + 16 + r, both in this lane: h index 16 cw + r
      uint16_t* h = reinterpret_cast<uint16_t*>(p.out);
      const int colA = tl.mb * 64 + 16 * cw + g, colB = colA + 8;
      if (t0 < tl.nrows) {
        const size_t o = static_cast<size_t>(tl.row0 + t0) * p.ldo;
        h[o + colA] = f32_to_bf16(acc[0] / (1.0f + expf(-acc[0])) * acc[4]);
        h[o + colB] = f32_to_bf16(acc[2] / (1.0f + expf(-acc[2])) * acc[6]);
      }
      if (t1 < tl.nrows) {
        const size_t o = static_cast<size_t>(tl.row0 + t1) * p.ldo;
        h[o + colA] = f32_to_bf16(acc[1] / (1.0f + expf(-acc[1])) * acc[5]);
        h[o + colB] = f32_to_bf16(acc[3] / (1.0f + expf(-acc[3])) * acc[7]);
      }
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Tensor map; dims/strides innermost first.  Encoding costs several
// microseconds of host time, so maps are cached by everything they encode
// (address, type, swizzle, rank, dims, strides, box).  A map holds no data,
// so a cached map stays valid for any buffer later placed at the same address
// with the same shape.
struct MapKey {
  const void* ptr;
  int rank;
  int dtype;
  int swizzle;
  cuuint64_t dims[5];
  cuuint64_t strides[4];
  cuuint32_t box[5];
  bool operator<(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) < 0; }
};

bool make_map(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
              const cuuint32_t* box, CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  MapKey key;
  std::memset(&key, 0, sizeof key);
  key.ptr = ptr;
  key.rank = rank;
  key.dtype = static_cast<int>(dtype);
  key.swizzle = static_cast<int>(swizzle);
  for (int i = 0; i < rank; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
    if (i + 1 < rank) key.strides[i] = strides_bytes[i];
  }
  static std::mutex mu;
  static std::map<MapKey, CUtensorMap> cache;
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
      *m = it->second;
      return true;
    }
  }
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, dtype, rank, const_cast<void*>(ptr), dims, strides_bytes, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() > 4096) cache.clear();
  cache.emplace(key, *m);
  return true;
}

// Row-major bf16 [rows, K] operand, boxes of 64 columns x box_rows rows.
bool make_rows_map(CUtensorMap* m, const void* ptr, int K, int rows, int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t str[1] = {static_cast<cuuint64_t>(K) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  return make_map(m, ptr, 2, dims, str, box);
}

template <int NMAX, int KIND, int AMODE, int G>
cudaError_t run_bf16(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& args, cudaStream_t st) {
  using C = CfgB<NMAX, G>;
  auto kern = grouped_gemm_kernel<NMAX, KIND, AMODE, G>;
  cudaError_t e = ensure_smem(kern, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = sm_count();
  if (grid <= 0) return cudaErrorNoDevice;
  return launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmemBytes, st, a, b, args);
}

template <int NMAX, int KIND, int QG>
cudaError_t run_q4_g(const CUtensorMap& b, const GemmArgs& args, cudaStream_t st) {
  using C = CfgQ<NMAX>;
  auto kern = grouped_gemm_q4_kernel<NMAX, KIND, QG>;
  cudaError_t e = ensure_smem(kern, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = sm_count();
  if (grid <= 0) return cudaErrorNoDevice;
  return launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmemBytes, st, b, args);
}

template <int NMAX, int KIND>
cudaError_t run_q4(const CUtensorMap& b, const GemmArgs& args, cudaStream_t st) {
  return args.qgroup == 2 ? run_q4_g<NMAX, KIND, 2>(b, args, st) : run_q4_g<NMAX, KIND, 1>(b, args, st);
}

// Token rows per tile: small when experts see few rows (decode), so the
// B operand and TMEM footprint stay small and the rings can run deeper.
int pick_nmax(int rows_hint) {
  if (rows_hint <= 320) return 16;
  if (rows_hint <= 1280) return 32;
  if (rows_hint <= 5120) return 64;
  return 128;
}

template <int KIND, int QG>
cudaError_t run_gemv_q4_g(const GemmArgs& args, cudaStream_t st) {
  auto kern = gemv_q4_kernel<KIND, QG>;
  cudaError_t e = ensure_smem(kern, CfgV::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = sm_count();
  if (grid <= 0) return cudaErrorNoDevice;
  return launch_pdl(kern, dim3(grid), dim3(kGvThreads), CfgV::kSmemBytes, st, args);
}

template <int KIND>
cudaError_t run_gemv_q4(const GemmArgs& args, cudaStream_t st) {
  return args.qgroup == 2 ? run_gemv_q4_g<KIND, 2>(args, st) : run_gemv_q4_g<KIND, 1>(args, st);
}

// Decode-sized int4 launches (few rows per expert, K within the token-row
// stage) go to the CUDA-core kernel.
bool use_gemv_q4(int fmt, int R, int K) {
  return fmt == MOE_W_INT4_G64_TILED && pick_nmax(R) == 16 && K <= kGvMaxK;
}

template <int KIND>
cudaError_t run_fmt(int fmt, int nmax, const CUtensorMap& a, const CUtensorMap& b, GemmArgs args,
                    cudaStream_t st) {
  if (fmt == MOE_W_INT4_G64_TILED) {
    args.qgroup = args.ksteps % 2 == 0 ? 2 : 1;  // 8.7 KB bulk copies
    if (KIND != 2 && use_gemv_q4(fmt, args.R, args.ksteps * kBK)) return run_gemv_q4<KIND>(args, st);
    switch (nmax) {
      case 16: return run_q4<16, KIND>(b, args, st);
      case 32: return run_q4<32, KIND>(b, args, st);
      case 64: return run_q4<64, KIND>(b, args, st);
      default: return run_q4<128, KIND>(b, args, st);
    }
  }
  if (fmt == MOE_W_BF16_TILED && args.ksteps % 2 == 0) {
    switch (nmax) {
      case 16: return run_bf16<16, KIND, 1, 2>(a, b, args, st);
      case 32: return run_bf16<32, KIND, 1, 2>(a, b, args, st);
      case 64: return run_bf16<64, KIND, 1, 2>(a, b, args, st);
      default: return run_bf16<128, KIND, 1, 2>(a, b, args, st);
    }
  }
  if (fmt == MOE_W_BF16_TILED) {
    switch (nmax) {
      case 16: return run_bf16<16, KIND, 1, 1>(a, b, args, st);
      case 32: return run_bf16<32, KIND, 1, 1>(a, b, args, st);
      case 64: return run_bf16<64, KIND, 1, 1>(a, b, args, st);
      default: return run_bf16<128, KIND, 1, 1>(a, b, args, st);
    }
  }
  switch (nmax) {
    case 16: return run_bf16<16, KIND, 0, 1>(a, b, args, st);
    case 32: return run_bf16<32, KIND, 0, 1>(a, b, args, st);
    case 64: return run_bf16<64, KIND, 0, 1>(a, b, args, st);
    default: return run_bf16<128, KIND, 0, 1>(a, b, args, st);
  }
}


template <int NMAX, int GG, bool CACHED>
cudaError_t run_fused(const CUtensorMap& mx, const CUtensorMap& mh, const FusedArgs& args, cudaStream_t st) {
  using C = CfgF<NMAX, GG, CACHED>;
  auto kern = grouped_swiglu_fused_kernel<NMAX, GG, CACHED>;
  cudaError_t e = ensure_smem(kern, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = sm_count();
  if (grid <= 0) return cudaErrorNoDevice;
  return launch_pdl(kern, dim3(grid), dim3(kCoreThreads + (CACHED ? 32 * kFetchWarps : 0)), C::kSmemBytes, st, mx,
                    mh, args);
}

}  // namespace

cudaError_t launch_swiglu_fused(const uint16_t* x, int k, const int32_t* perm, uint16_t* x_perm,
                                const int32_t* offsets, int E, int R, int H, int I, const void* w_gateup,
                                const void* w_down, const FusedCache* cache, uint16_t* h, float* y, int32_t* ready,
                                int32_t* st_word, cudaStream_t st) {
  CUtensorMap mx, mh;
  if (!make_rows_map(&mx, x_perm, H, R, kBoxRows)) return cudaErrorInvalidValue;
  if (!make_rows_map(&mh, h, I, R, kBoxRows)) return cudaErrorInvalidValue;
  FusedArgs a{};
  a.offsets = offsets;
  a.E = E;
  a.R = R;
  a.tiles_gu = static_cast<const uint8_t*>(w_gateup);
  a.tiles_dn = static_cast<const uint8_t*>(w_down);
  a.ks_gu = H / kBK;
  a.ks_dn = I / kBK;
  a.mb_gu = I / 64;
  a.mb_dn = H / kBM;
  a.h = h;
  a.y = y;
  a.I = I;
  a.H = H;
  a.ready = ready;
  a.status = st_word;
  a.x = x;
  a.x_perm = x_perm;
  a.perm = perm;
  a.k = k > 0 ? k : 1;
  if (cache != nullptr) {
    // slot pools; with host records the launch also fetches the planned misses
    if (a.ks_gu % 2 != 0 || a.ks_dn % 2 != 0) return cudaErrorNotSupported;
    a.slot_of = cache->slot_of;
    a.S = cache->S;
    if (cache->host_gu != nullptr) {
      a.host_gu = static_cast<const uint8_t*>(cache->host_gu);
      a.host_dn = static_cast<const uint8_t*>(cache->host_dn);
      a.pool_gu = static_cast<uint8_t*>(const_cast<void*>(w_gateup));
      a.pool_dn = static_cast<uint8_t*>(const_cast<void*>(w_down));
      a.rec_gu = static_cast<size_t>(4) * I * H;
      a.rec_dn = static_cast<size_t>(2) * I * H;
      a.nch_gu = static_cast<int>((a.rec_gu + kFetchChunk - 1) / kFetchChunk);
      a.nch_dn = static_cast<int>((a.rec_dn + kFetchChunk - 1) / kFetchChunk);
      a.miss_list = cache->miss_list;
      a.miss_slot = cache->miss_slot;
      a.stats = cache->stats;
      a.wave = cache->wave;
    }
    switch (pick_nmax(R)) {
      case 16: return run_fused<16, 2, true>(mx, mh, a, st);
      case 32: return run_fused<32, 2, true>(mx, mh, a, st);
      case 64: return run_fused<64, 2, true>(mx, mh, a, st);
      default: return run_fused<128, 2, true>(mx, mh, a, st);
    }
  }
  if (a.ks_gu % 2 == 0 && a.ks_dn % 2 == 0) {
    switch (pick_nmax(R)) {
      case 16: return run_fused<16, 2, false>(mx, mh, a, st);
      case 32: return run_fused<32, 2, false>(mx, mh, a, st);
      case 64: return run_fused<64, 2, false>(mx, mh, a, st);
      default: return run_fused<128, 2, false>(mx, mh, a, st);
    }
  }
  switch (pick_nmax(R)) {
    case 16: return run_fused<16, 1, false>(mx, mh, a, st);
    case 32: return run_fused<32, 1, false>(mx, mh, a, st);
    case 64: return run_fused<64, 1, false>(mx, mh, a, st);
    default: return run_fused<128, 1, false>(mx, mh, a, st);
  }
}

cudaError_t launch_grouped_gemm(GemmKind kind, int fmt, const void* w, const uint16_t* scales, const uint16_t* b_rows,
                                const int32_t* offsets, int E, int R, int H, int I, int router_E, void* out,
                                int32_t* st_word, cudaStream_t st) {
  (void)scales;
  CUtensorMap ma, mb;
  GemmArgs args{};
  args.offsets = offsets;
  args.E = E;
  args.R = R;
  args.status = st_word;
  args.out = out;
  args.tiles = static_cast<const uint8_t*>(w);
  args.brows = b_rows;
  args.qgroup = 1;
  const bool plain = (fmt == MOE_W_BF16);
  if (!plain && fmt != MOE_W_BF16_TILED && fmt != MOE_W_INT4_G64_TILED) return cudaErrorInvalidValue;
  switch (kind) {
    case GemmKind::kGateUp: {
      if (plain) {
        // A: [E][2][I][H] bf16 viewed 4-D, box = 16 gate rows + the 16 matching up rows
        cuuint64_t dims[4] = {(cuuint64_t)H, (cuuint64_t)I, 2, (cuuint64_t)E};
        cuuint64_t str[3] = {(cuuint64_t)H * 2, (cuuint64_t)I * H * 2, (cuuint64_t)2 * I * H * 2};
        cuuint32_t box[4] = {(cuuint32_t)kBK, (cuuint32_t)kBoxRows, 2, 1};
        if (!make_map(&ma, w, 4, dims, str, box)) return cudaErrorInvalidValue;
      }
      if (!make_rows_map(&mb, b_rows, H, R, kBoxRows)) return cudaErrorInvalidValue;
      args.ksteps = H / kBK;
      args.mblocks = I / 64;
      args.seg_rows = 2 * I;
      args.ldo = I;
      return run_fmt<0>(fmt, pick_nmax(R), plain ? ma : mb, mb, args, st);
    }
    case GemmKind::kDown: {
      if (plain && !make_rows_map(&ma, w, I, E * H, kBM)) return cudaErrorInvalidValue;
      if (!make_rows_map(&mb, b_rows, I, R, kBoxRows)) return cudaErrorInvalidValue;
      args.ksteps = I / kBK;
      args.mblocks = H / kBM;
      args.seg_rows = H;
      args.ldo = H;
      return run_fmt<1>(fmt, pick_nmax(R), plain ? ma : mb, mb, args, st);
    }
    case GemmKind::kRouter: {
      // one dense segment: all T token rows against all router_E expert rows
      if (!make_rows_map(&ma, w, H, router_E, kBM)) return cudaErrorInvalidValue;
      if (!make_rows_map(&mb, b_rows, H, R, kBoxRows)) return cudaErrorInvalidValue;
      args.offsets = nullptr;
      args.E = 1;
      args.ksteps = H / kBK;
      args.mblocks = router_E / kBM;
      args.seg_rows = router_E;
      args.ldo = router_E;
      return run_bf16<128, 2, 0, 1>(ma, mb, args, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
