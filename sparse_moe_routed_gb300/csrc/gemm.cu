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
//  * Warp roles: warp 0 = TMA producer, warp 1 = MMA issuer (and TMEM owner),
//    warps 2..5 = epilogue, and for int4 weights warps 6..13 = dequantisers.
//    A STAGES-deep shared-memory ring (mbarriers) feeds the tensor core; two
//    TMEM accumulators let the epilogue of one tile overlap the main loop of
//    the next.
//  * Gate/up tiles interleave 16 gate rows with the 16 matching up rows (a 4-D
//    TMA box over [E][2][I][K]), so each epilogue warp holds g in lanes 0..15
//    and u in lanes 16..31 of the same intermediate index: SwiGLU needs one
//    shuffle, no shared-memory exchange.
//  * int4 g64 weights (AFN-001 "Porting Qwen3.8-Flash-Next to Hebrus", section
//    "Phase 2": affine4 with group size 64, read as symmetric codes with one
//    bf16 scale per group): TMA brings the packed codes (4 KB per stage instead
//    of 16 KB) and the group's scales into a staging area; eight dequantiser
//    warps turn them into the 128-byte-swizzled bf16 operand tile
//    (w = bf16(code * scale)), fence the generic-proxy writes for the async
//    proxy and arrive on the stage's barrier; the MMA and epilogue are shared
//    with the bf16 path.
//  * Every mbarrier wait is bounded (2 s of globaltimer); on expiry the CTA
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

constexpr int kBM = 128;                              // weight rows per tile (MMA M)
constexpr int kBK = 64;                               // K per stage: one 128-byte swizzled row of bf16
constexpr int kUK = 16;                               // K per MMA instruction
constexpr int kABytes = kBM * kBK * 2;                // 16 KB bf16 operand tile
constexpr int kBoxRows = 16;                          // token rows per B TMA box
constexpr int kBBoxBytes = kBoxRows * kBK * 2;        // 2 KB
constexpr int kGUBoxBytes = 2 * kBoxRows * kBK * 2;   // 16 gate + 16 up rows: 4 KB
constexpr int kQBytes = kBM * kBK / 2;                // int4 codes of one stage: 4 KB
constexpr int kQGUBoxBytes = 2 * kBoxRows * kBK / 2;  // codes of 16 gate + 16 up rows: 1 KB
constexpr int kSBytes = kBM * 2;                      // one bf16 scale per row: 256 B
constexpr int kCoreThreads = 192;                     // producer, MMA, 4 epilogue warps
constexpr int kQuantWarps = 8;                        // dequantiser warps (int4 only)
constexpr uint64_t kWaitNs = 2000000000ull;

template <int NMAX, bool Q4>
struct Cfg {
  static constexpr int kThreads = kCoreThreads + (Q4 ? 32 * kQuantWarps : 0);
  static constexpr int kBBytes = NMAX * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes + (Q4 ? kQBytes + kSBytes : 0);
  static constexpr int kStagesBf16 = NMAX <= 32 ? 10 : (NMAX <= 64 ? 8 : (NMAX <= 128 ? 6 : 4));
  static constexpr int kStagesQ4 = NMAX <= 32 ? 8 : (NMAX <= 64 ? 7 : 5);
  static constexpr int kStages = Q4 ? kStagesQ4 : kStagesBf16;
  static constexpr int kTmemCols = 2 * NMAX < 32 ? 32 : 2 * NMAX;
  static constexpr int kNumBars = (Q4 ? 3 : 2) * kStages + 5;
  static constexpr int kMiscBytes = 16;
  // tile prefix [E+1] and clamped segment offsets [E+1]
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kNumBars * 8 + kMiscBytes + 2 * (kMaxE + 1) * 4;
  static_assert(kBBytes % 1024 == 0, "B stage must keep 1024-byte alignment");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct GemmArgs {
  const int32_t* offsets;  // [E+1] segment starts (null for one dense segment)
  int E;                   // segments
  int R;                   // rows of the B operand
  int ksteps;              // K / 64
  int mblocks;             // 128-row weight blocks per segment
  int seg_rows;            // weight rows per segment in the A map (down: H)
  int seg_groups;          // scale groups per weight row (int4 down: I / 64)
  void* out;
  int ldo;                 // leading dimension of out (elements)
  int32_t* status;
};

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                             int32_t* status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitNs) {
        *abort_flag = 1;
        set_status(status, MOE_DEV_TIMEOUT);
        return false;
      }
    }
  }
}

// Drain wait used during teardown after an abort: ignores the abort flag.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitNs) return;
  }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Eight signed 4-bit codes (one 32-bit word, element 0 in the low nibble)
// times one bf16 scale -> eight bf16 (a 16-byte chunk, element 0 first).
// Code q is placed in the mantissa of 128 + (q + 8) (exact in bf16), the
// offset is removed exactly, and the product with the scale is rounded once.
__device__ __forceinline__ uint4 dequant8(uint32_t word, __nv_bfloat162 scale2) {
  const uint32_t v = word ^ 0x88888888u;  // two's complement nibble -> q + 8
  const __nv_bfloat162 one2 = __floats2bfloat162_rn(1.0f, 1.0f);
  const __nv_bfloat162 off2 = __floats2bfloat162_rn(-136.0f, -136.0f);
  uint32_t out[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint32_t t = v >> (8 * p);
    const uint32_t bits = 0x43004300u | (t & 0xFu) | ((t & 0xF0u) << 12);
    __nv_bfloat162 b;
    std::memcpy(&b, &bits, 4);
    const __nv_bfloat162 q = __hfma2(b, one2, off2);
    const __nv_bfloat162 w = __hmul2(q, scale2);
    std::memcpy(&out[p], &w, 4);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

struct Tile {
  int e, mb, row0, nrows;
};

template <int NMAX, int KIND, bool Q4>
__global__ void __launch_bounds__(Cfg<NMAX, Q4>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmS, GemmArgs p) {
  using C = Cfg<NMAX, Q4>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;                         // [S][16 KB] bf16 operand tiles (swizzled)
  uint8_t* sB = sA + S * kABytes;             // [S][NMAX x 128 B] token rows (swizzled)
  uint8_t* sQ = sB + S * C::kBBytes;          // [S][4 KB] int4 codes (Q4)
  uint8_t* sS = sQ + (Q4 ? S * kQBytes : 0);  // [S][256 B] scales (Q4)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sS + (Q4 ? S * kSBytes : 0));
  const uint32_t full0 = ptx::smem_u32(bars);  // operand tiles ready for the MMA
  const uint32_t empty0 = full0 + 8 * S;       // MMA finished with a stage
  const uint32_t accf0 = empty0 + 8 * S;
  const uint32_t acce0 = accf0 + 16;
  const uint32_t drain = acce0 + 16;
  const uint32_t tfull0 = drain + 8;  // Q4: codes + scales + token rows landed
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(bars + C::kNumBars);
  int* prefix = const_cast<int*>(reinterpret_cast<volatile int*>(misc + 4));
  int* soff = prefix + (kMaxE + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool dense = (p.offsets == nullptr);
  const int E = dense ? 1 : p.E;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(full0 + 8 * s, Q4 ? kQuantWarps : 1);
      ptx::mbar_init(empty0 + 8 * s, 1);
      if (Q4) ptx::mbar_init(tfull0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(accf0 + 8 * a, 1);
      ptx::mbar_init(acce0 + 8 * a, 128);
    }
    ptx::mbar_init(drain, 1);
    misc[1] = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    if (Q4) ptx::prefetch_tmap(&tmS);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(const_cast<uint32_t*>(&misc[0])), C::kTmemCols);
    ptx::tmem_relinquish();
  }
  // Everything above overlaps the previous kernel's tail; from here on the
  // kernel reads upstream data (offsets, activation rows) and writes outputs.
  pdl_wait();
  pdl_trigger();
  // Segment offsets into shared memory, clamped into [0, R] (a segment's
  // length is never negative), so that corrupt offsets can never address rows
  // outside the buffers; then the per-segment tile prefix (warp 0).
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

  const uint32_t tmem_base = misc[0];
  const int total = prefix[E];

  auto tile_of = [&](int t) {
    int lo = 0, hi = E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= t) lo = mid; else hi = mid;
    }
    const int local = t - prefix[lo];
    const int chunk = local / p.mblocks;
    const int start = soff[lo];
    const int len = max(soff[lo + 1] - start, 0);
    Tile tl;
    tl.e = lo;
    tl.mb = local - chunk * p.mblocks;
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
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile tl = tile_of(t);
      const int nblk = (tl.nrows + kBoxRows - 1) / kBoxRows;
      for (int ks = 0; ks < p.ksteps; ++ks) {
        if (!wait_bounded(empty0 + 8 * s, ph ^ 1u, misc + 1, p.status)) {
          ok = false;
          break;
        }
        const uint32_t b_dst = ptx::smem_u32(sB + s * C::kBBytes);
        if (!Q4) {
          const uint32_t fb = full0 + 8 * s;
          ptx::mbar_arrive_expect_tx(fb, kABytes + nblk * kBBoxBytes);
          armed[s] = static_cast<int>(ph);
          const uint32_t a_dst = ptx::smem_u32(sA + s * kABytes);
          if (KIND == 0) {
#pragma unroll
            for (int b = 0; b < 4; ++b)
              ptx::tma_load_4d(a_dst + b * kGUBoxBytes, &tmA, fb, ks * kBK, tl.mb * 64 + b * 16, 0, tl.e, pol_w);
          } else if (KIND == 1) {
            ptx::tma_load_2d(a_dst, &tmA, fb, ks * kBK, tl.e * p.seg_rows + tl.mb * kBM, pol_w);
          } else {
            ptx::tma_load_2d(a_dst, &tmA, fb, ks * kBK, tl.mb * kBM, pol_w);
          }
          for (int b = 0; b < nblk; ++b)
            ptx::tma_load_2d(b_dst + b * kBBoxBytes, &tmB, fb, ks * kBK, tl.row0 + b * kBoxRows, pol_x);
        } else {
          const uint32_t fb = tfull0 + 8 * s;
          ptx::mbar_arrive_expect_tx(fb, kQBytes + kSBytes + nblk * kBBoxBytes);
          armed[s] = static_cast<int>(ph);
          const uint32_t q_dst = ptx::smem_u32(sQ + s * kQBytes);
          const uint32_t s_dst = ptx::smem_u32(sS + s * kSBytes);
          if (KIND == 0) {
            // codes [E][2][I][K/2] bytes, scales group-major [E][K/64][2][I]
#pragma unroll
            for (int b = 0; b < 4; ++b)
              ptx::tma_load_4d(q_dst + b * kQGUBoxBytes, &tmA, fb, ks * (kBK / 2), tl.mb * 64 + b * 16, 0, tl.e,
                               pol_w);
            ptx::tma_load_4d(s_dst, &tmS, fb, tl.mb * 64, 0, ks, tl.e, pol_w);
          } else {
            // codes [E*H][I/2] bytes, scales group-major [E][I/64][H]
            ptx::tma_load_2d(q_dst, &tmA, fb, ks * (kBK / 2), tl.e * p.seg_rows + tl.mb * kBM, pol_w);
            ptx::tma_load_2d(s_dst, &tmS, fb, tl.mb * kBM, tl.e * p.seg_groups + ks, pol_w);
          }
          for (int b = 0; b < nblk; ++b)
            ptx::tma_load_2d(b_dst + b * kBBoxBytes, &tmB, fb, ks * kBK, tl.row0 + b * kBoxRows, pol_x);
        }
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok || misc[1]) {
      // abort: let every copy already issued land before the CTA exits
      const uint32_t landed0 = Q4 ? tfull0 : full0;
#pragma unroll
      for (int q = 0; q < S; ++q)
        if (armed[q] >= 0) wait_drain(landed0 + 8 * q, static_cast<uint32_t>(armed[q]));
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
      const Tile tl = tile_of(t);
      const uint32_t npad = static_cast<uint32_t>((tl.nrows + 15) & ~15);
      const uint32_t idesc = ptx::idesc_bf16_f32(kBM, npad);
      if (!wait_bounded(acce0 + 8 * acc, aph ^ 1u, misc + 1, p.status)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * NMAX);
      for (int ks = 0; ks < p.ksteps; ++ks) {
        if (!wait_bounded(full0 + 8 * s, ph, misc + 1, p.status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t a0 = ptx::smem_u32(sA + s * kABytes);
        const uint32_t b0 = ptx::smem_u32(sB + s * C::kBBytes);
#pragma unroll
        for (int kk = 0; kk < kBK / kUK; ++kk) {
          ptx::umma_bf16(d_tmem, ptx::sdesc_k_sw128(a0 + kk * kUK * 2), ptx::sdesc_k_sw128(b0 + kk * kUK * 2),
                         idesc, (ks | kk) != 0 ? 1u : 0u);
        }
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
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row_in_tile = q * 32 + lane;
    int acc = 0;
    uint32_t aph = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = tile_of(t);
      bool ok = wait_bounded(accf0 + 8 * acc, aph, misc + 1, p.status);
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
  } else if (Q4 && warp >= 6) {
    // ------------------------------------------------------------ dequantisers
    // 256 threads, two per weight row: each turns 32 codes (16 bytes) of its
    // row into 4 swizzled 16-byte chunks of the bf16 operand tile.
    const int tt = threadIdx.x - kCoreThreads;
    const int row = tt >> 1;
    const int half = tt & 1;
    // scale slot of this row: gate/up tiles hold [2][64] (gate rows, up rows)
    // for the tile's four 16-row block pairs; down tiles hold one per row
    const int sidx = (KIND == 0) ? (((row >> 4) & 1) * 64 + (row >> 5) * 16 + (row & 15)) : row;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      for (int ks = 0; ks < p.ksteps; ++ks) {
        const bool got = wait_bounded(tfull0 + 8 * s, ph, misc + 1, p.status);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const uint4 pk = *reinterpret_cast<const uint4*>(sQ + s * kQBytes + row * 32 + half * 16);
        const uint16_t sbits = reinterpret_cast<const uint16_t*>(sS + s * kSBytes)[sidx];
        __nv_bfloat16 sc;
        std::memcpy(&sc, &sbits, 2);
        const __nv_bfloat162 sc2 = __halves2bfloat162(sc, sc);
        uint8_t* arow = sA + s * kABytes + row * 128;
        const uint32_t words[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int chunk = (4 * half + w) ^ (row & 7);
          *reinterpret_cast<uint4*>(arow + chunk * 16) = dequant8(words[w], sc2);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(full0 + 8 * s);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
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

template <int NMAX, int KIND, bool Q4>
cudaError_t run(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& sc, const GemmArgs& args,
                cudaStream_t st) {
  using C = Cfg<NMAX, Q4>;
  auto kern = grouped_gemm_kernel<NMAX, KIND, Q4>;
  cudaError_t e = ensure_smem(kern, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = sm_count();
  if (grid <= 0) return cudaErrorNoDevice;
  return launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmemBytes, st, a, b, sc, args);
}

template <int KIND, bool Q4>
cudaError_t run_nmax(int nmax, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& sc,
                     const GemmArgs& args, cudaStream_t st) {
  switch (nmax) {
    case 16: return run<16, KIND, Q4>(a, b, sc, args, st);
    case 32: return run<32, KIND, Q4>(a, b, sc, args, st);
    case 64: return run<64, KIND, Q4>(a, b, sc, args, st);
    default: return run<128, KIND, Q4>(a, b, sc, args, st);
  }
}

// Token rows per tile: small when experts see few rows (decode), so the
// B operand and TMEM footprint stay small and the ring can run deeper.
int pick_nmax(int rows_hint) {
  if (rows_hint <= 320) return 16;
  if (rows_hint <= 1280) return 32;
  if (rows_hint <= 5120) return 64;
  return 128;
}

}  // namespace

cudaError_t launch_grouped_gemm(GemmKind kind, int fmt, const void* w, const uint16_t* scales, const uint16_t* b_rows,
                                const int32_t* offsets, int E, int R, int H, int I, int router_E, void* out,
                                int32_t* st_word, cudaStream_t st) {
  CUtensorMap ma, mb, ms;
  GemmArgs args{};
  args.offsets = offsets;
  args.E = E;
  args.R = R;
  args.status = st_word;
  args.out = out;
  const bool q4 = (fmt == MOE_W_INT4_G64);
  switch (kind) {
    case GemmKind::kGateUp: {
      if (!q4) {
        // A: [E][2][I][H] bf16 viewed 4-D, box = 16 gate rows + the 16 matching up rows
        cuuint64_t dims[4] = {(cuuint64_t)H, (cuuint64_t)I, 2, (cuuint64_t)E};
        cuuint64_t str[3] = {(cuuint64_t)H * 2, (cuuint64_t)I * H * 2, (cuuint64_t)2 * I * H * 2};
        cuuint32_t box[4] = {(cuuint32_t)kBK, (cuuint32_t)kBoxRows, 2, 1};
        if (!make_map(&ma, w, 4, dims, str, box)) return cudaErrorInvalidValue;
      } else {
        // codes: [E][2][I][H/2] bytes, same 16 + 16 row box, 32 bytes (64 codes) wide
        cuuint64_t dims[4] = {(cuuint64_t)H / 2, (cuuint64_t)I, 2, (cuuint64_t)E};
        cuuint64_t str[3] = {(cuuint64_t)H / 2, (cuuint64_t)I * H / 2, (cuuint64_t)2 * I * H / 2};
        cuuint32_t box[4] = {(cuuint32_t)kBK / 2, (cuuint32_t)kBoxRows, 2, 1};
        if (!make_map(&ma, w, 4, dims, str, box, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_NONE))
          return cudaErrorInvalidValue;
        // scales: group-major [E][H/64][2][I] bf16; box = 64 rows of gate and of up for one group
        cuuint64_t sd[4] = {(cuuint64_t)I, 2, (cuuint64_t)H / 64, (cuuint64_t)E};
        cuuint64_t ss[3] = {(cuuint64_t)I * 2, (cuuint64_t)2 * I * 2, (cuuint64_t)(H / 64) * 2 * I * 2};
        cuuint32_t sb[4] = {64, 2, 1, 1};
        if (!make_map(&ms, scales, 4, sd, ss, sb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_NONE))
          return cudaErrorInvalidValue;
      }
      if (!make_rows_map(&mb, b_rows, H, R, kBoxRows)) return cudaErrorInvalidValue;
      args.ksteps = H / kBK;
      args.mblocks = I / 64;
      args.seg_rows = 2 * I;
      args.seg_groups = H / 64;
      args.ldo = I;
      if (q4) return run_nmax<0, true>(pick_nmax(R), ma, mb, ms, args, st);
      return run_nmax<0, false>(pick_nmax(R), ma, mb, ma, args, st);
    }
    case GemmKind::kDown: {
      if (!q4) {
        if (!make_rows_map(&ma, w, I, E * H, kBM)) return cudaErrorInvalidValue;
      } else {
        cuuint64_t dims[2] = {(cuuint64_t)I / 2, (cuuint64_t)E * H};
        cuuint64_t str[1] = {(cuuint64_t)I / 2};
        cuuint32_t box[2] = {(cuuint32_t)kBK / 2, (cuuint32_t)kBM};
        if (!make_map(&ma, w, 2, dims, str, box, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_NONE))
          return cudaErrorInvalidValue;
        // scales: group-major [E][I/64][H] bf16; box = 128 rows of one group
        cuuint64_t sd[2] = {(cuuint64_t)H, (cuuint64_t)E * (I / 64)};
        cuuint64_t ss[1] = {(cuuint64_t)H * 2};
        cuuint32_t sb[2] = {(cuuint32_t)kBM, 1};
        if (!make_map(&ms, scales, 2, sd, ss, sb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_NONE))
          return cudaErrorInvalidValue;
      }
      if (!make_rows_map(&mb, b_rows, I, R, kBoxRows)) return cudaErrorInvalidValue;
      args.ksteps = I / kBK;
      args.mblocks = H / kBM;
      args.seg_rows = H;
      args.seg_groups = I / 64;
      args.ldo = H;
      if (q4) return run_nmax<1, true>(pick_nmax(R), ma, mb, ms, args, st);
      return run_nmax<1, false>(pick_nmax(R), ma, mb, ma, args, st);
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
      args.seg_groups = 0;
      args.ldo = router_E;
      return run<128, 2, false>(ma, mb, ma, args, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
