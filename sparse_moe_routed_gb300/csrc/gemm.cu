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

#include "gemm_common.cuh"

namespace moe {

using namespace gk;

namespace {

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
      constexpr int BR = box_rows_for(NMAX);
      const int nblk = (tl.nrows + BR - 1) / BR;
      for (int ks = 0; ks < p.ksteps; ks += G) {
        if (!wait_bounded<kSpin>(empty0 + 8 * s, ph ^ 1u, misc + 1, p.status)) {
          ok = false;
          break;
        }
        const uint32_t fb = full0 + 8 * s;
        ptx::mbar_arrive_expect_tx(fb, G * (kABytes + nblk * BR * kBK * 2));
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
            ptx::tma_load_2d(b_dst + j * C::kBBytes + b * BR * kBK * 2, &tmB, fb, (ks + j) * kBK,
                             tl.row0 + b * BR, pol_x);
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
      constexpr int BR = box_rows_for(NMAX);
      const int nblk = (tl.nrows + BR - 1) / BR;
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
          ptx::mbar_arrive_expect_tx(fb, nblk * BR * kBK * 2);
          const uint32_t b_dst = ptx::smem_u32(sB + s * C::kBBytes);
          for (int b = 0; b < nblk; ++b)
            ptx::tma_load_2d(b_dst + b * BR * kBK * 2, &tmB, fb, ks * kBK, tl.row0 + b * BR, pol);
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

template <int KIND>
cudaError_t run_fmt(int fmt, int nmax, const CUtensorMap& a, const CUtensorMap& b, GemmArgs args,
                    cudaStream_t st) {
  if (fmt == MOE_W_INT4_G64_TILED) {
    args.qgroup = args.ksteps % 2 == 0 ? 2 : 1;  // 8.7 KB bulk copies
    if (KIND != 2 && use_gemv_q4(fmt, args.R, args.ksteps * kBK)) return launch_gemv_q4(KIND, args, st);
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

}  // namespace

namespace gk {

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

// Token rows per tile: small when experts see few rows (decode), so the
// B operand and TMEM footprint stay small and the rings can run deeper.
int pick_nmax(int rows_hint) {
  if (rows_hint <= 320) return 16;
  if (rows_hint <= 1280) return 32;
  if (rows_hint <= 5120) return 64;
  return 128;
}

}  // namespace gk

namespace gk {

cudaError_t launch_int4_slots(int kind, const uint16_t* rows, const int32_t* offsets, int E, int R, int H, int I,
                              const void* pool, int S, const int32_t* slot_of, void* out, int32_t* st_word,
                              cudaStream_t st) {
  const int K = kind == 0 ? H : I;
  if (!use_gemv_q4(MOE_W_INT4_G64_TILED, R, K)) return cudaErrorNotSupported;
  GemmArgs args{};
  args.offsets = offsets;
  args.E = E;
  args.R = R;
  args.status = st_word;
  args.out = out;
  args.tiles = static_cast<const uint8_t*>(pool);
  args.brows = rows;
  args.slot_of = slot_of;
  args.S = S;
  args.ksteps = K / kBK;
  args.mblocks = kind == 0 ? I / 64 : H / kBM;
  args.seg_rows = kind == 0 ? 2 * I : H;
  args.ldo = kind == 0 ? I : H;
  args.qgroup = args.ksteps % 2 == 0 ? 2 : 1;
  return launch_gemv_q4(kind, args, st);
}

cudaError_t launch_int4_fetch(const uint16_t* rows, const int32_t* offsets, int E, int R, int H, int I, void* pool_gu,
                              void* pool_dn, int S, const int32_t* slot_of, const void* host_gu, const void* host_dn,
                              const int32_t* miss_list, const int32_t* miss_slot, const int32_t* stats, uint16_t* h,
                              int32_t* fsync, int32_t* st_word, cudaStream_t st) {
  if (!use_gemv_q4(MOE_W_INT4_G64_TILED, R, H)) return cudaErrorNotSupported;
  GemmArgs args{};
  args.offsets = offsets;
  args.E = E;
  args.R = R;
  args.status = st_word;
  args.out = h;
  args.tiles = static_cast<const uint8_t*>(pool_gu);
  args.brows = rows;
  args.slot_of = slot_of;
  args.S = S;
  args.ksteps = H / kBK;
  args.mblocks = I / 64;
  args.seg_rows = 2 * I;
  args.ldo = I;
  args.qgroup = args.ksteps % 2 == 0 ? 2 : 1;
  args.host_gu = static_cast<const uint8_t*>(host_gu);
  args.host_dn = static_cast<const uint8_t*>(host_dn);
  args.pool_dn = static_cast<uint8_t*>(pool_dn);
  args.rec_gu = static_cast<size_t>(args.mblocks) * args.ksteps * kQChunk;
  args.rec_dn = static_cast<size_t>(H / kBM) * (I / kBK) * kQChunk;
  int cpp = 1;  // chunks per gate/up piece: the largest divisor of the K steps up to 8
  for (int c = 8; c >= 1; --c)
    if (args.ksteps % c == 0) {
      cpp = c;
      break;
    }
  args.cpp = cpp;
  args.miss_list = miss_list;
  args.miss_slot = miss_slot;
  args.stats = stats;
  args.fsync = fsync;
  return launch_gemv_q4(0, args, st);
}

}  // namespace gk

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
      if (!make_rows_map(&mb, b_rows, H, R, box_rows_for(pick_nmax(R)))) return cudaErrorInvalidValue;
      args.ksteps = H / kBK;
      args.mblocks = I / 64;
      args.seg_rows = 2 * I;
      args.ldo = I;
      return run_fmt<0>(fmt, pick_nmax(R), plain ? ma : mb, mb, args, st);
    }
    case GemmKind::kDown: {
      if (plain && !make_rows_map(&ma, w, I, E * H, kBM)) return cudaErrorInvalidValue;
      if (!make_rows_map(&mb, b_rows, I, R, box_rows_for(pick_nmax(R)))) return cudaErrorInvalidValue;
      args.ksteps = I / kBK;
      args.mblocks = H / kBM;
      args.seg_rows = H;
      args.ldo = H;
      return run_fmt<1>(fmt, pick_nmax(R), plain ? ma : mb, mb, args, st);
    }
    case GemmKind::kRouter: {
      // one dense segment: all T token rows against all router_E expert rows
      if (!make_rows_map(&ma, w, H, router_E, kBM)) return cudaErrorInvalidValue;
      if (!make_rows_map(&mb, b_rows, H, R, box_rows_for(128))) return cudaErrorInvalidValue;
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
