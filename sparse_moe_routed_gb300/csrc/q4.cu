// int4 g64 matrix-vector contraction for decode-sized launches (a few token
// rows per expert): codes from tile-packed records become bf16 MMA operands in
// registers.  AFN-001 "Porting Qwen3.8-Flash-Next to Hebrus", section
// "Phase 2": affine4 with group size 64, read as symmetric codes with one
// bf16 scale per group.  Shared tile machinery: gemm_common.cuh.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_common.cuh"

namespace moe {

using namespace gk;

namespace {

// ============================================================ int4 GEMV
// Decode-sized int4 tiles.  With about one token row per expert a tile is a
// matrix-vector product, and what limits it is instructions per weight, not
// MMA throughput: a tcgen05 MMA must read its operands from shared or tensor
// memory, so the codes of each K step would be expanded into a 16 KB bf16
// tile and read back (measured: ~0.35 us per 4.3 KB step), while a CUDA-core
// dot product spends ~6 instructions per weight.  Here the weights go from
// registers straight into warp-level MMAs (mma.sync m16n8k16, fp16 in, fp32
// accumulate): the codes of a packed word become exact fp16 pairs over the
// exponent of 1024 (1024 + c, or 1024 + 16c for the codes in bits 4-7 of a
// half-word), four logic instructions and one shift per word; the token
// values that meet the 16c codes are staged divided by 16 (exact in fp16), and
// one MMA instruction consumes 256 weights against up to 8 token rows.
//
// Warps: 0 streams packed chunks (bulk copies, deep ring); 1 stages each
// tile's token rows (one bulk copy per row, double-buffered), converts them
// to fp16 in place and writes each step's bias correction (from the row sums)
// into a table; the rest compute in groups.  The groups take ring slots (a
// slot holds four K steps, or two of each block of a multi-block tile) in
// turn, so each warp has several steps' time for the latency chain of one
// (wait, loads, conversion, MMAs); one wait and one release per slot.  Warp w
// of a group owns tile rows 32w .. 32w + 31 of one 128-row block as two MMA
// row tiles that share the token fragments: per K step (one scale group of
// 64 inputs) it runs eight MMAs, the first of each chain starting from the
// step's correction, and adds scale x partial to its fp32 accumulators.  The
// MMA's k slots run over the step's inputs in a permuted order (the same for
// weights and tokens), chosen so that each lane reads 16 consecutive inputs:
// one 8-byte load per weight row, two 16-byte loads of token values, and
// every code pair at a fixed nibble position.  In a gate/up record rows
// 32w .. 32w + 15 are gate and 32w + 16 .. 32w + 31 the up rows of the same h
// columns, so each lane ends a tile holding gate and up of the same outputs.
// At the end of a tile the other groups hand their sums (valid token columns
// only) through shared memory to the group that took the tile's last ring
// slot, which adds them in a fixed order (the same bits every call) and
// stores y, or h = silu(gate) * up.  Token columns past the tile's rows read
// stale staged rows and are never stored (an MMA column depends on its own B
// column only).
//
// Tiles span several 128-row blocks where the record's block count allows:
// gate/up tiles two (two groups of eight warps), down tiles (K = I = 640: ten
// K steps, so the per-tile staging and hand-over weigh more) four (one group
// of all sixteen warps, no hand-over) or two; each warp owns 32 rows of one
// block, and a ring slot holds the same K steps of every block of the tile.
constexpr int kGvRows = 4;                     // token rows per tile
constexpr int kGvN = 8;                        // MMA N: token columns (those past kGvRows are never stored)
constexpr int kGvGroups = 4;
constexpr int kGvWpg = 4;                      // compute warps per group, 32 rows each
constexpr int kGvWarps = 2 + kGvWpg * kGvGroups;
constexpr int kGvThreads = 32 * kGvWarps;
constexpr int kGvMaxK = 2560;                  // inputs per row the token-row stage holds
static_assert(kGvRows <= kGvN, "a tile's token rows fit the MMA's columns");

struct CfgV {
  static constexpr int SQmax = 36;  // packed chunks in flight
  // one tile's token rows, each row padded by 16 bytes so that the four
  // rows' MMA fragment words fall in different shared-memory banks
  static constexpr int kXBytes = kGvRows * (kGvMaxK * 2 + 16);
  static constexpr int kUpFloats = 0;
  static constexpr int kRedFloats = (kGvGroups - 1) * kBM * kGvRows;  // other groups' sums: [G-1][128][4]
  // per K step, each staged token row's bias correction in the MMA
  // accumulator layout of the two lane classes:
  // [K steps][c0, c1, c0, c1, c2, c3, c2, c3]
  static constexpr int kXsFloats = kGvMaxK / 64 * 8;
  static constexpr int kNumBars = 2 * SQmax + 12;
  // in-launch fetch: the tile order's expert at each position, and a bit per
  // expert being fetched
  static constexpr int kFetchTail = kMaxE * 4 + 2 * (kMaxE / 8);
  static constexpr int kSmemBytes = 1024 + SQmax * kQChunk + 2 * kXBytes + 2 * kUpFloats * 4 +
                                    2 * kRedFloats * 4 + 2 * kXsFloats * 4 + kNumBars * 8 + kSmemTail + kFetchTail;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ void mma_16816_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same MMA from the accumulator c (read only) into d.
__device__ __forceinline__ void mma_16816_f16_first(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                                    const float4& c) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c.x), "f"(c.y), "f"(c.z), "f"(c.w));
}

// Codes of a packed word as exact fp16 pairs over the exponent of 1024: in
// v = word (pairs 0, 1) or word >> 8 (pairs 2, 3), the codes in bits 0-3 and
// 16-19 give (1024 + stored code) x 2 (lo = true) and those in bits 4-7 and
// 20-23 give (1024 + 16 stored code) x 2 (lo = false): one three-input
// logic instruction each (mask as the immediate, `magic` = 0x64006400 held
// in a register).  The stored code is the weight code + 8.
__device__ __forceinline__ uint32_t code_pair_f16(uint32_t v, bool lo, uint32_t magic) {
  uint32_t d;
  if (lo)
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(v), "n"(0x000F000F), "r"(magic));
  else
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(v), "n"(0x00F000F0), "r"(magic));
  return d;
}

constexpr int kGvFetchWarps = 2;     // FETCH launches: warps that copy the misses' records
constexpr int kGvFetchBytes = 32768;  // a down-record piece

template <int KIND, int QG, int BPT, bool FETCH = false>
__global__ void __launch_bounds__(kGvThreads + (FETCH ? 32 * kGvFetchWarps : 0), 1)
    gemv_q4_kernel(GemmArgs p, int early) {
  static_assert(!FETCH || KIND == 0, "the gate/up launch fetches both components");
  using C = CfgV;
  static_assert(kGvGroups % BPT == 0, "groups");
  constexpr int G = kGvGroups / BPT;               // K-step groups
  constexpr int WPG = BPT * kGvWpg;                // compute warps per group, 32 rows each
  constexpr int RT = 32 * WPG;                     // weight rows per tile
  constexpr int CPS = BPT * QG;                    // chunks per ring slot
  constexpr int SQ = C::SQmax / CPS;               // ring slots
  constexpr int S = QG;                            // K steps per ring slot (one group reads them all)
  static_assert(SQ >= 2, "ring depth");
  static_assert(G * WPG == kGvGroups * kGvWpg, "all compute warps");
  static_assert((G - 1) * RT * kGvRows <= C::kRedFloats, "hand-over buffer");
  const int K = p.ksteps * kBK;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;                                  // [SQ][CPS x 4,352 B] packed codes + scales
  uint8_t* sX = sQ + C::SQmax * kQChunk;               // [2][8 rows][K] bf16 token rows of a tile
  float* sRed = reinterpret_cast<float*>(sX + 2 * C::kXBytes);  // [2][G-1][128][4] other groups' sums
  float* sXs = sRed + 2 * C::kRedFloats;  // [2][K steps][8]: each token row's bias correction per K step
  uint64_t* bars = reinterpret_cast<uint64_t*>(sXs + 2 * C::kXsFloats);
  const uint32_t qfull0 = ptx::smem_u32(bars);
  const uint32_t qempty0 = qfull0 + 8 * C::SQmax;
  const uint32_t xfull0 = qempty0 + 8 * C::SQmax;  // token rows of a tile staged (2 buffers)
  const uint32_t xempty0 = xfull0 + 16;            // every compute warp done with them
  const uint32_t redf0 = xempty0 + 16;             // other groups' sums written (2 buffers)
  const uint32_t rede0 = redf0 + 16;               // group 0 done with them (2 buffers)
  const uint32_t xland0 = rede0 + 16;              // token-row copies landed (2 buffers)
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(bars + C::kNumBars);
  int* prefix = const_cast<int*>(reinterpret_cast<volatile int*>(misc + 4));
  int* soff = prefix + (kMaxE + 1);
  int* eord = soff + (kMaxE + 1);                                   // FETCH: tile order
  uint32_t* mbits = reinterpret_cast<uint32_t*>(eord + kMaxE);      // FETCH: experts being fetched
  uint32_t* mseen = mbits + kMaxE / 32;                             // FETCH: placed in the order

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int E = p.E;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SQ; ++s) {
      ptx::mbar_init(qfull0 + 8 * s, 1);
      ptx::mbar_init(qempty0 + 8 * s, WPG);  // a slot is read by the warps of one group
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(xfull0 + 8 * b, 1);
      ptx::mbar_init(xland0 + 8 * b, 1);
      ptx::mbar_init(xempty0 + 8 * b, WPG * G);
      if (G > 1) {
        ptx::mbar_init(redf0 + 8 * b, WPG * (G - 1));
        ptx::mbar_init(rede0 + 8 * b, WPG);
      }
    }
    misc[1] = 0;
    ptx::fence_mbar_init();
  }
  // A launch over resident records right after a launch that left this
  // launch's offsets as its stream's token (early: the gate/up launch before
  // a down launch, the row gather before a gate/up launch) reads only its
  // token rows (h or x_perm) from that launch; its weights and its routes
  // (offsets, complete before that launch started, read here past L1) are
  // ready at its start.  Its token-row warp alone waits for the launch
  // before, so the weight stream starts on each SM as soon as one of that
  // launch's CTAs leaves it.
  const bool late_wait = !FETCH && early != 0 && p.slot_of == nullptr;
  if (!late_wait) pdl_wait();
  pdl_trigger();
  GemmArgs ps = p;  // the schedule counts tiles of RT rows
  ps.mblocks = p.mblocks / BPT;
  const int total = build_schedule<kGvRows>(ps, false, E, prefix, soff);
  Sched sc{prefix, soff, E, ps.mblocks, kGvRows};
  const int nmiss = FETCH ? min(max(p.stats[1], 0), min(E, p.S)) : 0;
  if constexpr (FETCH) {
    // The experts being fetched come last in the tile order (in plan order),
    // so that no CTA holds resident work behind a tile that waits for the
    // link; the prefix is recomputed over that order.
    for (int i = threadIdx.x; i < (E + 31) / 32; i += blockDim.x) {
      mbits[i] = 0u;
      mseen[i] = 0u;
    }
    __syncthreads();
    for (int m = threadIdx.x; m < nmiss; m += blockDim.x) {
      const int e = p.miss_list[m];
      if (e >= 0 && e < E) atomicOr(&mbits[e >> 5], 1u << (e & 31));
    }
    __syncthreads();
    if (warp == 0) {
      int run = 0;
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const bool keep = e < E && !((mbits[e0 >> 5] >> lane) & 1u);
        const unsigned bal = __ballot_sync(0xffffffffu, keep);
        if (keep) eord[run + __popc(bal & ((1u << lane) - 1u))] = e;
        run += __popc(bal);
      }
      // then the fetched ones in plan order, each once (an ID outside
      // [0, E) is flagged by the fetch warps and left out here): the
      // resident ones and these make up every expert exactly once
      if (lane == 0) {
        for (int m = 0; m < nmiss; ++m) {
          const int e = p.miss_list[m];
          if (e < 0 || e >= E || ((mseen[e >> 5] >> (e & 31)) & 1u)) continue;
          mseen[e >> 5] |= 1u << (e & 31);
          if (run < E) eord[run++] = e;
        }
      }
      __syncwarp();
      int running = 0;
      for (int j0 = 0; j0 < E; j0 += 32) {
        const int j = j0 + lane;
        int n = 0;
        if (j < E) {
          const int e = eord[j];
          n = max(soff[e + 1] - soff[e], 0);
        }
        const int tiles = ((n + kGvRows - 1) / kGvRows) * ps.mblocks;
        int incl = tiles;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += y;
        }
        if (j < E) prefix[j] = running + incl - tiles;
        running += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) prefix[E] = running;
    }
    __syncthreads();
    sc.order = eord;
  }

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ packed chunk producer
    const uint64_t pol = ptx::policy_evict_first();
    static_assert(SQ <= 64, "armed-slot masks");
    uint64_t armed_mask = 0, armed_ph = 0;  // slots with a copy issued, and the phase it completes
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile tl = sc.tile(t);
      // the expert's record: its own, or its slot in a cache pool (a routed
      // expert without a slot reads slot 0 and flags MOE_DEV_CACHE_FULL)
      int rec = tl.e;
      if (p.slot_of != nullptr) {
        rec = p.slot_of[tl.e];
        if (rec < 0 || rec >= p.S) {
          set_status(p.status, MOE_DEV_CACHE_FULL);
          rec = 0;
        }
      }
      if (FETCH && ((mbits[tl.e >> 5] >> (tl.e & 31)) & 1u)) {
        // a fetched expert: wait until the pieces of the tile's blocks have
        // landed in its slot (bounded)
        const int target = p.ksteps / p.cpp;
        for (int bb = 0; bb < BPT && ok; ++bb) {
          const int* word = p.fsync + 2 + tl.e * p.mblocks + BPT * tl.mb + bb;
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
        }
        if (!ok) break;
        fence_proxy_async_global();
      }
      for (int ks = 0; ks < p.ksteps; ks += QG) {
        if (!wait_bounded<kSpin>(qempty0 + 8 * s, ph ^ 1u, misc + 1, p.status)) {
          ok = false;
          break;
        }
        const uint32_t fb = qfull0 + 8 * s;
        armed_mask |= 1ull << s;
        armed_ph = (armed_ph & ~(1ull << s)) | (static_cast<uint64_t>(ph) << s);
        ptx::mbar_arrive_expect_tx(fb, CPS * kQChunk);
        // K steps ks .. ks + QG - 1 of each of the tile's BPT 128-row blocks
        const size_t c0 = (static_cast<size_t>(rec) * p.mblocks + BPT * tl.mb) * p.ksteps + ks;
#pragma unroll
        for (int bb = 0; bb < BPT; ++bb)
          ptx::bulk_load(ptx::smem_u32(sQ + (s * CPS + bb * QG) * kQChunk), p.tiles + (c0 + bb * p.ksteps) * kQChunk,
                         QG * kQChunk, fb, pol);
        if (++s == SQ) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok || misc[1]) {
      for (int q = 0; q < SQ; ++q)
        if ((armed_mask >> q) & 1u) wait_drain(qfull0 + 8 * q, static_cast<uint32_t>((armed_ph >> q) & 1u));
    }
  } else if (warp == 1) {
    // ------------------------------------------------ token-row producer
    // Lane 0 stages each tile's token rows (one bulk copy per row); once they
    // have landed the warp converts them to fp16 in place and sums every row
    // over every 64-input K step (fp32, input order) into the tile's table,
    // which supplies the correction of the biased codes, and then marks the
    // stage full.
    const uint64_t pol = ptx::policy_evict_last();
    uint32_t armed_mask = 0, armed_ph = 0;
    bool ok = true;
    int ntile = 0;
    if (late_wait) pdl_wait();
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++ntile) {
      const Tile tl = sc.tile(t);
      const int b = ntile & 1;
      const uint32_t use = static_cast<uint32_t>(ntile >> 1) & 1u;
      const int n = min(tl.nrows, kGvRows);
      if (lane == 0) {
        ok = wait_bounded<kSpin>(xempty0 + 8 * b, use ^ 1u, misc + 1, p.status);
        if (ok) {
          const uint32_t lb = xland0 + 8 * b;
          armed_mask |= 1u << b;
          armed_ph = (armed_ph & ~(1u << b)) | (use << b);
          ptx::mbar_arrive_expect_tx(lb, static_cast<uint32_t>(n * K * 2));
          for (int j = 0; j < n; ++j)
            ptx::bulk_load(ptx::smem_u32(sX + b * C::kXBytes + j * (K * 2 + 16)),
                           p.brows + static_cast<size_t>(tl.row0 + j) * K, static_cast<uint32_t>(K * 2), lb, pol);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const bool landed = wait_bounded<kSleepEpi>(xland0 + 8 * b, use, misc + 1, p.status);
      if (!__all_sync(0xffffffffu, landed)) {
        ok = false;
        break;
      }
      float* xs = sXs + b * C::kXsFloats;
      for (int it = lane; it < p.ksteps * kGvRows; it += 32) {  // item = (K step, token row)
        const int ks = it / kGvRows, j = it % kGvRows;
        // The step's 64 bf16 values become fp16 in place, those at inputs
        // with bit 1 set (odd pair words) divided by 16 (they meet codes
        // scaled by 16); both are exact inside fp16's normal range, and
        // magnitudes of 65,520 and more become infinite.  s1 sums the stored
        // values, s16 the token values themselves (fp32, input order).
        float s1 = 0.f, s16 = 0.f;
        if (j < n) {
          uint4* src = reinterpret_cast<uint4*>(sX + b * C::kXBytes + j * (K * 2 + 16) + ks * (kBK * 2));
#pragma unroll
          for (int v = 0; v < kBK / 8; ++v) {
            const uint4 w = src[v];
            uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float sc = (e & 1) ? 0.0625f : 1.0f;
              const __half2 h2 = __floats2half2_rn(__uint_as_float(ws[e] << 16) * sc,
                                                   __uint_as_float(ws[e] & 0xFFFF0000u) * sc);
              const float f0 = __low2float(h2), f1 = __high2float(h2);
              s1 += f0;
              s1 += f1;
              s16 += (e & 1) ? 16.0f * (f0 + f1) : (f0 + f1);
              std::memcpy(&ws[e], &h2, 4);
            }
            src[v] = make_uint4(ws[0], ws[1], ws[2], ws[3]);
          }
        }
        // sum over the step of A x B = 1024 s1 + sum(stored code x x), and
        // stored code = code + 8: the MMAs start from -(1024 s1 + 8 s16)
        const float c = -(1024.0f * s1 + 8.0f * s16);
        xs[ks * 8 + 4 * (j >> 1) + (j & 1)] = c;
        xs[ks * 8 + 4 * (j >> 1) + (j & 1) + 2] = c;
      }
      // the stage was rewritten by ordinary stores; a later bulk copy into it
      // (async proxy) must be ordered after them
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(xfull0 + 8 * b);
    }
    if (lane == 0 && (!ok || misc[1])) {
      for (int q = 0; q < 2; ++q)
        if ((armed_mask >> q) & 1u) wait_drain(xland0 + 8 * q, (armed_ph >> q) & 1u);
    }
  } else if (FETCH && warp >= kGvWarps) {
    // ---------------------------------------------------------- fetch
    // Each warp claims the next piece of the plan: every gate/up piece of
    // the misses (in plan order), then every down piece; copies it host ->
    // slot with eight 16-byte loads in flight per lane, fences for the bulk
    // copies of other CTAs, and counts a gate/up piece as landed in its
    // block's word.
    const int nblk = p.mblocks;
    const int ppb = p.ksteps / p.cpp;                       // pieces per gate/up block
    const int pg = nblk * ppb;                              // pieces per gate/up record
    const int pd = static_cast<int>((p.rec_dn + kGvFetchBytes - 1) / kGvFetchBytes);
    const int totalp = nmiss * (pg + pd);
    for (;;) {
      int qi = 0;
      if (lane == 0) qi = atomicAdd(p.fsync, 1);
      qi = __shfl_sync(0xffffffffu, qi, 0);
      if (qi >= totalp || misc[1]) break;
      const bool gu = qi < nmiss * pg;
      const int m = gu ? qi / pg : (qi - nmiss * pg) / pd;
      const int c = gu ? qi % pg : (qi - nmiss * pg) % pd;
      const int e = p.miss_list[m], sl = p.miss_slot[m];
      const bool valid = e >= 0 && e < E && sl >= 0 && sl < p.S;
      if (valid) {
        const size_t rec = gu ? p.rec_gu : p.rec_dn;
        const size_t off = gu ? static_cast<size_t>(c) * p.cpp * kQChunk : static_cast<size_t>(c) * kGvFetchBytes;
        const size_t len = gu ? static_cast<size_t>(p.cpp) * kQChunk : min(rec - off, size_t(kGvFetchBytes));
        const int nv = static_cast<int>(len / 16);
        const uint4* src = reinterpret_cast<const uint4*>((gu ? p.host_gu : p.host_dn) + e * rec + off);
        uint4* dst = reinterpret_cast<uint4*>((gu ? const_cast<uint8_t*>(p.tiles) : p.pool_dn) + sl * rec + off);
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
      if (lane == 0 && valid && gu) atomicAdd(p.fsync + 2 + e * nblk + c / ppb, 1);
    }
  } else if (warp >= 2) {
    // ---------------------------------------------------------- compute
    const int grp = (warp - 2) / WPG;  // takes the ring slots gu with gu % G == grp
    const int cwg = (warp - 2) % WPG;  // owns tile rows 32 cwg .. 32 cwg + 31
    const int blk = cwg / kGvWpg;      // the 128-row block (chunk) of those rows
    const int cw = cwg % kGvWpg;       // rows 32 cw .. 32 cw + 31 of that block
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
      // 0x64006400 (fp16 1024 pair), opaque to the compiler so that it stays in a register
      const uint32_t magic = 0x64006400u | (static_cast<uint32_t>(p.ksteps) >> 31);
      const uint8_t* xrow = sX + b * C::kXBytes + (g & (kGvRows - 1)) * (K * 2 + 16) + 32 * q;
      // the corrections of token columns 2q, 2q + 1 in accumulator order
      // (columns past the tile's rows read another column's and are never
      // stored)
      const float* xsum = sXs + b * C::kXsFloats + 4 * (q & 1);
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      // The MMA's k slots run over a step's 64 inputs in a permuted order
      // (the same for weights and tokens, so the products and their sum are
      // unchanged): in k16 block j, lane q's slots 2q, 2q + 1 take inputs
      // 16q + 4j, +1 and slots 2q + 8, 2q + 9 take inputs 16q + 4j + 2, +3.
      // Lane q thus reads inputs 16q .. 16q + 15 only: 8 code bytes per
      // weight row and 32 bytes of each token row, and every code pair sits
      // at a fixed nibble position.  A group takes whole ring slots (S
      // consecutive K steps): one wait and one release per slot.
      const int nslot = p.ksteps / S;
      const uint32_t sbase = gbase / S;  // this CTA's running ring-slot index at the tile's start
      for (int u = static_cast<int>((static_cast<uint32_t>(grp) + G - sbase % G) % G); u < nslot; u += G) {
        const uint32_t gu = sbase + u;
        const uint32_t sq = gu % SQ;
        got = wait_bounded<kSpin>(qfull0 + 8 * sq, (gu / SQ) & 1u, misc + 1, p.status);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
#pragma unroll 2  // two steps interleaved: more would spill
        for (int st = 0; st < S; ++st) {
          uint2 cw[4];  // code words of rows r0 + 8i, inputs 16q .. 16q + 15 of the step
          float sc[4];  // their group scales
          const uint8_t* chunk = sQ + (sq * CPS + blk * S + st) * kQChunk;
          const uint16_t* scl = reinterpret_cast<const uint16_t*>(chunk + kQBytes);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            cw[i] = *reinterpret_cast<const uint2*>(chunk + (r0 + 8 * i) * 32 + 8 * q);
            sc[i] = bf16_to_f32(scl[r0 + 8 * i]);
          }
          if (st == S - 1) {  // the slot's last reads are done: release it
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(qempty0 + 8 * sq);
          }
          const uint4* xk = reinterpret_cast<const uint4*>(xrow + (u * S + st) * (kBK * 2));
          const uint4 x0 = xk[0], x1 = xk[1];
          const uint32_t xb[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          // The MMAs take the codes as exact fp16 pairs (1024 + stored code
          // against the token value, 1024 + 16 stored code against a sixteenth
          // of it) and start from the step's correction in the table, so
          // they end at sum(code x).
          const float4 xs = *reinterpret_cast<const float4*>(xsum + (u * S + st) * 8);
          float d0[4], d1[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // word j/2 of a row holds inputs 16q + 8(j/2) .. +7; its pair
            // 2(j%2) is inputs 16q + 4j, +1 and pair 2(j%2) + 1 the next two
            const uint32_t sh = (j & 1) ? 8u : 0u;  // pairs 2(j%2), 2(j%2) + 1 sit 8 bits up for odd j
            const uint32_t v0 = ((j >> 1) ? cw[0].y : cw[0].x) >> sh, v1 = ((j >> 1) ? cw[1].y : cw[1].x) >> sh;
            const uint32_t v2 = ((j >> 1) ? cw[2].y : cw[2].x) >> sh, v3 = ((j >> 1) ? cw[3].y : cw[3].x) >> sh;
            const uint32_t a0[4] = {code_pair_f16(v0, true, magic), code_pair_f16(v1, true, magic),
                                    code_pair_f16(v0, false, magic),
                                    code_pair_f16(v1, false, magic)};  // rows r0, r0 + 8
            const uint32_t a1[4] = {code_pair_f16(v2, true, magic), code_pair_f16(v3, true, magic),
                                    code_pair_f16(v2, false, magic),
                                    code_pair_f16(v3, false, magic)};  // rows r0 + 16, r0 + 24
            if (j == 0) {
              mma_16816_f16_first(d0, a0, xb[0], xb[1], xs);
              mma_16816_f16_first(d1, a1, xb[0], xb[1], xs);
            } else {
              mma_16816_f16(d0, a0, xb[2 * j], xb[2 * j + 1]);
              mma_16816_f16(d1, a1, xb[2 * j], xb[2 * j + 1]);
            }
          }
          acc[0] = fmaf(sc[0], d0[0], acc[0]);  // row r0, token 2q
          acc[1] = fmaf(sc[0], d0[1], acc[1]);  // row r0, token 2q + 1
          acc[2] = fmaf(sc[1], d0[2], acc[2]);  // row r0 + 8
          acc[3] = fmaf(sc[1], d0[3], acc[3]);
          acc[4] = fmaf(sc[2], d1[0], acc[4]);  // row r0 + 16
          acc[5] = fmaf(sc[2], d1[1], acc[5]);
          acc[6] = fmaf(sc[3], d1[2], acc[6]);  // row r0 + 24
          acc[7] = fmaf(sc[3], d1[3], acc[7]);
        }
      }
      if (!ok) break;
      gbase += static_cast<uint32_t>(p.ksteps);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(xempty0 + 8 * b);
      if constexpr (G > 1) {  // (one group: it holds the whole sums)
        // The group that took the tile's last ring slot (it finishes last)
        // reduces and stores; the others hand it their sums of the valid token
        // columns (lanes q < 2), slot ri = their distance after it - 1.
        const int eg = static_cast<int>((sbase + static_cast<uint32_t>(nslot) - 1u) % G);
        if (grp != eg) {
          got = wait_bounded<kSleepEpi>(rede0 + 8 * b, use ^ 1u, misc + 1, p.status);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          if (q < kGvRows / 2) {
            const int ri = (grp - eg - 1 + G) % G;
            float* red = sRed + b * C::kRedFloats + ri * (RT * kGvRows) + blk * (kBM * kGvRows);
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
          for (int gi = 0; gi < G - 1; ++gi) {
            const float* red = sRed + b * C::kRedFloats + gi * (RT * kGvRows) + blk * (kBM * kGvRows);
  #pragma unroll
            for (int i = 0; i < 4; ++i) {
              acc[2 * i] += red[(r0 + 8 * i) * kGvRows + 2 * q];
              acc[2 * i + 1] += red[(r0 + 8 * i) * kGvRows + 2 * q + 1];
            }
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(rede0 + 8 * b);
      }
      const int t0 = 2 * q, t1 = 2 * q + 1;
      if (KIND == 1) {
        float* y = reinterpret_cast<float*>(p.out);
        const int col = tl.mb * RT + blk * kBM;
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
      const int colA = (tl.mb * BPT + blk) * 64 + 16 * cw + g, colB = colA + 8;
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
  if constexpr (FETCH) {
    // the last CTA out resets the piece queue, the exit count and the landed
    // counts of the fetched experts for the next call
    if (threadIdx.x == 0) {
      __threadfence();
      misc[2] = atomicAdd(p.fsync + 1, 1) == static_cast<int>(gridDim.x) - 1;
    }
    __syncthreads();
    if (misc[2]) {
      __threadfence();
      for (int i = threadIdx.x; i < nmiss * p.mblocks; i += blockDim.x) {
        const int e = p.miss_list[i / p.mblocks];
        if (e >= 0 && e < E) p.fsync[2 + e * p.mblocks + i % p.mblocks] = 0;
      }
      if (threadIdx.x == 0) {
        p.fsync[0] = 0;
        p.fsync[1] = 0;
      }
      __threadfence();
    }
  }
}

template <int KIND, int QG, int BPT, bool FETCH = false>
cudaError_t run_gemv_q4_g(const GemmArgs& args, cudaStream_t st) {
  auto kern = gemv_q4_kernel<KIND, QG, BPT, FETCH>;
  cudaError_t e = ensure_smem(kern, CfgV::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = sm_count();
  if (grid <= 0) return cudaErrorNoDevice;
  // the gate/up launch leaves its offsets as its stream's token (so does
  // the row gather); a launch that finds its own offsets there follows
  // such a launch directly
  const int early = stream_token_get(st) == args.offsets ? 1 : 0;
  e = launch_pdl(kern, dim3(grid), dim3(kGvThreads + (FETCH ? 32 * kGvFetchWarps : 0)), CfgV::kSmemBytes, st, args,
                 early);
  if (e == cudaSuccess && KIND == 0) stream_token_set(st, args.offsets);
  return e;
}

// Gate/up with the in-launch fetch: the same tile shapes as run_gemv_q4<0>.
cudaError_t run_gemv_q4_fetch(const GemmArgs& args, cudaStream_t st) {
  const bool even = args.ksteps % 2 == 0;
  if (args.mblocks % 2 == 0 && args.ksteps % 4 == 0) return run_gemv_q4_g<0, 4, 2, true>(args, st);
  if (args.ksteps % 4 == 0) return run_gemv_q4_g<0, 4, 1, true>(args, st);
  return even ? run_gemv_q4_g<0, 2, 1, true>(args, st) : run_gemv_q4_g<0, 1, 1, true>(args, st);
}

// A ring slot holds as many consecutive K steps as divide the record's
// (four, two or one).  Down tiles span four 128-row blocks (one group of all
// sixteen warps: no hand-over of sums) or two when the block count allows,
// and a slot then holds two steps of each block.
template <int KIND>
cudaError_t run_gemv_q4(const GemmArgs& args, cudaStream_t st) {
  const bool even = args.ksteps % 2 == 0;
  if (KIND == 1 && args.mblocks % 4 == 0)
    return even ? run_gemv_q4_g<1, 2, 4>(args, st) : run_gemv_q4_g<1, 1, 4>(args, st);
  if (KIND == 1 && args.mblocks % 2 == 0)
    return even ? run_gemv_q4_g<1, 2, 2>(args, st) : run_gemv_q4_g<1, 1, 2>(args, st);
  if (KIND == 0 && args.mblocks % 2 == 0 && args.ksteps % 4 == 0) return run_gemv_q4_g<0, 4, 2>(args, st);
  if (args.ksteps % 4 == 0) return run_gemv_q4_g<KIND, 4, 1>(args, st);
  return even ? run_gemv_q4_g<KIND, 2, 1>(args, st) : run_gemv_q4_g<KIND, 1, 1>(args, st);
}

}  // namespace

namespace gk {

// Decode-sized int4 launches (few rows per expert, K within the token-row
// stage) go to the CUDA-core kernel.
bool use_gemv_q4(int fmt, int R, int K) {
  return fmt == MOE_W_INT4_G64_TILED && pick_nmax(R) == 16 && K <= kGvMaxK;
}

cudaError_t launch_gemv_q4(int kind, const GemmArgs& args, cudaStream_t st) {
  if (kind == 0 && args.host_gu != nullptr) return run_gemv_q4_fetch(args, st);
  return kind == 1 ? run_gemv_q4<1>(args, st) : run_gemv_q4<0>(args, st);
}

}  // namespace gk

}  // namespace moe
