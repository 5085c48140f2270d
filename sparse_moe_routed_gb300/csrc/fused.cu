// Gate/up + SwiGLU + down of every routed expert in one persistent launch
// (tile-packed bf16 records), with the row gather of a decode block and, for
// the expert cache, slot tables and in-launch fetch warps.  AFN-019 "Hide SSD
// misses before the router knows they exist", section "Hypothesis H4": gate
// and up of an expert together, down once its SwiGLU intermediate exists;
// fetched records consumed as they land.  Shared tile machinery:
// gemm_common.cuh.
#include <cuda.h>
#include <cuda_bf16.h>

#include "gemm_common.cuh"

namespace moe {

using namespace gk;

namespace {

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
  float* y;                 // [R, H] fp32 expert outputs, or (yw != nullptr) unused
  // Weighted outputs (yw != nullptr): the down epilogue multiplies slot s's
  // row by its route weight topk_w[perm[s]] and stores it rounded to bf16 in
  // yw [R, H], which halves the bytes written here and read by the combine.
  const float* topk_w;
  uint16_t* yw;
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
// launches up to this many rows, and every launch of 256-row token tiles,
// claim tiles dynamically
constexpr int kFusedDynamicRows = 4096;
constexpr int kFetchChunk = 32768;
// launches of at least this many routes per expert (on average) take
// 256-row token tiles
constexpr int kFusedWideRowsPerExpert = 256;

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
  // token rows per TMA box: 16 (a decode block's rows), or 64 for 256-row
  // tiles, which then take at most four copies per K step instead of 16
  static constexpr int kBoxR = NMAX >= 256 ? 128 : box_rows_for(NMAX);
  static constexpr int kBoxB = kBoxR * kBK * 2;
  static constexpr int kNumBars = 2 * kStages + 5 + 2 * kTileRing;
  // misc words and the tile-id ring; offsets and the two tile prefixes;
  // cached: also slots and the expert order; then the epilogue warps' route
  // weights of the current tile's columns (weighted outputs)
  static constexpr int kTail = 32 + (CACHED ? 5 : 3) * (kMaxE + 1) * 4 + 16 + 4 * NMAX * 4;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kNumBars * 8 + kTail;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

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
// decode launch); on large launches of 128-row tiles the static order
// measured faster, on 256-row tiles the queue.  A down tile waits for the gate/up
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

// The in-launch row gather of a decode-sized launch: this CTA's contiguous
// share of the permuted token rows (x_perm[s] = x[perm[s] / k]), eight
// 16-byte loads in flight per thread, by the 128 epilogue threads (et = 0 ..
// 127); then fenced for the async proxy and counted once per CTA, so that
// the producers can start their token-row loads once every CTA has counted.
__device__ __forceinline__ void gather_share(const FusedArgs& p, int E, int et) {
  constexpr int kEpiThreads = 128;
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
  fence_proxy_async_global();
  __threadfence();
  asm volatile("bar.sync 2, %0;" ::"n"(kEpiThreads) : "memory");
  if (et == 0) atomicAdd(p.ready + E + 1, 1);
}

// Tile counts per position of the expert order: pre_gu[j] / pre_dn[j] =
// the gate/up / down tiles of the experts before position j (one warp).
// Chunk counts go to pre_dn in position order (coalesced); lane l then sums
// its run of consecutive positions (starting at a lane-dependent offset so
// that the lanes' reads fall in different banks), one warp scan places the
// runs, each lane writes its run's prefixes in order, and a last coalesced
// pass scales them by the blocks per expert.
template <int NMAX, bool CACHED>
__device__ __forceinline__ void tile_prefix(const FusedArgs& p, int E, const int* soff, const int* eord, int* pre_gu,
                                            int* pre_dn, int lane) {
  for (int j = lane; j < E; j += 32) {
    const int e = CACHED ? eord[j] : j;
    pre_dn[j] = (max(soff[e + 1] - soff[e], 0) + NMAX - 1) / NMAX;
  }
  __syncwarp();
  const int per = (E + 31) / 32;
  const int j0 = min(E, lane * per), j1 = min(E, j0 + per);
  const int n = j1 - j0;
  int c = 0;
  int kk = n > 0 ? lane % n : 0;
  for (int i = 0; i < n; ++i) {
    c += pre_dn[j0 + kk];
    kk = kk + 1 == n ? 0 : kk + 1;
  }
  int incl = c;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  int run = incl - c;
  for (int j = j0; j < j1; ++j) {
    const int cj = pre_dn[j];
    pre_gu[j] = run;
    run += cj;
  }
  __syncwarp();
  for (int j = lane; j < E; j += 32) {
    const int r = pre_gu[j];
    pre_gu[j] = r * p.mb_gu;
    pre_dn[j] = r * p.mb_dn;
  }
  if (lane == 0) {
    pre_gu[E] = total * p.mb_gu;
    pre_dn[E] = total * p.mb_dn;
  }
}

// One CTA's check-out from the launch's sync words (one thread): once every
// CTA has checked out, no producer will read them and no epilogue will count
// in them again, so the CTA that checks out last zeroes them for the next
// launch.
__device__ __forceinline__ void sync_words_check_out(const FusedArgs& p, int E) {
  __threadfence();
  if (atomicAdd(p.ready + E, 1) == static_cast<int>(gridDim.x) - 1) {
    __threadfence();
    for (int e = 0; e < E + 3; ++e) p.ready[e] = 0;
    __threadfence();
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
  // [4 epilogue warps][NMAX] route weights of the current tile's columns
  // (16-byte aligned: the epilogue reads it four floats at a time)
  float* swt = reinterpret_cast<float*>(
      (reinterpret_cast<uintptr_t>(soff + (CACHED ? 3 : 1) * (kMaxE + 1)) + 15) & ~static_cast<uintptr_t>(15));

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
    misc[3] = 0;  // uncached: roles done with the sync words (producer + 4 epilogue warps)
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
  if constexpr (!CACHED) {
    // Every thread reads the segment offsets; then the epilogue warps gather
    // the token rows while warp 0 builds the tile prefix and warp 1 asks L2
    // for the first weight stages of gate/up tile blockIdx.x (the tile this
    // CTA takes first in the static order, and one of the first wave's on
    // the queue), so that HBM starts streaming before the producer's first
    // claim.  Warp 0 arrives on named barrier 3, where warp 1 waits for the
    // prefix; warps 0 and 1 arrive on barrier 4, where the epilogue warps
    // wait.
    for (int i = threadIdx.x; i <= E; i += kCoreThreads) soff[i] = min(max(p.offsets[i], 0), p.R);
    __syncthreads();
    if (warp >= 2) {
      if (p.x != nullptr) gather_share(p, E, threadIdx.x - 64);
      asm volatile("bar.sync 4, %0;" ::"n"(kCoreThreads) : "memory");
    } else if (warp == 0) {
      tile_prefix<NMAX, CACHED>(p, E, soff, eord, pre_gu, pre_dn, lane);
      ptx::tc_fence_before();
      asm volatile("bar.arrive 3, 64;" ::: "memory");
      asm volatile("bar.arrive 4, %0;" ::"n"(kCoreThreads) : "memory");
    } else {
      // gate/up tile g = blockIdx.x: the expert whose tile range holds it,
      // walking the experts 32 at a time
      const int g = blockIdx.x;
      int run = 0;
      bool found = false;
      for (int e0 = 0; e0 < E && !found; e0 += 32) {
        const int e = e0 + lane;
        const int n = e < E ? max(soff[e + 1] - soff[e], 0) : 0;
        const int tiles = ((n + NMAX - 1) / NMAX) * p.mb_gu;
        int incl = tiles;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += y;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, tiles > 0 && g >= run + incl - tiles && g < run + incl);
        if (hit != 0u) {
          found = true;
          const int src = __ffs(hit) - 1;
          const int local = g - run - __shfl_sync(0xffffffffu, incl - tiles, src);
          const int mb = local % p.mb_gu;
          if (lane == 0) {
            const size_t chunk0 = (static_cast<size_t>(e0 + src) * p.mb_gu + mb) * p.ks_gu;
            const int ks = min(p.ks_gu, C::kStages * G);
            ptx::bulk_prefetch_l2(p.tiles_gu + chunk0 * kABytes, static_cast<uint32_t>(ks * kABytes));
          }
        }
        run += __shfl_sync(0xffffffffu, incl, 31);
      }
      ptx::tc_fence_before();
      asm volatile("bar.sync 3, 64;" ::: "memory");
      asm volatile("bar.arrive 4, %0;" ::"n"(kCoreThreads) : "memory");
    }
    ptx::tc_fence_after();
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
    tile_prefix<NMAX, CACHED>(p, E, soff, eord, pre_gu, pre_dn, lane);
  }
  ptx::tc_fence_before();
  compute_sync();
  ptx::tc_fence_after();
  }
  const uint32_t tmem_base = misc[0];
  const int total_gu = pre_gu[E];
  const int total = total_gu + pre_dn[E];
  const int jB = E - nmiss;  // first position of a fetched expert
  const int tguA = pre_gu[jB], tdnA = pre_dn[jB], tguB = total_gu - tguA;
  int* const queue = p.ready + E + 2;  // device-wide tile queue
  // 256-row tiles: an expert's rows span several chunks that read the same
  // weight tiles; claimed from the queue, the tiles of one expert run at
  // nearly the same time on different SMs and share those weights in L2
  // (the static order lets the CTAs drift apart and re-read them from HBM)
  const bool dynamic = p.R <= kFusedDynamicRows || NMAX == 256;
  const FSeq seq1(blockIdx.x, gridDim.x, total_gu, pre_dn[E], p.ks_gu, p.ks_dn);
  const FOrder seq2(blockIdx.x, gridDim.x, tguA, tdnA, tguB, pre_dn[E] - tdnA, p.ks_gu, p.ks_dn);
  // Uncached launches check out of the sync words early: the producer once
  // it has claimed its last tile, each epilogue warp once it reaches its
  // first down tile (its gate/up counts are all made); the fifth part checks
  // the CTA out, so the last CTA zeroes the words while others still compute.
  auto check_out_part = [&]() {
    __threadfence();
    if (atomicAdd(const_cast<uint32_t*>(&misc[3]), 1u) == 4u) sync_words_check_out(p, E);
  };
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
    // weights: read once when the expert's rows fit one tile, else once per
    // row chunk (kept in L2 for the other chunks' tiles)
    const uint64_t pol_w1 = ptx::policy_evict_first();
    const uint64_t pol_wn = ptx::policy_evict_normal();
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
            ptx::tma_load_2d(pend_dst[q] + j * C::kBBytes + b * C::kBoxB, &tmX, pend_bar[q], (pend_ks[q] + j) * kBK,
                             pend_row[q] + b * C::kBoxR, pol_x);
      npend = 0;
      return true;
    };
    int qs = 0;
    uint32_t qph = 0;
    // Decode-sized launches claim their next tile only once the current
    // one's stages are all issued: the stage ring hides the claim's round
    // trip, and at the end of the queue no CTA holds a claimed tile that an
    // idle one could take (measured 0.2 us per decode step).  With an expert
    // cache, and for 256-row tiles (0.3 % faster so), the next claim goes
    // out while a tile's loads do.
    constexpr bool kClaimAhead = CACHED || NMAX == 256;
    int next = (dynamic && kClaimAhead) ? atomicAdd(queue, 1) : 0;
    for (int n = 0; ok; ++n) {
      int t;
      if (dynamic) {
        const int g = kClaimAhead ? next : atomicAdd(queue, 1);
        t = g < total ? (CACHED ? fused_tile_at(g, tguA, tdnA, tguB, total_gu) : g) : -1;
        if (kClaimAhead && t >= 0) next = atomicAdd(queue, 1);
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
      const int nblk = (tl.nrows + C::kBoxR - 1) / C::kBoxR;
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
      const uint64_t pol_w = soff[tl.e + 1] - soff[tl.e] > NMAX ? pol_wn : pol_w1;
      for (int ks = 0; ks < KS; ks += G) {
        if (!wait_bounded<kSpin>(empty0 + 8 * s, ph ^ 1u, misc + 1, p.status)) {
          ok = false;
          break;
        }
        const uint32_t fb = full0 + 8 * s;
        ptx::mbar_arrive_expect_tx(fb, G * (kABytes + nblk * C::kBoxB));
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
              ptx::tma_load_2d(b_dst + j * C::kBBytes + b * C::kBoxB, tb, fb, (ks + j) * kBK,
                               tl.row0 + b * C::kBoxR, pol_x);
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
    if constexpr (!CACHED) check_out_part();
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
    if (CACHED && p.x != nullptr) gather_share(p, E, threadIdx.x - 64);
    const int q = warp & 3;
    const int row_in_tile = q * 32 + lane;
    int acc = 0;
    uint32_t aph = 0;
    int qs = 0;
    uint32_t qph = 0;
    bool out = CACHED;  // checked out of the sync words (uncached launches)
    for (;;) {
      int t = -1;
      if (!__all_sync(0xffffffffu, read_tile(qs, qph, &t))) break;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(tqe0 + 8 * qs);
      if (++qs == QR) {
        qs = 0;
        qph ^= 1u;
      }
      if (!out && (t < 0 || t >= total_gu)) {
        out = true;
        if (lane == 0) check_out_part();
      }
      if (t < 0) break;
      const FTile tl = tile_of(t);
      // weighted outputs: the route weight of every column of a gate/up
      // tile into this warp's row of swt, loaded before the wait for the
      // accumulator so that the two dependent loads overlap the tile's MMAs
      float* wrow = swt + q * NMAX;
      if (tl.kind == 0 && p.yw != nullptr) {
        for (int c = lane; c < tl.nrows; c += 32) {
          float wv = 0.f;
          const int r = p.perm[tl.row0 + c];
          if (r >= 0 && r < p.R) {
            wv = p.topk_w[r];
          } else {
            set_status(p.status, MOE_DEV_BAD_EXPERT);
          }
          wrow[c] = wv;
        }
        __syncwarp();
      }
      const bool ok = wait_bounded<kSleepEpi>(accf0 + 8 * acc, aph, misc + 1, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      ptx::tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * NMAX);
      if (tl.kind == 0 && p.yw != nullptr) {
        // weighted: h[s] = bf16(w_s * silu(g) * u), so the down tile's
        // accumulator is already w_s * (W_down h[s])
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
          const float4 wa = *reinterpret_cast<const float4*>(wrow + c0 + (up_lane ? 8 : 0));
          const float4 wb = *reinterpret_cast<const float4*>(wrow + c0 + (up_lane ? 12 : 4));
          const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int col = c0 + (up_lane ? 8 : 0) + jj;
            const float g = up_lane ? recv[jj] : v[jj];
            const float u = up_lane ? v[8 + jj] : recv[jj];
            if (col < tl.nrows)
              p.h[static_cast<size_t>(tl.row0 + col) * p.I + i] =
                  __bfloat16_as_ushort(__float2bfloat16_rn(wv[jj] * (g / (1.0f + expf(-g)) * u)));
          }
        }
      } else if (tl.kind == 0) {
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
      }
      if (tl.kind == 0) {
        // publish this warp's h rows to TMA loads in other CTAs: each lane
        // fences its own stores, then one arrival per warp (4 per tile)
        fence_proxy_async_global();
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(p.ready + tl.e, 1);
      } else if (p.yw == nullptr) {
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
      } else {
        // weighted: the accumulator already carries the route weight (it
        // was applied to h); bf16 rows
        const int j = tl.mb * kBM + row_in_tile;
        for (int c0 = 0; c0 < tl.nrows; c0 += 16) {
          float v[16];
          ptx::tmem_ld16(taddr + static_cast<uint32_t>(c0), v);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int col = c0 + jj;
            if (col < tl.nrows)
              p.yw[static_cast<size_t>(tl.row0 + col) * p.H + j] = __bfloat16_as_ushort(__float2bfloat16_rn(v[jj]));
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
  if constexpr (!CACHED) {
    // a role that left on an error path: complete the CTA's check-out here
    if (threadIdx.x == 0 && misc[3] < 5u) {
      misc[3] = 5u;
      sync_words_check_out(p, E);
    }
    return;
  }
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

template <int NMAX, int GG, bool CACHED>
cudaError_t run_fused(const FusedArgs& args, cudaStream_t st) {
  using C = CfgF<NMAX, GG, CACHED>;
  // token-row maps with this variant's box height
  CUtensorMap mx, mh;
  if (!make_rows_map(&mx, args.x_perm, args.H, args.R, C::kBoxR)) return cudaErrorInvalidValue;
  if (!make_rows_map(&mh, args.h, args.I, args.R, C::kBoxR)) return cudaErrorInvalidValue;
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
                                const void* w_down, const FusedCache* cache, uint16_t* h, float* y,
                                const float* topk_w, uint16_t* yw, int32_t* ready, int32_t* st_word,
                                cudaStream_t st) {
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
  a.topk_w = topk_w;
  a.yw = yw;
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
      case 16: return run_fused<16, 2, true>(a, st);
      case 32: return run_fused<32, 2, true>(a, st);
      case 64: return run_fused<64, 2, true>(a, st);
      default: return run_fused<128, 2, true>(a, st);
    }
  }
  // Compute-bound launches (hundreds of token rows per expert): 256-row
  // token tiles (MMA N = 256, both accumulators filling the 512 TMEM
  // columns), which halve how often an expert's weights are streamed and
  // take 48 KB of operands per 128 x 256 x 64 step instead of 32 KB per
  // 128 x 128 x 64; one K step per stage keeps four stages in 196 KB.
  if (static_cast<long long>(R) >= static_cast<long long>(kFusedWideRowsPerExpert) * E)
    return run_fused<256, 1, false>(a, st);
  if (a.ks_gu % 2 == 0 && a.ks_dn % 2 == 0) {
    switch (pick_nmax(R)) {
      case 16: return run_fused<16, 2, false>(a, st);
      case 32: return run_fused<32, 2, false>(a, st);
      case 64: return run_fused<64, 2, false>(a, st);
      default: return run_fused<128, 2, false>(a, st);
    }
  }
  switch (pick_nmax(R)) {
    case 16: return run_fused<16, 1, false>(a, st);
    case 32: return run_fused<32, 1, false>(a, st);
    case 64: return run_fused<64, 1, false>(a, st);
    default: return run_fused<128, 1, false>(a, st);
  }
}

}  // namespace moe
