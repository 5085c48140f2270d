// Expert weight packing: the one-time reordering of expert records into the
// tile order the grouped contraction streams.
//
// AFN-019 "Hide SSD misses before the router knows they exist", section
// "Hypothesis H4": ExpertMajor gives each expert one contiguous record with
// explicit component extents.  The packed records keep that (each expert's
// gate/up component and its down component stay contiguous) and order the
// bytes inside a component by (128-row weight block, 64-wide K step), so that
// every pipeline stage of the contraction is one contiguous chunk that a
// single bulk copy moves from HBM:
//
//   bf16 (MOE_W_BF16_TILED): 16,384-byte chunks, the exact shared-memory
//     image of a 128 x 64 bf16 tile with the 128-byte swizzle applied
//     (16-byte piece c of row r stored at r*128 + (c ^ (r % 8))*16);
//   int4 g64 (MOE_W_INT4_G64_TILED): 4,352-byte chunks, the 128 rows' 32 code
//     bytes (row-major) followed by the rows' 128 bf16 scales of that group.
//     Inside each 32-bit word the eight codes are stored offset by +8 (0..15)
//     with nibble j holding element 0,2,4,6,1,3,5,7 (j = 0..7), so that the
//     contraction's dequantiser extracts two neighbouring elements with one
//     mask-and-or.
//
// Gate/up tiles hold, for intermediate block mb (64 indices), 16 gate rows
// then the 16 matching up rows, four times (row r: q = r / 32, up = (r / 16)
// % 2, i = mb * 64 + q * 16 + r % 16).  Down tiles hold hidden rows
// mb * 128 .. mb * 128 + 127.  Integer data movement only: one thread per
// 16-byte piece, grid-stride over the whole component.
#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

// Source row (within the expert) of tile row r of gate/up block mb.
__device__ __forceinline__ int gu_src_row(int r, int mb, int I) {
  const int q = r >> 5;
  const int up = (r >> 4) & 1;
  return up * I + mb * 64 + q * 16 + (r & 15);
}

// bf16: one thread per 16-byte piece of the packed component.
__global__ void pack_bf16_kernel(const uint16_t* __restrict__ w, int E, int H, int I, int which,
                                 uint16_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int K = which == 0 ? H : I;                  // inputs per row
  const int rows = which == 0 ? 2 * I : H;           // rows per expert
  const int MB = which == 0 ? I / 64 : H / 128;      // 128-row blocks per expert
  const int KS = K / 64;
  const size_t pieces = static_cast<size_t>(E) * MB * KS * 128 * 8;
  for (size_t p = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; p < pieces;
       p += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(p & 7);           // 16-byte piece of the 128-byte row
    const int r = static_cast<int>((p >> 3) & 127);  // tile row
    size_t t = p >> 10;                              // chunk index = ((e * MB) + mb) * KS + ks
    const int ks = static_cast<int>(t % KS);
    t /= KS;
    const int mb = static_cast<int>(t % MB);
    const int e = static_cast<int>(t / MB);
    const int src_row = which == 0 ? gu_src_row(r, mb, I) : mb * 128 + r;
    const uint4 v = reinterpret_cast<const uint4*>(
        w + (static_cast<size_t>(e) * rows + src_row) * K + static_cast<size_t>(ks) * 64)[c];
    uint4* dst = reinterpret_cast<uint4*>(out + (p >> 10) * (128 * 64)) + r * 8 + (c ^ (r & 7));
    *dst = v;
  }
}

// Eight two's-complement codes (element e in nibble e) -> the packed order:
// element e offset by +8 in nibble (e even ? e/2 : 4 + e/2).
__device__ __forceinline__ uint32_t repack_codes(uint32_t src) {
  uint32_t dst = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const uint32_t n = ((src >> (4 * e)) & 0xFu) ^ 0x8u;
    const int pos = (e & 1) ? 4 + (e >> 1) : (e >> 1);
    dst |= n << (4 * pos);
  }
  return dst;
}

// int4 g64: one thread per 16-byte piece of codes, plus the scale of its row.
__global__ void pack_int4_kernel(const uint8_t* __restrict__ q, const uint16_t* __restrict__ s, int E, int H, int I,
                                 int which, uint8_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int K = which == 0 ? H : I;
  const int rows = which == 0 ? 2 * I : H;
  const int MB = which == 0 ? I / 64 : H / 128;
  const int KS = K / 64;
  constexpr int kChunk = 128 * 32 + 128 * 2;
  const size_t pieces = static_cast<size_t>(E) * MB * KS * 128 * 2;  // two 16-byte code pieces per row
  for (size_t p = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; p < pieces;
       p += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int half = static_cast<int>(p & 1);
    const int r = static_cast<int>((p >> 1) & 127);
    size_t t = p >> 8;
    const int ks = static_cast<int>(t % KS);
    t /= KS;
    const int mb = static_cast<int>(t % MB);
    const int e = static_cast<int>(t / MB);
    const int src_row = which == 0 ? gu_src_row(r, mb, I) : mb * 128 + r;
    const size_t row_g = static_cast<size_t>(e) * rows + src_row;
    uint4 v = reinterpret_cast<const uint4*>(q + row_g * (K / 2) + static_cast<size_t>(ks) * 32)[half];
    v.x = repack_codes(v.x);
    v.y = repack_codes(v.y);
    v.z = repack_codes(v.z);
    v.w = repack_codes(v.w);
    uint8_t* chunk = out + (p >> 8) * kChunk;
    reinterpret_cast<uint4*>(chunk + r * 32)[half] = v;
    if (half == 0) reinterpret_cast<uint16_t*>(chunk + 128 * 32)[r] = s[row_g * (K / 64) + ks];
  }
}

}  // namespace

size_t packed_component_bytes(int fmt_tiled, int E, int H, int I, int which) {
  const size_t MB = which == 0 ? I / 64 : H / 128;
  const size_t KS = (which == 0 ? H : I) / 64;
  const size_t chunk = fmt_tiled == MOE_W_BF16_TILED ? 128 * 64 * 2 : 128 * 32 + 128 * 2;
  return static_cast<size_t>(E) * MB * KS * chunk;
}

cudaError_t launch_pack(int fmt_in, const void* w, const uint16_t* s, int E, int H, int I, int which, void* out,
                        cudaStream_t st) {
  const int MB = which == 0 ? I / 64 : H / 128;
  const int KS = (which == 0 ? H : I) / 64;
  const size_t chunks = static_cast<size_t>(E) * MB * KS;
  const size_t pieces = chunks * (fmt_in == MOE_W_BF16 ? 1024 : 256);
  const int threads = 256;
  size_t blocks = (pieces + threads - 1) / threads;
  const size_t cap = static_cast<size_t>(sm_count() > 0 ? sm_count() : 148) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks == 0) blocks = 1;
  if (fmt_in == MOE_W_BF16)
    return launch_pdl(pack_bf16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, st,
                      static_cast<const uint16_t*>(w), E, H, I, which, static_cast<uint16_t*>(out));
  return launch_pdl(pack_int4_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, st,
                    static_cast<const uint8_t*>(w), s, E, H, I, which, static_cast<uint8_t*>(out));
}

}  // namespace moe
