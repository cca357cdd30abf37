// Helpers of the tensor-core kernels that contract 0/1 bit planes with real
// vectors (internal).  A packed plane word W holds 32 coordinates (or tokens)
// as bits; expand_word turns it into eight 32-bit TMEM words, four e4m3 values
// each, every value an exact power of two: byte bit 3 + (o % 4) of output word
// o, i.e. 2^-6, 2^-5, 2^-3 or 2.  The other operand of an MMA carries the
// reciprocal power (c_comp) of the position it meets.  K index kk of an
// expanded plane is TMEM column kk / 4, byte kk % 4; column 8 w + o holds bit
// 8 (kk % 4) + c_src[o] of word w.
#pragma once

#include <cuda_fp8.h>

#include "ptx_sm100.cuh"

namespace tq {
namespace {

using namespace ptx;

constexpr int kSlices = 4;          // e4m3 slices of the real operand
constexpr int kPlaneCols = 32;      // TMEM columns of one expanded plane (128 e4m3)

// reciprocal of the e4m3 value of bit 3 + i of a byte (2^-6, 2^-5, 2^-3, 2)
__constant__ float c_comp[4] = {64.f, 32.f, 8.f, 0.5f};
// source bit (within each byte of the plane word) of expanded word o
__constant__ int c_src[8] = {3, 4, 5, 6, 0, 1, 2, 7};

// Eight TMEM words (32 e4m3 values) from one 32-coordinate plane word.
__device__ __forceinline__ void expand_word(uint32_t W, uint32_t* o) {
  const uint32_t b = W << 3, c = W >> 1;
  o[0] = W & 0x08080808u;
  o[1] = W & 0x10101010u;
  o[2] = W & 0x20202020u;
  o[3] = W & 0x40404040u;
  o[4] = b & 0x08080808u;
  o[5] = b & 0x10101010u;
  o[6] = b & 0x20202020u;
  o[7] = c & 0x40404040u;
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f8f6f4 (e4m3 x e4m3, fp32 accumulate)
__device__ __forceinline__ void mma_f8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Warp-converged form (see mma_f16_ts_w): every lane passes the same operands,
// one elected lane issues.
__device__ __forceinline__ void mma_f8_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 r;\n\telect.sync r|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor, kind::f8f6f4: e4m3 A and B, fp32 accumulate, K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(uint32_t M, uint32_t N) {
  return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Position in a ring of n entries: index and the parity of the pass over it.
struct Ring {
  uint32_t idx = 0, phase = 0;
  __device__ __forceinline__ void advance(uint32_t by, uint32_t n) {
    idx += by;
    while (idx >= n) {
      idx -= n;
      phase ^= 1u;
    }
  }
};

// (group, block) of a tile, advanced without divisions.
struct TilePos {
  uint32_t g = 0, blk = 0;
  __device__ __forceinline__ void init(int64_t tile, int64_t nb) {
    g = (uint32_t)(tile / nb);
    blk = (uint32_t)(tile - (int64_t)g * nb);
  }
  __device__ __forceinline__ void advance(uint32_t by, uint32_t nb) {
    blk += by;
    while (blk >= nb) {
      blk -= nb;
      ++g;
    }
  }
};

__device__ __forceinline__ float slice_weight(int sl) {
  return sl == 0 ? 1.f : sl == 1 ? 0.0625f : sl == 2 ? 0.00390625f : 0.000244140625f;
}

// Byte offset of element (row n, K index k) of an image of rows x 128 e4m3
// (one 128-byte swizzle atom column), as the tensor cores read a K-major operand.
__device__ __forceinline__ uint32_t img_offset(int n, int k) {
  return (uint32_t)(n >> 3) * 1024u + (uint32_t)(n & 7) * 128u + (uint32_t)(((k >> 4) ^ (n & 7)) << 4) +
         (uint32_t)(k & 15);
}

__device__ __forceinline__ float e4m3_value(__nv_fp8_storage_t x) {
  return __half2float(__half(__nv_cvt_fp8_to_halfraw(x, __NV_E4M3)));
}

// One term's accumulators (N <= 32 columns), every TMEM load issued before a
// single wait: acc[h] = sum over slices of D[slice * HP + h] / 16^slice.
template <int HP>
__device__ __forceinline__ void load_term_all(uint32_t taddr, float (&acc)[HP]) {
  constexpr int N = kSlices * HP;
  static_assert(N <= 32, "at most 32 columns in flight");
  uint32_t v[N / 16][16];
#pragma unroll
  for (int c = 0; c < N / 16; ++c) tmem_ld16(taddr + 16 * c, v[c]);
  tmem_ld_wait();
#pragma unroll
  for (int h = 0; h < HP; ++h) acc[h] = 0.f;
#pragma unroll
  for (int c = 0; c < N / 16; ++c)
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int col = 16 * c + e, sl = col / HP, h = col % HP;
      acc[h] = fmaf(__uint_as_float(v[c][e]), slice_weight(sl), acc[h]);
    }
}

// Tokens' accumulators of one term: sum over slices of D[slice * HP + h] / 16^slice.
template <int HP>
__device__ __forceinline__ void load_term(uint32_t taddr, float (&acc)[HP]) {
  constexpr int N = kSlices * HP;
#pragma unroll
  for (int h = 0; h < HP; ++h) acc[h] = 0.f;
#pragma unroll
  for (int c0 = 0; c0 < N; c0 += 16) {
    uint32_t v[16];
    tmem_ld16(taddr + c0, v);
    tmem_ld_wait();
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int col = c0 + e, sl = col / HP, h = col % HP;
      const float w = sl == 0 ? 1.f : sl == 1 ? 0.0625f : sl == 2 ? 0.00390625f : 0.000244140625f;
      acc[h] = fmaf(__uint_as_float(v[e]), w, acc[h]);
    }
  }
}

}  // namespace
}  // namespace tq
