// Attention of one decode step on the compressed cache, and the value layout
// it reads.
//
// "Google acelera LLM 8 veces" ties the speed-up to attention logits computed
// directly on the compressed keys; the values of the same cache are
// TurboQuantMSE codes ("turboquant-pytorch 소개", "1단계"; its 58 MB figure
// covers K and V at 3 bits), reconstructed as v_hat = ||v|| Pi_v^T c[idx].
// One decode step computes, per group g and query head h,
//     out[g][h] = sum_t softmax_t(scale * logit[g][h][t]) v_hat[g][t],
// the logits being tq_score's estimates.
//
// Value layout (tq_encode_values).  The MSE encode writes token-major blocks
// (a token's 128 coordinates per 16-byte chunk).  The value contraction
// sum_t w_t c[idx_{t,j}] runs over tokens, so the values are stored
// coordinate-major instead: per 128-token block, for each code plane p and
// coordinate j, 16 bytes hold bit p of coordinate j of the block's 128 tokens
// (token t = bit t % 32 of little-endian word t / 32); the norms follow as in
// the MSE layout.  The kernel below converts blocks in place with a 32 x 32
// bit transpose per warp (five exchange steps of __shfl_xor_sync).
//
// Attention (tq_attend) runs three kernels:
//  1. the tensor-core score (query preparation + score_tc_kernel) writes the
//     logits to the caller's workspace;
//  2. attend_values_kernel, one CTA per (group, split of its tokens): the
//     weight warpgroup reads the split's logits once for each head's maximum
//     m, then per 128-token tile forms w = exp(scale (l - m)) ||v|| as four
//     e4m3 slices (the B operand, rows = slice x head, K = tokens); the value
//     warpgroup expands the tile's value bit planes (coordinate-major: one
//     16-byte chunk per coordinate and plane) to e4m3 in TMEM (the A operand,
//     rows = coordinates); tcgen05 MMAs accumulate, per parity plane T of the
//     codebook, sum_t x_T[j][t] w[t] over every tile of the split in TMEM;
//     at the end the same warpgroup combines planes and slices into
//     o[h][j] = sum_t w_t c[idx_{t,j}] in the rotated frame;
//  3. attend_combine_kernel merges the splits of a group (max-rescaled sums)
//     and rotates back, out = Pi_v^T o / sum_t exp(scale (l - m)).
// The packed keys and values are each read once; the logits make one round
// trip through memory (the workspace), which at decode-step sizes stays in L2.
#include <cuda_fp8.h>

#include "ptx_sm100.cuh"
#include "tq_internal.cuh"

namespace tq {
namespace {

using namespace ptx;

// 32 x 32 bit transpose across a warp: lane r holds row r (bit c = column c);
// on return lane c holds column c (bit r = element (r, c)).  Each step swaps
// the off-diagonal s x s sub-blocks of every 2s x 2s block.
__device__ __forceinline__ uint32_t transpose32(uint32_t x, int lane) {
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) {
    const uint32_t m = s == 16 ? 0x0000FFFFu : s == 8 ? 0x00FF00FFu : s == 4 ? 0x0F0F0F0Fu : s == 2 ? 0x33333333u : 0x55555555u;
    const uint32_t y = __shfl_xor_sync(0xffffffffu, x, s);
    x = (lane & s) ? ((x & ~m) | ((y >> s) & m)) : ((x & m) | ((y & m) << s));
  }
  return x;
}

// One CTA of 128 threads per 128-token block: every plane chunk of the block
// is read (thread t = token t), transposed into shared memory, and written
// back coordinate-major (thread j = coordinate j of a chunk).  In place: the
// whole block is read before any of it is written.
__global__ void __launch_bounds__(128) values_to_coordinate_major_kernel(uint8_t* __restrict__ packed,
                                                                         int64_t block_bytes, int planes, int C) {
  extern __shared__ uint32_t vt_sm[];  // [planes][C][128 coordinates][4 token words]
  uint8_t* blk = packed + (int64_t)blockIdx.x * block_bytes;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  for (int pc = 0; pc < planes * C; ++pc) {
    const uint4 v = *reinterpret_cast<const uint4*>(blk + ((int64_t)pc * kTokensPerBlock + t) * 16);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      // rows: tokens 32 warp + r; columns: coordinates 32 b + c of the chunk
      const uint32_t col = transpose32(w[b], lane);
      vt_sm[((pc * kTokensPerBlock) + 32 * b + lane) * 4 + warp] = col;
    }
  }
  __syncthreads();
  for (int pc = 0; pc < planes * C; ++pc) {
    const uint32_t* src = vt_sm + ((pc * kTokensPerBlock) + t) * 4;
    // plane p, coordinate 128 c + t: offset ((p d) + 128 c + t) 16 = ((p C + c) 128 + t) 16
    *reinterpret_cast<uint4*>(blk + ((int64_t)pc * kTokensPerBlock + t) * 16) = make_uint4(src[0], src[1], src[2], src[3]);
  }
}

}  // namespace

cudaError_t launch_values_layout(const tq_plan* p, uint8_t* packed, int64_t n_blocks, cudaStream_t s) {
  if (n_blocks == 0) return cudaSuccess;
  const int planes = p->lay.planes, C = p->lay.C;
  const size_t smem = (size_t)planes * C * kTokensPerBlock * 16;
  cudaError_t e = cudaFuncSetAttribute(values_to_coordinate_major_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  for (int64_t b0 = 0; b0 < n_blocks; b0 += 0x7fffffff) {
    const int64_t nb = n_blocks - b0 < 0x7fffffff ? n_blocks - b0 : 0x7fffffff;
    values_to_coordinate_major_kernel<<<(unsigned)nb, 128, smem, s>>>(packed + b0 * p->lay.block_bytes,
                                                                       p->lay.block_bytes, planes, C);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace tq
