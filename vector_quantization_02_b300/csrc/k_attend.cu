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
//  3. attend_combine_kernel (one CTA per group, every head) merges the splits
//     (max-rescaled sums) and rotates back, out = Pi_v^T o / sum_t exp(scale (l - m)).
// The packed keys and values are each read once; the logits make one round
// trip through memory (the workspace), which at decode-step sizes stays in L2.
#include <cuda_fp8.h>

#include "ptx_sm100.cuh"
#include "tc_planes.cuh"
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

// ------------------------------------------------------------------ attention
constexpr int kAttStages = 16;          // value-block ring
constexpr int kAttThreads = 608;        // 19 warps: producer, 2 issuers, 2 value WGs, 2 weight WGs
constexpr int kAttProducer = 0, kAttIssuer0 = 1, kAttValWarp0 = 3, kAttWgtWarp0 = 11;
enum {
  AB_FULL = 0,
  AB_EMPTY = AB_FULL + kAttStages,   // both value warpgroups (256) + the tile's weight warpgroup (128)
  AB_PFULL = AB_EMPTY + kAttStages,  // [2] value planes of TMEM entry e (tile i: e = i % 2)
  AB_WFULL = AB_PFULL + 2,           // [4] weight image slot i % 4 in shared memory
  AB_MDONE = AB_WFULL + 4,           // [4] MMAs of tile i complete (slot i % 4)
  AB_DONE = AB_MDONE + 4,            // [2] all MMAs of issuer e complete
  AB_COUNT = AB_DONE + 2
};

struct AttArgs {
  Layout lay;              // value layout (coordinate-major, d = 128)
  int64_t N, nb;
  int H, Hp, splits;
  const float* logits;     // [G][H][N]
  const uint8_t* vpacked;
  float scale;
  ParityExpansion px;      // value codebook
  float* part_o;           // [G][splits][Hp][128]: sum_t w_t c[idx_t] (rotated frame)
  float* part_ml;          // [G][splits][Hp][2]: max of scale * logit, sum_t exp(scale logit - max)
  int* err;
};

// TMEM: accumulators of entry e (NT planes x N columns) from column e NT N;
// value planes of entry e (NT x 32 columns) after both entries' accumulators.
template <int HP, int KV>
__global__ void __launch_bounds__(kAttThreads, 1) attend_values_kernel(const AttArgs a) {
  constexpr int N = kSlices * HP;
  constexpr int NT = KV == 3 ? 4 : KV;             // parity planes of an odd-symmetric codebook
  constexpr uint32_t kAcc = NT * N, kSlot0 = 2 * kAcc, kSlotCols = NT * kPlaneCols;
  constexpr uint32_t kImg = ((uint32_t)N * 128u + 1023u) & ~1023u;  // weight image: N rows x 128 tokens
  static_assert(kSlot0 + 2 * kSlotCols <= 512, "TMEM");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(smem);
  const uint32_t blk_bytes = (uint32_t)a.lay.block_bytes;
  const uint32_t off_ring = 4 * kImg;
  const uint32_t off_bar = off_ring + kAttStages * blk_bytes;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float s_red[8][HP][3];   // cross-warp reductions of the two weight warpgroups
  __shared__ float s_m[HP], s_sigma;  // per-head max of scale * logit; weight normalisation
  __shared__ float s_P[HP];           // sum_t w_t ||v_t|| per head
  auto bar = [&](int i) { return sb + off_bar + 8u * (uint32_t)i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int64_t g = blockIdx.x / a.splits, sp = blockIdx.x % a.splits;
  const int64_t t0 = sp * a.nb / a.splits, t1 = (sp + 1) * a.nb / a.splits;  // tiles of this split
  const uint32_t n_t = (uint32_t)(t1 - t0);
  const uint8_t* vblk0 = a.vpacked + (g * a.nb + t0) * a.lay.block_bytes;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kAttStages; ++s) {
      mbar_init(bar(AB_FULL + s), 1);
      mbar_init(bar(AB_EMPTY + s), 384);
    }
    for (int e = 0; e < 2; ++e) {
      mbar_init(bar(AB_PFULL + e), 256);
      mbar_init(bar(AB_DONE + e), 1);
    }
    for (int k = 0; k < 4; ++k) {
      mbar_init(bar(AB_WFULL + k), 128);
      mbar_init(bar(AB_MDONE + k), 1);
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort = &abort_flag;

  if (warp == kAttProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t issued = 0;
      bool ok = true;
      Ring slot;
      for (uint32_t i = 0; i < n_t; ++i, slot.advance(1, kAttStages)) {
        if (!mbar_wait_suspend(bar(AB_EMPTY + slot.idx), slot.phase ^ 1u, abort)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(AB_FULL + slot.idx), blk_bytes);
        bulk_load(sb + off_ring + slot.idx * blk_bytes, vblk0 + (int64_t)i * blk_bytes, blk_bytes,
                  bar(AB_FULL + slot.idx));
        issued = i + 1;
      }
      if (!ok) {
        *abort = 1;
        atomicExch(a.err, 1);
      }
      int dummy = 0;
      for (uint32_t i = issued > kAttStages ? issued - kAttStages : 0; i < issued; ++i)
        mbar_wait(bar(AB_FULL + i % kAttStages), (i / kAttStages) & 1u, &dummy);
    }
  } else if (warp < kAttValWarp0) {
    // ------------------------------------------------------------ MMA issuers
    // issuer e takes the tiles i with i % 2 == e: value planes of TMEM entry e
    // times weight image i % 4, accumulated per parity plane into accumulator
    // set e; the commit for tile i lands on MDONE[i % 4].  The whole warp runs
    // the loop (its operands stay warp-uniform); one elected lane issues each
    // MMA and commit.
    {
      const uint32_t e = (uint32_t)(warp - kAttIssuer0);
      constexpr uint32_t idesc = idesc_e4m3(128, N);
      const uint64_t bdesc0 = sdesc_k_sw128(sb + e * kImg), bdesc1 = sdesc_k_sw128(sb + (e + 2) * kImg);
      const uint32_t d0 = tmem + e * kAcc, at0 = tmem + kSlot0 + e * kSlotCols;
      bool ok = true;
      uint32_t use = 0;
      for (uint32_t i = e; i < n_t; i += 2, ++use) {
        const uint32_t k = i & 3u;  // e or e + 2
        if (!__all_sync(0xffffffffu, mbar_wait(bar(AB_PFULL + e), use & 1u, abort) &&
                                         mbar_wait(bar(AB_WFULL + k), (i >> 2) & 1u, abort))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int T = 0; T < NT; ++T)
#pragma unroll
          for (uint32_t kb = 0; kb < 4; ++kb)
            mma_f8_ts_w(d0 + (uint32_t)(T * N), at0 + (uint32_t)(T * kPlaneCols) + 8u * kb,
                      (k == e ? bdesc0 : bdesc1) + 2u * kb, idesc,
                      (use > 0 || kb > 0) ? 1u : 0u);
        mma_commit_w(bar(AB_MDONE + k));
      }
      if (!ok && lane == 0) {
        *abort = 1;
        atomicExch(a.err, 1);
      }
      mma_commit_w(bar(AB_DONE + e));
      int dummy = 0;
      mbar_wait(bar(AB_DONE + e), 0, &dummy);
    }
  } else if (warp < kAttWgtWarp0) {
    // ------------------------------------------------------------ value planes
    // Both value warpgroups expand every tile, warpgroup v the parity planes
    // T with T % 2 == v, into TMEM entry i % 2 (one warp moves only ~32 bytes
    // per cycle to TMEM, so a tile's planes are spread over eight warps).
    // Thread (warp w, lane l) owns coordinate j = 32 (w % 4) + l: its 16-byte
    // chunk of each code plane holds the block's 128 tokens.
    const uint32_t v = (uint32_t)(warp - kAttValWarp0) >> 2;
    const int quad = warp & 3;
    const int j = quad * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16) + kSlot0;
    Ring slot;
    for (uint32_t i = 0; i < n_t; ++i, slot.advance(1, kAttStages)) {
      const uint32_t e = i & 1u;  // TMEM entry of tile i
      if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(AB_FULL + slot.idx), slot.phase, abort))) {
        *abort = 1;
        atomicExch(a.err, 1);
        break;
      }
      const uint8_t* blkp = smem + off_ring + slot.idx * blk_bytes;
      uint4 w[NT];
#pragma unroll
      for (int q = 0; q < KV; ++q) w[q] = *reinterpret_cast<const uint4*>(blkp + ((q * 128) + j) * 16);
      if constexpr (KV == 3)
        w[3] = make_uint4(w[0].x ^ w[1].x ^ w[2].x, w[0].y ^ w[1].y ^ w[2].y, w[0].z ^ w[1].z ^ w[2].z,
                          w[0].w ^ w[1].w ^ w[2].w);
      mbar_arrive(bar(AB_EMPTY + slot.idx));
      // TMEM entry e was last used by tile i - 2 (MDONE slot (i + 2) % 4; a
      // fresh barrier's preceding phase for i < 2)
      if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(AB_MDONE + ((i + 2) & 3u)), (((i + 2) >> 2) & 1u) ^ 1u,
                                                     abort))) {
        *abort = 1;
        atomicExch(a.err, 1);
        break;
      }
      tc_fence_after();
      const uint32_t taddr = lane_base + e * kSlotCols;
#pragma unroll
      for (int T = 0; T < NT; ++T) {
        if ((uint32_t)(T & 1) != v) continue;  // this warpgroup's planes
        uint32_t o[32];
        expand_word(w[T].x, o);
        expand_word(w[T].y, o + 8);
        expand_word(w[T].z, o + 16);
        expand_word(w[T].w, o + 24);
        tmem_st32(taddr + (uint32_t)(T * kPlaneCols), o);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(AB_PFULL + e));
    }
  } else {
    // ------------------------------------------------------------ weights, then the result
    // Two weight warpgroups: warpgroup x takes the tiles i with i % 2 == x
    // (TMEM entry and weight image x).  Thread wt of a warpgroup owns token wt
    // of each of its tiles, and at the end (warpgroup 0) coordinate wt.
    const int wt256 = threadIdx.x - kAttWgtWarp0 * 32;  // 0..255 over both warpgroups
    const int x = wt256 >> 7, wt = wt256 & 127, wq8 = wt256 >> 5;
    const float sl2 = a.scale * 1.4426950408889634f;    // scale log2(e): weights are exp2 of it
    // pass 1: the split's max of scale * logit (in log2 units) per head and max value norm
    float mh[HP], nmax = 0.f;
#pragma unroll
    for (int h = 0; h < HP; ++h) mh[h] = -INFINITY;
    const int64_t tok0 = t0 * kTokensPerBlock, tok1 = t1 * kTokensPerBlock < a.N ? t1 * kTokensPerBlock : a.N;
    // Four consecutive tokens per thread per pass, read as one float4 of each
    // head's logits and two float4 of norm pairs, every load issued before the
    // first use (the logits come from L2; dependent loads would serialise one
    // round trip per token).  Rows whose length is not a multiple of four, and
    // the ragged end, take single loads.
    const bool vec = (a.N & 3) == 0;
    for (int64_t tok = tok0 + 4 * (int64_t)wt256; tok < tok1; tok += 4 * 256) {
      float l[HP][4], nv[4];
      if (vec && tok + 4 <= tok1) {
#pragma unroll
        for (int h = 0; h < HP; ++h) {
          const float4 f = h < a.H ? __ldg(reinterpret_cast<const float4*>(a.logits + (g * a.H + h) * a.N + tok))
                                   : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
          l[h][0] = f.x;
          l[h][1] = f.y;
          l[h][2] = f.z;
          l[h][3] = f.w;
        }
        // tokens tok .. tok + 3 lie in one 128-token block (tok is a multiple of 4)
        const int64_t r = tok - tok0;
        const float4* np = reinterpret_cast<const float4*>(vblk0 + (r >> 7) * a.lay.block_bytes + a.lay.norms_off +
                                                           (r & 127) * 8);
        const float4 n01 = __ldg(np), n23 = __ldg(np + 1);
        nv[0] = n01.x;
        nv[1] = n01.z;
        nv[2] = n23.x;
        nv[3] = n23.z;
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t t = tok + u;
          const bool in = t < tok1;
#pragma unroll
          for (int h = 0; h < HP; ++h)
            l[h][u] = (in && h < a.H) ? __ldg(a.logits + (g * a.H + h) * a.N + t) : -INFINITY;
          const int64_t r = t - tok0;
          nv[u] = in ? __ldg(reinterpret_cast<const float*>(vblk0 + (r >> 7) * a.lay.block_bytes +
                                                            a.lay.norms_off + (r & 127) * 8))
                     : 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
#pragma unroll
        for (int h = 0; h < HP; ++h)
          if (h < a.H && l[h][u] > -INFINITY) mh[h] = fmaxf(mh[h], sl2 * l[h][u]);
        nmax = fmaxf(nmax, nv[u]);
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
#pragma unroll
      for (int h = 0; h < HP; ++h) mh[h] = fmaxf(mh[h], __shfl_xor_sync(0xffffffffu, mh[h], o));
      nmax = fmaxf(nmax, __shfl_xor_sync(0xffffffffu, nmax, o));
    }
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < HP; ++h) s_red[wq8][h][0] = mh[h];
      s_red[wq8][0][1] = nmax;
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (wt256 < HP) {
      float m = -INFINITY;
      for (int q = 0; q < 8; ++q) m = fmaxf(m, s_red[q][wt256][0]);
      s_m[wt256] = m;
    }
    if (wt256 == 0) {
      // weights w ||v|| <= nmax scaled below 4: with the compensation (at most
      // 64) every e4m3 slice stays below 256
      float nm = 0.f;
      for (int q = 0; q < 8; ++q) nm = fmaxf(nm, s_red[q][0][1]);
      int ex = 0;
      if (nm > 0.f) frexpf(nm, &ex);
      s_sigma = ldexpf(1.f, 2 - ex);
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
#pragma unroll
    for (int h = 0; h < HP; ++h) mh[h] = s_m[h];
    const float sigma = s_sigma;
    // this thread's token t = wt of every tile: its K index in the expanded
    // value planes and the compensation of that position
    const int tw = wt >> 5, tb = wt & 31, tbyte = tb >> 3, tbit = tb & 7;
    const int o_of_bit = tbit == 7 ? 7 : tbit >= 3 ? tbit - 3 : tbit + 4;  // inverse of c_src
    const int kk = 4 * (8 * tw + o_of_bit) + tbyte;
    const float comp = c_comp[o_of_bit & 3];
    // image slot i % 4 (x or x + 2): the image of tile i + 2 is written while
    // the MMAs of tile i still read theirs
    float L[HP], P[HP];
#pragma unroll
    for (int h = 0; h < HP; ++h) L[h] = P[h] = 0.f;
    // the logits of this thread's token in its warpgroup's next tile, loaded
    // one tile ahead
    auto load_logits = [&](uint32_t i, float (&l)[HP]) {
      const int64_t tok = (t0 + i) * kTokensPerBlock + wt;
#pragma unroll
      for (int h = 0; h < HP; ++h)
        l[h] = (i < n_t && h < a.H && tok < a.N) ? __ldg(a.logits + (g * a.H + h) * a.N + tok) : -INFINITY;
    };
    float lc[HP];
    load_logits((uint32_t)x, lc);
    Ring slot;
    slot.advance((uint32_t)x, kAttStages);
    bool ok = true;
    uint32_t use = 0;
    for (uint32_t i = (uint32_t)x; i < n_t; i += 2, ++use, slot.advance(2, kAttStages)) {
      float ln[HP];
      load_logits(i + 2, ln);
      if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(AB_FULL + slot.idx), slot.phase, abort))) {
        ok = false;
        break;
      }
      const float nv = *reinterpret_cast<const float*>(smem + off_ring + slot.idx * blk_bytes + a.lay.norms_off + wt * 8);
      mbar_arrive(bar(AB_EMPTY + slot.idx));
      const float bscale = nv * sigma * comp;
      float b[HP];
#pragma unroll
      for (int h = 0; h < HP; ++h) {
        const float w = exp2f(fmaf(sl2, lc[h], -mh[h]));  // 0 for a masked token (logit -inf)
        L[h] += w;
        P[h] = fmaf(w, nv, P[h]);
        b[h] = w * bscale;
      }
      // image slot i % 4 was last read by the MMAs of tile i - 4
      if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(AB_MDONE + (i & 3u)), ((i >> 2) & 1u) ^ 1u, abort))) {
        ok = false;
        break;
      }
      uint8_t* img = smem + (i & 3u) * kImg;
      // four e4m3 slices of each weight, two heads per conversion
#pragma unroll
      for (int h = 0; h < HP; h += 2) {
        float2 val = make_float2(b[h], b[h + 1]);
        float sc = 1.f;
#pragma unroll
        for (int sl = 0; sl < kSlices; ++sl) {
          const __nv_fp8x2_storage_t x2 =
              __nv_cvt_float2_to_fp8x2(make_float2(val.x * sc, val.y * sc), __NV_SATFINITE, __NV_E4M3);
          img[img_offset(sl * HP + h, kk)] = (uint8_t)(x2 & 0xffu);
          img[img_offset(sl * HP + h + 1, kk)] = (uint8_t)(x2 >> 8);
          const float2 back = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(x2, __NV_E4M3)));
          const float inv = 1.f / sc;
          val.x = fmaf(-back.x, inv, val.x);
          val.y = fmaf(-back.y, inv, val.y);
          sc *= 16.f;
        }
      }
      // the MMAs read the image through the async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(bar(AB_WFULL + (i & 3u)));
#pragma unroll
      for (int h = 0; h < HP; ++h) lc[h] = ln[h];
    }
    if (!ok) {
      *abort = 1;
      atomicExch(a.err, 1);
    }
    // sums over the split's tokens: L (softmax denominator) and P = sum w ||v||
#pragma unroll
    for (int o = 16; o; o >>= 1)
#pragma unroll
      for (int h = 0; h < HP; ++h) {
        L[h] += __shfl_xor_sync(0xffffffffu, L[h], o);
        P[h] += __shfl_xor_sync(0xffffffffu, P[h], o);
      }
    // both warpgroups are past their loops: every phase of both MMA barriers
    // before the last has been waited for
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (lane == 0)
#pragma unroll
      for (int h = 0; h < HP; ++h) {
        s_red[wq8][h][1] = L[h];
        s_red[wq8][h][2] = P[h];
      }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    float* ml = a.part_ml + (blockIdx.x * (int64_t)a.Hp) * 2;
    if (wt256 < HP) {
      float Lh = 0.f, Ph = 0.f;
      for (int q = 0; q < 8; ++q) {
        Lh += s_red[q][wt256][1];
        Ph += s_red[q][wt256][2];
      }
      s_P[wt256] = Ph;
      // the combine works in the natural scale: max of scale * logit
      ml[2 * wt256] = s_m[wt256] * 0.6931471805599453f;
      ml[2 * wt256 + 1] = Lh;
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");
    if (x != 0) goto done;  // the result is read out by warpgroup 0
    // the result: thread = coordinate j (TMEM lane 32 (warp % 4) + lane)
    const int quad = warp & 3;
    const int j = quad * 32 + lane;
    float o_h[HP];
#pragma unroll
    for (int h = 0; h < HP; ++h) o_h[h] = a.px.c0 * s_P[h];
    int dummy = 0;
    for (uint32_t e = 0; e < 2 && e < n_t; ++e) {
      const uint32_t last = e + 2 * ((n_t - 1 - e) / 2);  // the last tile of entry e
      if (!mbar_wait(bar(AB_MDONE + (last & 3u)), (last >> 2) & 1u, &dummy)) atomicExch(a.err, 1);
    }
    tc_fence_after();
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    for (uint32_t e = 0; e < 2 && e < n_t; ++e) {
#pragma unroll
      for (int T = 0; T < NT; ++T) {
        float acc[HP];
        if constexpr (N <= 32) load_term_all<HP>(lane_base + e * kAcc + (uint32_t)(T * N), acc);
        else load_term<HP>(lane_base + e * kAcc + (uint32_t)(T * N), acc);
#pragma unroll
        for (int h = 0; h < HP; ++h) o_h[h] = fmaf(a.px.coef[T], acc[h] / sigma, o_h[h]);
      }
    }
    float* po = a.part_o + blockIdx.x * (int64_t)a.Hp * 128;
#pragma unroll
    for (int h = 0; h < HP; ++h)
      if (h < a.H) po[h * 128 + j] = o_h[h];
  }

done:
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// One CTA of 512 threads per group: merge the splits' partial sums of every
// head (max-rescaled), divide by the softmax denominator and rotate back,
// out = Pi_v^T o, reading Pi_v once for all heads of the group.  Thread
// (quarter r, coordinate j) sums rows i in [32 r, 32 r + 32) of Pi_v with its
// 32 loads in flight together; the four quarters are added in shared memory.
constexpr int kCombThreads = 512;
template <int HP>
__global__ void __launch_bounds__(kCombThreads) attend_combine_kernel(const float* __restrict__ part_o,
                                                                      const float* __restrict__ part_ml, int splits,
                                                                      int H, int Hp, const float* __restrict__ Pi_v,
                                                                      float* __restrict__ out) {
  __shared__ float s_o[HP][128];
  __shared__ float s_q[4][HP][128];
  const int64_t g = blockIdx.x;
  for (int p = threadIdx.x; p < HP * 128; p += kCombThreads) {
    const int h = p >> 7, j = p & 127;
    float o = 0.f;
    if (h < H) {
      float M = -INFINITY;
      for (int sp = 0; sp < splits; ++sp) M = fmaxf(M, part_ml[((g * splits + sp) * Hp + h) * 2]);
      float num = 0.f, den = 0.f;
      for (int sp = 0; sp < splits; ++sp) {
        const int64_t r = (g * splits + sp) * Hp + h;
        const float f = __expf(part_ml[r * 2] - M);
        num = fmaf(f, part_o[r * 128 + j], num);
        den = fmaf(f, part_ml[r * 2 + 1], den);
      }
      o = num / den;
    }
    s_o[h][j] = o;
  }
  // out_j = sum_i Pi_v[i][j] o_i  (Pi_v row-major, y = Pi_v u)
  const int r = threadIdx.x >> 7, j = threadIdx.x & 127;
  float pv[32];
#pragma unroll
  for (int ii = 0; ii < 32; ++ii) pv[ii] = __ldg(Pi_v + (32 * r + ii) * 128 + j);
  __syncthreads();
  float acc[HP];
#pragma unroll
  for (int h = 0; h < HP; ++h) acc[h] = 0.f;
#pragma unroll
  for (int ii = 0; ii < 32; ++ii)
#pragma unroll
    for (int h = 0; h < HP; ++h) acc[h] = fmaf(pv[ii], s_o[h][32 * r + ii], acc[h]);
#pragma unroll
  for (int h = 0; h < HP; ++h) s_q[r][h][j] = acc[h];
  __syncthreads();
  for (int p = threadIdx.x; p < H * 128; p += kCombThreads) {
    const int h = p >> 7, jj = p & 127;
    out[(g * H + h) * 128 + jj] = (s_q[0][h][jj] + s_q[1][h][jj]) + (s_q[2][h][jj] + s_q[3][h][jj]);
  }
}

}  // namespace

namespace {

bool odd_symmetric_masks(const ParityExpansion& px, int k) {
  static const uint32_t want[3][4] = {{1u}, {1u, 2u}, {1u, 2u, 4u, 7u}};
  const int n = k == 3 ? 4 : k;
  if (k < 1 || k > 3 || px.n != n) return false;
  for (int i = 0; i < n; ++i)
    if (px.mask[i] != want[k - 1][i]) return false;
  return true;
}

int att_hp(int H, int kv) { return H <= 4 ? 4 : H <= 8 ? 8 : (H <= 16 && kv <= 2) ? 16 : 0; }

int att_splits(int64_t G, int64_t nb) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t s = G >= sms ? 1 : sms / G;
  return (int)(s < 1 ? 1 : s > nb ? nb : s);
}

size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

template <int HP, int KV>
cudaError_t launch_att(const AttArgs& a, int64_t grid, cudaStream_t s) {
  constexpr int N = kSlices * HP;
  constexpr uint32_t kImg = ((uint32_t)N * 128u + 1023u) & ~1023u;
  const size_t smem = 4 * kImg + kAttStages * (size_t)a.lay.block_bytes + AB_COUNT * 8 + 1024;
  auto kern = attend_values_kernel<HP, KV>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)grid, kAttThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool attend_supported(const tq_plan* kp, const tq_plan* vp, int H) {
  if (!kp || !vp || kp->d != 128 || vp->d != 128 || !kp->lay.prod || vp->lay.prod || vp->lay.frac) return false;
  if (!score_tc_supported(kp, H) && !score_wide_supported(kp, H)) return false;  // the logits
  const int kv = vp->lay.k;
  return kv <= 3 && odd_symmetric_masks(vp->px, kv) && att_hp(H, kv) != 0;
}

size_t attend_workspace_bytes(const tq_plan* kp, const tq_plan* vp, int64_t G, int H, int64_t N) {
  if (!attend_supported(kp, vp, H)) return 0;
  const int64_t nb = (N + kTokensPerBlock - 1) / kTokensPerBlock;
  const int S = att_splits(G, nb), Hp = att_hp(H, vp->lay.k);
  return al256(score_workspace_bytes(kp, G, H, N, 0)) + al256((size_t)G * H * N * 4) +
         al256((size_t)G * S * Hp * 128 * 4) + al256((size_t)G * S * Hp * 2 * 4);
}

cudaError_t launch_attend(const tq_plan* kp, const tq_plan* vp, const float* q, int64_t G, int H,
                          const uint8_t* kpacked, const uint8_t* vpacked, int64_t N, float scale, float* out,
                          void* ws, cudaStream_t s) {
  if (!attend_supported(kp, vp, H)) return cudaErrorNotSupported;
  if (G * N == 0) return cudaSuccess;
  const int64_t nb = (N + kTokensPerBlock - 1) / kTokensPerBlock;
  const int S = att_splits(G, nb), kv = vp->lay.k, Hp = att_hp(H, kv);
  uint8_t* w = static_cast<uint8_t*>(ws);
  const size_t ws_score = al256(score_workspace_bytes(kp, G, H, N, 0));
  float* logits = reinterpret_cast<float*>(w + ws_score);
  float* part_o = reinterpret_cast<float*>(w + ws_score + al256((size_t)G * H * N * 4));
  float* part_ml = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(part_o) + al256((size_t)G * S * Hp * 128 * 4));
  cudaError_t e = score_run(kp, q, G, H, kpacked, N, logits, 0, nullptr, nullptr, w, s);
  if (e != cudaSuccess) return e;
  AttArgs a;
  a.lay = vp->lay;
  a.N = N;
  a.nb = nb;
  a.H = H;
  a.Hp = Hp;
  a.splits = S;
  a.logits = logits;
  a.vpacked = vpacked;
  a.scale = scale;
  a.px = vp->px;
  a.part_o = part_o;
  a.part_ml = part_ml;
  a.err = vp->err;
  const int64_t grid = G * S;
  switch (Hp * 4 + kv) {
    case 17: e = launch_att<4, 1>(a, grid, s); break;
    case 18: e = launch_att<4, 2>(a, grid, s); break;
    case 19: e = launch_att<4, 3>(a, grid, s); break;
    case 33: e = launch_att<8, 1>(a, grid, s); break;
    case 34: e = launch_att<8, 2>(a, grid, s); break;
    case 35: e = launch_att<8, 3>(a, grid, s); break;
    case 65: e = launch_att<16, 1>(a, grid, s); break;
    case 66: e = launch_att<16, 2>(a, grid, s); break;
    default: return cudaErrorNotSupported;
  }
  if (e != cudaSuccess) return e;
  switch (Hp) {
    case 4: attend_combine_kernel<4><<<(unsigned)G, kCombThreads, 0, s>>>(part_o, part_ml, S, H, Hp, vp->Pi, out); break;
    case 8: attend_combine_kernel<8><<<(unsigned)G, kCombThreads, 0, s>>>(part_o, part_ml, S, H, Hp, vp->Pi, out); break;
    default: attend_combine_kernel<16><<<(unsigned)G, kCombThreads, 0, s>>>(part_o, part_ml, S, H, Hp, vp->Pi, out); break;
  }
  return cudaGetLastError();
}

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
