// Decode on the 5th-generation tensor cores for any d above 128 (a multiple
// of 128):
//   x_hat = n Pi^T c[idx] + rho sqrt(pi/2)/m S^T (2z - 1)
// ("turboquant-pytorch 소개", usage listing ``decompress``; TurboQuantMSE keeps
// the first term only).  For a tile of 128 keys both terms are contractions
// over the d code coordinates, D1 = C Pi and D2 = Z S with C[key][i] =
// c[idx_i] and Z[key][i] = 2 z_i - 1, done in jobs of 128 output coordinates
// (columns j of D1 and D2), K = d in stages of 64 coordinates.
//
// Exactness as in the d = 128 decode: A is 2^8 c[idx] split into fp16 hi + lo
// (and the signs, exact), B is 2^8 Pi^T and 2^8 S^T split hi + lo; D1 takes
// three products per k step and D2 two, about 2^-22 relative per product.
//
// Work per CTA (persistent, one CTA per SM, tiles blockIdx.x + i gridDim.x):
//  warp 0     producer: TMA loads of the B operand into a 3-stage ring; a
//             stage holds 128 rows (output coordinates) x 64 K values of
//             2^8 Pi^T hi and lo and, for Prod, of 2^8 S^T hi and lo (128-byte
//             swizzle, 64 KB);
//  warp 1     TMEM owner (512 columns) and MMA issuer (one thread);
//  warps 2-5  A operand: thread = key row; per stage the code bits of its 64
//             coordinates (read from the packed block in global memory) become
//             fp16 hi, lo and sign words in a 2-stage TMEM ring.  The codes do
//             not depend on the job, but TMEM cannot hold all of K, so every
//             job expands them again (cheap beside the job's MMAs);
//  warps 6-9  epilogue: thread = key row; per job it reads D1 and D2 and
//             writes the job's 128 fp32 coordinates of the key's row.
// TMEM columns: D1 [0, 128), D2 [128, 256), A stage s at 256 + 96 s: hi 32,
// lo 32, signs 32 columns of fp16 pairs (k step kb at column 8 kb).
// Every wait is bounded: on expiry the kernel raises the plan's error word,
// drains what it issued and frees its TMEM.
#include <cuda.h>
#include <cuda_fp16.h>

#include "ptx_sm100.cuh"
#include "tc_planes.cuh"
#include "tq_internal.cuh"

namespace tq {
namespace {

using namespace ptx;

constexpr int kDWThreads = 320;
constexpr int kDWStages = 3;
constexpr int kDWAStages = 2;
constexpr int kDWStageK = 64;                     // K values per stage
constexpr uint32_t kDWPart = 128 * 128;           // 128 rows x 64 fp16 (one 128-byte swizzle row each)
constexpr uint32_t kDWStageBytes = 4 * kDWPart;   // Pi^T hi, lo, (Prod) S^T hi, lo
constexpr uint32_t kDWColD1 = 0, kDWColD2 = 128, kDWColA = 256, kDWAStageCols = 96;
enum {
  DW_FULL = 0,
  DW_EMPTY = DW_FULL + kDWStages,
  DW_AFULL = DW_EMPTY + kDWStages,
  DW_AEMPTY = DW_AFULL + kDWAStages,
  DW_DFULL = DW_AEMPTY + kDWAStages,
  DW_DEMPTY,
  DW_DONE,
  DW_COUNT
};
constexpr uint32_t kDWOffBar = kDWStages * kDWStageBytes;
constexpr uint32_t kDWSmem = kDWOffBar + DW_COUNT * 8 + 1024;  // + alignment slack

struct DecWideArgs {
  Layout lay;
  int64_t N, nb, n_tiles;
  int J, S;            // jobs per tile (d / 128), stages per job (d / 64)
  uint32_t ctab[16];   // level i: fp16 bits of hi (low half) and lo (high half) of 2^8 c_i
  float kappa;
  const uint8_t* packed;
  float* out;
  int* err;
};

__device__ __forceinline__ void raise_dw(int* err, volatile int* abort) {
  *abort = 1;
  atomicExch(err, 1);
}

template <int K, bool PROD>
__global__ void __launch_bounds__(kDWThreads, 1)
    decode_wide_kernel(const __grid_constant__ CUtensorMap tmPiT, const __grid_constant__ CUtensorMap tmST,
                       const DecWideArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(smem);
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  // k >= 3: a pair of coordinates' code bits (key = sum_p (2 bits of plane p)
  // << 2p) -> {hi pair, lo pair}; k <= 2 keeps the levels in registers
  __shared__ uint2 s_tab[K >= 3 ? (1 << (2 * K)) : 1];
  auto bar = [&](int i) { return sb + kDWOffBar + 8u * (uint32_t)i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.lay.d, J = a.J, S = a.S;

  if constexpr (K >= 3) {
    for (int e = threadIdx.x; e < (1 << (2 * K)); e += blockDim.x) {
      uint32_t c[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        uint32_t idx = 0;
#pragma unroll
        for (int p = 0; p < K; ++p) idx |= (uint32_t)((e >> (2 * p + u)) & 1) << p;
        c[u] = a.ctab[idx];
      }
      s_tab[e] = make_uint2(__byte_perm(c[0], c[1], 0x5410), __byte_perm(c[0], c[1], 0x7632));
    }
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kDWStages; ++s) {
      mbar_init(bar(DW_FULL + s), 1);
      mbar_init(bar(DW_EMPTY + s), 1);
    }
    for (int s = 0; s < kDWAStages; ++s) {
      mbar_init(bar(DW_AFULL + s), 128);
      mbar_init(bar(DW_AEMPTY + s), 1);
    }
    mbar_init(bar(DW_DFULL), 1);
    mbar_init(bar(DW_DEMPTY), 128);
    mbar_init(bar(DW_DONE), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort = &abort_flag;
  const int64_t n_my = blockIdx.x < a.n_tiles ? (a.n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmPiT);
      if constexpr (PROD) prefetch_tmap(&tmST);
      uint32_t b = 0, ph = 0, issued = 0;
      bool ok = true;
      for (int64_t i = 0; ok && i < n_my; ++i)
        for (int jb = 0; ok && jb < J; ++jb)
          for (int st = 0; st < S; ++st) {
            if (!mbar_wait_suspend(bar(DW_EMPTY + b), ph ^ 1u, abort)) {
              ok = false;
              break;
            }
            const uint32_t base = sb + b * kDWStageBytes;
            mbar_arrive_expect_tx(bar(DW_FULL + b), (PROD ? 4 : 2) * kDWPart);
            // rows j of the images: hi at j, lo at d + j
            tma_load_2d(base, &tmPiT, st * kDWStageK, jb * 128, bar(DW_FULL + b));
            tma_load_2d(base + kDWPart, &tmPiT, st * kDWStageK, d + jb * 128, bar(DW_FULL + b));
            if constexpr (PROD) {
              tma_load_2d(base + 2 * kDWPart, &tmST, st * kDWStageK, jb * 128, bar(DW_FULL + b));
              tma_load_2d(base + 3 * kDWPart, &tmST, st * kDWStageK, d + jb * 128, bar(DW_FULL + b));
            }
            ++issued;
            if (++b == kDWStages) {
              b = 0;
              ph ^= 1u;
            }
          }
      if (!ok) raise_dw(a.err, abort);
      // no copy may still be landing when the CTA exits: the last fills
      int dummy = 0;
      for (uint32_t k = 0; k < (issued < kDWStages ? issued : (uint32_t)kDWStages); ++k) {
        b = b == 0 ? kDWStages - 1 : b - 1;
        if (b == kDWStages - 1) ph ^= 1u;
        mbar_wait(bar(DW_FULL + b), ph, &dummy);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(0u, 128, 128);
      const uint32_t d1 = tmem + kDWColD1, d2 = tmem + kDWColD2;
      uint32_t b = 0, bph = 0, s = 0, aph = 0, q = 0;
      bool ok = true;
      for (int64_t i = 0; ok && i < n_my; ++i)
        for (int jb = 0; ok && jb < J; ++jb, ++q) {
          // the epilogue has read the previous job's accumulators
          if (!mbar_wait(bar(DW_DEMPTY), (q & 1u) ^ 1u, abort)) {
            ok = false;
            break;
          }
          for (int st = 0; st < S; ++st) {
            if (!mbar_wait(bar(DW_FULL + b), bph, abort) || !mbar_wait(bar(DW_AFULL + s), aph, abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t bq = sb + b * kDWStageBytes;
            const uint64_t ph_ = sdesc_k_sw128(bq), pl_ = sdesc_k_sw128(bq + kDWPart);
            const uint64_t sh_ = sdesc_k_sw128(bq + 2 * kDWPart), sl_ = sdesc_k_sw128(bq + 3 * kDWPart);
            const uint32_t at = tmem + kDWColA + s * kDWAStageCols;
#pragma unroll
            for (uint32_t ks = 0; ks < 4; ++ks) {
              // k step ks: 16 values, 32 bytes into the 128-byte swizzle rows
              // (descriptor units of 16 bytes); A columns 8 ks
              const uint32_t acc = (st > 0 || ks > 0) ? 1u : 0u;
              mma_f16_ts(d1, at + 8 * ks, ph_ + 2u * ks, idesc, acc);
              mma_f16_ts(d1, at + 8 * ks, pl_ + 2u * ks, idesc, 1u);
              mma_f16_ts(d1, at + 32 + 8 * ks, ph_ + 2u * ks, idesc, 1u);
              if constexpr (PROD) {
                mma_f16_ts(d2, at + 64 + 8 * ks, sh_ + 2u * ks, idesc, acc);
                mma_f16_ts(d2, at + 64 + 8 * ks, sl_ + 2u * ks, idesc, 1u);
              }
            }
            mma_commit(bar(DW_EMPTY + b));
            mma_commit(bar(DW_AEMPTY + s));
            if (++b == kDWStages) {
              b = 0;
              bph ^= 1u;
            }
            if (++s == kDWAStages) {
              s = 0;
              aph ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit(bar(DW_DFULL));
        }
      if (!ok) raise_dw(a.err, abort);
      // all issued MMAs complete before TMEM is freed
      mma_commit(bar(DW_DONE));
      int dummy = 0;
      mbar_wait(bar(DW_DONE), 0, &dummy);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ A operand
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16) + kDWColA;
    // k <= 2: the fp16 bytes of levels 0..3, hi and lo parts (levels 0, 1 in
    // x, 2, 3 in y), picked by byte permutes (see the d = 128 decode)
    const uint32_t thx = __byte_perm(a.ctab[0], a.ctab[1], 0x5410), thy = __byte_perm(a.ctab[2], a.ctab[3], 0x5410);
    const uint32_t tlx = __byte_perm(a.ctab[0], a.ctab[1], 0x7632), tly = __byte_perm(a.ctab[2], a.ctab[3], 0x7632);
    uint32_t s = 0, aph = 0;
    bool ok = true;
    for (int64_t i = 0; ok && i < n_my; ++i) {
      const int64_t tile = blockIdx.x + i * gridDim.x;
      const uint8_t* blk = a.packed + tile * a.lay.block_bytes;
      for (int jb = 0; ok && jb < J; ++jb)
        for (int st = 0; st < S; ++st) {
          // coordinates 64 st .. 64 st + 63: words 2 (st % 2), + 1 of chunk st / 2
          const int c = st >> 1, w0 = 2 * (st & 1);
          uint2 pw[K];
#pragma unroll
          for (int p = 0; p < K; ++p)
            pw[p] = __ldg(reinterpret_cast<const uint2*>(blk + a.lay.plane_off(p, c, row) + 4 * w0));
          uint2 zw = make_uint2(0u, 0u);
          if constexpr (PROD) zw = __ldg(reinterpret_cast<const uint2*>(blk + a.lay.plane_off(K, c, row) + 4 * w0));
          if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(DW_AEMPTY + s), aph ^ 1u, abort))) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t hi[32], lo[32];
#pragma unroll
          for (int ww = 0; ww < 2; ++ww) {
            uint32_t wp[K];
#pragma unroll
            for (int p = 0; p < K; ++p) wp[p] = ww ? pw[p].y : pw[p].x;
            if constexpr (K <= 2) {
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4) {
                uint32_t S4 = (((wp[0] >> (4 * q4)) & 0xFu) * 0x00204081u) & 0x01010101u;
                if constexpr (K == 2) S4 |= (((wp[1] >> (4 * q4)) & 0xFu) * 0x00408102u) & 0x02020202u;
                const uint32_t T = S4 * 0x22u + 0x10101010u;
                hi[16 * ww + 2 * q4] = __byte_perm(thx, thy, T);
                hi[16 * ww + 2 * q4 + 1] = __byte_perm(thx, thy, T >> 16);
                lo[16 * ww + 2 * q4] = __byte_perm(tlx, tly, T);
                lo[16 * ww + 2 * q4 + 1] = __byte_perm(tlx, tly, T >> 16);
              }
            } else {
#pragma unroll
              for (int m = 0; m < 16; ++m) {
                uint32_t key = 0;
#pragma unroll
                for (int p = 0; p < K; ++p) key |= ((wp[p] >> (2 * m)) & 3u) << (2 * p);
                const uint2 e = s_tab[key];
                hi[16 * ww + m] = e.x;
                lo[16 * ww + m] = e.y;
              }
            }
          }
          const uint32_t col = t_lane + s * kDWAStageCols;
          tmem_st32(col, hi);
          tmem_st32(col + 32, lo);
          if constexpr (PROD) {
            // 2 z - 1 as fp16 (+1 = 0x3C00, -1 = 0xBC00), four coordinates per permute pair
            uint32_t sg[32];
#pragma unroll
            for (int ww = 0; ww < 2; ++ww) {
              const uint32_t nz = ~(ww ? zw.y : zw.x);
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4) {
                const uint32_t S4 = (((nz >> (4 * q4)) & 0xFu) * 0x00204081u) & 0x01010101u;
                const uint32_t T = (S4 << 4) | 0x02020202u;
                sg[16 * ww + 2 * q4] = __byte_perm(0x0000BC3Cu, 0u, T);
                sg[16 * ww + 2 * q4 + 1] = __byte_perm(0x0000BC3Cu, 0u, T >> 16);
              }
            }
            tmem_st32(col + 64, sg);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(DW_AFULL + s));
          if (++s == kDWAStages) {
            s = 0;
            aph ^= 1u;
          }
        }
    }
    if (!ok) raise_dw(a.err, abort);
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    uint32_t q = 0;
    bool ok = true;
    for (int64_t i = 0; ok && i < n_my; ++i) {
      const int64_t tile = blockIdx.x + i * gridDim.x;
      const int64_t g = tile / a.nb, tok = (tile - g * a.nb) * kTokensPerBlock + row;
      const float2 nr = __ldg(reinterpret_cast<const float2*>(a.packed + tile * a.lay.block_bytes + a.lay.norms_off +
                                                              row * 8));
      const float s1 = nr.x * (1.f / 65536.f), s2 = nr.y * a.kappa * (1.f / 256.f);
      float* dst_row = a.out + (g * a.N + tok) * (int64_t)d;
      for (int jb = 0; jb < J; ++jb, ++q) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(DW_DFULL), q & 1u, abort))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float4* dst = reinterpret_cast<float4*>(dst_row + jb * 128);
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t v1[32], v2[32];
          tmem_ld32(t_lane + kDWColD1 + 32 * q4, v1);
          if constexpr (PROD) tmem_ld32(t_lane + kDWColD2 + 32 * q4, v2);
          tmem_ld_wait();
          if (q4 == 3) {  // both accumulators read: the next job's MMAs may write them
            tc_fence_before();
            mbar_arrive(bar(DW_DEMPTY));
          }
          if (tok < a.N) {
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              float o[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                o[u] = s1 * __uint_as_float(v1[4 * t + u]);
                if constexpr (PROD) o[u] = fmaf(s2, __uint_as_float(v2[4 * t + u]), o[u]);
              }
              dst[8 * q4 + t] = make_float4(o[0], o[1], o[2], o[3]);
            }
          }
        }
      }
    }
    if (!ok) raise_dw(a.err, abort);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int K, bool PROD>
cudaError_t launch_dw(const tq_plan* p, const uint8_t* packed, int64_t G, int64_t N, float* out, cudaStream_t s) {
  const int d = p->d;
  DecWideArgs a;
  a.lay = p->lay;
  a.N = N;
  a.nb = (N + kTokensPerBlock - 1) / kTokensPerBlock;
  a.n_tiles = G * a.nb;
  a.J = d / 128;
  a.S = d / kDWStageK;
  for (int i = 0; i < 16; ++i) a.ctab[i] = i < p->cp.L ? p->dec_ctab[i] : 0u;
  a.kappa = p->kappa;
  a.packed = packed;
  a.out = out;
  a.err = p->err;
  // B operands: [hi rows; lo rows] of 2^8 Pi^T and (Prod) 2^8 S^T, fp16 [2d][d]
  const size_t dd = (size_t)d * d;
  CUtensorMap tp, ts;
  cudaError_t e = make_tmap_2d(&tp, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p->dec_wide_ops, (uint64_t)d, 2 * (uint64_t)d,
                               (uint64_t)d * 2, kDWStageK, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e == cudaSuccess && PROD)
    e = make_tmap_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p->dec_wide_ops + 2 * dd, (uint64_t)d, 2 * (uint64_t)d,
                     (uint64_t)d * 2, kDWStageK, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  else
    ts = tp;  // an MSE decode has no second product and never reads this map
  if (e != cudaSuccess) return e;
  auto kern = decode_wide_kernel<K, PROD>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDWSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t grid = a.n_tiles < sms ? a.n_tiles : sms;
  kern<<<(unsigned)grid, kDWThreads, kDWSmem, s>>>(tp, ts, a);
  return cudaGetLastError();
}

}  // namespace

bool decode_wide_supported(const tq_plan* p) {
  return p->dec_wide_ops != nullptr && p->d > 128 && p->d % 128 == 0 && !p->lay.frac && p->cp.L >= 2 &&
         p->cp.L <= (p->lay.prod ? 8 : 16);
}

cudaError_t launch_decode_wide(const tq_plan* p, const uint8_t* packed, int64_t G, int64_t N, float* out,
                               cudaStream_t s) {
  if (G * N == 0) return cudaSuccess;
  if (!decode_wide_supported(p)) return cudaErrorInvalidValue;
  if (p->lay.prod) {
    switch (p->lay.k) {
      case 1: return launch_dw<1, true>(p, packed, G, N, out, s);
      case 2: return launch_dw<2, true>(p, packed, G, N, out, s);
      case 3: return launch_dw<3, true>(p, packed, G, N, out, s);
    }
  } else {
    switch (p->lay.k) {
      case 1: return launch_dw<1, false>(p, packed, G, N, out, s);
      case 2: return launch_dw<2, false>(p, packed, G, N, out, s);
      case 3: return launch_dw<3, false>(p, packed, G, N, out, s);
      case 4: return launch_dw<4, false>(p, packed, G, N, out, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace tq
