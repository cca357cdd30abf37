// Decode on the 5th-generation tensor cores (tcgen05 + TMEM), d = 128:
//   x_hat = n Pi^T c[idx] + rho sqrt(pi/2)/m S^T (2z - 1)
// ("turboquant-pytorch 소개", usage listing ``decompress``; TurboQuantMSE keeps
// the first term only).  For a tile of 128 keys both terms are contractions
// over the d code coordinates: D1 = C Pi (C[key][i] = c[idx_i]) and
// D2 = Z S (Z[key][i] = 2 z_i - 1).
//
// Exactness on fp16 tensor cores (fp32 accumulate): the A operands are
// 2^8 c[idx] split into fp16 hi + lo (the codebook has at most 16 values, split
// once per plan) and the signs +-1 (exact); the B operands are 2^8 Pi^T and
// 2^8 S^T split hi + lo.  D1 = A_hi B_hi + A_hi B_lo + A_lo B_hi and
// D2 = Z B_hi + Z B_lo leave ~2^-22 relative per product; the powers of two
// keep every lo part out of fp16's subnormal range and are undone in the
// epilogue (n 2^-16 D1 + rho kappa 2^-8 D2).
//
// Work per CTA (persistent, one CTA per SM, one packed block = 128 keys per tile):
//  warp 0     bulk copies: once the B images, then each tile's packed block
//             into a 2-stage ring;
//  warp 1     TMEM owner (512 columns) and MMA issuer (one thread);
//  warps 2-5  expansion: thread = key row; code bits -> A operands in TMEM;
//  warps 6-9  epilogue: thread = key row; accumulators -> fp32 rows of out.
// TMEM columns: D1 [0, 128), D2 [128, 256), A hi [256, 320), A lo [320, 384),
// signs [384, 448); A columns hold fp16 pairs, k step kb at column 8 kb.
// Every wait is bounded: on expiry the kernel raises the plan's error word,
// drains what it issued and frees its TMEM.
#include <cuda.h>
#include <cuda_fp16.h>

#include "ptx_sm100.cuh"
#include "tq_internal.cuh"

namespace tq {
namespace {

using namespace ptx;

constexpr int kDecThreads = 320;
constexpr int kDecStages = 2;
constexpr uint32_t kDecImg = 128 * 128 * 2;   // one 128 x 128 fp16 operand image
constexpr uint32_t kDecAtom = 128 * 128;      // 128 rows x 64 elements (128 B) per swizzle atom
constexpr uint32_t kOffPtHi = 0, kOffPtLo = kDecImg, kOffStHi = 2 * kDecImg, kOffStLo = 3 * kDecImg;
constexpr uint32_t kBlkMax = 4 * 2048 + 1024;  // largest d = 128 block: four planes + norms
constexpr uint32_t kOffBlk = 4 * kDecImg;
constexpr uint32_t kOffDecBar = kOffBlk + kDecStages * kBlkMax;
enum {
  DB_OPS = 0,
  DB_SFULL = 1,
  DB_SEMPTY = DB_SFULL + kDecStages,  // expansion (128) + epilogue (128) arrivals
  DB_AFULL = DB_SEMPTY + kDecStages,
  DB_AEMPTY,
  DB_DFULL,
  DB_DEMPTY,
  DB_DONE,
  DB_COUNT
};
constexpr uint32_t kDecSmem = kOffDecBar + DB_COUNT * 8 + 1024;  // + alignment slack
constexpr uint32_t kColD1 = 0, kColD2 = 128, kColAHi = 256, kColALo = 320, kColSg = 384;

struct DecTcArgs {
  Layout lay;
  int64_t N, nb, n_tiles;
  uint32_t ctab[16];  // level i: fp16 bits of hi (low half) and lo (high half) of 2^8 c_i
  uint32_t ctab_lo[16];  // the same for the lower codebook of a fractional width (coordinates 64..127)
  float kappa;
  const uint8_t* packed;
  const uint8_t* pit;  // 2^8 Pi^T images: hi, lo
  const uint8_t* st;   // 2^8 S^T images: hi, lo (PROD)
  float* out;
  int* err;
};

__device__ __forceinline__ void raise_dec(int* err, volatile int* abort) {
  *abort = 1;
  atomicExch(err, 1);
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int w) {
  return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
}

template <int K, bool PROD>
__global__ void __launch_bounds__(kDecThreads, 1) decode_tc_kernel(const DecTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(smem);
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ uint32_t s_ctab[32];  // [0, 16): coordinates 0..63; [16, 32): 64..127
  auto bar = [&](int i) { return sb + kOffDecBar + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < 16) {
    s_ctab[threadIdx.x] = a.ctab[threadIdx.x];
    s_ctab[16 + threadIdx.x] = a.lay.frac ? a.ctab_lo[threadIdx.x] : a.ctab[threadIdx.x];
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar(DB_OPS), 1);
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(bar(DB_SFULL + s), 1);
      mbar_init(bar(DB_SEMPTY + s), 256);
    }
    mbar_init(bar(DB_AFULL), 128);
    mbar_init(bar(DB_AEMPTY), 1);
    mbar_init(bar(DB_DFULL), 1);
    mbar_init(bar(DB_DEMPTY), 128);
    mbar_init(bar(DB_DONE), 1);
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
  const uint32_t bb = (uint32_t)a.lay.block_bytes;

  if (warp == 0) {
    // ------------------------------------------------------------ bulk copies
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(DB_OPS), (PROD ? 4 : 2) * kDecImg);
      bulk_load(sb + kOffPtHi, a.pit, kDecImg, bar(DB_OPS));
      bulk_load(sb + kOffPtLo, a.pit + kDecImg, kDecImg, bar(DB_OPS));
      if constexpr (PROD) {
        bulk_load(sb + kOffStHi, a.st, kDecImg, bar(DB_OPS));
        bulk_load(sb + kOffStLo, a.st + kDecImg, kDecImg, bar(DB_OPS));
      }
      int64_t issued = 0;
      for (int64_t i = 0; i < n_my; ++i) {
        const int s = (int)(i % kDecStages);
        if (!mbar_wait(bar(DB_SEMPTY + s), ((uint32_t)(i / kDecStages) & 1u) ^ 1u, abort)) {
          raise_dec(a.err, abort);
          break;
        }
        const int64_t tile = blockIdx.x + i * gridDim.x;
        mbar_arrive_expect_tx(bar(DB_SFULL + s), bb);
        bulk_load(sb + kOffBlk + s * kBlkMax, a.packed + tile * a.lay.block_bytes, bb, bar(DB_SFULL + s));
        issued = i + 1;
      }
      // no copy may still be landing when the CTA exits
      int dummy = 0;
      for (int64_t i = issued > kDecStages ? issued - kDecStages : 0; i < issued; ++i)
        mbar_wait(bar(DB_SFULL + (int)(i % kDecStages)), (uint32_t)(i / kDecStages) & 1u, &dummy);
      mbar_wait(bar(DB_OPS), 0, &dummy);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(0u, 128, 128);
      bool ok = mbar_wait(bar(DB_OPS), 0, abort);
      for (int64_t i = 0; ok && i < n_my; ++i) {
        const uint32_t ph = (uint32_t)i & 1u;
        if (!mbar_wait(bar(DB_AFULL), ph, abort) || !mbar_wait(bar(DB_DEMPTY), ph ^ 1u, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
          const uint32_t off = (kb >> 2) * kDecAtom + (kb & 3) * 32;
          const uint64_t bh = sdesc_k_sw128(sb + kOffPtHi + off), bl = sdesc_k_sw128(sb + kOffPtLo + off);
          const uint32_t ahi = tmem + kColAHi + 8 * kb, alo = tmem + kColALo + 8 * kb;
          mma_f16_ts(tmem + kColD1, ahi, bh, idesc, kb > 0);
          mma_f16_ts(tmem + kColD1, ahi, bl, idesc, 1u);
          mma_f16_ts(tmem + kColD1, alo, bh, idesc, 1u);
          if constexpr (PROD) {
            const uint64_t sh = sdesc_k_sw128(sb + kOffStHi + off), sl = sdesc_k_sw128(sb + kOffStLo + off);
            const uint32_t sg = tmem + kColSg + 8 * kb;
            mma_f16_ts(tmem + kColD2, sg, sh, idesc, kb > 0);
            mma_f16_ts(tmem + kColD2, sg, sl, idesc, 1u);
          }
        }
        mma_commit(bar(DB_DFULL));
        mma_commit(bar(DB_AEMPTY));
      }
      if (!ok) raise_dec(a.err, abort);
      // all issued MMAs complete before TMEM is freed
      mma_commit(bar(DB_DONE));
      int dummy = 0;
      mbar_wait(bar(DB_DONE), 0, &dummy);
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ expansion
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    bool ok = true;
    for (int64_t i = 0; ok && i < n_my; ++i) {
      const int s = (int)(i % kDecStages);
      // every lane polls; the warp proceeds (or gives up) as one, because the
      // tcgen05 stores below are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(bar(DB_SFULL + s), (uint32_t)(i / kDecStages) & 1u, abort)) ||
          !__all_sync(0xffffffffu, mbar_wait(bar(DB_AEMPTY), ((uint32_t)i & 1u) ^ 1u, abort))) {
        ok = false;
        break;
      }
      tc_fence_after();
      // this key's 16-byte chunk of every plane (d = 128: one chunk per plane)
      const uint8_t* blk = smem + kOffBlk + s * kBlkMax;
      uint4 pw[K];
#pragma unroll
      for (int p = 0; p < K; ++p) {
        if (p == K - 1 && a.lay.frac) {  // a fractional width's half plane: coordinates 0..63
          const uint2 h = *reinterpret_cast<const uint2*>(blk + a.lay.top_off + row * 8);
          pw[p] = make_uint4(h.x, h.y, 0u, 0u);
        } else {
          pw[p] = *reinterpret_cast<const uint4*>(blk + ((int64_t)p * kTokensPerBlock + row) * 16);
        }
      }
      uint4 zw = make_uint4(0u, 0u, 0u, 0u);
      if constexpr (PROD) zw = *reinterpret_cast<const uint4*>(blk + a.lay.sign_off + row * 16);
      mbar_arrive(bar(DB_SEMPTY + s));
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        // coordinates 32 w + e, e = 0..31: bit e of word w of each plane
        uint32_t wp[K];
#pragma unroll
        for (int p = 0; p < K; ++p) wp[p] = word_of(pw[p], w);
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          uint32_t i0 = 0, i1 = 0;
#pragma unroll
          for (int p = 0; p < K; ++p) {
            i0 |= ((wp[p] >> (2 * m)) & 1u) << p;
            i1 |= ((wp[p] >> (2 * m + 1)) & 1u) << p;
          }
          const uint32_t c0 = s_ctab[(w >> 1) * 16 + i0], c1 = s_ctab[(w >> 1) * 16 + i1];
          hi[m] = __byte_perm(c0, c1, 0x5410);  // (hi of coordinate 2m, hi of 2m + 1)
          lo[m] = __byte_perm(c0, c1, 0x7632);
        }
        tmem_st16(t_lane + kColAHi + 16 * w, hi);
        tmem_st16(t_lane + kColALo + 16 * w, lo);
        if constexpr (PROD) {
          // 2 z - 1 as fp16 (+1 = 0x3C00, -1 = 0xBC00)
          const uint32_t z = word_of(zw, w);
          uint32_t sg[16];
#pragma unroll
          for (int m = 0; m < 16; ++m)
            sg[m] = 0x3C003C00u | ((~(z >> (2 * m)) & 1u) << 15) | ((~(z >> (2 * m + 1)) & 1u) << 31);
          tmem_st16(t_lane + kColSg + 16 * w, sg);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(DB_AFULL));
    }
    if (!ok) raise_dec(a.err, abort);
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    bool ok = true;
    for (int64_t i = 0; ok && i < n_my; ++i) {
      const int s = (int)(i % kDecStages);
      const int64_t tile = blockIdx.x + i * gridDim.x;
      const int64_t g = tile / a.nb, tok = (tile - g * a.nb) * kTokensPerBlock + row;
      // the key's norms, read from the staged block (this role waits on the
      // stage itself, so the block cannot be refilled before it is read)
      if (!__all_sync(0xffffffffu, mbar_wait(bar(DB_SFULL + s), (uint32_t)(i / kDecStages) & 1u, abort))) {
        ok = false;
        break;
      }
      const float2 nr =
          *reinterpret_cast<const float2*>(smem + kOffBlk + s * kBlkMax + a.lay.norms_off + row * 8);
      mbar_arrive(bar(DB_SEMPTY + s));
      const float s1 = nr.x * (1.f / 65536.f), s2 = nr.y * a.kappa * (1.f / 256.f);
      if (!__all_sync(0xffffffffu, mbar_wait(bar(DB_DFULL), (uint32_t)i & 1u, abort))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float4* dst = reinterpret_cast<float4*>(a.out + (g * a.N + tok) * 128);
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        uint32_t v1[32], v2[32];
        tmem_ld32(t_lane + kColD1 + 32 * q, v1);
        if constexpr (PROD) tmem_ld32(t_lane + kColD2 + 32 * q, v2);
        tmem_ld_wait();
        if (q == 3) {  // both accumulators read: the next tile's MMAs may write them
          tc_fence_before();
          mbar_arrive(bar(DB_DEMPTY));
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
            dst[8 * q + t] = make_float4(o[0], o[1], o[2], o[3]);
          }
        }
      }
    }
    if (!ok) raise_dec(a.err, abort);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int K, bool PROD>
cudaError_t launch_dec(const tq_plan* p, const uint8_t* packed, int64_t G, int64_t N, float* out, cudaStream_t s) {
  DecTcArgs a;
  a.lay = p->lay;
  a.N = N;
  a.nb = (N + kTokensPerBlock - 1) / kTokensPerBlock;
  a.n_tiles = G * a.nb;
  for (int i = 0; i < 16; ++i) a.ctab[i] = i < p->cp.L ? p->dec_ctab[i] : 0u;
  for (int i = 0; i < 16; ++i) a.ctab_lo[i] = p->lay.frac && i < p->cp_lo.L ? p->dec_ctab_lo[i] : 0u;
  a.kappa = p->kappa;
  a.packed = packed;
  a.pit = p->tc_ops + tc_dec_image(p, 0) * kDecImg;
  a.st = PROD ? p->tc_ops + tc_dec_image(p, 2) * kDecImg : nullptr;
  a.out = out;
  a.err = p->err;
  auto kern = decode_tc_kernel<K, PROD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t grid = a.n_tiles < sms ? a.n_tiles : sms;
  kern<<<(unsigned)grid, kDecThreads, kDecSmem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool decode_tc_supported(const tq_plan* p) {
  return p->tc_ops != nullptr && p->d == 128 && p->lay.block_bytes <= kBlkMax && p->cp.L >= 2 &&
         p->cp.L <= (p->lay.prod ? 8 : 16);
}

cudaError_t launch_decode_tc(const tq_plan* p, const uint8_t* packed, int64_t G, int64_t N, float* out,
                             cudaStream_t s) {
  if (G * N == 0) return cudaSuccess;
  if (p->lay.prod) {
    switch (p->lay.k) {
      case 1: return launch_dec<1, true>(p, packed, G, N, out, s);
      case 2: return launch_dec<2, true>(p, packed, G, N, out, s);
      case 3: return launch_dec<3, true>(p, packed, G, N, out, s);
    }
  } else {
    switch (p->lay.k) {
      case 1: return launch_dec<1, false>(p, packed, G, N, out, s);
      case 2: return launch_dec<2, false>(p, packed, G, N, out, s);
      case 3: return launch_dec<3, false>(p, packed, G, N, out, s);
      case 4: return launch_dec<4, false>(p, packed, G, N, out, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace tq
