// Score on the tensor cores for any head dimension d (a multiple of 128) and up
// to 256 query heads per group: the shape of a vector-search index (d = 1536,
// 256 queries), where the estimate is a long dense contraction per key.
//
// Same estimate as the other score kernels ("turboquant-pytorch 소개", usage
// listing ``tq.inner_product(query, compressed)`` and "2단계"):
//     logit = n <Pi q, c[idx]> + rho sqrt(pi/2)/m <S q, 2z - 1>.
// Here the per-key factors are folded into the key operand, so one fp32
// accumulator holds the logit itself:
//     logit = sum_j (n c[idx_j]) (Pi q)_j + sum_j (kappa rho (2 z_j - 1)) (S q)_j.
//
// Exactness on bf16 tensor cores (fp32 accumulate): every operand is split
// into a bf16 pair v = v_hi + v_lo (about 2^-17 relative), and three products
// per term are issued (hi hi, hi lo, lo hi; the dropped lo lo is ~2^-17 of a
// term's lo parts).  The sign operand kappa rho (2z - 1) is the split of
// kappa rho with the sign of each coordinate applied to both parts.
//
// Tile: M = 128 keys (one packed block), N = the group's heads padded to a
// multiple of 16 (<= 256), K = d in stages of 32 coordinates.
//  warp 0     producer: TMA loads of the query operand (4 parts: (Pi q)_hi,
//             (Pi q)_lo, (S q)_hi, (S q)_lo, each N rows x 32 bf16, 64-byte
//             swizzle) into a 3-stage ring.
//  warp 1     TMEM owner (512 columns: the accumulator in [0, 256), the key
//             operand ring in [256, 512)) and MMA issuer (one thread).
//  warps 2-5  key decoders: thread (warp w, lane l) owns key row 32 (w % 4) + l;
//             per stage it reads its 32 coordinates' code bits and sign bits,
//             looks up n c[idx] (a per-key table of bf16 pairs in shared
//             memory) and writes the key operand parts into TMEM (4-stage ring).
//  warps 6-9  epilogue: the tile's accumulator -> H logits per key.
// Every wait is bounded: on expiry the kernel raises the plan's error word,
// drains what it issued and frees its TMEM.
#include <cuda_bf16.h>

#include "ptx_sm100.cuh"
#include "tq_internal.cuh"

namespace tq {
namespace {

using namespace ptx;

constexpr int kWThreads = 320;
constexpr int kEpiWarp0 = 6;  // warps 2-5 decode keys
constexpr int kBStages = 3;
constexpr int kAStages = 4;
constexpr int kStageK = 32;        // coordinates per stage
constexpr int kAccCols = 256;      // accumulator columns (N <= 256)
constexpr int kAPartCols = 16;     // TMEM columns of one key-operand part per stage (32 bf16)

enum {
  BAR_BFULL = 0,
  BAR_BEMPTY = BAR_BFULL + kBStages,
  BAR_AFULL = BAR_BEMPTY + kBStages,
  BAR_AEMPTY = BAR_AFULL + kAStages,
  BAR_DFULL = BAR_AEMPTY + kAStages,
  BAR_DEMPTY = BAR_DFULL + 1,
  BAR_DONE = BAR_DEMPTY + 1,
  BAR_COUNT = BAR_DONE + 1
};

struct WideArgs {
  Layout lay;
  int H, N;                 // heads, MMA N (heads padded to a multiple of 16)
  int L;                    // codebook levels
  float c[kMaxLevels];      // codebook (unit-norm scale)
  float kappa;
  int64_t Ntok, nb, n_tiles;
  const uint8_t* packed;
  float* logits;
  int* err;
};

__device__ __forceinline__ void raise(int* err, volatile int* abort) {
  *abort = 1;
  atomicExch(err, 1);
}

// Shared-memory descriptor, K-major, 64-byte swizzle: rows of 64 B, 8-row
// groups 512 B apart.
__device__ __forceinline__ uint64_t sdesc_k_sw64(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(512u >> 4) << 32) | ((uint64_t)1 << 46) |
         ((uint64_t)4 << 61);
}

// v = hi + lo with hi, lo bf16 (round to nearest each): returns hi | lo << 16
__device__ __forceinline__ uint32_t split_pair(float v) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  const __nv_bfloat16 l = __float2bfloat16_rn(v - __bfloat162float(h));
  return (uint32_t)__bfloat16_as_ushort(h) | ((uint32_t)__bfloat16_as_ushort(l) << 16);
}

template <int K, int PROD>
__global__ void __launch_bounds__(kWThreads, 1)
score_wide_kernel(const __grid_constant__ CUtensorMap tmQ, const WideArgs a) {
  constexpr int NPART_B = PROD ? 4 : 2;  // query operand parts
  constexpr int NPART_A = PROD ? 4 : 2;  // key operand parts: (n c)_hi, (n c)_lo [, (k rho s)_hi, (k rho s)_lo]
  constexpr int LV = 1 << K;             // table entries (levels)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(smem);
  const uint32_t part_bytes = (uint32_t)a.N * 64u;           // N rows x 32 bf16
  const uint32_t stage_bytes = NPART_B * part_bytes;
  const uint32_t off_lut = kBStages * stage_bytes;            // [LV][128] bf16 pairs of n c[i]
  const uint32_t off_bar = off_lut + LV * 128 * 4;
  uint32_t* lut = reinterpret_cast<uint32_t*>(smem + off_lut);
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  auto bar = [&](int i) { return sb + off_bar + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(bar(BAR_BFULL + s), 1);
      mbar_init(bar(BAR_BEMPTY + s), 1);
    }
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(bar(BAR_AFULL + s), 128);
      mbar_init(bar(BAR_AEMPTY + s), 1);
    }
    mbar_init(bar(BAR_DFULL), 1);
    mbar_init(bar(BAR_DEMPTY), 128);
    mbar_init(bar(BAR_DONE), 1);
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

  const int S = a.lay.d / kStageK;  // stages per tile
  const int64_t n_my = blockIdx.x < a.n_tiles ? (a.n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      uint32_t b = 0, ph = 0, issued = 0;
      bool ok = true;
      for (int64_t i = 0; ok && i < n_my; ++i) {
        const int64_t g = (blockIdx.x + i * gridDim.x) / a.nb;
        for (int st = 0; st < S; ++st) {
          if (!mbar_wait_suspend(bar(BAR_BEMPTY + b), ph ^ 1u, abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(BAR_BFULL + b), stage_bytes);
#pragma unroll
          for (int p = 0; p < NPART_B; ++p)
            tma_load_2d(sb + b * stage_bytes + p * part_bytes, &tmQ, st * kStageK,
                        (int32_t)((g * NPART_B + p) * a.N), bar(BAR_BFULL + b));
          ++issued;
          if (++b == kBStages) {
            b = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) raise(a.err, abort);
      // no copy may still be landing when the CTA exits
      int dummy = 0;
      for (uint32_t k = 0; k < (issued < kBStages ? issued : kBStages); ++k) {
        b = b == 0 ? kBStages - 1 : b - 1;
        if (b == kBStages - 1) ph ^= 1u;
        mbar_wait(bar(BAR_BFULL + b), ph, &dummy);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(1u, 128, (uint32_t)a.N);
      uint32_t b = 0, bph = 0, s = 0, aph = 0;
      bool ok = true;
      for (int64_t i = 0; ok && i < n_my; ++i) {
        if (!mbar_wait_suspend(bar(BAR_DEMPTY), ((uint32_t)i & 1u) ^ 1u, abort)) {
          ok = false;
          break;
        }
        for (int st = 0; st < S; ++st) {
          if (!mbar_wait_suspend(bar(BAR_BFULL + b), bph, abort) ||
              !mbar_wait_suspend(bar(BAR_AFULL + s), aph, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t bq = sb + b * stage_bytes;
          const uint32_t at = tmem + kAccCols + s * (NPART_A * kAPartCols);
#pragma unroll
          for (int ks = 0; ks < 2; ++ks) {
            // K step ks: 16 coordinates, 32 bytes into each 64-byte row, 8 TMEM columns
            const uint64_t pq_hi = sdesc_k_sw64(bq + 0 * part_bytes) + 2u * ks;
            const uint64_t pq_lo = sdesc_k_sw64(bq + 1 * part_bytes) + 2u * ks;
            const uint32_t nc_hi = at + 0 * kAPartCols + 8 * ks, nc_lo = at + 1 * kAPartCols + 8 * ks;
            const uint32_t first = (st == 0 && ks == 0) ? 0u : 1u;
            mma_f16_ts(tmem, nc_hi, pq_hi, idesc, first);
            mma_f16_ts(tmem, nc_hi, pq_lo, idesc, 1u);
            mma_f16_ts(tmem, nc_lo, pq_hi, idesc, 1u);
            if constexpr (PROD) {
              const uint64_t sq_hi = sdesc_k_sw64(bq + 2 * part_bytes) + 2u * ks;
              const uint64_t sq_lo = sdesc_k_sw64(bq + 3 * part_bytes) + 2u * ks;
              const uint32_t z_hi = at + 2 * kAPartCols + 8 * ks, z_lo = at + 3 * kAPartCols + 8 * ks;
              mma_f16_ts(tmem, z_hi, sq_hi, idesc, 1u);
              mma_f16_ts(tmem, z_hi, sq_lo, idesc, 1u);
              mma_f16_ts(tmem, z_lo, sq_hi, idesc, 1u);
            }
          }
          mma_commit(bar(BAR_BEMPTY + b));
          mma_commit(bar(BAR_AEMPTY + s));
          if (++b == kBStages) {
            b = 0;
            bph ^= 1u;
          }
          if (++s == kAStages) {
            s = 0;
            aph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(bar(BAR_DFULL));
      }
      if (!ok) raise(a.err, abort);
      mma_commit(bar(BAR_DONE));
      int dummy = 0;
      mbar_wait(bar(BAR_DONE), 0, &dummy);
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------------ key decoders
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16) + kAccCols;
    uint32_t s = 0, aph = 0;
    bool ok = true;
    for (int64_t i = 0; ok && i < n_my; ++i) {
      const int64_t tile = blockIdx.x + i * gridDim.x;
      const uint8_t* blk = a.packed + tile * a.lay.block_bytes;
      const float2 nr = *reinterpret_cast<const float2*>(blk + a.lay.norms_off + row * 8);
      // this key's table of n c[i] as bf16 pairs (column `row` of each entry:
      // the 32 lanes of a warp read 32 consecutive words whatever their codes)
      __syncwarp();
#pragma unroll
      for (int e = 0; e < LV; ++e) lut[e * 128 + row] = e < a.L ? split_pair(nr.x * a.c[e]) : 0u;
      __syncwarp();
      const uint32_t rk = split_pair(nr.y * a.kappa);
      const uint32_t rk_hi2 = (rk & 0xFFFFu) * 0x10001u, rk_lo2 = (rk >> 16) * 0x10001u;
      for (int c = 0; ok && c < a.lay.C; ++c) {
        uint4 w[K + PROD];
#pragma unroll
        for (int p = 0; p < K + PROD; ++p)
          w[p] = __ldg(reinterpret_cast<const uint4*>(blk + a.lay.plane_off(p, c, row)));
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(BAR_AEMPTY + s), aph ^ 1u, abort))) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t W[K + PROD];
#pragma unroll
          for (int p = 0; p < K + PROD; ++p) W[p] = q == 0 ? w[p].x : q == 1 ? w[p].y : q == 2 ? w[p].z : w[p].w;
          uint32_t nh[16], nl[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            uint32_t i0 = 0, i1 = 0;
#pragma unroll
            for (int p = 0; p < K; ++p) {
              i0 |= ((W[p] >> e) & 1u) << p;
              i1 |= ((W[p] >> (e + 1)) & 1u) << p;
            }
            const uint32_t v0 = lut[i0 * 128 + row], v1 = lut[i1 * 128 + row];
            nh[e >> 1] = __byte_perm(v0, v1, 0x5410);
            nl[e >> 1] = __byte_perm(v0, v1, 0x7632);
          }
          const uint32_t col = t_lane + s * (NPART_A * kAPartCols);
          tmem_st16(col + 0 * kAPartCols, nh);
          tmem_st16(col + 1 * kAPartCols, nl);
          if constexpr (PROD) {
            // 2z - 1: z = 0 sets the sign bit of both halves' coordinate
            const uint32_t nz = ~W[K];
            uint32_t zh[16], zl[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const uint32_t t = nz >> e;
              const uint32_t m = ((t & 1u) << 15) | ((t & 2u) << 30);
              zh[e >> 1] = rk_hi2 ^ m;
              zl[e >> 1] = rk_lo2 ^ m;
            }
            tmem_st16(col + 2 * kAPartCols, zh);
            tmem_st16(col + 3 * kAPartCols, zl);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(BAR_AFULL + s));
          if (++s == kAStages) {
            s = 0;
            aph ^= 1u;
          }
        }
      }
    }
    if (!ok) raise(a.err, abort);
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    for (int64_t i = 0; i < n_my; ++i) {
      const int64_t tile = blockIdx.x + i * gridDim.x;
      const int64_t g = tile / a.nb, blk = tile - g * a.nb;
      const int64_t tok = blk * kTokensPerBlock + row;
      if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(BAR_DFULL), (uint32_t)i & 1u, abort))) {
        raise(a.err, abort);
        break;
      }
      tc_fence_after();
      float* out = a.logits + (g * a.H) * a.Ntok + tok;
      for (int c0 = 0; c0 < a.N; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(t_lane + c0, v);
        tmem_ld_wait();
        if (tok < a.Ntok) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c0 + e < a.H) out[(int64_t)(c0 + e) * a.Ntok] = __uint_as_float(v[e]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(BAR_DEMPTY));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// qs [nv][G][H][d] fp32 (Pi q, S q) -> ops [G][NPART][N][d] bf16 parts
// (Pi q)_hi, (Pi q)_lo [, (S q)_hi, (S q)_lo]; heads H..N-1 are zero.
__global__ void wide_split_kernel(const float* __restrict__ qs, int64_t G, int H, int N, int d, int nv,
                                  __nv_bfloat16* __restrict__ ops) {
  const int64_t total = G * (int64_t)N * d;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int j = (int)(i % d);
    const int64_t r = i / d;
    const int h = (int)(r % N);
    const int64_t g = r / N;
    for (int v = 0; v < nv; ++v) {
      const float x = h < H ? qs[((v * G + g) * H + h) * d + j] : 0.f;
      const __nv_bfloat16 hi = __float2bfloat16_rn(x);
      const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
      ops[(((g * 2 * nv) + 2 * v + 0) * N + h) * (int64_t)d + j] = hi;
      ops[(((g * 2 * nv) + 2 * v + 1) * N + h) * (int64_t)d + j] = lo;
    }
  }
}

int wide_n(int H) { return ((H + 15) / 16) * 16; }

size_t wide_smem_bytes(const tq_plan* p, int H) {
  const int nparts = p->lay.prod ? 4 : 2;
  const size_t stage = (size_t)nparts * wide_n(H) * 64;
  return kBStages * stage + (size_t)(1 << p->lay.k) * 128 * 4 + BAR_COUNT * 8 + 1024;
}

template <int K, int PROD>
cudaError_t launch_wide_kernel(const CUtensorMap& tm, const WideArgs& a, size_t smem, cudaStream_t s) {
  auto kern = score_wide_kernel<K, PROD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t grid = a.n_tiles < sms ? a.n_tiles : sms;
  kern<<<(unsigned)grid, kWThreads, smem, s>>>(tm, a);
  return cudaGetLastError();
}

}  // namespace

bool score_wide_supported(const tq_plan* p, int H) {
  return !p->lay.frac && p->d % 128 == 0 && H >= 1 && H <= 256 && p->lay.k >= 1 && p->lay.k <= 4 &&
         wide_smem_bytes(p, H) <= 227 * 1024;
}

// [Pi q, S q fp32 | bf16 operand parts]
size_t score_wide_workspace_bytes(const tq_plan* p, int64_t G, int H) {
  const int nv = p->lay.prod ? 2 : 1;
  const size_t qs = ((size_t)G * H * nv * p->d * sizeof(float) + 255) & ~(size_t)255;
  return qs + (size_t)G * 2 * nv * wide_n(H) * p->d * sizeof(__nv_bfloat16);
}

cudaError_t launch_score_wide(const tq_plan* p, const float* queries, int64_t G, int H, const uint8_t* packed,
                              int64_t N, float* logits, void* ws, cudaStream_t s) {
  if (G == 0 || N == 0) return cudaSuccess;
  const int nv = p->lay.prod ? 2 : 1;
  const int Np = wide_n(H);
  float* qs = static_cast<float*>(ws);
  __nv_bfloat16* ops = reinterpret_cast<__nv_bfloat16*>(
      static_cast<char*>(ws) + (((size_t)G * H * nv * p->d * sizeof(float) + 255) & ~(size_t)255));
  // Pi q and S q of every query: products with matrices shared by all groups
  cudaError_t e = launch_rows_times_shared(queries, p->Pi, nv == 2 ? p->S : nullptr, G, H, p->d, p->d, qs,
                                           qs + (size_t)G * H * p->d, s);
  if (e != cudaSuccess) return e;
  wide_split_kernel<<<1184, 256, 0, s>>>(qs, G, H, Np, p->d, nv, ops);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  CUtensorMap tm;
  e = make_tmap_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ops, (uint64_t)p->d, (uint64_t)G * 2 * nv * Np,
                   (uint64_t)p->d * 2, kStageK, (uint32_t)Np, CU_TENSOR_MAP_SWIZZLE_64B);
  if (e != cudaSuccess) return e;
  WideArgs a;
  a.lay = p->lay;
  a.H = H;
  a.N = Np;
  a.L = p->cp.L;
  for (int i = 0; i < kMaxLevels; ++i) a.c[i] = p->cp.c[i];
  a.kappa = p->kappa;
  a.Ntok = N;
  a.nb = (N + kTokensPerBlock - 1) / kTokensPerBlock;
  a.n_tiles = G * a.nb;
  a.packed = packed;
  a.logits = logits;
  a.err = p->err;
  const size_t smem = wide_smem_bytes(p, H);
  const int k = p->lay.k;
  if (p->lay.prod) {
    switch (k) {
      case 1: return launch_wide_kernel<1, 1>(tm, a, smem, s);
      case 2: return launch_wide_kernel<2, 1>(tm, a, smem, s);
      case 3: return launch_wide_kernel<3, 1>(tm, a, smem, s);
    }
  } else {
    switch (k) {
      case 1: return launch_wide_kernel<1, 0>(tm, a, smem, s);
      case 2: return launch_wide_kernel<2, 0>(tm, a, smem, s);
      case 3: return launch_wide_kernel<3, 0>(tm, a, smem, s);
      case 4: return launch_wide_kernel<4, 0>(tm, a, smem, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace tq
