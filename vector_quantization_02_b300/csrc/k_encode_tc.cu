// Encode on the 5th-generation tensor cores (tcgen05 + TMA + TMEM), d = 128,
// fp16 or bf16 keys, TurboQuantProd; TurboQuantMSE ("turboquant-pytorch 소개",
// "1단계" alone) runs E1-E3 and E6 only, with up to 16 levels and rho = 0.
//
// The computation ("turboquant-pytorch 소개", "1단계" then "2단계"):
// y = Pi x, codes idx_j = #{i : n t_i < y_j},
// r = y - n c[idx] (rotated frame, unnormalised), rho = ||r||,
// z = [M r >= 0] with M = S Pi^T, so that sign(M r) = sign(S (x - n Pi^T c[idx])).
//
// Exactness of the two contractions on fp16/bf16 tensor cores (fp32 accumulate):
//  E2  keys are exact in their own 16-bit type; Pi is split Pi = Pi_hi + Pi_lo
//      in that type (fp16: Pi_lo is mostly subnormal, still exact to 2^-24),
//      so Y = X Pi_hi^T + X Pi_lo^T carries ~2^-17 relative error or better;
//  E5  the residual and M are split in bf16: P = R_hi M_hi^T + R_hi M_lo^T +
//      R_lo M_hi^T (the dropped R_lo M_lo^T term is ~2^-18 relative).
//
// Work per CTA (persistent, one CTA per SM, 128 keys = one packed block per tile):
//  warp 0      TMA producer: key tiles (K-major, 128-byte swizzle) into a
//              2-stage ring; once, the swizzled images of Pi_hi/lo and M_hi/lo.
//  warp 1      TMEM owner (512 columns) and E2 issuer;
//  warp 10     E5 issuer.  Two issuers, because one issuing warp puts out a
//              tcgen05.mma only every ~50-80 cycles and E5 of tile i must not
//              wait behind E2 of tile i + 1.  Each issuer warp runs its loop
//              converged and one elected lane issues.
//  warps 2-9   two epilogue warpgroups; tile i goes to warpgroup i % 2, which
//              owns TMEM columns [256 b, 256 b + 256): Y/R in the first 128
//              (the bf16 residual split is written back over the Y columns it
//              was computed from and is the A operand of E5), P in the last 128.
//              Thread (warp w, lane l) owns key row 32 (w % 4) + l.
// Every wait is bounded: on expiry the kernel raises the plan's error word,
// drains what it issued and frees its TMEM.
#include <cuda.h>

#include "ptx_sm100.cuh"
#include "tq_internal.cuh"

namespace tq {
namespace {

using namespace ptx;

constexpr int kThreads = 352;
constexpr int kE5Warp = 10;
constexpr int kStages = 2;
constexpr uint32_t kOpBytes = 128 * 128 * 2;  // one 128 x 128 16-bit operand image
constexpr uint32_t kAtomBytes = 128 * 128;    // 128 rows x 64 elements (128 B) per swizzle atom
constexpr uint32_t kOffPiHi = 0, kOffPiLo = kOpBytes, kOffMHi = 2 * kOpBytes, kOffMLo = 3 * kOpBytes;
constexpr uint32_t kOffX = 4 * kOpBytes;
constexpr uint32_t kOffBar = kOffX + kStages * kOpBytes;
enum {
  BAR_OPS = 0,
  BAR_XFULL = 1,
  BAR_XEMPTY = BAR_XFULL + kStages,
  BAR_YFULL = BAR_XEMPTY + kStages,
  BAR_RFULL = BAR_YFULL + 2,       // [stage][half]: residual of coordinates 64 h .. 64 h + 63 written
  BAR_PFULL = BAR_RFULL + 4,
  BAR_ACCEMPTY = BAR_PFULL + 2,
  BAR_DONE = BAR_ACCEMPTY + 2,
  BAR_DONE5 = BAR_DONE + 1,
  BAR_COUNT = BAR_DONE5 + 1
};
constexpr uint32_t kSmemBytes = kOffBar + BAR_COUNT * 8 + 16 + 1024;  // + slot, + alignment slack

struct EncTcArgs {
  Layout lay;
  CodeParams cp;
  ParityExpansion px;
  int64_t G, N, nb, n_tiles;
  const uint8_t* pi_hi;
  const uint8_t* pi_lo;
  const uint8_t* m_hi;
  const uint8_t* m_lo;
  uint8_t* packed;
  int* err;
  // 1 for a Walsh-Hadamard plan: the rotation is one exact product with the
  // +-1 matrix (pi_hi), whose scale c is folded into cp, px and M; rho = c ||r'||
  int e2_single;
  float rho_scale;
  // fractional width: coordinates 64..127 use the lower codebook (padded to
  // the same number of code bits; its top bit is never set), and code plane
  // K - 1 is stored as a half plane (coordinates 0..63, 8 bytes per token)
  int frac;
  CodeParams cp_lo;
  ParityExpansion px_lo;
  // error-path self-test only (tq_selftest_encode_drain): CTA 0's producer
  // withholds the copy of its first key tile, so the waits on it run out
  int drop_first;
};

__device__ __forceinline__ void raise(int* err, volatile int* abort) {
  *abort = 1;
  atomicExch(err, 1);
}

template <bool kBF16>
__device__ __forceinline__ float2 pair_to_float2(uint32_t w) {
  if constexpr (kBF16) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  } else {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  }
}

// PX: the codebook's parity expansion has the odd-weight masks of a symmetric
// codebook ({1}, {1, 2} or {1, 2, 4, 7}); the centroid n c[idx] is then summed
// from the code bits' sign words (one LOP3 and one FADD per term) instead of
// selected threshold by threshold.
template <int L, bool kBF16, bool PX, bool PROD>
__global__ void __launch_bounds__(kThreads, 1)
encode_tc_kernel(const __grid_constant__ CUtensorMap tmX, const EncTcArgs a) {
  constexpr int K = L == 2 ? 1 : L == 4 ? 2 : L == 8 ? 3 : 4;  // code planes
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(smem);
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  auto bar = [&](int i) { return sb + kOffBar + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar(BAR_OPS), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(BAR_XFULL + s), 1);
      mbar_init(bar(BAR_XEMPTY + s), 1 + 128);  // MMA commit + the owning warpgroup's norm pass
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(BAR_YFULL + b), 1);
      mbar_init(bar(BAR_RFULL + 2 * b), 128);
      mbar_init(bar(BAR_RFULL + 2 * b + 1), 128);
      mbar_init(bar(BAR_PFULL + b), 1);
      mbar_init(bar(BAR_ACCEMPTY + b), 128);
    }
    mbar_init(bar(BAR_DONE), 1);
    mbar_init(bar(BAR_DONE5), 1);
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
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tmX);
      mbar_arrive_expect_tx(bar(BAR_OPS), (PROD ? 4 : 2) * kOpBytes);
      bulk_load(sb + kOffPiHi, a.pi_hi, kOpBytes, bar(BAR_OPS));
      bulk_load(sb + kOffPiLo, a.pi_lo, kOpBytes, bar(BAR_OPS));
      if constexpr (PROD) {
        bulk_load(sb + kOffMHi, a.m_hi, kOpBytes, bar(BAR_OPS));
        bulk_load(sb + kOffMLo, a.m_lo, kOpBytes, bar(BAR_OPS));
      }
      int64_t issued = 0, withheld = -1;
      for (int64_t i = 0; i < n_my; ++i) {
        const int s = (int)(i % kStages);
        const uint32_t use = (uint32_t)(i / kStages);
        if (!mbar_wait_suspend(bar(BAR_XEMPTY + s), (use & 1) ^ 1, abort)) {
          raise(a.err, abort);
          break;
        }
        if (i == 0 && a.drop_first && blockIdx.x == 0) {  // self-test: no copy, no arrival
          withheld = 0;
          issued = 1;
          continue;
        }
        const int64_t tile = blockIdx.x + i * gridDim.x;
        const int64_t g = tile / a.nb, blk = tile % a.nb;
        const int32_t row = (int32_t)(g * a.N + blk * kTokensPerBlock);
        mbar_arrive_expect_tx(bar(BAR_XFULL + s), kOpBytes);
        tma_load_2d(sb + kOffX + s * kOpBytes, &tmX, 0, row, bar(BAR_XFULL + s));
        tma_load_2d(sb + kOffX + s * kOpBytes + kAtomBytes, &tmX, 64, row, bar(BAR_XFULL + s));
        issued = i + 1;
      }
      // no copy may still be landing when the CTA exits: wait for the last loads
      int dummy = 0;
      for (int64_t i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
        if (i != withheld) mbar_wait(bar(BAR_XFULL + (int)(i % kStages)), (uint32_t)(i / kStages) & 1, &dummy);
      mbar_wait(bar(BAR_OPS), 0, &dummy);
    }
  } else if (warp == 1 || warp == kE5Warp) {
    // ------------------------------------------------------------ MMA issuers
    // The whole warp runs the loop (its operands stay warp-uniform); one
    // elected lane issues each MMA and commit.
    {
      constexpr uint32_t idesc_x = idesc_f16(kBF16 ? 1u : 0u, 128, 128);
      constexpr uint32_t idesc_r = idesc_f16(1u, 128, 128);
      const bool e2 = warp == 1;
      // shared-memory descriptors computed once: every MMA below takes one of
      // these plus a compile-time offset (descriptor units of 16 B), so the
      // issuing thread does no address arithmetic between MMAs
      const uint64_t dx0 = sdesc_k_sw128(sb + kOffX), dpih = sdesc_k_sw128(sb + kOffPiHi),
                     dpil = sdesc_k_sw128(sb + kOffPiLo), dmh = sdesc_k_sw128(sb + kOffMHi),
                     dml = sdesc_k_sw128(sb + kOffMLo);
      const int64_t n_iss = (PROD || e2) ? n_my : 0;  // MSE has no E5
      bool ok = __all_sync(0xffffffffu, mbar_wait_suspend(bar(BAR_OPS), 0, abort));
      for (int64_t i = 0; ok && i < n_iss; ++i) {
        const int b = (int)(i & 1);
        const uint32_t j = (uint32_t)(i >> 1);
        if (e2) {
          // E2: Y = X Pi^T, Pi split hi + lo
          const int s = (int)(i % kStages);
          if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(BAR_XFULL + s), (uint32_t)(i / kStages) & 1, abort) &&
                                           mbar_wait_suspend(bar(BAR_ACCEMPTY + b), (j & 1) ^ 1, abort))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + 256u * b;
          const uint64_t dx = dx0 + (uint64_t)(((uint32_t)s * kOpBytes) >> 4);
#pragma unroll
          for (int kb = 0; kb < 8; ++kb) {
            const uint32_t off16 = ((kb >> 2) * kAtomBytes + (kb & 3) * 32) >> 4;
            mma_f16_ss_w(d, dx + off16, dpih + off16, idesc_x, kb > 0);
            if (!a.e2_single) mma_f16_ss_w(d, dx + off16, dpil + off16, idesc_x, 1);
          }
          mma_commit_w(bar(BAR_YFULL + b));
          mma_commit_w(bar(BAR_XEMPTY + s));
        } else {
          // E5: P = R' M^T with R' = R_hi + R_lo and M = M_hi + M_lo (bf16), R_lo M_lo dropped;
          // the first 64 coordinates' MMAs start while the epilogue still
          // quantises the last 64
          const uint32_t r = tmem + 256u * b, d = r + 128;
#pragma unroll
          for (int kb = 0; kb < 8; ++kb) {
            if ((kb & 3) == 0) {
              if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(BAR_RFULL + 2 * b + (kb >> 2)), j & 1, abort))) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            const uint32_t off16 = ((kb >> 2) * kAtomBytes + (kb & 3) * 32) >> 4;
            const uint32_t a_hi = r + 32 * (kb >> 1) + 8 * (kb & 1), a_lo = a_hi + 16;
            mma_f16_ts_w(d, a_hi, dmh + off16, idesc_r, kb > 0);
            mma_f16_ts_w(d, a_hi, dml + off16, idesc_r, 1);
            mma_f16_ts_w(d, a_lo, dmh + off16, idesc_r, 1);
          }
          if (!ok) break;
          mma_commit_w(bar(BAR_PFULL + b));
        }
      }
      if (!ok && lane == 0) raise(a.err, abort);
      // all issued MMAs complete before TMEM is freed
      const int done = e2 ? BAR_DONE : BAR_DONE5;
      mma_commit_w(bar(done));
      int dummy = 0;
      mbar_wait(bar(done), 0, &dummy);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int wg = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16) + 256u * wg;
    for (int64_t i = wg; i < n_my; i += 2) {
      const int s = (int)(i % kStages);
      const uint32_t j = (uint32_t)(i >> 1);
      const int64_t tile = blockIdx.x + i * gridDim.x;
      const int64_t blk = tile % a.nb;
      const bool live = blk * kTokensPerBlock + row < a.N;

      // E1: ||x|| from the staged key row (two 128-byte-swizzled K halves)
      // every lane polls; the warp proceeds (or gives up) as one, because the
      // tcgen05 loads and stores below are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(BAR_XFULL + s), (uint32_t)(i / kStages) & 1, abort))) {
        raise(a.err, abort);
        break;
      }
      float n2;
      {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const uint8_t* xr = smem + kOffX + s * kOpBytes + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 q = *reinterpret_cast<const uint4*>(xr + h * kAtomBytes + ((c ^ (row & 7)) << 4));
            const float2 f0 = pair_to_float2<kBF16>(q.x), f1 = pair_to_float2<kBF16>(q.y);
            const float2 f2 = pair_to_float2<kBF16>(q.z), f3 = pair_to_float2<kBF16>(q.w);
            acc[0] = fmaf(f0.x, f0.x, acc[0]);
            acc[1] = fmaf(f0.y, f0.y, acc[1]);
            acc[2] = fmaf(f1.x, f1.x, acc[2]);
            acc[3] = fmaf(f1.y, f1.y, acc[3]);
            acc[4] = fmaf(f2.x, f2.x, acc[4]);
            acc[5] = fmaf(f2.y, f2.y, acc[5]);
            acc[6] = fmaf(f3.x, f3.x, acc[6]);
            acc[7] = fmaf(f3.y, f3.y, acc[7]);
          }
        }
        n2 = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
      }
      mbar_arrive(bar(BAR_XEMPTY + s));
      const float n = sqrtf(n2);
      // thresholds scaled by n (a zero key compares 0 with the unscaled
      // boundaries: idx = #{t_i < 0}); centroids scaled by n
      const float sc = n > 0.f ? n : 1.f;
      float nt[L - 1], nc[L];
      // signed-form terms: -n half[t] as bits (the sign flips where the term's
      // parity is 1), and n mid
      constexpr int NT = K == 1 ? 1 : K == 2 ? 2 : 4;
      uint32_t nhalf[NT];
      float nmid;
      // the constants of one codebook (the lower one for coordinates 64..127
      // of a fractional width)
      auto set_codebook = [&](const CodeParams& cp, const ParityExpansion& px) {
#pragma unroll
        for (int q = 0; q < L - 1; ++q) nt[q] = sc * cp.t[q];
#pragma unroll
        for (int q = 0; q < L; ++q) nc[q] = n * cp.c[q];
#pragma unroll
        for (int t = 0; t < NT; ++t) nhalf[t] = __float_as_uint(-(n * px.half[t]));
        nmid = n * px.mid;
      };
      set_codebook(a.cp, a.px);

      // E2 result -> E3 codes, E4 residual; the residual's bf16 split goes back
      // into the same TMEM columns as the A operand of E5
      if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(BAR_YFULL + wg), j & 1, abort))) {
        raise(a.err, abort);
        break;
      }
      tc_fence_after();
      // plane words of the four 32-coordinate chunks shift through pl[p][0..3]
      // (the chunk loop is not unrolled: the unrolled body overflows the
      // instruction cache)
      uint32_t pl[K][4];
#pragma unroll
      for (int p = 0; p < K; ++p) pl[p][0] = pl[p][1] = pl[p][2] = pl[p][3] = 0;
      float rr = 0.f;
      // one 32-coordinate chunk: codes into pl (shifted in), residual split
      // written back over the chunk's own Y columns
      auto chunk = [&](const uint32_t (&v)[32], int cc) {
        uint32_t w[K];
#pragma unroll
        for (int p = 0; p < K; ++p) w[p] = 0;
        uint32_t hi[16], lo[16];
        // coordinates from 31 down to 0: each funnel shift appends one bit, so
        // coordinate e ends at bit e
#pragma unroll
        for (int e = 30; e >= 0; e -= 2) {
          float r2[2];
#pragma unroll
          for (int u = 1; u >= 0; --u) {
            const float y = __uint_as_float(v[e + u]);
            // sb[q] = n t_q - y: its sign bit is [y > n t_q] (a tie gives +0)
            uint32_t sbit[L - 1];
            float cv = nc[0];
#pragma unroll
            for (int q = 0; q < L - 1; ++q) {
              sbit[q] = __float_as_uint(nt[q] - y);
              if constexpr (!PX) cv = (int)sbit[q] < 0 ? nc[q + 1] : cv;
            }
            // bit p of idx = #{q : y > n t_q} is the XOR of the sign bits of
            // the thresholds q with (q + 1) % 2^p == 0 (the count is monotone)
            uint32_t xb[K];
#pragma unroll
            for (int p = 0; p < K; ++p) {
              uint32_t x = 0;
#pragma unroll
              for (int q = 0; q < L - 1; ++q)
                if (((q + 1) & ((1 << p) - 1)) == 0) x ^= sbit[q];
              xb[p] = x;
              w[p] = __funnelshift_l(x, w[p], 1);
            }
            if constexpr (PX) {
              // term t contributes +n half[t] where its parity (bit 31 of the
              // XOR of its bits' sign words) is 1, else -n half[t]
              constexpr uint32_t kS = 0x80000000u;
              cv = nmid + __uint_as_float(nhalf[0] ^ (xb[0] & kS));
              if constexpr (K >= 2) cv += __uint_as_float(nhalf[1] ^ (xb[1] & kS));
              if constexpr (K == 3) {
                cv += __uint_as_float(nhalf[2] ^ (xb[2] & kS));
                cv += __uint_as_float(nhalf[3] ^ ((xb[0] ^ xb[1] ^ xb[2]) & kS));
              }
            }
            if constexpr (PROD) {
              const float rv = y - cv;
              rr = fmaf(rv, rv, rr);
              r2[u] = rv;
            }
          }
          if constexpr (PROD) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(r2[0], r2[1]);
            const float2 hf = __bfloat1622float2(h);
            const __nv_bfloat162 l = __floats2bfloat162_rn(r2[0] - hf.x, r2[1] - hf.y);
            hi[e >> 1] = *reinterpret_cast<const uint32_t*>(&h);
            lo[e >> 1] = *reinterpret_cast<const uint32_t*>(&l);
          }
        }
        if constexpr (PROD) {
          tmem_st16(t_lane + 32 * cc, hi);
          tmem_st16(t_lane + 32 * cc + 16, lo);
        }
#pragma unroll
        for (int p = 0; p < K; ++p) {
          pl[p][0] = pl[p][1];
          pl[p][1] = pl[p][2];
          pl[p][2] = pl[p][3];
          pl[p][3] = w[p];
        }
      };
      // the next chunk's TMEM load is in flight while a chunk is processed
      uint32_t va[32], vb[32];
      tmem_ld32(t_lane, va);
      tmem_ld_wait();
#pragma unroll 1
      for (int cc = 0; cc < 4; cc += 2) {
        if (cc == 2 && a.frac) set_codebook(a.cp_lo, a.px_lo);
        tmem_ld32(t_lane + 32 * (cc + 1), vb);
        chunk(va, cc);
        tmem_ld_wait();
        if (cc + 2 < 4) tmem_ld32(t_lane + 32 * (cc + 2), va);
        chunk(vb, cc + 1);
        if constexpr (PROD) {
          // this half of the residual is in TMEM: E5 may start on it
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(BAR_RFULL + 2 * wg + (cc >> 1)));
        }
        if (cc + 2 < 4) tmem_ld_wait();
      }
      const float rho = PROD ? sqrtf(rr) * a.rho_scale : 0.f;

      uint32_t zs[4] = {0u, 0u, 0u, 0u};
      if constexpr (PROD) {
        // E5 result -> sign plane
        if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(BAR_PFULL + wg), j & 1, abort))) {
          raise(a.err, abort);
          break;
        }
        tc_fence_after();
        uint32_t v[4][32];
        tmem_ld32(t_lane + 128, v[0]);
        tmem_ld32(t_lane + 160, v[1]);
        tmem_ld32(t_lane + 192, v[2]);
        tmem_ld32(t_lane + 224, v[3]);
        tmem_ld_wait();
        // shift in the sign bits (coordinate e at bit e), then invert: z = [p >= 0]
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t z = 0;
#pragma unroll
          for (int e = 31; e >= 0; --e) z = __funnelshift_l(v[cc][e], z, 1);
          zs[cc] = n > 0.f ? ~z : 0xFFFFFFFFu;
        }
      }
      // (MSE: every Y column has been read) the accumulator is free
      tc_fence_before();
      mbar_arrive(bar(BAR_ACCEMPTY + wg));

      // E6: this key's 16-byte chunks and norms (consecutive rows -> consecutive 16 B)
      uint8_t* out = a.packed + tile * a.lay.block_bytes;
#pragma unroll
      for (int p = 0; p < K; ++p) {
        if (p == K - 1 && a.frac) {  // the half plane: coordinates 0..63
          *reinterpret_cast<uint2*>(out + a.lay.top_off + row * 8) =
              live ? make_uint2(pl[p][0], pl[p][1]) : make_uint2(0, 0);
          continue;
        }
        const uint4 val = live ? make_uint4(pl[p][0], pl[p][1], pl[p][2], pl[p][3])
                               : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(out + ((int64_t)p * kTokensPerBlock + row) * 16) = val;
      }
      if constexpr (PROD)
        *reinterpret_cast<uint4*>(out + a.lay.sign_off + row * 16) =
            live ? make_uint4(zs[0], zs[1], zs[2], zs[3]) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<float2*>(out + a.lay.norms_off + row * 8) = live ? make_float2(n, rho) : make_float2(0.f, 0.f);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// The expansion's masks are those of a symmetric codebook with k code bits.
bool odd_masks(const ParityExpansion& px, int k) {
  static const uint32_t want[3][4] = {{1u}, {1u, 2u}, {1u, 2u, 4u, 7u}};
  const int n = k == 3 ? 4 : k;
  if (k < 1 || k > 3 || px.n != n) return false;
  for (int i = 0; i < n; ++i)
    if (px.mask[i] != want[k - 1][i]) return false;
  return true;
}

template <int L, bool kBF16, bool PX, bool PROD>
cudaError_t launch_tc(const tq_plan* p, const void* keys, int64_t G, int64_t N, uint8_t* packed, cudaStream_t s,
                      bool drop_first) {
  CUtensorMap tm;
  const cudaError_t te = make_tmap_2d(&tm, kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                                      keys, 128, (uint64_t)(G * N), 256, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  if (te != cudaSuccess) return te;
  EncTcArgs a;
  a.lay = p->lay;
  a.cp = p->cp_enc;
  a.px = p->px_enc;
  a.e2_single = p->hadamard;
  a.rho_scale = p->rot_scale;
  a.frac = p->lay.frac;
  a.cp_lo = p->cp_enc_lo;
  a.px_lo = p->px_enc_lo;
  a.G = G;
  a.N = N;
  a.nb = (N + kTokensPerBlock - 1) / kTokensPerBlock;
  a.n_tiles = G * a.nb;
  const uint8_t* ops = p->tc_ops;
  a.pi_hi = ops + (kBF16 ? 2 : 0) * kOpBytes;
  a.pi_lo = ops + (kBF16 ? 3 : 1) * kOpBytes;
  a.m_hi = PROD ? ops + 4 * kOpBytes : nullptr;  // an MSE plan holds the Pi images only
  a.m_lo = PROD ? ops + 5 * kOpBytes : nullptr;
  a.packed = packed;
  a.err = p->err;
  a.drop_first = drop_first ? 1 : 0;
  auto kern = encode_tc_kernel<L, kBF16, PX, PROD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t grid = a.n_tiles < sms ? a.n_tiles : sms;
  kern<<<(unsigned)grid, kThreads, kSmemBytes, s>>>(tm, a);
  return cudaGetLastError();
}

}  // namespace

bool encode_tc_supported(const tq_plan* p, tq_dtype dt) {
  return p->tc_ops != nullptr && p->d == 128 && (dt == TQ_F16 || dt == TQ_BF16) && p->cp.L >= 2 &&
         p->cp.L <= (p->lay.prod ? 8 : 16);
}

cudaError_t launch_encode_tc(const tq_plan* p, const void* keys, tq_dtype dt, int64_t G, int64_t N, uint8_t* packed,
                             cudaStream_t s, bool drop_first) {
  const bool bf = dt == TQ_BF16;
  const int k = p->cp.L == 2 ? 1 : p->cp.L == 4 ? 2 : p->cp.L == 8 ? 3 : 4;
  const bool px = odd_masks(p->px, k);
  const bool prod = p->lay.prod != 0;
#define TQ_ENC_CASE(LV, PR)                                                                                    \
  if (px) return bf ? launch_tc<LV, true, true, PR>(p, keys, G, N, packed, s, drop_first)                                  \
                    : launch_tc<LV, false, true, PR>(p, keys, G, N, packed, s, drop_first);                                \
  return bf ? launch_tc<LV, true, false, PR>(p, keys, G, N, packed, s, drop_first)                                         \
            : launch_tc<LV, false, false, PR>(p, keys, G, N, packed, s, drop_first);
  switch (p->cp.L) {
    case 2:
      if (prod) { TQ_ENC_CASE(2, true) }
      TQ_ENC_CASE(2, false)
    case 4:
      if (prod) { TQ_ENC_CASE(4, true) }
      TQ_ENC_CASE(4, false)
    case 8:
      if (prod) { TQ_ENC_CASE(8, true) }
      TQ_ENC_CASE(8, false)
    case 16:  // 4-bit MSE codebooks: no parity expansion of that size
      if (!prod) return bf ? launch_tc<16, true, false, false>(p, keys, G, N, packed, s, drop_first)
                           : launch_tc<16, false, false, false>(p, keys, G, N, packed, s, drop_first);
      break;
  }
#undef TQ_ENC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace tq
