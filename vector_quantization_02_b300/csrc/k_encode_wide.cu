// Encode on the tensor cores for any head dimension d (a multiple of 128) and
// any key dtype: the shape of a vector-search index (10^6 fp32 keys of
// d = 1536), where the two d x d projections are long dense contractions.
// TurboQuantProd runs both projections; TurboQuantMSE ("turboquant-pytorch
// 소개", "1단계" alone) runs E2 only and stores ||r|| = 0 with no sign plane.
//
// Same computation as the other encode kernels ("turboquant-pytorch 소개",
// "1단계" then "2단계"): y = Pi x, codes idx_j = #{i : n t_i < y_j},
// r = y - n c[idx] (rotated frame, unnormalised), rho = ||r||,
// z = [M r >= 0] with M = S Pi^T.
//
// Exactness on fp16 tensor cores (fp32 accumulate): every operand is split
// into an fp16 pair v = hi + lo (22 significant bits) and each product is
// issued three times (hi hi, hi lo, lo hi; lo lo is ~2^-22 of a term).  At
// d = 1536 the error of y reaches p = M r amplified by the norm of M's rows
// (~d^1/2), so the operands carry powers of two that keep every lo part in
// fp16's normal range: the key enters as u = 2^8 x / ||x|| (the loaders sum
// ||x||^2 over the row first), Pi as 2^8 Pi, so Y = 2^16 Pi u, compared with
// 2^16 t; the residual enters E5 as 2^10 r'.  Signs do not see the scales.
//
// A tile is 128 keys (one packed block).  Its work is a sequence of jobs,
// each 128 keys x 128 coordinates (one chunk) over K = d in stages of 64
// coordinates, accumulated in TMEM per 128-coordinate slice of K and summed in
// fp32 by the epilogue (one tensor-core accumulator over K = 1536 loses too
// much):
//   d / NC E2 jobs  Y[:, chunk] = X Pi[chunk]^T, then quantised: code bits
//                   into the packed block, the residual's split into the
//                   cluster's scratch rows,
//   d / NC E5 jobs  P[:, chunk] = R M[chunk]^T, then the sign bits.
// A thread-block cluster of CL CTAs (one per SM) works on each tile: CTA r
// takes the chunks r, r + CL, ...  Every job re-reads the whole key tile (E2)
// or residual tile (E5); shared by the cluster, the tiles being worked on fit
// in L2, and those re-reads stay out of DRAM.  The CTAs meet twice per tile:
// every CTA's residual columns are written before any CTA's E5 stages load the
// residual (a barrier each CTA arrives on in every CTA), and rank 0 adds the
// CTAs' partial ||r||^2 (sent to its shared memory) into rho.
// The scratch slot of a cluster is its rank-0 SM's id: this kernel needs a
// whole SM (all 512 TMEM columns, more than half of the shared memory), so no
// two of its CTAs, from any launch, share one at a time.
// ||x|| comes from a pre-pass (key_norm_kernel) that writes it into the packed
// block's norm slot.
//  warp 0       producer: TMA loads into a 3-stage shared-memory ring; a stage
//               holds the B operand (hi and lo rows of 2^8 Pi or M for the
//               job's 128 columns, 64 coordinates, 128-byte swizzle) and the A
//               source: the key tile (E2) or the residual tile from the scratch
//               (E5, read by the MMA straight from shared memory).
//  warp 1       TMEM owner (two partial accumulators in [0, 256), the E2 key
//               operand of each ring stage in [256, 448)) and MMA issuer (the
//               warp runs the loop converged, one elected lane issues): one
//               wait and one commit per stage of 12 MMAs.
//  warps 2-5    E2 key operand: thread (warp w, lane l) owns key row
//               32 (w % 4) + l; per stage it reads its 64 coordinates from the
//               staged key tile and writes u = 2^8 x / ||x|| as fp16 hi, lo into
//               the stage's TMEM columns.
//  warps 6-13   epilogue: two warpgroups, each taking half of a job's columns.
// Every wait is bounded: on expiry the kernel raises the plan's error word,
// drains what it issued and frees its TMEM; the CTAs of a cluster leave
// together.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx_sm100.cuh"
#include "tq_internal.cuh"

namespace tq {
namespace {

using namespace ptx;

constexpr int kEThreads = 448;
constexpr int kEpiWarp0 = 6;       // warps 2-5 load the A operand
constexpr int kStages = 3;         // shared-memory ring (B operand + A source)
constexpr uint32_t kPartBytes = 128 * 128;  // 128 rows x 64 16-bit values (one 128-byte swizzle row each)
constexpr uint32_t kStageBytes = 4 * kPartBytes;  // B hi, B lo, A source (two parts): 64 KB
constexpr int kStageK = 64;        // coordinates per stage
constexpr int kARing = 256;        // first TMEM column of the E2 key operand, one slot per ring stage
constexpr int kAPartCols = 32;     // TMEM columns of one A part per stage (64 16-bit values)
constexpr int kSliceCols = 128;    // output columns of a job (two partial accumulators of 128 columns)
constexpr int kSliceStages = 2;    // stages (128 coordinates of K) per partial accumulator
constexpr int kMaxCluster = 4;     // CTAs per cluster at most

enum {
  BAR_FULL = 0,                       // E5 stage landed: B operand and residual tile (only E5 fills advance it)
  BAR_XFULL = BAR_FULL + kStages,     // E2 stage landed: B operand and key tile (only E2 fills advance it)
  BAR_EMPTY = BAR_XFULL + kStages,
  BAR_AFULL = BAR_EMPTY + kStages,    // E2 key operand of the stage written to TMEM
  BAR_DFULL = BAR_AFULL + kStages,    // [2] partial accumulators
  BAR_DEMPTY = BAR_DFULL + 2,
  BAR_RREADY = BAR_DEMPTY + 2,
  BAR_RHO = BAR_RREADY + 1,
  BAR_DONE = BAR_RHO + 1,
  BAR_COUNT = BAR_DONE + 1
};

struct EncWideArgs {
  Layout lay;
  CodeParams cp;
  ParityExpansion px;
  int NC, J, S;               // chunk columns, jobs per phase, stages per job
  int CL;                     // CTAs per cluster (a divisor of J): CTA r of a cluster takes chunks r, r + CL, ...
  int nslots;                 // scratch slots (SM ids)
  int64_t G, N, nb, n_tiles;
  const void* keys;
  uint8_t* packed;
  void* scratch;              // [slot][2][128][d] fp16 residual 2^10 r' hi, lo
  int* err;
};

__device__ __forceinline__ void raise(int* err, volatile int* abort) {
  *abort = 1;
  atomicExch(err, 1);
}


__device__ __forceinline__ uint32_t smid() {
  uint32_t v;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(v));
  return v;
}

// compensated sum (Neumaier) of squares
struct KSum {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float v = x * x;
    const float t = s + v;
    c += fabsf(s) >= fabsf(v) ? (s - t) + v : (v - t) + s;
    s = t;
  }
};

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// fp16 hi + lo words of the pairs (a0, a1)
__device__ __forceinline__ void split_h2(float a0, float a1, uint32_t& hi, uint32_t& lo) {
  hi = pack_h2(a0, a1);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  lo = pack_h2(a0 - f.x, a1 - f.y);
}

template <int DT>
__device__ __forceinline__ float2 key_pair(uint32_t w) {
  if constexpr (DT == 1) return __half22float2(*reinterpret_cast<const __half2*>(&w));
  else return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
}

constexpr float kYScale = 65536.f;      // Y = 2^16 Pi u
constexpr float kRScale = 1.f / 64.f;   // E5 operand 2^10 r' = 2^-6 (2^16 r')

// DT: key dtype, 0 fp32, 1 fp16, 2 bf16.
template <int L, int DT, bool PX, bool PROD>
__global__ void __launch_bounds__(kEThreads, 1)
encode_wide_kernel(const __grid_constant__ CUtensorMap tmPi, const __grid_constant__ CUtensorMap tmM,
                   const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmR,
                   const EncWideArgs a) {
  constexpr int K = L == 2 ? 1 : L == 4 ? 2 : L == 8 ? 3 : 4;  // code planes
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(smem);
  const int d = a.lay.d, NC = a.NC, J = a.J, S = a.S, CL = a.CL;
  const uint32_t rank = cluster_ctarank();
  // this CTA's jobs: its E2 chunks rank, rank + CL, ... (Jm of them), then (Prod)
  // the E5 jobs of the same chunks; the cluster's CTAs share each tile
  const int Jm = J / CL;
  const int MYJOBS = PROD ? 2 * Jm : Jm;
  auto job_of = [&](int t) { return t < Jm ? (int)rank + CL * t : J + (int)rank + CL * (t - Jm); };
  const uint32_t off_bar = kStages * kStageBytes;
  float* s_rr = reinterpret_cast<float*>(smem + off_bar + BAR_COUNT * 8);  // [2][128]
  float* s_rr_peer = s_rr + 256;  // [CL - 1][128] (rank 0): the other CTAs' partial ||r||^2 per row
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ uint32_t s_slot;
  auto bar = [&](int i) { return sb + off_bar + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    s_slot = smid();
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(BAR_FULL + s), 1);
      mbar_init(bar(BAR_XFULL + s), 1);
      mbar_init(bar(BAR_EMPTY + s), 1);
      mbar_init(bar(BAR_AFULL + s), 128);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(BAR_DFULL + b), 1);
      mbar_init(bar(BAR_DEMPTY + b), 256);
    }
    // the residual rows of a tile: every epilogue thread of every CTA of the cluster
    mbar_init(bar(BAR_RREADY), 256 * CL);
    // the tile's ||r||^2 partials: both local warpgroups, and on rank 0 one
    // warpgroup of each other CTA
    mbar_init(bar(BAR_RHO), rank == 0 ? 256 + 128 * (CL - 1) : 256);
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
  // every CTA of the cluster has initialised its barriers before any remote
  // arrival; the cluster's residual scratch slot is rank 0's SM id (no two
  // running CTAs of this kernel share an SM: its shared memory use rules it out)
  cluster_sync_all();
  if (threadIdx.x == 0 && rank != 0) s_slot = ld_cluster_u32(mapa_shared(smem_u32(&s_slot), 0));
  __syncthreads();
  const uint32_t tmem = tmem_slot;
  volatile int* abort = &abort_flag;
  // (Prod) cannot be out of range with a plan built on this device; the same
  // slot, so the same decision, in every CTA of the cluster
  if (PROD && s_slot >= (uint32_t)a.nslots) {
    if (threadIdx.x == 0) raise(a.err, abort);
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
    cluster_sync_all();
    return;
  }
  uint16_t* scr = PROD ? static_cast<uint16_t*>(a.scratch) + (size_t)s_slot * 2 * 128 * d : nullptr;

  // tiles of this cluster: c, c + P, ... (P clusters)
  const int64_t cid = blockIdx.x / CL, P = gridDim.x / CL;
  const int64_t n_my = cid < a.n_tiles ? (a.n_tiles - 1 - cid) / P + 1 : 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmPi);
      prefetch_tmap(&tmM);
      prefetch_tmap(&tmX);
      prefetch_tmap(&tmR);
      constexpr uint32_t kXBytes = DT == 0 ? 2 * kPartBytes : kPartBytes;  // key tile: 128 rows x 64 values
      uint32_t b = 0, ph = 0, issued = 0;
      // per slot: parity of its next E2 fill, of its next E5 fill; its last fill was E2
      uint32_t xmask = 0, fmask = 0, last_e2 = 0;
      bool ok = true;
      for (int64_t i = 0; ok && i < n_my; ++i) {
        const int64_t tile = cid + i * P;
        const int64_t g = tile / a.nb, blk = tile - g * a.nb;
        const int32_t xrow0 = (int32_t)(g * a.N + blk * kTokensPerBlock);
        for (int t = 0; ok && t < MYJOBS; ++t) {
          const int job = job_of(t);
          const bool e2 = t < Jm;
          if (t == Jm) {  // every CTA of the cluster has written its residual columns of this tile
            if (!mbar_wait_suspend_cluster(bar(BAR_RREADY), (uint32_t)i & 1u, abort)) {
              ok = false;
              break;
            }
            // the other CTAs' generic stores, read next by the async proxy
            asm volatile("fence.proxy.async.global;" ::: "memory");
          }
          const CUtensorMap* map = e2 ? &tmPi : &tmM;
          const int row0 = (job % J) * NC;
          for (int st = 0; st < S; ++st) {
            if (!mbar_wait_suspend(bar(BAR_EMPTY + b), ph ^ 1u, abort)) {
              ok = false;
              break;
            }
            const uint32_t base = sb + b * kStageBytes;
            // an E2 stage (B operand and key tile) lands on XFULL, which the
            // key-operand warps wait for; an E5 stage (B operand and residual
            // tile) on FULL, which the issuer waits for
            const uint32_t fb = bar((e2 ? BAR_XFULL : BAR_FULL) + b);
            mbar_arrive_expect_tx(fb, e2 ? 2 * kPartBytes + kXBytes : 4 * kPartBytes);
            tma_load_2d(base, map, st * kStageK, row0, fb);
            tma_load_2d(base + kPartBytes, map, st * kStageK, d + row0, fb);
            if (e2) {
              // fp32 keys: two boxes of 32 values (128-byte rows); 16-bit keys: one of 64
              tma_load_2d(base + 2 * kPartBytes, &tmX, st * kStageK, xrow0, fb);
              if constexpr (DT == 0) tma_load_2d(base + 3 * kPartBytes, &tmX, st * kStageK + 32, xrow0, fb);
              xmask ^= 1u << b;
              last_e2 |= 1u << b;
            } else {
              tma_load_2d(base + 2 * kPartBytes, &tmR, st * kStageK, (int32_t)(s_slot * 256), fb);
              tma_load_2d(base + 3 * kPartBytes, &tmR, st * kStageK, (int32_t)(s_slot * 256 + 128), fb);
              fmask ^= 1u << b;
              last_e2 &= ~(1u << b);
            }
            ++issued;
            if (++b == kStages) {
              b = 0;
              ph ^= 1u;
            }
          }
        }
      }
      if (!ok) raise(a.err, abort);
      // no copy may still be landing when the CTA exits
      int dummy = 0;
      for (uint32_t k = 0; k < (issued < kStages ? issued : kStages); ++k) {
        b = b == 0 ? kStages - 1 : b - 1;
        if ((last_e2 >> b) & 1u)
          mbar_wait(bar(BAR_XFULL + b), ((xmask >> b) & 1u) ^ 1u, &dummy);
        else
          mbar_wait(bar(BAR_FULL + b), ((fmask >> b) & 1u) ^ 1u, &dummy);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (its operands stay warp-uniform); one
    // elected lane issues each MMA and commit.
    {
      const uint32_t idesc = idesc_f16(0u, 128, (uint32_t)NC);
      // ring slot; per slot, parity of its next E2 fill and of its next E5 fill
      uint32_t b = 0, xmask = 0, fmask = 0, cq = 0;
      bool ok = true;
      for (int64_t i = 0; ok && i < n_my; ++i) {
        for (int t = 0; ok && t < MYJOBS; ++t) {
          const bool e2 = t < Jm;
          // K in slices of 128 coordinates, each into a fresh partial accumulator
          for (int c = 0; ok && c < S / kSliceStages; ++c, ++cq) {
            const uint32_t pb = cq & 1u, d_acc = tmem + pb * kSliceCols;
            if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(BAR_DEMPTY + pb), ((cq >> 1) & 1u) ^ 1u, abort))) {
              ok = false;
              break;
            }
            for (int st = 0; st < kSliceStages; ++st) {
              // E2: the key-operand warps saw the stage land and wrote its
              // A operand (one wait covers both); E5: the stage landed
              const bool got = e2 ? mbar_wait_suspend(bar(BAR_AFULL + b), (xmask >> b) & 1u, abort)
                                  : mbar_wait_suspend(bar(BAR_FULL + b), (fmask >> b) & 1u, abort);
              if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t bq = sb + b * kStageBytes;
              const uint32_t at = tmem + kARing + b * (2 * kAPartCols);
              // k steps of 16 values: 32 bytes within the 128-byte swizzle rows
              // (descriptor address units of 16 bytes)
              const uint64_t bh0 = sdesc_k_sw128(bq), bl0 = sdesc_k_sw128(bq + kPartBytes);
              const uint64_t rh0 = sdesc_k_sw128(bq + 2 * kPartBytes), rl0 = sdesc_k_sw128(bq + 3 * kPartBytes);
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                const uint64_t b_hi = bh0 + 2u * ks, b_lo = bl0 + 2u * ks;
                const uint32_t acc = (st == 0 && ks == 0) ? 0u : 1u;
                if (e2) {
                  const uint32_t a_hi = at + 8 * ks, a_lo = at + kAPartCols + 8 * ks;
                  mma_f16_ts_w(d_acc, a_hi, b_hi, idesc, acc);
                  mma_f16_ts_w(d_acc, a_hi, b_lo, idesc, 1u);
                  mma_f16_ts_w(d_acc, a_lo, b_hi, idesc, 1u);
                } else {
                  const uint64_t r_hi = rh0 + 2u * ks, r_lo = rl0 + 2u * ks;
                  mma_f16_ss_w(d_acc, r_hi, b_hi, idesc, acc);
                  mma_f16_ss_w(d_acc, r_hi, b_lo, idesc, 1u);
                  mma_f16_ss_w(d_acc, r_lo, b_hi, idesc, 1u);
                }
              }
              // frees the slot's shared memory and its TMEM A columns: the
              // key-operand warps rewrite those only after the slot's next
              // fill lands, which the producer issues after this commit
              mma_commit_w(bar(BAR_EMPTY + b));
              if (e2)
                xmask ^= 1u << b;
              else
                fmask ^= 1u << b;
              if (++b == kStages) b = 0;
            }
            if (!ok) break;
            mma_commit_w(bar(BAR_DFULL + pb));
          }
        }
      }
      if (!ok && lane == 0) raise(a.err, abort);
      mma_commit_w(bar(BAR_DONE));
      int dummy = 0;
      mbar_wait(bar(BAR_DONE), 0, &dummy);
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------------ E2 key operand
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16) + kARing;
    uint32_t b = 0, xmask = 0;  // ring slot, per-slot parity of its next E2 fill
    bool ok = true;
    for (int64_t i = 0; ok && i < n_my; ++i) {
      const int64_t tile = cid + i * P;
      // ||x|| from the pre-pass (0 for padded rows, whose staged rows may hold
      // another group's keys)
      const float n = *reinterpret_cast<const float*>(a.packed + tile * a.lay.block_bytes + a.lay.norms_off + row * 8);
      const float inv = n > 0.f ? 256.f / n : 0.f;
      for (int t = 0; ok && t < Jm * S; ++t) {
        // the stage landed; its TMEM A columns are free (the MMAs that last
        // read them completed before the producer refilled the slot)
        if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(BAR_XFULL + b), (xmask >> b) & 1u, abort))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* xs = smem + b * kStageBytes + 2 * kPartBytes;
        const uint32_t col = t_lane + b * (2 * kAPartCols);
        // 128-byte rows, 16-byte chunk c at position c ^ (row % 8); values in
        // two halves of 32, each one 16-column TMEM store per part
#pragma unroll
        for (int hv = 0; hv < 2; ++hv) {
          uint32_t hi[16], lo[16];
          if constexpr (DT == 0) {
            // fp32: half hv is its own box of 32 values
            const uint8_t* xr = xs + hv * kPartBytes + row * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const float4 f = *reinterpret_cast<const float4*>(xr + ((c ^ (row & 7)) << 4));
              split_h2(f.x * inv, f.y * inv, hi[2 * c], lo[2 * c]);
              split_h2(f.z * inv, f.w * inv, hi[2 * c + 1], lo[2 * c + 1]);
            }
          } else {
            // 16-bit: chunks 4 hv .. 4 hv + 3 of the row (8 values each)
            const uint8_t* xr = xs + row * 128;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              const int c = 4 * hv + cc;
              const uint4 w = *reinterpret_cast<const uint4*>(xr + ((c ^ (row & 7)) << 4));
              const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 f = key_pair<DT>(ws[e]);
                split_h2(f.x * inv, f.y * inv, hi[4 * cc + e], lo[4 * cc + e]);
              }
            }
          }
          tmem_st16(col + 16 * hv, hi);
          tmem_st16(col + kAPartCols + 16 * hv, lo);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(BAR_AFULL + b));
        xmask ^= 1u << b;
        if (++b == kStages) b = 0;
      }
      // the tile's E5 stages pass through the ring without this role
      if constexpr (PROD) b = (uint32_t)((b + (uint32_t)(Jm * S)) % kStages);
    }
    if (!ok) raise(a.err, abort);
  } else {
    // ------------------------------------------------------------ epilogue
    const int wg = (warp - kEpiWarp0) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    constexpr int half = kSliceCols / 2;  // columns of this warpgroup per job
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(wg * half);
    __half* rhi = reinterpret_cast<__half*>(scr) + (size_t)row * d;
    __half* rlo = reinterpret_cast<__half*>(scr) + (size_t)(128 + row) * d;
    constexpr int NT = K == 1 ? 1 : K == 2 ? 2 : 4;
    uint32_t cq = 0;
    bool ok = true;
    for (int64_t i = 0; ok && i < n_my; ++i) {
      const int64_t tile = cid + i * P;
      const int64_t blk = tile % a.nb;
      const bool live = blk * kTokensPerBlock + row < a.N;
      uint8_t* out = a.packed + tile * a.lay.block_bytes;
      float n = 0.f, rr = 0.f;
      float nt[L - 1], nc[L];
      uint32_t nhalf[NT];
      float nmid = 0.f;
      for (int t = 0; ok && t < MYJOBS; ++t) {
        const int job = job_of(t);
        const bool e2 = t < Jm;
        if (t == 0) {
          n = *reinterpret_cast<const float*>(out + a.lay.norms_off + row * 8);
          // thresholds and centroids in the scale of Y = 2^16 Pi u (exact)
#pragma unroll
          for (int q = 0; q < L - 1; ++q) nt[q] = kYScale * a.cp.t[q];
#pragma unroll
          for (int q = 0; q < L; ++q) nc[q] = kYScale * a.cp.c[q];
#pragma unroll
          for (int q = 0; q < NT; ++q) nhalf[q] = __float_as_uint(-(kYScale * a.px.half[q]));
          nmid = kYScale * a.px.mid;
        }
        // the job's sums: partial accumulators of 128-coordinate K slices,
        // added here in fp32 with round-to-nearest
        float yv[half];
#pragma unroll
        for (int e = 0; e < half; ++e) yv[e] = 0.f;
        for (int c = 0; ok && c < S / kSliceStages; ++c, ++cq) {
          const uint32_t pb = cq & 1u;
          if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(BAR_DFULL + pb), (cq >> 1) & 1u, abort))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int g32 = 0; g32 < half / 32; ++g32) {
            uint32_t v[32];
            tmem_ld32(t_lane + pb * kSliceCols + 32 * g32, v);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) yv[32 * g32 + e] += __uint_as_float(v[e]);
          }
          tc_fence_before();
          mbar_arrive(bar(BAR_DEMPTY + pb));
        }
        if (!ok) break;
        const int cbase = (job % J) * NC + wg * half;  // first coordinate of this warpgroup's columns
        uint32_t pl[K + 1][half / 32];
#pragma unroll
        for (int g32 = 0; g32 < half / 32; ++g32) {
          const float* v = yv + 32 * g32;
          if (e2) {
            uint32_t w[K];
#pragma unroll
            for (int p = 0; p < K; ++p) w[p] = 0;
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int e = 30; e >= 0; e -= 2) {
              float r2[2];
#pragma unroll
              for (int u = 1; u >= 0; --u) {
                const float y = v[e + u];
                uint32_t sbit[L - 1];
                float cv = nc[0];
#pragma unroll
                for (int q = 0; q < L - 1; ++q) {
                  sbit[q] = __float_as_uint(nt[q] - y);
                  if constexpr (!PX) cv = (int)sbit[q] < 0 ? nc[q + 1] : cv;
                }
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
                  constexpr uint32_t kS = 0x80000000u;
                  cv = nmid + __uint_as_float(nhalf[0] ^ (xb[0] & kS));
                  if constexpr (K >= 2) cv += __uint_as_float(nhalf[1] ^ (xb[1] & kS));
                  if constexpr (K == 3) {
                    cv += __uint_as_float(nhalf[2] ^ (xb[2] & kS));
                    cv += __uint_as_float(nhalf[3] ^ ((xb[0] ^ xb[1] ^ xb[2]) & kS));
                  }
                }
                const float rv = y - cv;
                rr = fmaf(rv, rv, rr);
                r2[u] = rv * kRScale;
              }
              if constexpr (PROD) split_h2(r2[0], r2[1], hi[e >> 1], lo[e >> 1]);
            }
            if constexpr (PROD) {
              uint4* dh = reinterpret_cast<uint4*>(rhi + cbase + 32 * g32);
              uint4* dl = reinterpret_cast<uint4*>(rlo + cbase + 32 * g32);
  #pragma unroll
              for (int q = 0; q < 4; ++q) {
                __stcg(dh + q, make_uint4(hi[4 * q], hi[4 * q + 1], hi[4 * q + 2], hi[4 * q + 3]));
                __stcg(dl + q, make_uint4(lo[4 * q], lo[4 * q + 1], lo[4 * q + 2], lo[4 * q + 3]));
              }
            }
#pragma unroll
            for (int p = 0; p < K; ++p) pl[p][g32] = w[p];
          } else {
            uint32_t z = 0;
#pragma unroll
            for (int e = 31; e >= 0; --e) z = __funnelshift_l(__float_as_uint(v[e]), z, 1);
            pl[K][g32] = n > 0.f ? ~z : 0xFFFFFFFFu;
          }
        }
        // this warpgroup's plane words 2 wg, 2 wg + 1 of the job's 128-coordinate chunk
        const int chunk = cbase / 128, w0 = (cbase % 128) / 32;
        for (int p = e2 ? 0 : K; p < (e2 ? K : K + 1); ++p) {
          uint8_t* dst = out + a.lay.plane_off(p, chunk, row) + 4 * w0;
          *reinterpret_cast<uint2*>(dst) = live ? make_uint2(pl[p][0], pl[p][1]) : make_uint2(0, 0);
        }
        if (PROD && t == Jm - 1) {
          // every residual column of the tile this thread writes is stored,
          // made visible to the TMA loads (async proxy) of every CTA of the
          // cluster.  The local arrival comes first: once a peer has seen this
          // thread's remote arrival, this CTA's phase has it too, so no
          // CTA's next-tile arrivals can reach a phase that is still open.
          asm volatile("fence.proxy.async.global;" ::: "memory");
          mbar_arrive(bar(BAR_RREADY));
          for (int q = 1; q < CL; ++q) mbar_arrive_cluster(mapa_shared(bar(BAR_RREADY), (rank + (uint32_t)q) % (uint32_t)CL));
        }
      }
      if (!ok) break;
      if constexpr (PROD) {
        // rho: the partial sums of both warpgroups of every CTA of the
        // cluster, added on rank 0.  No arrival can come a tile early: a
        // CTA's next tile needs that tile's residual columns from every
        // CTA, which rank 0's warpgroup 0 writes only after this exchange.
        s_rr[wg * 128 + row] = rr;
        mbar_arrive(bar(BAR_RHO));
        if (wg == 0) {
          const bool got = rank == 0 ? mbar_wait_suspend_cluster(bar(BAR_RHO), (uint32_t)i & 1u, abort)
                                     : mbar_wait_suspend(bar(BAR_RHO), (uint32_t)i & 1u, abort);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          float r2 = s_rr[row] + s_rr[128 + row];
          if (rank == 0) {
            for (int q = 1; q < CL; ++q) r2 += s_rr_peer[(q - 1) * 128 + row];
            const float rho = n * (sqrtf(r2) * (1.f / kYScale));
            *reinterpret_cast<float2*>(out + a.lay.norms_off + row * 8) = live ? make_float2(n, rho)
                                                                                 : make_float2(0.f, 0.f);
          } else {
            st_cluster_f32(mapa_shared(smem_u32(s_rr_peer + (rank - 1) * 128 + row), 0), r2);
            mbar_arrive_cluster(mapa_shared(bar(BAR_RHO), 0));
          }
        }
      } else if (wg == 0 && rank == 0) {
        // MSE stores ||r|| = 0 and needs no exchange (which, with one K slice
        // per tile at d = 128, would let warpgroup 1 lap this barrier)
        *reinterpret_cast<float2*>(out + a.lay.norms_off + row * 8) = live ? make_float2(n, 0.f)
                                                                             : make_float2(0.f, 0.f);
      }
    }
    if (!ok) raise(a.err, abort);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
  // no CTA leaves while another may still arrive on its barriers or write its
  // shared memory (on a bounded-wait abort; otherwise each CTA has waited for
  // every arrival aimed at it)
  cluster_sync_all();
}

__global__ void nsmid_kernel(int* out) {
  uint32_t v;
  asm volatile("mov.u32 %0, %%nsmid;" : "=r"(v));
  *out = (int)v;
}

// at least 120 KB, so that no two CTAs of this kernel share an SM (the
// residual scratch is indexed by an SM id)
size_t enc_wide_smem(int) {
  const size_t need = (size_t)kStages * kStageBytes + BAR_COUNT * 8 + (2 + kMaxCluster - 1) * 128 * sizeof(float) + 1024;
  return need > 120 * 1024 ? need : 120 * 1024;
}

// CTAs per cluster for J chunks per phase: the CTAs of a cluster split each
// tile's chunks, so that a key or residual tile, re-read once per chunk, is
// shared by them and the tiles being worked on fit in L2
int enc_wide_cluster(int J) {
  static constexpr int kPrefer[] = {4, 3, 2};
  for (int c : kPrefer)
    if (c <= kMaxCluster && J % c == 0) return c;
  return 1;
}

// ||x|| of every row of every 128-token block (0 for padded rows) into the
// packed block's norm slot: one warp per row, compensated sums per lane,
// combined across lanes with error-free additions.
template <int DT>
__global__ void key_norm_kernel(const void* __restrict__ keys, int64_t N, int d, int64_t nb, int64_t rows,
                                Layout lay, uint8_t* __restrict__ packed) {
  constexpr int kEsize = DT == 0 ? 4 : 2;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += nwarps) {
    const int64_t gb = r >> 7, g = gb / nb;
    const int t = (int)(r & 127);
    const int64_t tok = (gb - g * nb) * kTokensPerBlock + t;
    float n = 0.f;
    if (tok < N) {
      KSum acc;
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(keys) + (g * N + tok) * (int64_t)d * kEsize);
      for (int v = lane; v < d * kEsize / 16; v += 32) {
        const uint4 w = __ldg(src + v);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if constexpr (DT == 0) {
            acc.add(__uint_as_float(ws[e]));
          } else {
            const float2 f = key_pair<DT>(ws[e]);
            acc.add(f.x);
            acc.add(f.y);
          }
        }
      }
      float sum = acc.s, comp = acc.c;
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float s2 = __shfl_xor_sync(0xffffffffu, sum, o), c2 = __shfl_xor_sync(0xffffffffu, comp, o);
        const float tt = sum + s2;
        comp += c2 + (fabsf(sum) >= fabsf(s2) ? (sum - tt) + s2 : (s2 - tt) + sum);
        sum = tt;
      }
      n = sqrtf(sum + comp);
    }
    if (lane == 0) *reinterpret_cast<float*>(packed + gb * lay.block_bytes + lay.norms_off + t * 8) = n;
  }
}

int enc_wide_nc(int) { return kSliceCols; }

struct EncMaps {
  CUtensorMap pi, m, x, r;
};

template <int L, int DT, bool PX, bool PROD>
cudaError_t launch_ew(const tq_plan* p, const EncWideArgs& a, const EncMaps& mp, cudaStream_t s) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t rows = a.n_tiles * kTokensPerBlock;
  const int64_t nblk = (rows + 7) / 8;
  key_norm_kernel<DT><<<(unsigned)(nblk < 8 * sms ? nblk : 8 * sms), 256, 0, s>>>(a.keys, a.N, a.lay.d, a.nb, rows,
                                                                                    a.lay, a.packed);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto kern = encode_wide_kernel<L, DT, PX, PROD>;
  const size_t smem = enc_wide_smem(a.NC);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)a.CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kEThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // one persistent cluster per group of CL SMs that can hold one at a time
  cfg.gridDim = dim3((unsigned)(sms / a.CL * a.CL));
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  const int64_t n_cl = a.n_tiles < clusters ? a.n_tiles : clusters;
  cfg.gridDim = dim3((unsigned)(n_cl * a.CL));
  e = cudaLaunchKernelEx(&cfg, kern, mp.pi, mp.m, mp.x, mp.r, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int DT, bool PX, bool PROD>
cudaError_t launch_ew_l(const tq_plan* p, const EncWideArgs& a, const EncMaps& mp, cudaStream_t s) {
  switch (p->cp.L) {
    case 2: return launch_ew<2, DT, PX, PROD>(p, a, mp, s);
    case 4: return launch_ew<4, DT, PX, PROD>(p, a, mp, s);
    case 8: return launch_ew<8, DT, PX, PROD>(p, a, mp, s);
    case 16:  // 4-bit MSE codebooks take the threshold-by-threshold centroid
      if constexpr (!PX && !PROD) return launch_ew<16, DT, false, false>(p, a, mp, s);
      break;
  }
  return cudaErrorInvalidValue;
}

template <int DT, bool PX>
cudaError_t launch_ew_m(const tq_plan* p, const EncWideArgs& a, const EncMaps& mp, cudaStream_t s) {
  return p->lay.prod ? launch_ew_l<DT, PX, true>(p, a, mp, s) : launch_ew_l<DT, PX, false>(p, a, mp, s);
}

bool odd_masks_w(const ParityExpansion& px, int k) {
  static const uint32_t want[3][4] = {{1u}, {1u, 2u}, {1u, 2u, 4u, 7u}};
  const int n = k == 3 ? 4 : k;
  if (k < 1 || k > 3 || px.n != n) return false;
  for (int i = 0; i < n; ++i)
    if (px.mask[i] != want[k - 1][i]) return false;
  return true;
}

}  // namespace

int query_nsmid() {
  int* d = nullptr;
  int v = 0;
  if (cudaMalloc(&d, sizeof(int)) != cudaSuccess) return 0;
  nsmid_kernel<<<1, 1>>>(d);
  if (cudaMemcpy(&v, d, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) v = 0;
  cudaFree(d);
  return v;
}

bool encode_wide_supported(const tq_plan* p, tq_dtype dt) {
  (void)dt;
  const bool prod = p->lay.prod != 0;
  return !p->lay.frac && p->wide_ops && (!prod || p->wide_scratch) && p->d % 128 == 0 && p->cp.L >= 2 &&
         p->cp.L <= (prod ? 8 : 16) && enc_wide_smem(enc_wide_nc(p->d)) <= 227 * 1024;
}

cudaError_t launch_encode_wide(const tq_plan* p, const void* keys, tq_dtype dt, int64_t G, int64_t N,
                               uint8_t* packed, cudaStream_t s) {
  if (G * N == 0) return cudaSuccess;
  const int d = p->d;
  EncWideArgs a;
  a.lay = p->lay;
  a.cp = p->cp;
  a.px = p->px;
  a.NC = enc_wide_nc(d);
  a.J = d / a.NC;
  a.CL = enc_wide_cluster(a.J);
  a.S = d / kStageK;
  a.nslots = p->wide_slots;
  a.G = G;
  a.N = N;
  a.nb = (N + kTokensPerBlock - 1) / kTokensPerBlock;
  a.n_tiles = G * a.nb;
  a.keys = keys;
  a.packed = packed;
  a.scratch = p->wide_scratch;
  a.err = p->err;
  // B operands: [hi rows; lo rows] of 2^8 Pi and (Prod) of M (fp16)
  const size_t dd = (size_t)d * d;
  const uint16_t* pi = p->wide_ops;
  const uint16_t* m = p->lay.prod ? p->wide_ops + 2 * dd : nullptr;
  EncMaps mp;
  const uint32_t nc = (uint32_t)a.NC;
  cudaError_t e = make_tmap_2d(&mp.pi, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, pi, (uint64_t)d, 2 * (uint64_t)d,
                               (uint64_t)d * 2, kStageK, nc, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e == cudaSuccess && p->lay.prod)
    e = make_tmap_2d(&mp.m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, m, (uint64_t)d, 2 * (uint64_t)d, (uint64_t)d * 2, kStageK,
                     nc, CU_TENSOR_MAP_SWIZZLE_128B);
  else if (e == cudaSuccess)
    mp.m = mp.pi;  // an MSE plan holds no M; its encode has no E5 and never reads this map
  // key tiles: 128 rows x 64 values, in boxes of 128-byte rows (two per stage
  // for fp32 keys); rows past G N read as zero
  if (e == cudaSuccess) {
    const CUtensorMapDataType xt = dt == TQ_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : dt == TQ_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t es = dt == TQ_F32 ? 4 : 2;
    e = make_tmap_2d(&mp.x, xt, keys, (uint64_t)d, (uint64_t)(G * N), (uint64_t)d * es,
                     dt == TQ_F32 ? kStageK / 2 : kStageK, kTokensPerBlock, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  // residual rows of the per-SM scratch: [slot][hi, lo][128][d] fp16 (Prod; an
  // MSE encode has no E5 and never reads this map)
  if (e == cudaSuccess) {
    if (p->lay.prod)
      e = make_tmap_2d(&mp.r, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p->wide_scratch, (uint64_t)d,
                       (uint64_t)p->wide_slots * 256, (uint64_t)d * 2, kStageK, kTokensPerBlock,
                       CU_TENSOR_MAP_SWIZZLE_128B);
    else
      mp.r = mp.pi;
  }
  if (e != cudaSuccess) return e;
  const bool px = odd_masks_w(p->px, p->lay.k);
  if (dt == TQ_F32) return px ? launch_ew_m<0, true>(p, a, mp, s) : launch_ew_m<0, false>(p, a, mp, s);
  if (dt == TQ_F16) return px ? launch_ew_m<1, true>(p, a, mp, s) : launch_ew_m<1, false>(p, a, mp, s);
  return px ? launch_ew_m<2, true>(p, a, mp, s) : launch_ew_m<2, false>(p, a, mp, s);
}

}  // namespace tq
