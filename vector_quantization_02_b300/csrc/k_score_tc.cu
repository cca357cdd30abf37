// Score on the 5th-generation tensor cores (tcgen05, fp8 operands, A operand in
// TMEM), d = 128, up to 16 query heads per group.
//
// Computes the same estimate as the CUDA-core score ("turboquant-pytorch 소개",
// usage listing ``tq.inner_product(query, compressed)`` and "2단계"):
//     logit = n <Pi q, c[idx]> + rho sqrt(pi/2)/m <S q, 2z - 1>.
//
// Bit-plane form.  The codebook is written in its parity (Walsh) expansion over
// the k code bits, c[idx] = c0 + sum_T gamma_T x_T(idx), where x_T(idx) is the
// XOR of the bits of idx selected by the mask T.  For an odd-symmetric codebook
// (the Lloyd-Max codebook of a symmetric density) only odd-weight masks carry
// weight: {1} for k = 1, {1, 2} for k = 2, {1, 2, 4, 7} for k = 3.  Hence
//     <Pi q, c[idx]> = c0 sum(Pi q) + sum_T <gamma_T Pi q, x_T>,
//     <S q, 2z - 1>  = <2 S q, z> - sum(S q),
// i.e. per key a sum of dot products between 0/1 bit planes and real query
// vectors: a dense contraction [128 keys x 128 K] . [128 K x N] per plane.
//
// Exactness.  Each key bit becomes an e4m3 value that is an exact power of two:
// a 32-coordinate plane word W yields eight 32-bit TMEM words (four e4m3 each)
// with two shifts and eight ANDs; every byte of output word o holds one source
// bit at bit position 3 + o % 4 of the byte, i.e. the e4m3 value 2^-6, 2^-5,
// 2^-3 or 2.  The query side carries the reciprocal power of two and a
// per-(head, term) power-of-two normalisation, and is split into four e4m3
// slices q = s0 + s1/16 + s2/256 + s3/4096 (about 2^-16 relative), one group
// of N = 4 Hp columns each.  Every product is exact; the accumulation is fp32.
//
// Work per CTA (persistent, contiguous range of 128-token blocks), four roles
// that only meet at mbarriers, so expansion never waits for an epilogue:
//  warps 0-3    MMA issuers (one elected lane each: a single thread issues one
//               tcgen05.mma about every 50 cycles, and every mbarrier operation
//               costs it ~150 cycles).  A tile has one job per term - the
//               MMA-term planes into one accumulator, the sign plane into
//               another; tile i's jobs go to warps 2 (i % 2) and 2 (i % 2) + 1.
//               Warp 0 owns the TMEM allocation (512 columns).
//  warps 4-11   two expansion warpgroups; tile i goes to warpgroup i % 2.
//               Thread (warp w, lane l) owns key row 32 (w % 4) + l: it reads its
//               16-byte plane chunks from the staged block and writes all the
//               tile's expanded planes into one group of 32-column TMEM slots
//               (a ring of SG groups), then arrives once.
//  warps 12-19  two epilogue warpgroups; tile i goes to warpgroup i % 2.  They
//               read the accumulators of a tile (a ring of DS stages), combine
//               slices and terms with the key's norms, and store H logits (one
//               coalesced store per head).
//  warp 20      producer: bulk copies of packed blocks (8-stage ring) and of the
//               per-group query operand images (double-buffered).
// Ordering.  A parity wait cannot tell phase k of an mbarrier from phase k + 2,
// so every ring entry has exactly one consumer, which waits for its uses in
// sequence: with the ring sizes even, tile i's packed block, plane-slot group
// and accumulator stage are only ever waited for by the expansion warpgroup,
// the issuer pair and the epilogue warpgroup of parity i % 2.  (Barrier waits
// cost ~150 cycles even when the phase is complete, so serialising the waits
// of different consumers through counters would cap the tile rate.)
// Every wait is bounded: on expiry the kernel raises the plan's error word,
// drains what it issued and frees its TMEM.
#include <cuda_fp8.h>

#include <algorithm>

#include "ptx_sm100.cuh"
#include "tc_planes.cuh"
#include "tq_internal.cuh"

namespace tq {
namespace {

using namespace ptx;

constexpr int kMaxStages = 16;      // packed-block ring entries (a multiple of the warpgroups per role)
constexpr int kMaxR = 4;            // TMEM tiles in flight: plane-slot groups = accumulator stages = R
constexpr int kMaxIssuers = kMaxR;

// MMA-term planes of an odd-symmetric codebook with k code bits.
__host__ __device__ constexpr int planes_of(int k) { return k == 3 ? 4 : k; }

// TMEM tiles in flight R for a plane-slot group of gcols columns and an
// accumulator stage of dcols (512 columns in all); 0 if not even two fit.
__host__ __device__ constexpr int tiles_in_flight(int gcols, int dcols) {
  return 4 * (gcols + dcols) <= 512 ? 4 : 3 * (gcols + dcols) <= 512 ? 3 : 2 * (gcols + dcols) <= 512 ? 2 : 0;
}

// Roles of the kernel for H_p heads, k code bits, Prod or MSE.  Tile i of a
// CTA's range uses TMEM entry i % R (its plane slots and accumulators), MMA
// issuer i % I, expansion warpgroup i % WE, epilogue warpgroup i % WP and
// packed-block slot i % stages, with I, WE and WP dividing R and WE dividing
// stages: every entry of every ring then has a single waiter per role, which
// waits for each of its phases in turn.  (A parity wait cannot tell phase k
// from k - 2 or k + 2, so a waiter that skipped phases could take a stale
// completion for the one it wants.)
template <int HP, int K, int PROD>
struct TcRoles {
  static constexpr int N = kSlices * HP;
  static constexpr int NA = planes_of(K), NP = NA + PROD, NJ = 1 + PROD;
  // (a shape where fewer than two tiles fit is never launched: fits is false)
  static constexpr bool fits = tiles_in_flight(NP * kPlaneCols, NJ * N) >= 2;
  static constexpr int R = fits ? tiles_in_flight(NP * kPlaneCols, NJ * N) : 2;
  static constexpr int I = R;                     // MMA issuers
  static constexpr int WE = R == 3 ? 3 : 2;       // expansion warpgroups
  static constexpr int WP = R;                    // epilogue warpgroups (the slower role)
  static constexpr int kExpWarp0 = I, kEpiWarp0 = I + 4 * WE, kProducerWarp = I + 4 * WE + 4 * WP;
  static constexpr int kThreads = 32 * (kProducerWarp + 1);
};

enum {
  BAR_FULL = 0,
  BAR_EMPTY = BAR_FULL + kMaxStages,
  BAR_BFULL = BAR_EMPTY + kMaxStages,
  BAR_BEMPTY = BAR_BFULL + 2,
  BAR_PFULL = BAR_BEMPTY + 2,
  BAR_MDONE = BAR_PFULL + kMaxR,   // a tile's MMAs complete: plane slots free, accumulators full
  BAR_DEMPTY = BAR_MDONE + kMaxR,
  BAR_DONE = BAR_DEMPTY + kMaxR,
  BAR_COUNT = BAR_DONE + kMaxIssuers
};


struct ScoreTcArgs {
  Layout lay;
  int H, Hp;                  // heads, padded heads (4, 8 or 16)
  uint32_t stages;            // packed-block ring entries (a multiple of the warpgroups per role)
  uint32_t img_bytes;         // per group: planes x (4 Hp rows x 128 B)
  int64_t N, nb, n_tiles;
  const uint8_t* packed;
  const uint8_t* images;      // [G][img_bytes]
  const float4* consts;       // [G][Hp] {1/sigma_A, c0 sum(Pi q), 1/sigma_B, -sum(S q)}
  float kappa;
  float* logits;
  int* err;
};

__device__ __forceinline__ void raise(int* err, volatile int* abort) {
  *abort = 1;
  atomicExch(err, 1);
}


// Both terms' accumulators of a tile (NJ x N <= 64 columns): every TMEM load is
// issued before a single wait.
template <int HP, int NJ>
__device__ __forceinline__ void load_terms(uint32_t taddr, float (&accA)[HP], float (&accB)[HP]) {
  constexpr int N = kSlices * HP;
  uint32_t v[NJ * N / 16][16];
#pragma unroll
  for (int c = 0; c < NJ * N / 16; ++c) tmem_ld16(taddr + 16 * c, v[c]);
  tmem_ld_wait();
#pragma unroll
  for (int h = 0; h < HP; ++h) accA[h] = accB[h] = 0.f;
#pragma unroll
  for (int c = 0; c < NJ * N / 16; ++c)
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int col = 16 * c + e, term = col / N, sl = (col % N) / HP, h = col % HP;
      if (term == 0) accA[h] = fmaf(__uint_as_float(v[c][e]), slice_weight(sl), accA[h]);
      else accB[h] = fmaf(__uint_as_float(v[c][e]), slice_weight(sl), accB[h]);
    }
}


// One job's MMAs for one tile: planes [P0, P1) x 4 K steps into one
// accumulator.  Every operand is a per-tile base plus a compile-time offset,
// so the issuing thread does no address arithmetic between MMAs (a thread
// that computes its descriptors between MMAs issues one only every ~250
// cycles; this form, ~60).
template <int P0, int P1, int N>
__device__ __forceinline__ void issue_job(uint32_t d, uint32_t at, uint64_t b, uint32_t idesc) {
#pragma unroll
  for (int p = P0; p < P1; ++p)
#pragma unroll
    for (uint32_t kb = 0; kb < 4; ++kb)
      // plane p of the image: N rows x 128 B (one swizzle atom column), p N 128
      // bytes in; K step kb starts 32 bytes further (descriptor units of 16 B)
      mma_f8_ts_w(d, at + (uint32_t)(p * kPlaneCols) + 8u * kb,
                b + (uint64_t)(((uint32_t)p * (uint32_t)N * 128u) >> 4) + 2u * kb, idesc,
                (p > P0 || kb > 0) ? 1u : 0u);
}

template <int HP, int K, int PROD>
__global__ void __launch_bounds__(TcRoles<HP, K, PROD>::kThreads, 1) score_tc_kernel(const ScoreTcArgs a) {
  using Cfg = TcRoles<HP, K, PROD>;
  constexpr int N = Cfg::N, NA = Cfg::NA, NP = Cfg::NP, NJ = Cfg::NJ;
  constexpr uint32_t R = Cfg::R, I = Cfg::I, WE = Cfg::WE, WP = Cfg::WP;
  constexpr int kExpWarp0 = Cfg::kExpWarp0, kEpiWarp0 = Cfg::kEpiWarp0, kProducerWarp = Cfg::kProducerWarp;
  static_assert(R >= 2 && R % I == 0 && R % WE == 0 && R % WP == 0, "ring entries must have a single waiter each");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(smem);
  const uint32_t n_stages = a.stages;
  const uint32_t off_ring = 2 * a.img_bytes;
  const uint32_t blk_bytes = (uint32_t)a.lay.block_bytes;
  const uint32_t off_bar = (off_ring + n_stages * blk_bytes + 7) & ~7u;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float4 s_cst[4 * WP][HP];  // per-head constants of each epilogue warp's current group
  auto bar = [&](int i) { return sb + off_bar + 8u * (uint32_t)i; };
  // TMEM: accumulators of entry r at r NJ N; plane slots of entry r at kSlot0 + r NP 32
  constexpr uint32_t kSlot0 = R * (uint32_t)(NJ * N);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t nb = (uint32_t)a.nb;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (uint32_t s = 0; s < n_stages; ++s) {
      mbar_init(bar(BAR_FULL + s), 1);
      mbar_init(bar(BAR_EMPTY + s), 128);  // the expansion warpgroup that read it
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(BAR_BFULL + b), 1);
      mbar_init(bar(BAR_BEMPTY + b), I);
    }
    for (uint32_t r = 0; r < R; ++r) {
      mbar_init(bar(BAR_PFULL + r), 128);
      mbar_init(bar(BAR_MDONE + r), 1);
      mbar_init(bar(BAR_DEMPTY + r), 128);
    }
    for (uint32_t w = 0; w < I; ++w) mbar_init(bar(BAR_DONE + w), 1);
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

  const int64_t t_begin = blockIdx.x * a.n_tiles / gridDim.x;
  const uint32_t n_my = (uint32_t)((blockIdx.x + 1) * a.n_tiles / gridDim.x - t_begin);

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      TilePos pos;
      pos.init(t_begin, a.nb);
      uint32_t epoch = 0, issued = 0;
      bool ok = true, have_img = false;
      const uint8_t* src = a.packed + t_begin * a.lay.block_bytes;
      // the first ring's worth of packed blocks does not depend on the query
      // preparation: it streams while that kernel still runs (programmatic
      // dependent launch); the query images wait for it to complete
      const uint32_t pre = n_my < n_stages ? n_my : n_stages;
      for (uint32_t i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(bar(BAR_FULL + i), blk_bytes);
        bulk_load(sb + off_ring + i * blk_bytes, src + (int64_t)i * blk_bytes, blk_bytes, bar(BAR_FULL + i));
      }
      issued = pre;
      grid_dependency_wait();
      Ring slot;  // packed-block slot of tile i
      for (uint32_t i = 0; i < n_my; ++i, src += blk_bytes, slot.advance(1, n_stages)) {
        if (i > 0) {
          const uint32_t g0 = pos.g;
          pos.advance(1, nb);
          if (pos.g != g0) ++epoch;
        }
        if (i == 0 || pos.blk == 0) {  // a new group: its query operand image
          const uint32_t b = epoch & 1u;
          if (!mbar_wait_suspend(bar(BAR_BEMPTY + b), ((epoch >> 1) & 1u) ^ 1u, abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(BAR_BFULL + b), a.img_bytes);
          bulk_load(sb + b * a.img_bytes, a.images + (int64_t)pos.g * a.img_bytes, a.img_bytes, bar(BAR_BFULL + b));
          have_img = true;
        }
        if (i < pre) continue;  // issued above
        if (!mbar_wait_suspend(bar(BAR_EMPTY + slot.idx), slot.phase ^ 1u, abort)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(bar(BAR_FULL + slot.idx), blk_bytes);
        bulk_load(sb + off_ring + slot.idx * blk_bytes, src, blk_bytes, bar(BAR_FULL + slot.idx));
        issued = i + 1;
      }
      if (!ok) raise(a.err, abort);
      // no copy may still be landing when the CTA exits
      int dummy = 0;
      for (uint32_t i = issued > n_stages ? issued - n_stages : 0; i < issued; ++i)
        mbar_wait(bar(BAR_FULL + i % n_stages), (i / n_stages) & 1u, &dummy);
      if (have_img) {
        for (uint32_t e = epoch > 0 ? epoch - 1 : 0; e <= epoch; ++e)
          mbar_wait(bar(BAR_BFULL + (e & 1u)), (e >> 1) & 1u, &dummy);
      }
    }
  } else if (warp < (int)I) {
    // ------------------------------------------------------------ MMA issuers
    // warp w issues every MMA of the tiles i with i % I == w (TMEM entries
    // i % R), then one commit: the tile's plane slots are free and its
    // accumulators full (the expansion and the epilogue of that entry both
    // wait on it, each for every phase in turn).  The whole warp runs the loop
    // (its operands stay warp-uniform); one elected lane issues each MMA and
    // commit.
    {
      constexpr uint32_t idesc = idesc_e4m3(128, N);
      // descriptors of the two query-image buffers, computed once
      const uint64_t bdesc0 = sdesc_k_sw128(sb), bdesc1 = sdesc_k_sw128(sb + a.img_bytes);
      TilePos pos;
      pos.init(t_begin, a.nb);
      uint32_t epoch = 0;
      Ring ent;  // TMEM entry of tile i
      bool need_b = true, ok = true;
      for (uint32_t i = 0; ok && i < n_my; ++i, ent.advance(1, R)) {
        if (i > 0) {
          const uint32_t g0 = pos.g;
          pos.advance(1, nb);
          if (pos.g != g0) {
            // this warp's MMAs on the previous group's image are all issued
            mma_commit_w(bar(BAR_BEMPTY + (epoch & 1u)));
            ++epoch;
            need_b = true;
          }
        }
        // every issuer waits for every group's image, owning tiles there or
        // not, so that it sees each phase of the image barriers in turn
        if (need_b) {
          if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(BAR_BFULL + (epoch & 1u)), (epoch >> 1) & 1u, abort))) {
            ok = false;
            break;
          }
          need_b = false;
        }
        if (i % I != (uint32_t)warp) continue;
        // polled with a suspend hint: a spinning issuer takes issue slots from
        // the expansion and epilogue warps that share its SM sub-partition
        // (measured: 3 % faster on the decode cache, 7 % on the Llama cache)
        if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(BAR_PFULL + ent.idx), ent.phase, abort) &&
                                         mbar_wait_suspend(bar(BAR_DEMPTY + ent.idx), ent.phase ^ 1u, abort))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + ent.idx * (uint32_t)(NJ * N);
        const uint32_t at = tmem + kSlot0 + ent.idx * (uint32_t)(NP * kPlaneCols);
        const uint64_t b = (epoch & 1u) ? bdesc1 : bdesc0;
        issue_job<0, NA, N>(d, at, b, idesc);
        if constexpr (PROD) issue_job<NA, NP, N>(d + (uint32_t)N, at, b, idesc);
        mma_commit_w(bar(BAR_MDONE + ent.idx));
      }
      if (!ok && lane == 0) raise(a.err, abort);
      mma_commit_w(bar(BAR_DONE + warp));
      int dummy = 0;
      mbar_wait(bar(BAR_DONE + warp), 0, &dummy);
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------------ expansion
    // Thread (warp w, lane l) owns key row 32 (w % 4) + l of the tiles i with
    // i % WE == wg.  It reads the key's plane chunks from the staged block,
    // frees the ring entry at once and writes the expanded planes to TMEM.
    const uint32_t wg = (uint32_t)(warp - kExpWarp0) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16) + kSlot0;
    Ring ent, slot;
    ent.advance(wg, R);
    slot.advance(wg, n_stages);
    for (uint32_t i = wg; i < n_my; i += WE, ent.advance(WE, R), slot.advance(WE, n_stages)) {
      if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(BAR_FULL + slot.idx), slot.phase, abort))) {
        raise(a.err, abort);
        break;
      }
      const uint8_t* blkp = smem + off_ring + slot.idx * blk_bytes;
      uint4 w[NP];
#pragma unroll
      for (int q = 0; q < K; ++q) {
        if (q == K - 1 && a.lay.frac) {  // a fractional width's half plane: coordinates 0..63
          const uint2 h = *reinterpret_cast<const uint2*>(blkp + a.lay.top_off + row * 8);
          w[q] = make_uint4(h.x, h.y, 0u, 0u);
        } else {
          w[q] = *reinterpret_cast<const uint4*>(blkp + ((q * kTokensPerBlock) + row) * 16);
        }
      }
      if constexpr (K == 3) {  // the triple-product plane x0 ^ x1 ^ x2
        w[3] = make_uint4(w[0].x ^ w[1].x ^ w[2].x, w[0].y ^ w[1].y ^ w[2].y, w[0].z ^ w[1].z ^ w[2].z,
                          w[0].w ^ w[1].w ^ w[2].w);
      }
      if constexpr (PROD) w[NA] = *reinterpret_cast<const uint4*>(blkp + a.lay.sign_off + row * 16);
      mbar_arrive(bar(BAR_EMPTY + slot.idx));
      if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(BAR_MDONE + ent.idx), ent.phase ^ 1u, abort))) {
        raise(a.err, abort);
        break;
      }
      tc_fence_after();
      const uint32_t taddr = lane_base + ent.idx * (uint32_t)(NP * kPlaneCols);
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        uint32_t o[32];
        expand_word(w[p].x, o);
        expand_word(w[p].y, o + 8);
        expand_word(w[p].z, o + 16);
        expand_word(w[p].w, o + 24);
        tmem_st32(taddr + (uint32_t)(p * kPlaneCols), o);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(BAR_PFULL + ent.idx));
    }
  } else {
    // ------------------------------------------------------------ epilogue
    grid_dependency_wait();  // the per-head constants come from the query preparation
    // Thread (warp w, lane l) owns key row 32 (w % 4) + l of the tiles i with
    // i % WP == eg.  The key's norms come straight from the packed block in
    // global memory (one 8-byte load, issued before the accumulator wait; the
    // block has just been streamed, so it is read from L2).
    const uint32_t eg = (uint32_t)(warp - kEpiWarp0) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    float4* wcst = s_cst[warp - kEpiWarp0];
    TilePos pos;
    pos.init(t_begin + eg, a.nb);
    Ring ent;
    ent.advance(eg, R);
    uint32_t cst_g = 0xffffffffu;  // group whose per-head constants wcst holds
    const uint8_t* norm_src = a.packed + (t_begin + eg) * a.lay.block_bytes + a.lay.norms_off + row * 8;
    for (uint32_t i = eg; i < n_my; i += WP, ent.advance(WP, R), norm_src += WP * a.lay.block_bytes) {
      if (i != eg) pos.advance(WP, nb);
      const float2 nr = __ldg(reinterpret_cast<const float2*>(norm_src));
      const int64_t tok = (int64_t)pos.blk * kTokensPerBlock + row;
      if (pos.g != cst_g) {  // a new group: its per-head constants (each warp keeps its own copy)
        __syncwarp();        // every lane has read the previous group's
        if (lane < HP) wcst[lane] = __ldg(a.consts + (int64_t)pos.g * a.Hp + lane);
        __syncwarp();
        cst_g = pos.g;
      }
      if (!__all_sync(0xffffffffu, mbar_wait_suspend(bar(BAR_MDONE + ent.idx), ent.phase, abort))) {
        raise(a.err, abort);
        break;
      }
      tc_fence_after();
      const uint32_t d = lane_base + ent.idx * (uint32_t)(NJ * N);
      float accA[HP], accB[HP];
      // at most 32 accumulator registers in flight
      if constexpr (NJ * N <= 32) {
        load_terms<HP, NJ>(d, accA, accB);
      } else if constexpr (N <= 32) {
        load_term_all<HP>(d, accA);
        if constexpr (PROD) load_term_all<HP>(d + N, accB);
      } else {
        load_term<HP>(d, accA);
        if constexpr (PROD) load_term<HP>(d + N, accB);
      }
      tc_fence_before();
      mbar_arrive(bar(BAR_DEMPTY + ent.idx));
      if (tok < a.N) {
        const float rk = nr.y * a.kappa;
        float* out = a.logits + ((int64_t)pos.g * a.H) * a.N + tok;
#pragma unroll
        for (int h = 0; h < HP; ++h) {
          if (h < a.H) {
            const float4 c = wcst[h];
            float v = nr.x * fmaf(accA[h], c.x, c.y);
            if constexpr (PROD) v = fmaf(rk, fmaf(accB[h], c.z, c.w), v);
            out[(int64_t)h * a.N] = v;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- query operand images

constexpr int kPrepHeads = 4;      // heads per prep CTA
constexpr int kPrepThreads = 512;  // four threads per output coordinate (quarters of the sum)

// One CTA per (group, up to 4 heads).  Pi^T and S^T are read from global
// memory, where every CTA reads the same 128 KB (L2-resident): thread
// (quarter r, coordinate j) sums rows [32 r, 32 r + 32) with sixteen rows of
// each matrix in flight at a time.  Pi q and S q are formed in fp32, then every
// plane's image rows (4 slices x head) and the heads' constants are written.
// No shared-memory staging of the matrices: two CTAs fit on an SM.
__global__ void __launch_bounds__(kPrepThreads, 2)
score_tc_prep_kernel(const float* __restrict__ q, int H, int Hp, int nA, int prod, ParityExpansion px,
                     ParityExpansion px_lo, int frac, const float* __restrict__ PiT, const float* __restrict__ ST,
                     uint32_t img_bytes, uint8_t* __restrict__ images, float4* __restrict__ consts) {
  constexpr int d = 128;
  grid_dependents_launch();  // the score kernel may start streaming packed blocks now
  __shared__ float4 s_q[d];                          // the CTA's heads' queries, one float4 per coordinate
  __shared__ float s_part[4][2][kPrepHeads][d];      // quarter sums of Pi q and S q
  __shared__ float s_full[kPrepHeads][2][d];         // Pi q and S q
  __shared__ float red[kPrepHeads][4][4];            // [head][warp][sum c0 Pi q, sum S q, max |Pi q|, max |S q|]
  __shared__ float s_coef[kMaxTerms], s_coef_lo[kMaxTerms];  // coordinates 0..63 and 64..127
  const int quads = (H + kPrepHeads - 1) / kPrepHeads;
  const int64_t g = blockIdx.x / quads;
  const int h0 = (blockIdx.x % quads) * kPrepHeads;
  const int nh = min(kPrepHeads, H - h0);
  const int t = threadIdx.x, r = t >> 7, j = t & (d - 1), lane = t & 31;
  const int N = kSlices * Hp;
  if (t < d) {
    const float* qg = q + (g * H + h0) * d + t;
    s_q[t] = make_float4(qg[0], nh > 1 ? qg[d] : 0.f, nh > 2 ? qg[2 * d] : 0.f, nh > 3 ? qg[3 * d] : 0.f);
  }
  if (t < kMaxTerms) {
    s_coef[t] = t < px.n ? px.coef[t] : 0.f;
    // a fractional width's lower codebook (coordinates 64..127), its terms on
    // the same masks (zero where the top code bit is involved)
    s_coef_lo[t] = t < px.n ? (frac ? px_lo.coef[t] : px.coef[t]) : 0.f;
  }
  float qr[kPrepHeads], sq[kPrepHeads];
#pragma unroll
  for (int hh = 0; hh < kPrepHeads; ++hh) qr[hh] = sq[hh] = 0.f;
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const int i0 = 32 * r + 16 * b;
    float pv[16], sv[16];
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) {
      pv[ii] = __ldg(PiT + (i0 + ii) * d + j);
      sv[ii] = __ldg(ST + (i0 + ii) * d + j);
    }
    if (b == 0) __syncthreads();  // the queries are in shared memory
#pragma unroll
    for (int ii = 0; ii < 16; ++ii) {
      const float4 qq = s_q[i0 + ii];
      qr[0] = fmaf(pv[ii], qq.x, qr[0]);
      qr[1] = fmaf(pv[ii], qq.y, qr[1]);
      qr[2] = fmaf(pv[ii], qq.z, qr[2]);
      qr[3] = fmaf(pv[ii], qq.w, qr[3]);
      sq[0] = fmaf(sv[ii], qq.x, sq[0]);
      sq[1] = fmaf(sv[ii], qq.y, sq[1]);
      sq[2] = fmaf(sv[ii], qq.z, sq[2]);
      sq[3] = fmaf(sv[ii], qq.w, sq[3]);
    }
  }
#pragma unroll
  for (int hh = 0; hh < kPrepHeads; ++hh) {
    s_part[r][0][hh][j] = qr[hh];
    s_part[r][1][hh][j] = sq[hh];
  }
  __syncthreads();
  // thread (head hh = r, coordinate j) from here on: the full values, and per
  // head the sum and max |.| over the coordinates (the head's four warps)
  const int hh = r;
  const float vqr = (s_part[0][0][hh][j] + s_part[1][0][hh][j]) + (s_part[2][0][hh][j] + s_part[3][0][hh][j]);
  const float vsq = (s_part[0][1][hh][j] + s_part[1][1][hh][j]) + (s_part[2][1][hh][j] + s_part[3][1][hh][j]);
  s_full[hh][0][j] = vqr;
  s_full[hh][1][j] = vsq;
  // the c0 term: c0 of coordinate j's codebook times (Pi q)_j, summed below
  float v[4] = {((frac && j >= 64) ? px_lo.c0 : px.c0) * vqr, vsq, fabsf(vqr), fabsf(vsq)};
#pragma unroll
  for (int o = 16; o; o >>= 1)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float x = __shfl_xor_sync(0xffffffffu, v[c], o);
      v[c] = (c & 2) ? fmaxf(v[c], x) : v[c] + x;
    }
  if (lane == 0)
#pragma unroll
    for (int c = 0; c < 4; ++c) red[hh][(t >> 5) & 3][c] = v[c];
  __syncthreads();
  float gmax = 0.f;
  for (int p = 0; p < nA; ++p) gmax = fmaxf(gmax, fmaxf(fabsf(s_coef[p]), fabsf(s_coef_lo[p])));
  const int nP = nA + prod;
  uint8_t* img = images + g * img_bytes;
  // K index kk of a plane: TMEM column c = kk / 4 = 8 w + o, byte b = kk % 4,
  // coordinate 32 w + 8 b + src(o)
  const int kk = j, col = kk >> 2, bte = kk & 3;
  const int jc = 32 * (col >> 3) + 8 * bte + c_src[col & 7];
  const float comp = c_comp[col & 3];
  if (hh < nh) {
    const int h = h0 + hh;
    const float sum_qr = (red[hh][0][0] + red[hh][1][0]) + (red[hh][2][0] + red[hh][3][0]);
    const float sum_sq = (red[hh][0][1] + red[hh][1][1]) + (red[hh][2][1] + red[hh][3][1]);
    const float max_qr = fmaxf(fmaxf(red[hh][0][2], red[hh][1][2]), fmaxf(red[hh][2][2], red[hh][3][2]));
    const float max_sq = fmaxf(fmaxf(red[hh][0][3], red[hh][1][3]), fmaxf(red[hh][2][3], red[hh][3][3]));
    // sigma = 2^(2 - e) with max |value| < 2^e: normalised values below 4, so
    // with the compensation (at most 64) every slice stays below 256
    int eA = 0, eB = 0;
    const float mA = gmax * max_qr, mB = 2.f * max_sq;
    if (mA > 0.f) frexpf(mA, &eA);
    if (mB > 0.f) frexpf(mB, &eB);
    const float sA = ldexpf(1.f, 2 - eA), sB = ldexpf(1.f, 2 - eB);
    for (int p = 0; p < nP; ++p) {
      const float coef = jc < 64 ? s_coef[p] : s_coef_lo[p];
      float val = p < nA ? coef * s_full[hh][0][jc] * comp * sA : 2.f * s_full[hh][1][jc] * comp * sB;
      uint8_t* base = img + (uint32_t)p * (uint32_t)N * 128u;
      float scale = 1.f;
#pragma unroll
      for (int sl = 0; sl < kSlices; ++sl) {
        const __nv_fp8_storage_t x = __nv_cvt_float_to_fp8(val * scale, __NV_SATFINITE, __NV_E4M3);
        base[img_offset(sl * Hp + h, kk)] = x;
        val -= e4m3_value(x) / scale;
        scale *= 16.f;
      }
    }
    if (j == 0) consts[g * Hp + h] = make_float4(1.f / sA, sum_qr, 1.f / sB, -sum_sq);
  }
  if (h0 == 0) {  // zero rows of the padding heads
    for (int p = 0; p < nP; ++p) {
      uint8_t* base = img + (uint32_t)p * (uint32_t)N * 128u;
      for (int hz = H + r; hz < Hp; hz += 4)
        for (int sl = 0; sl < kSlices; ++sl) base[img_offset(sl * Hp + hz, kk)] = 0;
    }
  }
}

int hp_of(int H) { return H <= 4 ? 4 : H <= 8 ? 8 : 16; }

// The masks the kernels expand for k code bits (odd-symmetric codebook).
bool standard_masks(const ParityExpansion& px, int k) {
  static const uint32_t want[3][4] = {{1u}, {1u, 2u}, {1u, 2u, 4u, 7u}};
  if (k < 1 || k > 3 || px.n != planes_of(k)) return false;
  for (int i = 0; i < px.n; ++i)
    if (px.mask[i] != want[k - 1][i]) return false;
  return true;
}

struct TcGeom {
  int Hp, N, nA, nP, R;
  uint32_t img, smem, stages;
};

bool tc_geom(const tq_plan* p, int H, TcGeom* gm) {
  if (p->d != 128 || H < 1 || H > 16) return false;
  const int k = p->lay.k;
  if (!standard_masks(p->px, k)) return false;
  gm->Hp = hp_of(H);
  gm->N = kSlices * gm->Hp;
  gm->nA = planes_of(k);
  gm->nP = gm->nA + p->lay.prod;
  // TMEM tiles in flight, as the kernel's TcRoles computes them
  gm->R = tiles_in_flight(gm->nP * kPlaneCols, (1 + p->lay.prod) * gm->N);
  if (gm->R < 2) return false;
  const uint32_t W = gm->R == 3 ? 3 : 2;  // expansion warpgroups (TcRoles::WE)
  gm->img = ((uint32_t)gm->nP * (uint32_t)gm->N * 128u + 1023u) & ~1023u;
  // the deepest packed-block ring (a multiple of the W warpgroups per role, at
  // most 16 entries) that fits beside the two query images
  for (uint32_t st = (kMaxStages / W) * W; st >= 2 * W; st -= W) {
    gm->stages = st;
    gm->smem = 2 * gm->img + st * (uint32_t)p->lay.block_bytes + BAR_COUNT * 8 + 16 + 1024;
    if (gm->smem <= 190 * 1024) return true;
  }
  return false;
}

template <int HP, int K, int PROD>
cudaError_t launch_kernel(const ScoreTcArgs& a, const TcGeom& gm, int64_t grid, cudaStream_t s) {
  if (!TcRoles<HP, K, PROD>::fits) return cudaErrorInvalidValue;
  auto kern = score_tc_kernel<HP, K, PROD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gm.smem);
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the CTAs may start while the query
  // preparation runs; the roles that read its output wait for it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(TcRoles<HP, K, PROD>::kThreads);
  cfg.dynamicSmemBytes = gm.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int HP>
cudaError_t launch_hp(const ScoreTcArgs& a, const TcGeom& gm, int64_t grid, int k, int prod, cudaStream_t s) {
  switch (k * 2 + prod) {
    case 2: return launch_kernel<HP, 1, 0>(a, gm, grid, s);
    case 3: return launch_kernel<HP, 1, 1>(a, gm, grid, s);
    case 4: return launch_kernel<HP, 2, 0>(a, gm, grid, s);
    case 5: return launch_kernel<HP, 2, 1>(a, gm, grid, s);
    case 6: return launch_kernel<HP, 3, 0>(a, gm, grid, s);
    case 7: return launch_kernel<HP, 3, 1>(a, gm, grid, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool score_tc_supported(const tq_plan* p, int H) {
  TcGeom gm;
  return tc_geom(p, H, &gm);
}

size_t score_tc_workspace_bytes(const tq_plan* p, int64_t G, int H) {
  TcGeom gm;
  if (!tc_geom(p, H, &gm)) return 0;
  const size_t imgs = (size_t)G * gm.img;
  return ((imgs + 255) & ~(size_t)255) + (size_t)G * gm.Hp * sizeof(float4);
}

cudaError_t launch_score_tc(const tq_plan* p, const float* queries, int64_t G, int H, const uint8_t* packed,
                            int64_t N, float* logits, void* ws, cudaStream_t s) {
  TcGeom gm;
  if (!tc_geom(p, H, &gm)) return cudaErrorInvalidValue;
  if (G * N == 0) return cudaSuccess;
  uint8_t* images = static_cast<uint8_t*>(ws);
  float4* consts = reinterpret_cast<float4*>(images + (((size_t)G * gm.img + 255) & ~(size_t)255));
  const int64_t prep_blocks = G * ((H + kPrepHeads - 1) / kPrepHeads);
  score_tc_prep_kernel<<<(unsigned)prep_blocks, kPrepThreads, 0, s>>>(
      queries, H, gm.Hp, gm.nA, p->lay.prod, p->px, p->px_enc_lo, p->lay.frac, p->PiT, p->lay.prod ? p->ST : p->PiT,
      gm.img, images, consts);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  ScoreTcArgs a;
  a.lay = p->lay;
  a.H = H;
  a.Hp = gm.Hp;
  a.stages = gm.stages;
  a.img_bytes = gm.img;
  a.N = N;
  a.nb = (N + kTokensPerBlock - 1) / kTokensPerBlock;
  a.n_tiles = G * a.nb;
  a.packed = packed;
  a.images = images;
  a.consts = consts;
  a.kappa = p->kappa;
  a.logits = logits;
  a.err = p->err;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t grid = a.n_tiles < sms ? a.n_tiles : sms;
  const int k = p->lay.k, prod = p->lay.prod;
  if (gm.Hp == 4) return launch_hp<4>(a, gm, grid, k, prod, s);
  if (gm.Hp == 8) return launch_hp<8>(a, gm, grid, k, prod, s);
  return launch_hp<16>(a, gm, grid, k, prod, s);
}

}  // namespace tq
