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
//  warps 2-9  expansion: thread = (key row, half of the coordinates); code
//             bits -> A operands in TMEM: for k <= 2 the levels' fp16 bytes sit
//             in registers and byte permutes pick them for four coordinates at
//             a time; for k >= 3 a table built once per CTA maps the code bits
//             of two coordinates to their fp16 hi and lo words;
//  warps 10-17 epilogue: thread = (key row, half of the coordinates);
//             accumulators -> fp32 rows, staged in shared memory (128-byte
//             swizzle, conflict-free) and written by TMA tensor stores that
//             clip the rows past N of a ragged block.
// Two warps per TMEM lane quarter in each of these roles: one warp moves only
// about 32 bytes per cycle between its registers and TMEM, and the rate grows
// with the number of warps.
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

constexpr int kDecSplit = 2;                  // warps per TMEM lane quarter in the expansion and the epilogue
constexpr int kDecThreads = 64 + 256 * kDecSplit;
constexpr int kDecExpWarp0 = 2, kDecEpiWarp0 = 2 + 4 * kDecSplit;
constexpr int kDecEpi0 = 32 * kDecEpiWarp0;   // first epilogue thread
constexpr int kDecStages = 2;
constexpr uint32_t kDecImg = 128 * 128 * 2;   // one 128 x 128 fp16 operand image
constexpr uint32_t kDecAtom = 128 * 128;      // 128 rows x 64 elements (128 B) per swizzle atom
constexpr uint32_t kOffPtHi = 0, kOffPtLo = kDecImg, kOffStHi = 2 * kDecImg, kOffStLo = 3 * kDecImg;
constexpr uint32_t kBlkMax = 4 * 2048 + 1024;  // largest d = 128 block: four planes + norms
constexpr uint32_t kOffBlk = 4 * kDecImg;
// output staging: four boxes of 128 rows x 32 fp32 (128 B rows, 128-byte swizzle)
constexpr uint32_t kStageBox = 128 * 128;
constexpr uint32_t kOffStage = kOffBlk + kDecStages * kBlkMax;  // a multiple of 1024
constexpr uint32_t kOffTab = kOffStage + 4 * kStageBox;        // lookup tables: 2 x 256 x 16 B
constexpr uint32_t kOffDecBar = kOffTab + 2 * 256 * 16;
enum {
  DB_OPS = 0,
  DB_SFULL = 1,
  DB_SEMPTY = DB_SFULL + kDecStages,  // expansion + epilogue arrivals (every thread of both)
  DB_AFULL0 = DB_SEMPTY + kDecStages,  // A columns of k steps 0..3 written
  DB_AFULL1,  // A columns of k steps 4..7 written
  DB_H0DONE,  // the MMAs of k steps 0..3 complete: their A columns may be rewritten
  DB_MDONE,   // all of a tile's MMAs complete: A may be rewritten, D1 and D2 are full
  DB_DEMPTY,
  DB_SFREE,   // the staging buffer may be written (previous tile's stores have read it)
  DB_STAGED,  // the tile's rows are in the staging buffer (every epilogue thread)
  DB_DONE,
  DB_COUNT
};
constexpr uint32_t kDecSmem = kOffDecBar + DB_COUNT * 8 + 1024;  // + alignment slack
static_assert(kOffStage % 1024 == 0, "128-byte swizzled boxes start on 1024-byte boundaries");
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

// Lookup table of the expansion for k >= 3, built per CTA from the codebook's
// split levels ctab (coordinates 0..63) and ctab_lo (64..127, the lower
// codebook of a fractional width, else ctab again).  An entry covers two
// coordinates: key = sum_p (2 bits of plane p) << 2p, value = {hi pair, lo
// pair} in the first half of a uint4.  (k <= 2 keeps its levels in registers.)
template <int K>
__device__ __forceinline__ void build_dec_tables(const DecTcArgs& a, uint4* tab) {
  constexpr int kEnt = 1 << (2 * K);
  static_assert(kEnt <= 256, "table");
  for (int e = threadIdx.x; e < 2 * kEnt; e += blockDim.x) {
    const int t = e / kEnt, key = e % kEnt;
    const uint32_t* ct = (t == 1 && a.lay.frac) ? a.ctab_lo : a.ctab;
    uint32_t c[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      uint32_t idx = 0;
#pragma unroll
      for (int p = 0; p < K; ++p) idx |= (uint32_t)((key >> (2 * p + u)) & 1) << p;
      c[u] = ct[idx];
    }
    tab[t * 256 + key] = make_uint4(__byte_perm(c[0], c[1], 0x5410), __byte_perm(c[0], c[1], 0x7632), 0u, 0u);
  }
}

template <int K, bool PROD>
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmOut, const DecTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(smem);
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  uint4* tab = reinterpret_cast<uint4*>(smem + kOffTab);
  auto bar = [&](int i) { return sb + kOffDecBar + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if constexpr (K >= 3) build_dec_tables<K>(a, tab);
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar(DB_OPS), 1);
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(bar(DB_SFULL + s), 1);
      mbar_init(bar(DB_SEMPTY + s), 256 * kDecSplit);
    }
    mbar_init(bar(DB_AFULL0), 128);
    mbar_init(bar(DB_AFULL1), 128);
    mbar_init(bar(DB_H0DONE), 1);
    mbar_init(bar(DB_MDONE), 1);
    mbar_init(bar(DB_DEMPTY), 128 * kDecSplit);
    mbar_init(bar(DB_SFREE), 1);
    mbar_init(bar(DB_STAGED), 128 * kDecSplit);
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
    // The operand descriptors are built once; every MMA adds a compile-time
    // offset.  Two commits per tile, one per half of K: the expansion waits
    // on each (that half of A free), the epilogue on the second (D full).
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(0u, 128, 128);
      const uint64_t dph = sdesc_k_sw128(sb + kOffPtHi), dpl = sdesc_k_sw128(sb + kOffPtLo);
      const uint64_t dsh = sdesc_k_sw128(sb + kOffStHi), dsl = sdesc_k_sw128(sb + kOffStLo);
      const uint32_t d1 = tmem + kColD1, d2 = tmem + kColD2;
      const uint32_t ahi = tmem + kColAHi, alo = tmem + kColALo, sg = tmem + kColSg;
      bool ok = mbar_wait(bar(DB_OPS), 0, abort);
      for (int64_t i = 0; ok && i < n_my; ++i) {
        const uint32_t ph = (uint32_t)i & 1u;
        // two halves of K: the expansion rewrites the first half of A for the
        // next tile while the second half's MMAs run
#pragma unroll
        for (uint32_t h = 0; h < 2; ++h) {
          if (!mbar_wait(bar(h == 0 ? DB_AFULL0 : DB_AFULL1), ph, abort) ||
              (h == 0 && !mbar_wait(bar(DB_DEMPTY), ph ^ 1u, abort))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (uint32_t kb = 4 * h; kb < 4 * h + 4; ++kb) {
            // k step kb: swizzle atom kb / 4 of the image, 32 bytes per step within it
            // (descriptor address units of 16 bytes); A columns 8 kb
            const uint64_t off = (uint64_t)(((kb >> 2) * kDecAtom + (kb & 3) * 32) >> 4);
            mma_f16_ts(d1, ahi + 8 * kb, dph + off, idesc, kb > 0 ? 1u : 0u);
            mma_f16_ts(d1, ahi + 8 * kb, dpl + off, idesc, 1u);
            mma_f16_ts(d1, alo + 8 * kb, dph + off, idesc, 1u);
            if constexpr (PROD) {
              mma_f16_ts(d2, sg + 8 * kb, dsh + off, idesc, kb > 0 ? 1u : 0u);
              mma_f16_ts(d2, sg + 8 * kb, dsl + off, idesc, 1u);
            }
          }
          mma_commit(bar(h == 0 ? DB_H0DONE : DB_MDONE));
        }
      }
      if (!ok) raise_dec(a.err, abort);
      // all issued MMAs complete before TMEM is freed
      mma_commit(bar(DB_DONE));
      int dummy = 0;
      mbar_wait(bar(DB_DONE), 0, &dummy);
    }
  } else if (warp < kDecEpiWarp0) {
    // ------------------------------------------------------------ expansion
    // half hh of the coordinates: words 2 hh and 2 hh + 1 of each plane
    const int quad = warp & 3, hh = (warp - kDecExpWarp0) >> 2;
    // levels 0..3 of each codebook (k <= 2): fp16 hi (h) and lo (l) parts,
    // levels 0, 1 in x and 2, 3 in y
    struct {
      uint32_t hx0, hy0, lx0, ly0, hx1, hy1, lx1, ly1;
    } lv;
    {
      const uint32_t* c1 = a.lay.frac ? a.ctab_lo : a.ctab;
      lv.hx0 = __byte_perm(a.ctab[0], a.ctab[1], 0x5410);
      lv.hy0 = __byte_perm(a.ctab[2], a.ctab[3], 0x5410);
      lv.lx0 = __byte_perm(a.ctab[0], a.ctab[1], 0x7632);
      lv.ly0 = __byte_perm(a.ctab[2], a.ctab[3], 0x7632);
      lv.hx1 = __byte_perm(c1[0], c1[1], 0x5410);
      lv.hy1 = __byte_perm(c1[2], c1[3], 0x5410);
      lv.lx1 = __byte_perm(c1[0], c1[1], 0x7632);
      lv.ly1 = __byte_perm(c1[2], c1[3], 0x7632);
    }
    const int row = quad * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    bool ok = true;
    for (int64_t i = 0; ok && i < n_my; ++i) {
      const int s = (int)(i % kDecStages);
      // every lane polls; the warp proceeds (or gives up) as one, because the
      // tcgen05 stores below are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(bar(DB_SFULL + s), (uint32_t)(i / kDecStages) & 1u, abort))) {
        ok = false;
        break;
      }
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
      // half h of A (words 2 h, 2 h + 1: k steps 4 h .. 4 h + 3) once the
      // previous tile's MMAs on it are complete
#pragma unroll
      for (int hx = 0; hx < 2 / kDecSplit; ++hx) {
      const int h = (2 / kDecSplit) * hh + hx;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(h == 0 ? DB_H0DONE : DB_MDONE), ((uint32_t)i & 1u) ^ 1u, abort))) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int ww = 0; ww < 2; ++ww) {
        // coordinates 32 w + e, e = 0..31: bit e of word w of each plane;
        // the lower codebook's levels for coordinates 64..127
        const int w = 2 * h + ww;
        uint32_t wp[K];
#pragma unroll
        for (int p = 0; p < K; ++p) wp[p] = word_of(pw[p], w);
        uint32_t hi[16], lo[16];
        if constexpr (K <= 2) {
          // Levels in registers: the fp16 bytes of levels 0..3 (hi and lo
          // parts), picked by byte permutes.  For four coordinates, byte u of
          // S is coordinate u's level index, and byte u of T = 0x22 S +
          // 0x10101010 holds the selectors (2 idx, 2 idx + 1) of that level's
          // two bytes; T's low half selects coordinates 0, 1, its high half 2, 3.
          const uint32_t thx = w < 2 ? lv.hx0 : lv.hx1, thy = w < 2 ? lv.hy0 : lv.hy1;
          const uint32_t tlx = w < 2 ? lv.lx0 : lv.lx1, tly = w < 2 ? lv.ly0 : lv.ly1;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            // bit u of a nibble to bit 8 u: x * 0x204081 places the four
            // shifted copies without overlap
            uint32_t S = (((wp[0] >> (4 * q)) & 0xFu) * 0x00204081u) & 0x01010101u;
            if constexpr (K == 2) S |= (((wp[1] >> (4 * q)) & 0xFu) * 0x00408102u) & 0x02020202u;
            const uint32_t T = S * 0x22u + 0x10101010u;
            hi[2 * q] = __byte_perm(thx, thy, T);
            hi[2 * q + 1] = __byte_perm(thx, thy, T >> 16);
            lo[2 * q] = __byte_perm(tlx, tly, T);
            lo[2 * q + 1] = __byte_perm(tlx, tly, T >> 16);
          }
        } else {
          const uint4* tw = tab + (w >> 1) * 256;
#pragma unroll
          for (int m = 0; m < 16; ++m) {
            uint32_t key = 0;
#pragma unroll
            for (int p = 0; p < K; ++p) key |= ((wp[p] >> (2 * m)) & 3u) << (2 * p);
            const uint2 e = *reinterpret_cast<const uint2*>(tw + key);
            hi[m] = e.x;
            lo[m] = e.y;
          }
        }
        tmem_st16(t_lane + kColAHi + 16 * w, hi);
        tmem_st16(t_lane + kColALo + 16 * w, lo);
        if constexpr (PROD) {
          // 2 z - 1 as fp16 (+1 = 0x3C00, -1 = 0xBC00): byte u of S is 1 - z of
          // coordinate u; the selectors pick 0x00 for the low byte and 0x3C or
          // 0xBC for the high byte of each value
          const uint32_t nz = ~word_of(zw, w);
          uint32_t sg[16];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t S = (((nz >> (4 * q)) & 0xFu) * 0x00204081u) & 0x01010101u;
            const uint32_t T = (S << 4) | 0x02020202u;
            sg[2 * q] = __byte_perm(0x0000BC3Cu, 0u, T);
            sg[2 * q + 1] = __byte_perm(0x0000BC3Cu, 0u, T >> 16);
          }
          tmem_st16(t_lane + kColSg + 16 * w, sg);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(h == 0 ? DB_AFULL0 : DB_AFULL1));
      }
    }
    if (!ok) raise_dec(a.err, abort);
  } else {
    // ------------------------------------------------------------ epilogue
    // Thread = (key row, half hh of the coordinates).  Rows go to the staging
    // buffer (box q = fp32 columns 32 q .. 32 q + 31, 128-byte rows whose
    // 16-byte chunks are XOR-swizzled by row % 8), then thread kDecEpi0 writes
    // the tile with four TMA stores.
    const int quad = warp & 3, hh = (warp - kDecEpiWarp0) >> 2;
    const int row = quad * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    const bool leader = threadIdx.x == kDecEpi0;
    const uint32_t stage_row = sb + kOffStage + (uint32_t)row * 128u;
    if (leader) prefetch_tmap(&tmOut);
    bool ok = true;
    for (int64_t i = 0; ok && i < n_my; ++i) {
      const int s = (int)(i % kDecStages);
      const uint32_t ph = (uint32_t)i & 1u;
      const int64_t tile = blockIdx.x + i * gridDim.x;
      const int64_t g = tile / a.nb, tok0 = (tile - g * a.nb) * kTokensPerBlock;
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
      if (leader) {
        // the previous tile's stores have read the staging buffer
        bulk_wait_read_all();
        mbar_arrive(bar(DB_SFREE));
      }
      if (!__all_sync(0xffffffffu, mbar_wait(bar(DB_MDONE), ph, abort)) ||
          !__all_sync(0xffffffffu, mbar_wait(bar(DB_SFREE), ph, abort))) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int q = (4 / kDecSplit) * hh; q < (4 / kDecSplit) * (hh + 1); ++q) {
        uint32_t v1[32], v2[32];
        tmem_ld32(t_lane + kColD1 + 32 * q, v1);
        if constexpr (PROD) tmem_ld32(t_lane + kColD2 + 32 * q, v2);
        tmem_ld_wait();
        if (q == (4 / kDecSplit) * (hh + 1) - 1) {  // accumulators read: the next tile's MMAs may write them
          tc_fence_before();
          mbar_arrive(bar(DB_DEMPTY));
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float o[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            o[u] = s1 * __uint_as_float(v1[4 * j + u]);
            if constexpr (PROD) o[u] = fmaf(s2, __uint_as_float(v2[4 * j + u]), o[u]);
          }
          sts128(stage_row + (uint32_t)q * kStageBox + (uint32_t)((j ^ (row & 7)) << 4), __float_as_uint(o[0]),
                 __float_as_uint(o[1]), __float_as_uint(o[2]), __float_as_uint(o[3]));
        }
      }
      // the rows are visible to the TMA unit, then the leader stores the tile
      // (rows past N, in a ragged last block of a group, are clipped)
      fence_proxy_async_smem();
      mbar_arrive(bar(DB_STAGED));
      if (leader) {
        if (!mbar_wait(bar(DB_STAGED), ph, abort)) {
          ok = false;
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            tma_store_3d(&tmOut, sb + kOffStage + (uint32_t)q * kStageBox, 32 * q, (int32_t)tok0, (int32_t)g);
          bulk_commit_group();
        }
      }
    }
    if (!ok) raise_dec(a.err, abort);
    if (leader) bulk_wait_all();  // the output is written before the CTA exits
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
  // the output as [G][N][128] fp32, written in boxes of 128 rows x 32 values
  CUtensorMap tm;
  const uint64_t dims[3] = {128, (uint64_t)N, (uint64_t)G};
  const uint64_t strides[2] = {128 * sizeof(float), (uint64_t)N * 128 * sizeof(float)};
  // (a box no taller than the tensor; the staging rows keep their places)
  const uint32_t box[3] = {32, N < 128 ? (uint32_t)N : 128u, 1};
  cudaError_t e = make_tmap_3d(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, out, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  auto kern = decode_tc_kernel<K, PROD>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t grid = a.n_tiles < sms ? a.n_tiles : sms;
  kern<<<(unsigned)grid, kDecThreads, kDecSmem, s>>>(tm, a);
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
