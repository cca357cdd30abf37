// Plan derivation, the uncompressed fp32 baseline, and the bounded-wait self-test.
#include "ptx_sm100.cuh"
#include "tq_internal.cuh"

namespace tq {
namespace {

// Out = A B^T in fp64 accumulation, rounded to fp32; A, B, Out are [d][d].
// Also writes OutT = Out^T.  16x16 tiles.
__global__ void abt_f64_kernel(const float* __restrict__ A, const float* __restrict__ B, int d,
                               float* __restrict__ Out, float* __restrict__ OutT) {
  __shared__ double sa[16][17], sb[16][17];
  const int r = blockIdx.y * 16 + threadIdx.y;   // row of A
  const int c = blockIdx.x * 16 + threadIdx.x;   // row of B
  double acc = 0.0;
  for (int k0 = 0; k0 < d; k0 += 16) {
    sa[threadIdx.y][threadIdx.x] = A[(int64_t)(blockIdx.y * 16 + threadIdx.y) * d + k0 + threadIdx.x];
    sb[threadIdx.y][threadIdx.x] = B[(int64_t)(blockIdx.x * 16 + threadIdx.y) * d + k0 + threadIdx.x];
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 16; ++k) acc = fma(sa[threadIdx.y][k], sb[threadIdx.x][k], acc);
    __syncthreads();
  }
  Out[(int64_t)r * d + c] = (float)acc;
  OutT[(int64_t)c * d + r] = (float)acc;
}

__global__ void transpose_kernel(const float* __restrict__ A, int d, float* __restrict__ AT) {
  __shared__ float tile[32][33];
  const int x = blockIdx.x * 32 + threadIdx.x, y0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) tile[i][threadIdx.x] = A[(int64_t)(y0 + i) * d + x];
  __syncthreads();
  const int xo = blockIdx.y * 32 + threadIdx.x, yo0 = blockIdx.x * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) AT[(int64_t)(yo0 + i) * d + xo] = tile[threadIdx.x][i];
}

// fp32 baseline: a CTA stages KT keys of one group in shared memory (coalesced),
// then thread (key, head) computes the dot product; the key row is read with a
// rotated start so that a warp's 32 keys hit 32 banks.
template <int KT>
__global__ void __launch_bounds__(256)
score_fp32_kernel(const float* __restrict__ q, const float* __restrict__ x, int64_t G, int H, int64_t N, int d,
                  float* __restrict__ logits) {
  extern __shared__ float xs[];   // [KT][d]
  const int64_t ntile = (N + KT - 1) / KT;
  const int64_t g = blockIdx.x / ntile, tile = blockIdx.x % ntile;
  const int64_t tok0 = tile * KT;
  const int kn = (int)(N - tok0 < KT ? N - tok0 : KT);
  const float* src = x + (g * N + tok0) * d;
  for (int i = threadIdx.x; i < kn * d; i += blockDim.x) xs[i] = src[i];
  __syncthreads();
  const int k = threadIdx.x % KT;
  for (int h = threadIdx.x / KT; h < H; h += blockDim.x / KT) {
    if (k >= kn) continue;
    const float* qh = q + (g * H + h) * d;
    const float* xr = xs + k * d;
    float acc = 0.f;
    int j = k % d;
    for (int i = 0; i < d; ++i) {
      acc = fmaf(__ldg(qh + j), xr[j], acc);
      j = j + 1 == d ? 0 : j + 1;
    }
    logits[(g * H + h) * N + tok0 + k] = acc;
  }
}

// Streaming form for d % 4 == 0, d <= 1024: thread t of a block owns key t of
// its 128-key tile and reads it with 16-byte loads; the group's queries sit in
// shared memory and are read as broadcasts, eight heads per pass over the key.
// Logit stores are coalesced (consecutive threads, consecutive tokens).
constexpr int kF32Tile = 128;
constexpr int kF32Heads = 8;

__global__ void __launch_bounds__(kF32Tile)
score_fp32_stream_kernel(const float* __restrict__ q, const float* __restrict__ x, int64_t G, int H, int64_t N,
                         int d, int64_t n_tiles, float* __restrict__ logits) {
  extern __shared__ float4 qs4[];  // [H][d / 4]
  const int d4 = d >> 2;
  const int64_t tiles_per_group = (N + kF32Tile - 1) / kF32Tile;
  int64_t cur_g = -1;
  for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const int64_t g = tile / tiles_per_group;
    const int64_t tok = (tile - g * tiles_per_group) * kF32Tile + threadIdx.x;
    if (g != cur_g) {
      __syncthreads();
      const float4* qg = reinterpret_cast<const float4*>(q + g * H * d);
      for (int i = threadIdx.x; i < H * d4; i += kF32Tile) qs4[i] = __ldg(qg + i);
      __syncthreads();
      cur_g = g;
    }
    if (tok >= N) continue;
    const float4* xr = reinterpret_cast<const float4*>(x + (g * N + tok) * d);
    float* out = logits + (g * H) * N + tok;
    for (int h0 = 0; h0 < H; h0 += kF32Heads) {
      float acc[kF32Heads];
#pragma unroll
      for (int h = 0; h < kF32Heads; ++h) acc[h] = 0.f;
#pragma unroll 4
      for (int j = 0; j < d4; ++j) {
        const float4 xv = __ldg(xr + j);
#pragma unroll
        for (int h = 0; h < kF32Heads; ++h) {
          if (h0 + h < H) {
            const float4 qv = qs4[(h0 + h) * d4 + j];
            acc[h] = fmaf(qv.x, xv.x, fmaf(qv.y, xv.y, fmaf(qv.z, xv.z, fmaf(qv.w, xv.w, acc[h]))));
          }
        }
      }
#pragma unroll
      for (int h = 0; h < kF32Heads; ++h)
        if (h0 + h < H) out[(int64_t)(h0 + h) * N] = acc[h];
    }
  }
}

// d = 128: eight lanes share a key, lane c reading its 16-byte chunks c, c+8,
// c+16, c+24, so one load instruction covers four whole 128-byte key rows. Each
// lane forms partial dot products for eight heads (queries from shared memory,
// the eight lanes of a key reading eight distinct chunks), and a reduce-scatter
// across the eight lanes leaves lane c with head c's logit for its key. A warp
// takes sixteen keys (four loads of four rows in flight per chunk), a block
// 128 consecutive keys of one group, so the tiles spread evenly over a grid
// of resident blocks.
constexpr int kD128Sub = 4;  // groups of four keys per warp
constexpr int kD128Tile = 8 * 4 * kD128Sub;

__device__ __forceinline__ float dot4(float4 a, float4 b, float acc) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, fmaf(a.w, b.w, acc))));
}

// Eight partial sums per lane -> lane (c) of each 8-lane group holds the group's
// total for value index c. Round with offset s keeps the half whose index bit
// matches the lane's bit s and sends the other half to the partner lane.
__device__ __forceinline__ float reduce_scatter8(float (&v)[8], int c) {
  const bool u4 = c & 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = u4 ? v[i] : v[i + 4];
    const float keep = u4 ? v[i + 4] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  const bool u2 = c & 2;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = u2 ? v[i] : v[i + 2];
    const float keep = u2 ? v[i + 2] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  const bool u1 = c & 1;
  const float send = u1 ? v[0] : v[1];
  const float keep = u1 ? v[1] : v[0];
  return keep + __shfl_xor_sync(0xffffffffu, send, 1);
}

__global__ void __launch_bounds__(256, 2)
score_fp32_d128_kernel(const float* __restrict__ q, const float* __restrict__ x, int64_t G, int H, int64_t N,
                       int64_t n_tiles, float* __restrict__ logits) {
  extern __shared__ float4 qs4[];  // [H][32]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = lane & 7, tg = lane >> 3;
  const int64_t tiles_per_group = (N + kD128Tile - 1) / kD128Tile;
  int64_t cur_g = -1;
  for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const int64_t g = tile / tiles_per_group;
    const int64_t tile_tok = (tile - g * tiles_per_group) * kD128Tile;
    if (g != cur_g) {
      __syncthreads();
      const float4* qg = reinterpret_cast<const float4*>(q + g * H * 128);
      for (int i = threadIdx.x; i < H * 32; i += blockDim.x) qs4[i] = __ldg(qg + i);
      __syncthreads();
      cur_g = g;
    }
    const float4* xg = reinterpret_cast<const float4*>(x + g * N * 128);
    float* lg = logits + g * H * N;
    {
      const int64_t base = tile_tok + warp * 4 * kD128Sub;
      if (base >= N) continue;
      int64_t tok[kD128Sub];
      float4 xv[kD128Sub][4];
#pragma unroll
      for (int s2 = 0; s2 < kD128Sub; ++s2) {
        tok[s2] = base + s2 * 4 + tg;
        const bool ok = tok[s2] < N;
        const float4* row = xg + (ok ? tok[s2] : 0) * 32 + c;
#pragma unroll
        for (int j = 0; j < 4; ++j) xv[s2][j] = ok ? __ldg(row + 8 * j) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      for (int h0 = 0; h0 < H; h0 += 8) {
        float acc[kD128Sub][8];
#pragma unroll
        for (int s2 = 0; s2 < kD128Sub; ++s2)
#pragma unroll
          for (int h = 0; h < 8; ++h) acc[s2][h] = 0.f;
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          const int hh = h0 + h < H ? h0 + h : H - 1;  // padded heads repeat a real one, stored nowhere
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 qv = qs4[hh * 32 + c + 8 * j];
#pragma unroll
            for (int s2 = 0; s2 < kD128Sub; ++s2) acc[s2][h] = dot4(qv, xv[s2][j], acc[s2][h]);
          }
        }
#pragma unroll
        for (int s2 = 0; s2 < kD128Sub; ++s2) {
          const float r = reduce_scatter8(acc[s2], c);
          if (tok[s2] < N && h0 + c < H) lg[(int64_t)(h0 + c) * N + tok[s2]] = r;
        }
      }
    }
  }
}

// Many heads or long rows (e.g. 256 queries of d = 1536): a register-tiled
// fp32 product per group, logits[h][t] = sum_j q[h][j] x[t][j].  A block owns 64
// heads x 128 keys and walks d in steps of 16 through k-major shared tiles;
// thread (ty, tx) accumulates heads 4 ty .. 4 ty + 3 against keys 8 tx .. 8 tx + 7.
// Blocks of the same key tile are adjacent in the grid (head tile fastest), so
// a key row is fetched from HBM once and re-read from L2.
constexpr int kGH = 64, kGT = 128, kGK = 16;

__global__ void __launch_bounds__(256)
score_fp32_gemm_kernel(const float* __restrict__ q, const float* __restrict__ x0, const float* __restrict__ x1,
                       int64_t x_gstride, int H, int64_t N, int d, int h_tiles, int64_t t_tiles,
                       float* __restrict__ out0, float* __restrict__ out1) {
  // blockIdx.y picks the matrix (and output) when two products share one launch
  const float* __restrict__ x = blockIdx.y ? x1 : x0;
  float* __restrict__ logits = blockIdx.y ? out1 : out0;
  __shared__ __align__(16) float qs[kGK][kGH];
  __shared__ __align__(16) float xs[kGK][kGT];
  const int64_t bid = blockIdx.x;
  const int ht = (int)(bid % h_tiles);
  const int64_t rest = bid / h_tiles;
  const int64_t tt = rest % t_tiles, g = rest / t_tiles;
  const int h0 = ht * kGH;
  const int64_t t0 = tt * kGT;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const float* qg = q + (g * H) * (int64_t)d;
  const float* xg = x + g * x_gstride;
  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < d; k0 += kGK) {
    // q tile: 64 heads x 16 coordinates (one float4 per thread)
    {
      const int r = tid >> 2, c = (tid & 3) * 4;
      const float4 v = h0 + r < H ? __ldg(reinterpret_cast<const float4*>(qg + (int64_t)(h0 + r) * d + k0 + c))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
      qs[c + 0][r] = v.x;
      qs[c + 1][r] = v.y;
      qs[c + 2][r] = v.z;
      qs[c + 3][r] = v.w;
    }
    // key tile: 128 keys x 16 coordinates (two float4 per thread)
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int i = tid + u * 256, r = i >> 2, c = (i & 3) * 4;
      const float4 v = t0 + r < N ? __ldg(reinterpret_cast<const float4*>(xg + (t0 + r) * d + k0 + c))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
      xs[c + 0][r] = v.x;
      xs[c + 1][r] = v.y;
      xs[c + 2][r] = v.z;
      xs[c + 3][r] = v.w;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kGK; ++k) {
      const float4 a = *reinterpret_cast<const float4*>(&qs[k][ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&xs[k][tx * 8]);
      const float4 b1 = *reinterpret_cast<const float4*>(&xs[k][tx * 8 + 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int h = h0 + ty * 4 + i;
    if (h >= H) continue;
    float* out = logits + (g * H + h) * N + t0 + tx * 8;
    if (t0 + tx * 8 + 8 <= N && (N & 3) == 0) {
      reinterpret_cast<float4*>(out)[0] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      reinterpret_cast<float4*>(out)[1] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (t0 + tx * 8 + j < N) out[j] = acc[i][j];
    }
  }
}

// One mbarrier that nothing arrives on: thread 0 polls it with back-off, thread
// 32 with suspend hints; each gives up after its bounded number of polls.
__global__ void wait_expiry_kernel(int* err) {
  __shared__ __align__(8) unsigned long long bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  bool ok = true;
  if (threadIdx.x == 0) ok = ptx::mbar_wait(ptx::smem_u32(&bar), 0, &abort_flag);
  if (threadIdx.x == 32) ok = ptx::mbar_wait_suspend(ptx::smem_u32(&bar), 0, &abort_flag);
  if (!ok) atomicAdd(err, 1);
}

}  // namespace

cudaError_t launch_plan_derive(tq_plan* p, cudaStream_t s) {
  const int d = p->d;
  dim3 tb(32, 8), tg(d / 32, d / 32);
  transpose_kernel<<<tg, tb, 0, s>>>(p->Pi, d, p->PiT);
  if (p->lay.prod) {
    transpose_kernel<<<tg, tb, 0, s>>>(p->S, d, p->ST);
    dim3 b16(16, 16), g16(d / 16, d / 16);
    abt_f64_kernel<<<g16, b16, 0, s>>>(p->S, p->Pi, d, p->M, p->MT);
  }
  return cudaGetLastError();
}

template <int KT>
static cudaError_t launch_fp32_kt(const float* q, const float* x, int64_t G, int H, int64_t N, int d,
                                  float* logits, cudaStream_t s) {
  const size_t smem = (size_t)KT * d * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(score_fp32_kernel<KT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t ntile = (N + KT - 1) / KT;
  score_fp32_kernel<KT><<<(unsigned)(G * ntile), 256, smem, s>>>(q, x, G, H, N, d, logits);
  return cudaGetLastError();
}

// out0[g][h][t] = sum_j q[g][h][j] x0[t][j] (and out1 with x1, in the same
// launch, unless x1 is null) with matrices [N][d] shared by every group
// (d % 16 == 0): e.g. Pi q and S q for many queries at once.
cudaError_t launch_rows_times_shared(const float* q, const float* x0, const float* x1, int64_t G, int H, int64_t N,
                                     int d, float* out0, float* out1, cudaStream_t s) {
  if (G * N == 0 || H == 0) return cudaSuccess;
  if (d % kGK != 0) return cudaErrorInvalidValue;
  const int h_tiles = (H + kGH - 1) / kGH;
  const int64_t t_tiles = (N + kGT - 1) / kGT;
  const dim3 grid((unsigned)(G * t_tiles * h_tiles), x1 ? 2u : 1u);
  score_fp32_gemm_kernel<<<grid, 256, 0, s>>>(q, x0, x1 ? x1 : x0, 0, H, N, d, h_tiles, t_tiles, out0,
                                              x1 ? out1 : out0);
  return cudaGetLastError();
}

cudaError_t launch_wait_expiry(int* err, cudaStream_t s) {
  wait_expiry_kernel<<<1, 64, 0, s>>>(err);
  return cudaGetLastError();
}

cudaError_t launch_score_fp32(const float* q, const float* x, int64_t G, int H, int64_t N, int d,
                              float* logits, cudaStream_t s) {
  if (G * N == 0 || H == 0) return cudaSuccess;
  const size_t qbytes = (size_t)H * d * sizeof(float);
  if (d % kGK == 0 && (H > 16 || d > 1024)) {
    const int h_tiles = (H + kGH - 1) / kGH;
    const int64_t t_tiles = (N + kGT - 1) / kGT;
    const int64_t blocks = G * t_tiles * h_tiles;
    score_fp32_gemm_kernel<<<(unsigned)blocks, 256, 0, s>>>(q, x, x, N * (int64_t)d, H, N, d, h_tiles, t_tiles,
                                                            logits, logits);
    return cudaGetLastError();
  }
  if (d == 128 && qbytes <= 96 * 1024) {
    const int64_t n_tiles = G * ((N + kD128Tile - 1) / kD128Tile);
    cudaError_t e = cudaFuncSetAttribute(score_fp32_d128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)qbytes);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t grid = n_tiles < (int64_t)sms * 2 ? n_tiles : (int64_t)sms * 2;
    score_fp32_d128_kernel<<<(unsigned)grid, 256, qbytes, s>>>(q, x, G, H, N, n_tiles, logits);
    return cudaGetLastError();
  }
  if (d % 4 == 0 && d <= 1024 && qbytes <= 96 * 1024) {
    const int64_t n_tiles = G * ((N + kF32Tile - 1) / kF32Tile);
    cudaError_t e = cudaFuncSetAttribute(score_fp32_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)qbytes);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t grid = n_tiles < (int64_t)sms * 16 ? n_tiles : (int64_t)sms * 16;
    score_fp32_stream_kernel<<<(unsigned)grid, kF32Tile, qbytes, s>>>(q, x, G, H, N, d, n_tiles, logits);
    return cudaGetLastError();
  }
  if (d <= 1024) return launch_fp32_kt<32>(q, x, G, H, N, d, logits, s);
  return launch_fp32_kt<8>(q, x, G, H, N, d, logits, s);
}

}  // namespace tq
