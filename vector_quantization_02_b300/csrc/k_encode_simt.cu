// Encode, exact-fp32 CUDA-core version (any d that is a multiple of 128).
//
// Follows "turboquant-pytorch 소개" (discuss.pytorch.kr): "1단계" (normalise,
// rotate by Pi, quantise every coordinate with the Lloyd-Max codebook) and
// "2단계" (signs of a Gaussian projection of the quantisation residual).
// The residual projection is taken in the rotated frame: with y = Pi x / n and
// r' = y - c[idx],  S r = n S Pi^T r' = n M r'  (M = S Pi^T, derived once per
// plan), equal to S (x - n Pi^T c[idx]) for orthogonal Pi; and ||r|| = n ||r'||.
//
// One CTA (256 threads) takes KB keys at a time: keys are staged in shared
// memory as fp32; thread j computes output coordinate j of Y = X Pi^T for all
// KB keys (Pi^T rows read coalesced, keys broadcast from shared memory), so a
// warp holds 32 consecutive coordinates of a key and one ballot packs a
// 32-coordinate code word.  Then the same for P = R' M^T and the sign plane.
#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kThreads = 256;

template <int KB>
__global__ void __launch_bounds__(kThreads)
encode_simt_kernel(const void* __restrict__ keys, int dt, int64_t G, int64_t N, Layout lay,
                   CodeParams cp, const float* __restrict__ PiT, const float* __restrict__ MT,
                   uint8_t* __restrict__ packed) {
  extern __shared__ float smem[];
  const int d = lay.d;
  float* X = smem;                 // [KB][d] keys, then reused as nothing
  float* R = smem + KB * d;        // [KB][d] residual r' (unit scale)
  __shared__ float s_inv[KB], s_n[KB], s_rr[KB];

  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t nb = (N + kTokensPerBlock - 1) / kTokensPerBlock;
  const int tiles_per_block = kTokensPerBlock / KB;
  const int64_t n_tiles = G * nb * tiles_per_block;

  for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const int64_t gb = tile / tiles_per_block;          // (group, block)
    const int64_t g = gb / nb, blk = gb % nb;
    const int t0 = (int)(tile % tiles_per_block) * KB;  // first token of the tile within the block
    const int64_t tok0 = blk * kTokensPerBlock + t0;
    uint8_t* out = packed + gb * lay.block_bytes;

    // stage the keys (coalesced), zero for padded tokens
    for (int i = tid; i < KB * d; i += kThreads) {
      int kk = i / d, col = i - kk * d;
      int64_t tok = tok0 + kk;
      X[i] = tok < N ? load_key(keys, dt, (g * N + tok) * d + col) : 0.f;
    }
    if (tid < KB) s_rr[tid] = 0.f;
    __syncthreads();
    // norms: warp w takes keys w, w+8, ...; fp64 accumulation
    for (int kk = tid >> 5; kk < KB; kk += kThreads / 32) {
      double acc = 0.0;
      for (int col = lane; col < d; col += 32) acc += (double)X[kk * d + col] * X[kk * d + col];
      for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) {
        float n = (float)sqrt(acc);
        s_n[kk] = n;
        s_inv[kk] = n > 0.f ? 1.f / n : 0.f;
      }
    }
    __syncthreads();

    // Y = X Pi^T, quantise, residual, code planes
    float rr[KB];
#pragma unroll
    for (int kk = 0; kk < KB; ++kk) rr[kk] = 0.f;
    for (int j = tid; j < d; j += kThreads) {
      float acc[KB];
#pragma unroll
      for (int kk = 0; kk < KB; ++kk) acc[kk] = 0.f;
      for (int i = 0; i < d; ++i) {
        float w = __ldg(PiT + (int64_t)i * d + j);
#pragma unroll
        for (int kk = 0; kk < KB; ++kk) acc[kk] = fmaf(X[kk * d + i], w, acc[kk]);
      }
      const int c = j / kChunk, wd = (j % kChunk) / 32;
#pragma unroll
      for (int kk = 0; kk < KB; ++kk) {
        float y = acc[kk] * s_inv[kk];
        int idx = quantize_index(y, cp);
        float r = y - cp.c[idx];
        R[kk * d + j] = r;
        rr[kk] = fmaf(r, r, rr[kk]);
        const bool live = tok0 + kk < N;
        for (int p = 0; p < lay.k; ++p) {
          unsigned word = __ballot_sync(0xffffffffu, (idx >> p) & 1);
          if (lane == 0) {
            *reinterpret_cast<unsigned*>(out + lay.plane_off(p, c, t0 + kk) + 4 * wd) = live ? word : 0u;
          }
        }
      }
    }
#pragma unroll
    for (int kk = 0; kk < KB; ++kk) {
      float v = rr[kk];
      for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) atomicAdd(&s_rr[kk], v);
    }
    __syncthreads();

    if (lay.prod) {
      // P = R' M^T; z = [p >= 0] (forced to 1 for a zero key)
      for (int j = tid; j < d; j += kThreads) {
        float acc[KB];
#pragma unroll
        for (int kk = 0; kk < KB; ++kk) acc[kk] = 0.f;
        for (int i = 0; i < d; ++i) {
          float w = __ldg(MT + (int64_t)i * d + j);
#pragma unroll
          for (int kk = 0; kk < KB; ++kk) acc[kk] = fmaf(R[kk * d + i], w, acc[kk]);
        }
        const int c = j / kChunk, wd = (j % kChunk) / 32;
#pragma unroll
        for (int kk = 0; kk < KB; ++kk) {
          bool z = acc[kk] >= 0.f || s_n[kk] == 0.f;
          unsigned word = __ballot_sync(0xffffffffu, z);
          if (lane == 0) {
            const bool live = tok0 + kk < N;
            *reinterpret_cast<unsigned*>(out + lay.plane_off(lay.k, c, t0 + kk) + 4 * wd) = live ? word : 0u;
          }
        }
      }
    }
    if (tid < KB) {
      const bool live = tok0 + tid < N;
      float2 nr;
      nr.x = live ? s_n[tid] : 0.f;
      nr.y = (live && lay.prod) ? s_n[tid] * sqrtf(s_rr[tid]) : 0.f;
      *reinterpret_cast<float2*>(out + lay.norms_off + (int64_t)(t0 + tid) * 8) = nr;
    }
    __syncthreads();
  }
}

template <int KB>
cudaError_t launch_kb(const tq_plan* p, const void* keys, tq_dtype dt, int64_t G, int64_t N,
                      uint8_t* packed, cudaStream_t s) {
  const size_t smem = (size_t)2 * KB * p->d * sizeof(float);
  auto kern = encode_simt_kernel<KB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int per_sm = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
  const int64_t nb = (N + kTokensPerBlock - 1) / kTokensPerBlock;
  const int64_t tiles = G * nb * (kTokensPerBlock / KB);
  int64_t grid = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
  if (grid > tiles) grid = tiles;
  kern<<<(unsigned)grid, kThreads, smem, s>>>(keys, (int)dt, G, N, p->lay, p->cp, p->PiT, p->MT, packed);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_encode_simt(const tq_plan* p, const void* keys, tq_dtype dt, int64_t G, int64_t N,
                               uint8_t* packed, cudaStream_t s) {
  if (p->d <= 128) return launch_kb<32>(p, keys, dt, G, N, packed, s);
  if (p->d <= 256) return launch_kb<16>(p, keys, dt, G, N, packed, s);
  return launch_kb<8>(p, keys, dt, G, N, packed, s);
}

}  // namespace tq
