// Query preparation, score on packed keys (CUDA-core version) and top-k.
//
// Score follows the usage listing of "turboquant-pytorch 소개"
// (``tq.inner_product(query, compressed)``) and its "2단계" paragraph: the
// inner product is estimated without reconstructing the key,
//     <q, x> ~ n <Pi q, c[idx]> + rho sqrt(pi/2)/m <S q, sign(S r)>,
// which equals <q, n Pi^T c[idx]> + the QJL term because Pi is orthogonal.
// Each query is rotated and projected once (query prep); every packed key
// byte is then read once for all H query heads of its group (GQA batching).
#include "tq_internal.cuh"

namespace tq {
namespace {

// qs[g][h][0][:] = Pi q, qs[g][h][1][:] = S q (PROD only)
__global__ void query_prep_kernel(const float* __restrict__ q, int64_t GH, int d, int prod,
                                  const float* __restrict__ PiT, const float* __restrict__ ST,
                                  float* __restrict__ qs) {
  extern __shared__ float sq[];
  const int64_t row = blockIdx.x;
  if (row >= GH) return;
  for (int i = threadIdx.x; i < d; i += blockDim.x) sq[i] = q[row * d + i];
  __syncthreads();
  const int nv = prod ? 2 : 1;
  for (int j = threadIdx.x; j < d; j += blockDim.x) {
    float a = 0.f, b = 0.f;
    for (int i = 0; i < d; ++i) {
      a = fmaf(__ldg(PiT + (int64_t)i * d + j), sq[i], a);
      if (prod) b = fmaf(__ldg(ST + (int64_t)i * d + j), sq[i], b);
    }
    qs[(row * nv + 0) * d + j] = a;
    if (prod) qs[(row * nv + 1) * d + j] = b;
  }
}

// One CTA per (group, 128-token block); thread t scores token t against HC heads
// at a time.
template <int HC>
__global__ void __launch_bounds__(128)
score_simt_kernel(const float* __restrict__ qs, int64_t G, int H, Layout lay, CodeParams cp, float kappa,
                  const uint8_t* __restrict__ packed, int64_t N, float* __restrict__ logits) {
  extern __shared__ float sm[];
  const int d = lay.d;
  const int nv = lay.prod ? 2 : 1;
  float* s_qr = sm;              // [HC][d]
  float* s_sq = sm + HC * d;     // [HC][d]
  __shared__ float s_c[kMaxLevels];
  const int64_t nb = (N + kTokensPerBlock - 1) / kTokensPerBlock;
  const int64_t gb = blockIdx.x;
  const int64_t g = gb / nb, blk = gb % nb;
  const int t = threadIdx.x;
  const int64_t tok = blk * kTokensPerBlock + t;
  const uint8_t* in = packed + gb * lay.block_bytes;
  if (t < kMaxLevels) s_c[t] = t < cp.L ? cp.c[t] : 0.f;
  const float2 nr = *reinterpret_cast<const float2*>(in + lay.norms_off + (int64_t)t * 8);

  for (int h0 = 0; h0 < H; h0 += HC) {
    const int hc = min(HC, H - h0);
    __syncthreads();
    for (int i = t; i < hc * d; i += blockDim.x) {
      int h = i / d, j = i - h * d;
      const float* src = qs + (((g * H + h0 + h) * nv) * (int64_t)d);
      s_qr[i] = src[j];
      if (lay.prod) s_sq[i] = src[d + j];
    }
    __syncthreads();
    float A[HC], B[HC];
#pragma unroll
    for (int h = 0; h < HC; ++h) A[h] = B[h] = 0.f;
    for (int c = 0; c < lay.C; ++c) {
      uint4 w[5];
      for (int p = 0; p < lay.planes; ++p)
        w[p] = *reinterpret_cast<const uint4*>(in + lay.plane_off(p, c, t));
      for (int wd = 0; wd < 4; ++wd) {
        unsigned pw[5];
        for (int p = 0; p < lay.planes; ++p) pw[p] = wd == 0 ? w[p].x : wd == 1 ? w[p].y : wd == 2 ? w[p].z : w[p].w;
        for (int i = 0; i < 32; ++i) {
          const int j = c * kChunk + wd * 32 + i;
          int idx = 0;
          for (int p = 0; p < lay.k; ++p) idx |= ((pw[p] >> i) & 1u) << p;
          const float cv = s_c[idx];
          const bool pos = lay.prod ? ((pw[lay.k] >> i) & 1u) : false;
#pragma unroll
          for (int h = 0; h < HC; ++h) {
            if (h < hc) {
              A[h] = fmaf(s_qr[h * d + j], cv, A[h]);
              if (lay.prod) {
                float sv = s_sq[h * d + j];
                B[h] += pos ? sv : -sv;
              }
            }
          }
        }
      }
    }
    if (tok < N) {
#pragma unroll
      for (int h = 0; h < HC; ++h) {
        if (h < hc) {
          float v = nr.x * A[h];
          if (lay.prod) v = fmaf(nr.y * kappa, B[h], v);
          logits[((g * H) + h0 + h) * N + tok] = v;
        }
      }
    }
  }
}

// ---------------------------------------------------------------- top-k
// Stage 1: CTA (row, split) keeps, per thread, the best K of a strided slice,
// then merges them into the split's best K (written to the workspace).
// Stage 2: one CTA per row merges the splits.  Order: descending score, ties to
// the lower index.

__device__ __forceinline__ bool better(float a, int64_t ia, float b, int64_t ib) {
  return a > b || (a == b && ia < ib);
}

constexpr int kTopkThreads = 128;

__device__ void block_merge(float* cs, int64_t* ci, int* cnt, int K, float* out_s, int64_t* out_i) {
  // cs/ci: [kTopkThreads][K] sorted candidate lists (shared); cnt: per-thread lengths
  __shared__ float rs[kTopkThreads];
  __shared__ int64_t ri[kTopkThreads];
  __shared__ int rt[kTopkThreads];
  const int t = threadIdx.x;
  int head = 0;
  for (int r = 0; r < K; ++r) {
    rs[t] = head < cnt[t] ? cs[t * K + head] : -INFINITY;
    ri[t] = head < cnt[t] ? ci[t * K + head] : INT64_MAX;
    rt[t] = t;
    __syncthreads();
    for (int s = kTopkThreads / 2; s; s >>= 1) {
      if (t < s && better(rs[t + s], ri[t + s], rs[t], ri[t])) {
        rs[t] = rs[t + s];
        ri[t] = ri[t + s];
        rt[t] = rt[t + s];
      }
      __syncthreads();
    }
    if (t == 0) {
      out_s[r] = rs[0];
      out_i[r] = ri[0];
    }
    const int win = rt[0];
    __syncthreads();
    if (t == win) ++head;
  }
}

__global__ void __launch_bounds__(kTopkThreads)
topk_stage1(const float* __restrict__ x, int64_t N, int K, int splits, float* ws_s, int64_t* ws_i) {
  extern __shared__ unsigned char tk_sm[];
  float* cs = reinterpret_cast<float*>(tk_sm);
  int64_t* ci = reinterpret_cast<int64_t*>(cs + kTopkThreads * K + (kTopkThreads * K) % 2);
  __shared__ int cnt[kTopkThreads];
  const int64_t row = blockIdx.x / splits;
  const int sp = blockIdx.x % splits;
  const int64_t per = (N + splits - 1) / splits;
  const int64_t lo = sp * per, hi = min(N, lo + per);
  const float* xr = x + row * N;
  const int t = threadIdx.x;
  float* my_s = cs + t * K;
  int64_t* my_i = ci + t * K;
  int n = 0;
  // the thread's current k-th best, kept in registers (most values fail the test)
  float th_s = 0.f;
  int64_t th_i = 0;
  // eight independent loads in flight per step, then the tests in order
  constexpr int kU = 8;
  for (int64_t i0 = lo + t; i0 < hi; i0 += kU * kTopkThreads) {
    float vs[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t i = i0 + (int64_t)u * kTopkThreads;
      vs[u] = i < hi ? __ldg(xr + i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t i = i0 + (int64_t)u * kTopkThreads;
      const float v = vs[u];
      if (i >= hi || (n == K && !better(v, i, th_s, th_i))) continue;
      int pos = n < K ? n : K - 1;
      while (pos > 0 && better(v, i, my_s[pos - 1], my_i[pos - 1])) {
        my_s[pos] = my_s[pos - 1];
        my_i[pos] = my_i[pos - 1];
        --pos;
      }
      my_s[pos] = v;
      my_i[pos] = i;
      if (n < K) ++n;
      if (n == K) {
        th_s = my_s[K - 1];
        th_i = my_i[K - 1];
      }
    }
  }
  cnt[t] = n;
  __syncthreads();
  const int64_t o = (row * splits + sp) * K;
  block_merge(cs, ci, cnt, K, ws_s + o, ws_i + o);
}

__global__ void __launch_bounds__(kTopkThreads)
topk_stage2(const float* ws_s, const int64_t* ws_i, int splits, int K, float* out_s, int64_t* out_i) {
  extern __shared__ unsigned char tk_sm[];
  float* cs = reinterpret_cast<float*>(tk_sm);
  int64_t* ci = reinterpret_cast<int64_t*>(cs + kTopkThreads * K + (kTopkThreads * K) % 2);
  __shared__ int cnt[kTopkThreads];
  const int64_t row = blockIdx.x;
  const int t = threadIdx.x;
  // thread t owns splits t, t + 128, ...: merge them into its own sorted list
  int n = 0;
  for (int sp = t; sp < splits; sp += kTopkThreads) {
    const float* s = ws_s + (row * splits + sp) * K;
    const int64_t* ix = ws_i + (row * splits + sp) * K;
    for (int r = 0; r < K; ++r) {
      float v = s[r];
      int64_t i = ix[r];
      if (i == INT64_MAX) break;
      if (n == K && !better(v, i, cs[t * K + K - 1], ci[t * K + K - 1])) break;
      int pos = n < K ? n : K - 1;
      while (pos > 0 && better(v, i, cs[t * K + pos - 1], ci[t * K + pos - 1])) {
        cs[t * K + pos] = cs[t * K + pos - 1];
        ci[t * K + pos] = ci[t * K + pos - 1];
        --pos;
      }
      cs[t * K + pos] = v;
      ci[t * K + pos] = i;
      if (n < K) ++n;
    }
  }
  cnt[t] = n;
  __syncthreads();
  block_merge(cs, ci, cnt, K, out_s + row * K, out_i + row * K);
}

int topk_splits(int64_t rows, int64_t N, int K) {
  int64_t s = (1184 + rows - 1) / rows;    // about eight CTAs per SM in total
  int64_t cap = N / (4 * (int64_t)K * kTopkThreads);  // keep every thread busy
  if (s > cap) s = cap;
  if (s < 1) s = 1;
  if (s > 1024) s = 1024;
  return (int)s;
}

size_t topk_smem(int K) { return (size_t)kTopkThreads * K * (sizeof(float) + sizeof(int64_t)) + 8; }

}  // namespace

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t topk_workspace_bytes(int64_t rows, int64_t N, int k) {
  if (k <= 0) return 0;
  const size_t n = (size_t)rows * topk_splits(rows, N, k) * k;
  return align256(n * sizeof(float)) + n * sizeof(int64_t);
}

cudaError_t launch_query_prep(const tq_plan* p, const float* q, int64_t G, int H, float* qs, cudaStream_t s) {
  const int64_t GH = G * H;
  if (GH == 0) return cudaSuccess;
  query_prep_kernel<<<(unsigned)GH, 128, p->d * sizeof(float), s>>>(q, GH, p->d, p->lay.prod, p->PiT, p->ST, qs);
  return cudaGetLastError();
}

template <int HC>
static cudaError_t launch_score_hc(const tq_plan* p, const float* qs, int64_t G, int H, const uint8_t* packed,
                                   int64_t N, float* logits, cudaStream_t s) {
  const size_t smem = (size_t)2 * HC * p->d * sizeof(float);
  auto kern = score_simt_kernel<HC>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t nb = (N + kTokensPerBlock - 1) / kTokensPerBlock;
  kern<<<(unsigned)(G * nb), 128, smem, s>>>(qs, G, H, p->lay, p->cp, p->kappa, packed, N, logits);
  return cudaGetLastError();
}

cudaError_t launch_score_simt(const tq_plan* p, const float* qs, int64_t G, int H, const uint8_t* packed,
                              int64_t N, float* logits, cudaStream_t s) {
  if (G * N == 0) return cudaSuccess;
  if (p->d <= 512) return launch_score_hc<8>(p, qs, G, H, packed, N, logits, s);
  if (p->d <= 1024) return launch_score_hc<4>(p, qs, G, H, packed, N, logits, s);
  return launch_score_hc<2>(p, qs, G, H, packed, N, logits, s);
}

cudaError_t launch_topk(const float* logits, int64_t rows, int64_t N, int k, float* top_scores,
                        int64_t* top_idx, void* ws, cudaStream_t s) {
  if (rows == 0 || k == 0) return cudaSuccess;
  const int splits = topk_splits(rows, N, k);
  const size_t n = (size_t)rows * splits * k;
  float* ws_s = reinterpret_cast<float*>(ws);
  int64_t* ws_i = reinterpret_cast<int64_t*>(reinterpret_cast<char*>(ws) + align256(n * sizeof(float)));
  const size_t smem = topk_smem(k);
  cudaError_t e = cudaFuncSetAttribute(topk_stage1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(topk_stage2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  topk_stage1<<<(unsigned)(rows * splits), kTopkThreads, smem, s>>>(logits, N, k, splits, ws_s, ws_i);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  topk_stage2<<<(unsigned)rows, kTopkThreads, smem, s>>>(ws_s, ws_i, splits, k, top_scores, top_idx);
  return cudaGetLastError();
}

}  // namespace tq
