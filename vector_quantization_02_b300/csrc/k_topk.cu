// Top-k of each row of the logits (the vector-search step keeps the best 10
// keys per query): descending score, ties to the lower key index.
#include "tq_internal.cuh"

namespace tq {
namespace {

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
  // cs/ci: [kTopkThreads][K] sorted candidate lists (shared); cnt: per-thread lengths.
  // Each round takes the best head of all lists: a butterfly over each warp,
  // then the four warp winners; the winning thread advances its head.
  constexpr int kWarps = kTopkThreads / 32;
  __shared__ float ws_s[kWarps];
  __shared__ int64_t ws_i[kWarps];
  __shared__ int ws_t[kWarps];
  __shared__ int win;
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
  int head = 0;
  for (int r = 0; r < K; ++r) {
    float v = head < cnt[t] ? cs[t * K + head] : -INFINITY;
    int64_t ix = head < cnt[t] ? ci[t * K + head] : INT64_MAX;
    int tt = t;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
      const int64_t i2 = __shfl_xor_sync(0xffffffffu, ix, o);
      const int t2 = __shfl_xor_sync(0xffffffffu, tt, o);
      if (better(v2, i2, v, ix)) {
        v = v2;
        ix = i2;
        tt = t2;
      }
    }
    if (lane == 0) {
      ws_s[wid] = v;
      ws_i[wid] = ix;
      ws_t[wid] = tt;
    }
    __syncthreads();
    if (t == 0) {
      int b = 0;
      for (int w = 1; w < kWarps; ++w)
        if (better(ws_s[w], ws_i[w], ws_s[b], ws_i[b])) b = w;
      out_s[r] = ws_s[b];
      out_i[r] = ws_i[b];
      win = ws_t[b];
    }
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
