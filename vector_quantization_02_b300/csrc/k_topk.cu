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

// Elements of a row per split: rows of a multiple of 4 elements are split on
// multiples of 4, so that every split starts on a 16-byte boundary.
__host__ __device__ inline int64_t topk_per(int64_t N, int splits) {
  const int64_t per = (N + splits - 1) / splits;
  return (N & 3) == 0 ? (per + 3) & ~(int64_t)3 : per;
}

// Order-preserving code of a float (unsigned order = float order, -0 as +0):
// a value whose code is below another's is strictly smaller.
__device__ __forceinline__ uint32_t order_code(float v) {
  const uint32_t b = __float_as_uint(v + 0.f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__global__ void __launch_bounds__(kTopkThreads)
topk_stage1(const float* __restrict__ x, int64_t N, int K, int splits, float* ws_s, int64_t* ws_i) {
  extern __shared__ unsigned char tk_sm[];
  float* cs = reinterpret_cast<float*>(tk_sm);
  int64_t* ci = reinterpret_cast<int64_t*>(cs + kTopkThreads * K + (kTopkThreads * K) % 2);
  __shared__ int cnt[kTopkThreads];
  // a lower bound on the split's k-th best: the best of the full threads'
  // k-th bests (such a thread holds K values at least as good), as a code
  __shared__ uint32_t s_bound;
  if (threadIdx.x == 0) s_bound = 0u;
  __syncthreads();
  volatile uint32_t* bound = &s_bound;
  const int64_t row = blockIdx.x / splits;
  const int sp = blockIdx.x % splits;
  const int64_t per = topk_per(N, splits);
  const int64_t lo = min(N, sp * per), hi = min(N, lo + per);
  const float* xr = x + row * N;
  const int t = threadIdx.x;
  float* my_s = cs + t * K;
  int64_t* my_i = ci + t * K;
  int n = 0;
  // the thread's current k-th best, kept in registers (most values fail the test)
  float th_s = 0.f;
  int64_t th_i = 0;
  auto consider = [&](float v, int64_t i, uint32_t lb) {
    // below the split's bound (strictly), or not better than this thread's k-th
    if (order_code(v) < lb || (n == K && !better(v, i, th_s, th_i))) return;
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
      if (th_s == th_s) atomicMax(&s_bound, order_code(th_s));  // (a NaN bounds nothing)
    }
  };
  if (K <= 32) {
    // one list per warp, held in registers: lane l < K has the warp's l-th
    // best.  A value enters when it beats the warp's k-th best (lane K - 1)
    // and is not below the split's bound; the lanes offering one are taken in
    // turn (a ballot), and each insertion is a count of the entries ahead of
    // it and a shift of those behind (shuffles): a few warp instructions, not
    // every lane's insertion loop.  Every shuffle and ballot takes the whole
    // warp, so the loops below run on warp-uniform bounds; lanes past the end
    // offer nothing.
    constexpr unsigned kAll = 0xffffffffu;
    const int lane = t & 31, wid = t >> 5;
    float ls = -INFINITY;
    int64_t li = INT64_MAX;  // this lane's entry (an empty entry loses to every value)
    float tv = -INFINITY;
    int64_t tix = INT64_MAX;  // the warp's k-th best
    auto passes = [&](float v, int64_t i, uint32_t lb) { return order_code(v) >= lb && better(v, i, tv, tix); };
    auto offer = [&](float v, int64_t i, bool cand) {
      unsigned m = __ballot_sync(kAll, cand);
      while (m) {
        const int src = __ffs(m) - 1;
        m &= m - 1;
        const float cv = __shfl_sync(kAll, v, src);
        const int64_t cx = __shfl_sync(kAll, i, src);
        if (better(cv, cx, tv, tix)) {  // (the list may have improved since it was offered)
          const int pos = __popc(__ballot_sync(kAll, lane < K && better(ls, li, cv, cx)));
          const float us = __shfl_up_sync(kAll, ls, 1);
          const int64_t ux = __shfl_up_sync(kAll, li, 1);
          if (lane > pos) {
            ls = us;
            li = ux;
          } else if (lane == pos) {
            ls = cv;
            li = cx;
          }
          tv = __shfl_sync(kAll, ls, K - 1);
          tix = __shfl_sync(kAll, li, K - 1);
          if (lane == 0 && tix != INT64_MAX && tv == tv) atomicMax(&s_bound, order_code(tv));
        }
      }
    };
    if ((N & 3) == 0) {
      const float4* xr4 = reinterpret_cast<const float4*>(xr);
      const int64_t lo4 = lo >> 2, hi4 = hi >> 2;
      constexpr int kU = 4;
      for (int64_t jw = lo4 + wid * 32; jw < hi4; jw += kU * kTopkThreads) {
        float4 vs[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int64_t j = jw + lane + (int64_t)u * kTopkThreads;
          vs[u] = j < hi4 ? __ldg(xr4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int64_t j = jw + lane + (int64_t)u * kTopkThreads;
          const bool ok = j < hi4;
          const float4 v = vs[u];
          const uint32_t lb = *bound;
          if (!__any_sync(kAll, ok && passes(fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)), -1, lb))) continue;
          offer(v.x, 4 * j, ok && passes(v.x, 4 * j, lb));
          offer(v.y, 4 * j + 1, ok && passes(v.y, 4 * j + 1, lb));
          offer(v.z, 4 * j + 2, ok && passes(v.z, 4 * j + 2, lb));
          offer(v.w, 4 * j + 3, ok && passes(v.w, 4 * j + 3, lb));
        }
      }
    } else {
      constexpr int kU = 8;
      for (int64_t iw = lo + wid * 32; iw < hi; iw += kU * kTopkThreads) {
        float vs[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int64_t i = iw + lane + (int64_t)u * kTopkThreads;
          vs[u] = i < hi ? __ldg(xr + i) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int64_t i = iw + lane + (int64_t)u * kTopkThreads;
          offer(vs[u], i, i < hi && passes(vs[u], i, *bound));
        }
      }
    }
    // the warp's list becomes list number wid of the block merge
    if (lane < K) {
      cs[wid * K + lane] = ls;
      ci[wid * K + lane] = li;
    }
    const int filled = __popc(__ballot_sync(kAll, lane < K && li != INT64_MAX));
    cnt[t] = 0;
    __syncthreads();
    if (lane == 0) cnt[wid] = filled;
  } else {
    if ((N & 3) == 0) {
      // the row and the split start on 16-byte boundaries: four values per load,
      // four loads in flight per step, and four values rejected by one test of
      // their maximum against this thread's k-th best and the split's bound (a
      // value equal to either is still tested alone, for the lower-index rule;
      // a NaN never enters)
      const float4* xr4 = reinterpret_cast<const float4*>(xr);
      const int64_t lo4 = lo >> 2, hi4 = hi >> 2;
      constexpr int kU = 4;
      for (int64_t j0 = lo4 + t; j0 < hi4; j0 += kU * kTopkThreads) {
        float4 vs[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int64_t j = j0 + (int64_t)u * kTopkThreads;
          vs[u] = j < hi4 ? __ldg(xr4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int64_t j = j0 + (int64_t)u * kTopkThreads;
          if (j >= hi4) continue;
          const float4 v = vs[u];
          const float m = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
          const uint32_t lb = *bound;
          if ((n == K && m < th_s) || order_code(m) < lb) continue;
          consider(v.x, 4 * j, lb);
          consider(v.y, 4 * j + 1, lb);
          consider(v.z, 4 * j + 2, lb);
          consider(v.w, 4 * j + 3, lb);
        }
      }
    } else {
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
          if (i < hi) consider(vs[u], i, *bound);
        }
      }
    }
    cnt[t] = n;
  }
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
