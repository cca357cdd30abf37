// Internal declarations shared by libtq's CUDA sources (not installed).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tq.h"

namespace tq {

constexpr int kTokensPerBlock = 128;   // packed layout: tokens per block
constexpr int kChunk = 128;            // packed layout: coordinates per 16-byte chunk
constexpr int kMaxLevels = 16;
constexpr int kMaxD = 2048;

// Codebook and decision boundaries passed by value to kernels.
struct CodeParams {
  float c[kMaxLevels];      // ascending centroids (unit-norm scale)
  float t[kMaxLevels - 1];  // t_i = (c_i + c_{i+1}) / 2, fp32
  int L;                    // number of centroids
};

// Parity (Walsh) expansion of a codebook over its k index bits:
//   c[idx] = c0 + sum_t coef[t] * parity(idx & mask[t]),
// with only the terms whose coefficient is not zero.  Scoring contracts the
// XOR planes of the code bits against coef[t] Pi q.
constexpr int kMaxTerms = kMaxLevels - 1;
struct ParityExpansion {
  int n;
  uint32_t mask[kMaxTerms];
  float coef[kMaxTerms];
  float c0;
  // the same expansion in signed form, for arithmetic on sign bits:
  //   c[idx] = mid + sum_t (parity ? half[t] : -half[t]),
  // half[t] = coef[t] / 2 and mid = c0 + sum_t coef[t] / 2 (rounded from fp64)
  float half[kMaxTerms];
  float mid;
};

// Geometry of the packed layout for one plan.
struct Layout {
  int d;            // head dimension
  int k;            // code planes (code bits of the coordinates with the most)
  int planes;       // k (+1 sign plane in PROD)
  int C;            // 128-coordinate chunks per plane
  int prod;         // 1 for TurboQuantProd
  int frac;         // 1 for a fractional width: the first d/2 coordinates have k code
                    // bits, the others k - 1; code plane k - 1 is then a half plane
                    // of 8 bytes per 128 coordinates per token
  int64_t top_off;      // offset of code plane k - 1 inside a block
  int64_t sign_off;     // offset of the sign plane (PROD)
  int64_t block_bytes;  // bytes per 128-token block
  int64_t norms_off;    // offset of the norm pairs inside a block

  __host__ __device__ int64_t plane_off(int p, int c, int t) const {
    return ((int64_t)(p * C + c) * kTokensPerBlock + t) * 16;
  }
};

}  // namespace tq

struct tq_plan {
  int d, bits, mode;
  int device;
  tq::Layout lay;
  tq::CodeParams cp;
  tq::ParityExpansion px;  // codebook in parity form (tensor-core score)
  float kappa;        // sqrt(pi/2) / m
  int hadamard;       // 1: Pi = c H diag(signs), c = 1/sqrt(d) (tq_plan_create_hadamard)
  float rot_scale;    // c for a Hadamard plan, else 1
  tq::CodeParams cp_enc;       // the codebook as the d = 128 encode uses it: divided by c (Hadamard)
  tq::ParityExpansion px_enc;  // the same for the parity expansion
  // fractional width (lay.frac): the codebook of the last d/2 coordinates, with
  // 2^(k-1) levels (cp_lo, px_lo); padded to 2^k levels for the encode (never
  // reached thresholds at +inf, zero weights on the extra parity terms)
  tq::CodeParams cp_lo, cp_enc_lo;
  tq::ParityExpansion px_lo, px_enc_lo;
  uint32_t dec_ctab_lo[16];
  float* Pi;          // [d][d] row-major, y = Pi u
  float* PiT;         // [d][d] = Pi^T (coalesced column access in SIMT kernels)
  float* S;           // [d][d] (PROD)
  float* ST;          // [d][d] = S^T (PROD)
  float* M;           // [d][d] = S Pi^T (PROD)
  float* MT;          // [d][d] = M^T (PROD)
  uint16_t* wide_ops;  // row-major fp16 [4][d][d]: (2^8 Pi) hi, lo; (PROD) M hi, lo
  uint16_t* dec_wide_ops;  // d > 128: row-major fp16 [4][d][d]: (2^8 Pi^T) hi, lo; (PROD) (2^8 S^T) hi, lo
  void* wide_scratch;  // (PROD) residual rows of the wide encode: [wide_slots][2][128][d] bf16
  int wide_slots;      // SM ids of the device (%nsmid)
  uint8_t* tc_ops;    // tensor-core operand images (d = 128), 32 KB each, K-major
                      // 128-byte swizzle: Pi hi/lo fp16, Pi hi/lo bf16, (PROD) M hi/lo
                      // bf16; then for decode 2^8 Pi^T hi/lo and (PROD) 2^8 S^T hi/lo, fp16
  uint32_t dec_ctab[16];  // decode: fp16 bits of hi (low half) and lo (high half) of 2^8 c_i
  int* err;           // device error word
  uint64_t fingerprint;  // hash of d, bits, mode, kind and the bytes of Pi, S and the codebooks (packed-cache headers)
};

namespace tq {

// ---- launchers (one per kernel family); all return cudaGetLastError()
cudaError_t launch_plan_derive(tq_plan* p, cudaStream_t s);
bool encode_tc_supported(const tq_plan* p, tq_dtype dt);
// drop_first: error-path self-test only (CTA 0 withholds its first key tile)
cudaError_t launch_encode_tc(const tq_plan* p, const void* keys, tq_dtype dt, int64_t G, int64_t N, uint8_t* packed,
                             cudaStream_t s, bool drop_first = false);
cudaError_t launch_topk(const float* logits, int64_t rows, int64_t N, int k, float* top_scores,
                        int64_t* top_idx, void* ws, cudaStream_t s);
bool decode_tc_supported(const tq_plan* p);
bool decode_wide_supported(const tq_plan* p);
cudaError_t launch_decode_wide(const tq_plan* p, const uint8_t* packed, int64_t G, int64_t N, float* out,
                               cudaStream_t s);
cudaError_t launch_decode_tc(const tq_plan* p, const uint8_t* packed, int64_t G, int64_t N, float* out,
                             cudaStream_t s);
// index of decode image j in tc_ops (0, 1: Pi^T hi, lo; 2, 3: S^T hi, lo)
inline int tc_dec_image(const tq_plan* p, int j) { return (p->lay.prod ? 6 : 4) + j; }
cudaError_t launch_score_fp32(const float* q, const float* x, int64_t G, int H, int64_t N, int d,
                              float* logits, cudaStream_t s);
cudaError_t launch_wait_expiry(int* err, cudaStream_t s);
cudaError_t launch_rows_times_shared(const float* q, const float* x0, const float* x1, int64_t G, int H, int64_t N,
                                     int d, float* out0, float* out1, cudaStream_t s);

size_t topk_workspace_bytes(int64_t rows, int64_t N, int k);

bool score_tc_supported(const tq_plan* p, int H);
size_t score_tc_workspace_bytes(const tq_plan* p, int64_t G, int H);
cudaError_t launch_score_tc(const tq_plan* p, const float* queries, int64_t G, int H, const uint8_t* packed,
                            int64_t N, float* logits, void* ws, cudaStream_t s);

bool encode_wide_supported(const tq_plan* p, tq_dtype dt);
cudaError_t launch_encode_wide(const tq_plan* p, const void* keys, tq_dtype dt, int64_t G, int64_t N,
                               uint8_t* packed, cudaStream_t s);
int query_nsmid();
bool score_wide_supported(const tq_plan* p, int H);
size_t score_wide_workspace_bytes(const tq_plan* p, int64_t G, int H);
cudaError_t launch_score_wide(const tq_plan* p, const float* queries, int64_t G, int H, const uint8_t* packed,
                              int64_t N, float* logits, void* ws, cudaStream_t s);

// Attention of a decode step (k_attend.cu): keys of a Prod plan, values of an
// MSE plan in the coordinate-major value layout.
cudaError_t launch_values_layout(const tq_plan* p, uint8_t* packed, int64_t n_blocks, cudaStream_t s);
bool attend_supported(const tq_plan* kp, const tq_plan* vp, int H);
size_t attend_workspace_bytes(const tq_plan* kp, const tq_plan* vp, int64_t G, int H, int64_t N);
cudaError_t launch_attend(const tq_plan* kp, const tq_plan* vp, const float* q, int64_t G, int H,
                          const uint8_t* kpacked, const uint8_t* vpacked, int64_t N, float scale, float* out,
                          void* ws, cudaStream_t s);

// Scoring as tq_score performs it (query preparation, score kernel, optional
// top-k) on a caller-provided workspace of at least score_workspace_bytes().
size_t score_workspace_bytes(const tq_plan* p, int64_t G, int H, int64_t N, int top_k);
cudaError_t score_run(const tq_plan* p, const float* queries, int64_t G, int H, const uint8_t* packed, int64_t N,
                      float* logits, int top_k, float* top_scores, int64_t* top_idx, void* ws, cudaStream_t s);

__device__ __forceinline__ float load_key(const void* keys, int dt, int64_t i) {
  if (dt == TQ_F32) return reinterpret_cast<const float*>(keys)[i];
  if (dt == TQ_F16) return __half2float(reinterpret_cast<const __half*>(keys)[i]);
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(keys)[i]);
}

// idx = #{i : t_i < y} (a value on a boundary takes the lower index)
__device__ __forceinline__ int quantize_index(float y, const CodeParams& cp) {
  int idx = 0;
#pragma unroll
  for (int i = 0; i < kMaxLevels - 1; ++i)
    if (i < cp.L - 1) idx += (y > cp.t[i]) ? 1 : 0;
  return idx;
}

}  // namespace tq
