// The C ABI of libtq.so: argument checks, plan lifetime, dispatch.
// Declarations, layouts and error behaviour are documented in include/tq.h.
#include <cuda.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>
#include <type_traits>
#include <cstddef>
#include <vector>

#include "ptx_sm100.cuh"
#include "tq_internal.cuh"

using namespace tq;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

tq_status from_cuda(cudaError_t e) {
  return e == cudaSuccess ? TQ_OK : e == cudaErrorNotSupported ? TQ_EUNSUPPORTED : TQ_ECUDA;
}

void free_plan(tq_plan* p) {
  if (!p) return;
  float* bufs[] = {p->Pi, p->PiT, p->S, p->ST, p->M, p->MT};
  for (float* b : bufs)
    if (b) cudaFree(b);
  if (p->err) cudaFree(p->err);
  if (p->tc_ops) cudaFree(p->tc_ops);
  if (p->wide_ops) cudaFree(p->wide_ops);
  if (p->dec_wide_ops) cudaFree(p->dec_wide_ops);
  if (p->wide_scratch) cudaFree(p->wide_scratch);
  delete p;
}


// Byte offset of element (n, k) of a 128 x 128 16-bit matrix stored as the
// tensor cores read a K-major operand with the 128-byte swizzle: two 64-wide
// K halves of 16 KB; in each, row n at (n / 8) * 1024 + (n % 8) * 128 and its
// 16-byte chunk c at position c ^ (n % 8).
size_t sw128_offset(int n, int k) {
  return (size_t)(k / 64) * 16384 + (size_t)(n / 8) * 1024 + (n % 8) * 128 + ((((k % 64) / 8) ^ (n % 8)) * 16) +
         (k % 8) * 2;
}

// Splits a row-major 128 x 128 fp32 matrix into hi + lo in a 16-bit type and
// writes both swizzled images.
template <typename T>
void split_images(const float* A, uint8_t* hi, uint8_t* lo) {
  for (int n = 0; n < 128; ++n)
    for (int k = 0; k < 128; ++k) {
      const float v = A[n * 128 + k];
      T h, l;
      float hf;
      if constexpr (sizeof(T) == 2 && std::is_same<T, __half>::value) {
        h = __float2half_rn(v);
        hf = __half2float(h);
        l = __float2half_rn(v - hf);
      } else {
        h = __float2bfloat16_rn(v);
        hf = __bfloat162float(h);
        l = __float2bfloat16_rn(v - hf);
      }
      std::memcpy(hi + sw128_offset(n, k), &h, 2);
      std::memcpy(lo + sw128_offset(n, k), &l, 2);
    }
}

// Row-major fp16 hi + lo splits of 2^8 Pi and (Prod) of M for the wide
// tensor-core encode, and (Prod) its per-SM residual scratch; any d.  The power of two
// keeps the lo parts of Pi's entries (|Pi_ij| ~ d^-1/2) out of the fp16
// subnormal range; M = S Pi^T has entries of order 1.
cudaError_t build_wide_ops(tq_plan* p) {
  const size_t dd = (size_t)p->d * p->d;
  std::vector<float> Pi(dd), M(p->lay.prod ? dd : 0);
  cudaError_t e = cudaMemcpy(Pi.data(), p->Pi, dd * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && p->lay.prod) e = cudaMemcpy(M.data(), p->M, dd * 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return e;
  std::vector<uint16_t> host((p->lay.prod ? 4 : 2) * dd);
  auto split = [&](float v, size_t hi_at, size_t lo_at) {
    const __half h = __float2half_rn(v);
    const __half l = __float2half_rn(v - __half2float(h));
    std::memcpy(&host[hi_at], &h, 2);
    std::memcpy(&host[lo_at], &l, 2);
  };
  for (size_t i = 0; i < dd; ++i) {
    split(Pi[i] * 256.f, i, dd + i);
    if (p->lay.prod) split(M[i], 2 * dd + i, 3 * dd + i);
  }
  e = cudaMalloc(&p->wide_ops, host.size() * 2);
  if (e == cudaSuccess) e = cudaMemcpy(p->wide_ops, host.data(), host.size() * 2, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return e;
  if (p->d > 128) {
    // the tensor-core decode of larger d: 2^8 Pi^T and (Prod) 2^8 S^T, split
    // hi + lo in fp16 (row j holds column j of Pi and of S), and the split
    // levels 2^8 c_i
    std::vector<float> S(p->lay.prod ? dd : 0);
    if (p->lay.prod) e = cudaMemcpy(S.data(), p->S, dd * 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return e;
    const size_t d = (size_t)p->d;
    std::vector<uint16_t> dh((p->lay.prod ? 4 : 2) * dd);
    auto split_to = [&](float v, size_t hi_at, size_t lo_at) {
      const __half h = __float2half_rn(v);
      const __half l = __float2half_rn(v - __half2float(h));
      std::memcpy(&dh[hi_at], &h, 2);
      std::memcpy(&dh[lo_at], &l, 2);
    };
    for (size_t j = 0; j < d; ++j)
      for (size_t i = 0; i < d; ++i) {
        split_to(256.f * Pi[i * d + j], j * d + i, dd + j * d + i);
        if (p->lay.prod) split_to(256.f * S[i * d + j], 2 * dd + j * d + i, 3 * dd + j * d + i);
      }
    e = cudaMalloc(&p->dec_wide_ops, dh.size() * 2);
    if (e == cudaSuccess) e = cudaMemcpy(p->dec_wide_ops, dh.data(), dh.size() * 2, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return e;
    for (int i = 0; i < 16; ++i) {
      const float v = i < p->cp.L ? 256.f * p->cp.c[i] : 0.f;
      const __half h = __float2half_rn(v);
      const __half l = __float2half_rn(v - __half2float(h));
      uint16_t hb, lb;
      std::memcpy(&hb, &h, 2);
      std::memcpy(&lb, &l, 2);
      p->dec_ctab[i] = (uint32_t)hb | ((uint32_t)lb << 16);
    }
  }
  if (!p->lay.prod) return e;  // an MSE encode needs no residual scratch
  int slots = tq::query_nsmid();
  if (slots <= 0) return cudaErrorUnknown;
  p->wide_slots = slots;
  return cudaMalloc(&p->wide_scratch, (size_t)slots * 2 * 128 * p->d * 2);
}

// Operand images for the tensor-core encode and decode (d = 128): Pi hi/lo in
// fp16 and in bf16, (PROD) M hi/lo in bf16, then 2^8 Pi^T hi/lo and (PROD)
// 2^8 S^T hi/lo in fp16; and the decode's split codebook 2^8 c_i.
cudaError_t build_tc_ops(tq_plan* p) {
  constexpr size_t img = 128 * 128 * 2;
  const bool prod = p->lay.prod != 0;
  std::vector<float> Pi(128 * 128), M(prod ? 128 * 128 : 0), S(prod ? 128 * 128 : 0);
  std::vector<uint8_t> host((prod ? 10 : 6) * img);
  cudaError_t e = cudaMemcpy(Pi.data(), p->Pi, Pi.size() * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && prod) e = cudaMemcpy(M.data(), p->M, M.size() * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && prod) e = cudaMemcpy(S.data(), p->S, S.size() * 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return e;
  if (p->hadamard) {
    // the encode's rotation operand is the +-1 matrix Pi / c (exact in fp16
    // and bf16; the lo images stay zero), and its E5 operand c M: the encode
    // then works on y / c, with the codebook divided by c (cp_enc, px_enc)
    std::vector<float> U(128 * 128), cM(prod ? 128 * 128 : 0);
    for (int i = 0; i < 128 * 128; ++i) U[i] = Pi[i] < 0.f ? -1.f : 1.f;
    for (size_t i = 0; i < cM.size(); ++i) cM[i] = p->rot_scale * M[i];
    split_images<__half>(U.data(), host.data(), host.data() + img);
    split_images<__nv_bfloat16>(U.data(), host.data() + 2 * img, host.data() + 3 * img);
    if (prod) split_images<__nv_bfloat16>(cM.data(), host.data() + 4 * img, host.data() + 5 * img);
  } else {
    split_images<__half>(Pi.data(), host.data(), host.data() + img);
    split_images<__nv_bfloat16>(Pi.data(), host.data() + 2 * img, host.data() + 3 * img);
    if (prod) split_images<__nv_bfloat16>(M.data(), host.data() + 4 * img, host.data() + 5 * img);
  }
  // decode B operands: row j of the image holds column j of Pi (of S), scaled by 2^8
  std::vector<float> T(128 * 128);
  auto transposed_scaled = [&](const std::vector<float>& A) {
    for (int n = 0; n < 128; ++n)
      for (int k = 0; k < 128; ++k) T[n * 128 + k] = 256.f * A[k * 128 + n];
  };
  transposed_scaled(Pi);
  split_images<__half>(T.data(), host.data() + tq::tc_dec_image(p, 0) * img, host.data() + tq::tc_dec_image(p, 1) * img);
  if (prod) {
    transposed_scaled(S);
    split_images<__half>(T.data(), host.data() + tq::tc_dec_image(p, 2) * img,
                         host.data() + tq::tc_dec_image(p, 3) * img);
  }
  auto ctab = [](const CodeParams& cp, uint32_t* tab) {
    for (int i = 0; i < 16; ++i) {
      const float v = i < cp.L ? 256.f * cp.c[i] : 0.f;
      const __half h = __float2half_rn(v);
      const __half l = __float2half_rn(v - __half2float(h));
      uint16_t hb, lb;
      std::memcpy(&hb, &h, 2);
      std::memcpy(&lb, &l, 2);
      tab[i] = (uint32_t)hb | ((uint32_t)lb << 16);
    }
  };
  ctab(p->cp, p->dec_ctab);
  if (p->lay.frac) ctab(p->cp_lo, p->dec_ctab_lo);
  e = cudaMalloc(&p->tc_ops, host.size());
  if (e == cudaSuccess) e = cudaMemcpy(p->tc_ops, host.data(), host.size(), cudaMemcpyHostToDevice);
  return e;
}

}  // namespace

namespace tq {

// ---- tensor maps (host): cuTensorMapEncodeTiled through the runtime's
// driver entry point, looked up once (thread-safe static initialisation)
using EncodeTmapFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTmapFn tmap_encoder() {
  static const EncodeTmapFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTmapFn>(p);
    return static_cast<EncodeTmapFn>(nullptr);
  }();
  return fn;
}

cudaError_t make_tmap_2d(CUtensorMap* tm, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
                         uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
  EncodeTmapFn enc = tmap_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(tm, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_3d(CUtensorMap* tm, CUtensorMapDataType dt, const void* base, const uint64_t dims[3],
                         const uint64_t strides[2], const uint32_t box[3], CUtensorMapSwizzle sw) {
  EncodeTmapFn enc = tmap_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  const cuuint64_t st[2] = {strides[0], strides[1]};
  const cuuint32_t bx[3] = {box[0], box[1], box[2]};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(tm, dt, 3, const_cast<void*>(base), d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                         CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Workspace: [tensor-core query images and constants | Pi q, S q] [top-k candidates]
size_t score_workspace_bytes(const tq_plan* p, int64_t G, int H, int64_t N, int top_k) {
  const size_t prep = score_tc_supported(p, H)     ? score_tc_workspace_bytes(p, G, H)
                      : score_wide_supported(p, H) ? score_wide_workspace_bytes(p, G, H)
                                                   : 0;
  return align256(prep) + topk_workspace_bytes(G * H, N, top_k) + 256;
}

cudaError_t score_run(const tq_plan* p, const float* queries, int64_t G, int H, const uint8_t* packed, int64_t N,
                      float* logits, int top_k, float* top_scores, int64_t* top_idx, void* ws, cudaStream_t s) {
  cudaError_t e;
  size_t prep;
  if (score_tc_supported(p, H)) {
    prep = score_tc_workspace_bytes(p, G, H);
    e = launch_score_tc(p, queries, G, H, packed, N, logits, ws, s);
  } else if (score_wide_supported(p, H)) {
    prep = score_wide_workspace_bytes(p, G, H);
    e = launch_score_wide(p, queries, G, H, packed, N, logits, ws, s);
  } else {
    return cudaErrorNotSupported;  // every shape the API accepts fits one of the two
  }
  if (e == cudaSuccess && top_k > 0)
    e = launch_topk(logits, G * H, N, top_k, top_scores, top_idx, static_cast<char*>(ws) + align256(prep), s);
  return e;
}

}  // namespace tq

extern "C" {

const char* tq_status_string(tq_status s) {
  switch (s) {
    case TQ_OK: return "ok";
    case TQ_EINVAL: return "invalid argument";
    case TQ_EALIGN: return "pointer not 16-byte aligned";
    case TQ_EUNSUPPORTED: return "unsupported";
    case TQ_ECUDA: return "CUDA error";
    case TQ_ETIMEOUT: return "device wait timed out";
    case TQ_ENOMEM: return "out of device memory";
  }
  return "unknown status";
}

int tq_format_version(void) { return 1; }

tq_status tq_selftest_wait_expiry(tq_plan* p, void* stream) {
  if (!p) return TQ_EINVAL;
  return from_cuda(tq::launch_wait_expiry(p->err, static_cast<cudaStream_t>(stream)));
}

tq_status tq_selftest_encode_drain(tq_plan* p, const void* keys, tq_dtype dtype, int64_t G, int64_t N,
                                   void* packed, void* stream) {
  if (!p || G < 1 || N < 1 || !keys || !packed) return TQ_EINVAL;
  if (dtype != TQ_F16 && dtype != TQ_BF16) return TQ_EINVAL;
  if (!aligned16(keys) || !aligned16(packed)) return TQ_EALIGN;
  if (G * N >= (int64_t)INT32_MAX - 2 * kTokensPerBlock || !encode_tc_supported(p, dtype)) return TQ_EUNSUPPORTED;
  return from_cuda(launch_encode_tc(p, keys, dtype, G, N, static_cast<uint8_t*>(packed),
                                    static_cast<cudaStream_t>(stream), true));
}

int tq_score_path(const tq_plan* p, int H) {
  if (!p || H < 1 || H > 256) return TQ_EINVAL;
  if (tq::score_tc_supported(p, H)) return TQ_PATH_TENSOR_D128;
  if (tq::score_wide_supported(p, H)) return TQ_PATH_TENSOR_WIDE;
  return TQ_EUNSUPPORTED;
}

int tq_decode_path(const tq_plan* p) {
  if (!p) return TQ_EINVAL;
  return tq::decode_tc_supported(p)     ? TQ_PATH_TENSOR_D128
         : tq::decode_wide_supported(p) ? TQ_PATH_TENSOR_WIDE
                                        : TQ_EUNSUPPORTED;
}

int tq_encode_path(const tq_plan* p, tq_dtype dt) {
  if (!p || (dt != TQ_F32 && dt != TQ_F16 && dt != TQ_BF16)) return TQ_EINVAL;
  if (tq::encode_tc_supported(p, dt)) return TQ_PATH_TENSOR_D128;
  if (tq::encode_wide_supported(p, dt)) return TQ_PATH_TENSOR_WIDE;
  return TQ_EUNSUPPORTED;
}

}  // extern "C"

namespace {

// Plan creation shared by tq_plan_create and tq_plan_create_hadamard; a
// Hadamard plan passes hadamard = 1 (Pi already holds c H diag(signs)).
// Parity expansion of an ascending codebook of `levels` entries (host, fp64
// coefficients rounded to fp32), as tq_codebook_parity_expansion computes it.
bool expansion_of(int levels, const float* hc, ParityExpansion* px) {
  unsigned masks[kMaxTerms];
  double coefs[kMaxTerms], c0 = 0.0;
  int n = 0;
  if (tq_codebook_parity_expansion(levels, hc, &n, masks, coefs, &c0) != TQ_OK) return false;
  px->n = n;
  double mid = c0;
  for (int i = 0; i < kMaxTerms; ++i) {
    px->mask[i] = i < n ? masks[i] : 0u;
    px->coef[i] = i < n ? (float)coefs[i] : 0.f;
    px->half[i] = i < n ? (float)(0.5 * coefs[i]) : 0.f;
    if (i < n) mid += 0.5 * coefs[i];
  }
  px->c0 = (float)c0;
  px->mid = (float)mid;
  return true;
}

// A codebook of 2^(k-1) levels in the form of the k-bit one (fractional
// widths: the encode quantises both halves of the coordinates with k code
// bits): thresholds past the last at +inf, so the top bit is never set, and
// the parity terms of the k-bit masks with the lower codebook's coefficients
// (zero on the masks that involve the top bit).
void pad_lower_codebook(const CodeParams& lo, const ParityExpansion& pxlo, const ParityExpansion& pxhi,
                        CodeParams* cp, ParityExpansion* px) {
  *cp = lo;
  const int L = 2 * lo.L;
  cp->L = L;
  for (int i = lo.L; i < L && i < kMaxLevels; ++i) cp->c[i] = lo.c[lo.L - 1];
  for (int i = lo.L - 1; i + 1 < L && i < kMaxLevels - 1; ++i) cp->t[i] = INFINITY;
  *px = pxhi;
  double mid = pxlo.c0;
  for (int t = 0; t < pxhi.n; ++t) {
    float c = 0.f;
    for (int u = 0; u < pxlo.n; ++u)
      if (pxlo.mask[u] == pxhi.mask[t]) c = pxlo.coef[u];
    px->coef[t] = c;
    px->half[t] = 0.5f * c;
    mid += 0.5 * (double)c;
  }
  px->c0 = pxlo.c0;
  px->mid = (float)mid;
}

// 64-bit hash of bytes, eight at a time (a multiply-xorshift mix per word,
// then a final avalanche); identifies a plan's inputs in packed-cache headers
struct Hash64 {
  uint64_t h = 0x9E3779B97F4A7C15ull;
  void word(uint64_t w) {
    h ^= w + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
    h *= 0xBF58476D1CE4E5B9ull;
    h ^= h >> 31;
  }
  void bytes(const void* p, size_t n) {
    const unsigned char* b = static_cast<const unsigned char*>(p);
    size_t i = 0;
    for (; i + 8 <= n; i += 8) {
      uint64_t w;
      std::memcpy(&w, b + i, 8);
      word(w);
    }
    uint64_t t = 0;
    std::memcpy(&t, b + i, n - i);
    word(t ^ ((uint64_t)n << 56));
  }
  uint64_t done() const {
    uint64_t z = h;
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBull;
    return z ^ (z >> 31);
  }
};

cudaError_t plan_fingerprint(tq_plan* p, const float* codebook_host, const float* codebook_lo_host, cudaStream_t s) {
  Hash64 h;
  const int32_t head[5] = {p->d, p->bits, p->mode, p->hadamard, p->lay.frac};
  h.bytes(head, sizeof(head));
  const size_t mat = (size_t)p->d * p->d;
  std::vector<float> m(mat);
  cudaError_t e = cudaMemcpyAsync(m.data(), p->Pi, mat * sizeof(float), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  h.bytes(m.data(), mat * sizeof(float));
  if (p->lay.prod) {
    e = cudaMemcpyAsync(m.data(), p->S, mat * sizeof(float), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    h.bytes(m.data(), mat * sizeof(float));
  }
  h.bytes(codebook_host, (size_t)p->cp.L * sizeof(float));
  if (codebook_lo_host) h.bytes(codebook_lo_host, (size_t)p->cp_lo.L * sizeof(float));
  p->fingerprint = h.done();
  return cudaSuccess;
}

tq_status create_plan(int d, int bits, tq_mode mode, const float* Pi, const float* S, const float* codebook,
                      void* stream, int hadamard, tq_plan** out, const float* codebook_lo = nullptr) {
  if (!out) return TQ_EINVAL;
  *out = nullptr;
  if (d < 128 || d > kMaxD || d % 128 != 0) return TQ_EINVAL;
  if (mode != TQ_PROD && mode != TQ_MSE) return TQ_EINVAL;
  if (mode == TQ_PROD && (bits < 2 || bits > 4)) return TQ_EINVAL;
  if (mode == TQ_MSE && (bits < 1 || bits > 4)) return TQ_EINVAL;
  if (!Pi || !codebook || (mode == TQ_PROD && !S)) return TQ_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  tq_plan* p = new (std::nothrow) tq_plan();
  if (!p) return TQ_ENOMEM;
  std::memset(p, 0, sizeof(*p));
  p->d = d;
  p->bits = bits;
  p->mode = mode;
  cudaGetDevice(&p->device);
  const int k = mode == TQ_PROD ? bits - 1 : bits;
  Layout& L = p->lay;
  L.d = d;
  L.k = k;
  L.prod = mode == TQ_PROD;
  L.planes = k + L.prod;
  L.C = d / kChunk;
  L.frac = codebook_lo != nullptr;
  L.top_off = (int64_t)(k - 1) * L.C * kTokensPerBlock * 16;
  // a fractional width's top code plane holds the first d/2 coordinates only
  L.sign_off = L.top_off + (int64_t)L.C * kTokensPerBlock * (L.frac ? 8 : 16);
  L.norms_off = L.sign_off + (L.prod ? (int64_t)L.C * kTokensPerBlock * 16 : 0);
  L.block_bytes = L.norms_off + kTokensPerBlock * 8;
  p->kappa = (float)(std::sqrt(M_PI / 2.0) / d);
  p->hadamard = hadamard;
  p->rot_scale = hadamard ? (float)(1.0 / std::sqrt((double)d)) : 1.f;

  const size_t mat = (size_t)d * d * sizeof(float);
  bool ok = cudaMalloc(&p->Pi, mat) == cudaSuccess && cudaMalloc(&p->PiT, mat) == cudaSuccess &&
            cudaMalloc(&p->err, sizeof(int)) == cudaSuccess;
  if (ok && L.prod)
    ok = cudaMalloc(&p->S, mat) == cudaSuccess && cudaMalloc(&p->ST, mat) == cudaSuccess &&
         cudaMalloc(&p->M, mat) == cudaSuccess && cudaMalloc(&p->MT, mat) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    free_plan(p);
    return TQ_ENOMEM;
  }
  const int levels = 1 << k;
  float hc[kMaxLevels];
  cudaError_t e = cudaMemcpyAsync(p->Pi, Pi, mat, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && L.prod) e = cudaMemcpyAsync(p->S, S, mat, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(hc, codebook, levels * sizeof(float), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(p->err, 0, sizeof(int), s);
  if (e == cudaSuccess) e = launch_plan_derive(p, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    free_plan(p);
    return TQ_ECUDA;
  }
  CodeParams& cp = p->cp;
  cp.L = levels;
  for (int i = 0; i < kMaxLevels; ++i) cp.c[i] = i < levels ? hc[i] : 0.f;
  for (int i = 0; i + 1 < kMaxLevels; ++i) cp.t[i] = i + 1 < levels ? 0.5f * (hc[i] + hc[i + 1]) : 0.f;
  for (int i = 0; i + 1 < levels; ++i) {
    if (!(hc[i] < hc[i + 1])) {  // must be strictly ascending and finite
      free_plan(p);
      return TQ_EINVAL;
    }
  }
  {
    unsigned masks[kMaxTerms];
    double coefs[kMaxTerms], c0 = 0.0;
    int n = 0;
    if (tq_codebook_parity_expansion(levels, hc, &n, masks, coefs, &c0) != TQ_OK) {
      free_plan(p);
      return TQ_EINVAL;
    }
    p->px.n = n;
    double mid = c0;
    for (int i = 0; i < kMaxTerms; ++i) {
      p->px.mask[i] = i < n ? masks[i] : 0u;
      p->px.coef[i] = i < n ? (float)coefs[i] : 0.f;
      p->px.half[i] = i < n ? (float)(0.5 * coefs[i]) : 0.f;
      if (i < n) mid += 0.5 * coefs[i];
    }
    p->px.c0 = (float)c0;
    p->px.mid = (float)mid;
  }
  // the codebook as the d = 128 encode compares it: divided by the rotation's
  // scale for a Hadamard plan (the encode works on y / c there)
  if (L.frac) {
    // the codebook of the last d/2 coordinates: 2^(k-1) levels, ascending
    const int lv = levels / 2;
    float hl[kMaxLevels];
    if (cudaMemcpyAsync(hl, codebook_lo, lv * sizeof(float), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
      free_plan(p);
      return TQ_ECUDA;
    }
    CodeParams& lo = p->cp_lo;
    lo.L = lv;
    for (int i = 0; i < kMaxLevels; ++i) lo.c[i] = i < lv ? hl[i] : 0.f;
    for (int i = 0; i + 1 < kMaxLevels; ++i) lo.t[i] = i + 1 < lv ? 0.5f * (hl[i] + hl[i + 1]) : 0.f;
    for (int i = 0; i + 1 < lv; ++i)
      if (!(hl[i] < hl[i + 1])) {
        free_plan(p);
        return TQ_EINVAL;
      }
    if (!expansion_of(lv, hl, &p->px_lo)) {
      free_plan(p);
      return TQ_EINVAL;
    }
    pad_lower_codebook(p->cp_lo, p->px_lo, p->px, &p->cp_enc_lo, &p->px_enc_lo);
  }
  p->cp_enc = p->cp;
  p->px_enc = p->px;
  if (hadamard) {
    const float c = p->rot_scale;
    for (int i = 0; i < kMaxLevels; ++i) p->cp_enc.c[i] = p->cp.c[i] / c;
    for (int i = 0; i + 1 < kMaxLevels; ++i) p->cp_enc.t[i] = p->cp.t[i] / c;
    for (int i = 0; i < kMaxTerms; ++i) {
      p->px_enc.coef[i] = p->px.coef[i] / c;
      p->px_enc.half[i] = p->px.half[i] / c;
    }
    p->px_enc.c0 = p->px.c0 / c;
    p->px_enc.mid = p->px.mid / c;
  }
  if (d == 128) {
    if (build_tc_ops(p) != cudaSuccess) {
      free_plan(p);
      return TQ_ECUDA;
    }
  }
  {
    const cudaError_t we = build_wide_ops(p);
    if (we != cudaSuccess) {
      free_plan(p);
      return we == cudaErrorMemoryAllocation ? TQ_ENOMEM : TQ_ECUDA;
    }
  }
  if (plan_fingerprint(p, hc, codebook_lo ? p->cp_lo.c : nullptr, s) != cudaSuccess) {
    free_plan(p);
    return TQ_ECUDA;
  }
  *out = p;
  return TQ_OK;
}

}  // namespace

extern "C" {

tq_status tq_plan_create(int d, int bits, tq_mode mode, const float* Pi, const float* S, const float* codebook,
                         void* stream, tq_plan** out) {
  return create_plan(d, bits, mode, Pi, S, codebook, stream, 0, out);
}

tq_status tq_plan_create_hadamard(int d, int bits, tq_mode mode, const float* signs, const float* S,
                                  const float* codebook, void* stream, tq_plan** out) {
  if (!out) return TQ_EINVAL;
  *out = nullptr;
  if (d < 128 || d > kMaxD || (d & (d - 1)) != 0 || !signs) return TQ_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  std::vector<float> sg(d), Pi((size_t)d * d);
  if (cudaMemcpyAsync(sg.data(), signs, d * sizeof(float), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return TQ_ECUDA;
  for (int j = 0; j < d; ++j)
    if (sg[j] != 1.f && sg[j] != -1.f) return TQ_EINVAL;
  // Pi[i][j] = c (-1)^popcount(i & j) signs[j], c = 1/sqrt(d) rounded once to fp32
  const float c = (float)(1.0 / std::sqrt((double)d));
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < d; ++j) Pi[(size_t)i * d + j] = (__builtin_popcount((unsigned)(i & j)) & 1 ? -c : c) * sg[j];
  float* Pi_d = nullptr;
  if (cudaMalloc(&Pi_d, Pi.size() * sizeof(float)) != cudaSuccess) {
    cudaGetLastError();
    return TQ_ENOMEM;
  }
  tq_status st = cudaMemcpyAsync(Pi_d, Pi.data(), Pi.size() * sizeof(float), cudaMemcpyHostToDevice, s) ==
                         cudaSuccess
                     ? create_plan(d, bits, mode, Pi_d, S, codebook, stream, 1, out)
                     : TQ_ECUDA;
  cudaStreamSynchronize(s);
  cudaFree(Pi_d);
  return st;
}

tq_status tq_plan_create_fractional(int d, int half_bits, tq_mode mode, const float* Pi, const float* S,
                                    const float* codebook_hi, const float* codebook_lo, void* stream,
                                    tq_plan** out) {
  if (!out) return TQ_EINVAL;
  *out = nullptr;
  if (d != 128 || !codebook_lo) return TQ_EINVAL;
  if (mode == TQ_PROD && half_bits != 5 && half_bits != 7) return TQ_EINVAL;
  if (mode == TQ_MSE && half_bits != 3 && half_bits != 5) return TQ_EINVAL;
  const int k_hi = (half_bits + 1) / 2 - (mode == TQ_PROD ? 1 : 0);
  return create_plan(d, mode == TQ_PROD ? k_hi + 1 : k_hi, mode, Pi, S, codebook_hi, stream, 0, out, codebook_lo);
}

tq_status tq_plan_destroy(tq_plan* plan) {
  if (!plan) return TQ_EINVAL;
  free_plan(plan);
  return TQ_OK;
}

size_t tq_packed_bytes(const tq_plan* p, int64_t G, int64_t N) {
  if (!p || G < 0 || N < 0) return 0;
  const int64_t nb = (N + kTokensPerBlock - 1) / kTokensPerBlock;
  return (size_t)(G * nb) * (size_t)p->lay.block_bytes;
}

// Packed-cache header (64 bytes, little-endian): magic, format version, d,
// bits, mode, kind flags, G, N, block bytes, plan fingerprint, checksum of the
// first 56 bytes.
namespace {
constexpr uint32_t kHeaderMagic = 0x4B505154u;  // "TQPK"
struct PackedHeader {
  uint32_t magic, version, d, bits, mode, flags;
  int64_t G, N;
  uint64_t block_bytes, fingerprint, check;
};
static_assert(sizeof(PackedHeader) == TQ_PACKED_HEADER_BYTES, "header size");
uint64_t header_check(const PackedHeader& h) {
  Hash64 x;
  x.bytes(&h, offsetof(PackedHeader, check));
  return x.done();
}
}  // namespace

tq_status tq_packed_header_write(const tq_plan* p, int64_t G, int64_t N, void* header) {
  if (!p || G < 0 || N < 0 || !header) return TQ_EINVAL;
  PackedHeader h;
  std::memset(&h, 0, sizeof(h));
  h.magic = kHeaderMagic;
  h.version = (uint32_t)tq_format_version();
  h.d = (uint32_t)p->d;
  h.bits = (uint32_t)p->bits;
  h.mode = (uint32_t)p->mode;
  h.flags = (p->hadamard ? 1u : 0u) | (p->lay.frac ? 2u : 0u);
  h.G = G;
  h.N = N;
  h.block_bytes = (uint64_t)p->lay.block_bytes;
  h.fingerprint = p->fingerprint;
  h.check = header_check(h);
  std::memcpy(header, &h, sizeof(h));
  return TQ_OK;
}

tq_status tq_packed_header_read(const tq_plan* p, const void* header, int64_t* G, int64_t* N) {
  if (!p || !header) return TQ_EINVAL;
  PackedHeader h;
  std::memcpy(&h, header, sizeof(h));
  if (h.magic != kHeaderMagic || h.check != header_check(h)) return TQ_EINVAL;
  if (h.version != (uint32_t)tq_format_version() || h.d != (uint32_t)p->d || h.bits != (uint32_t)p->bits ||
      h.mode != (uint32_t)p->mode || h.flags != ((p->hadamard ? 1u : 0u) | (p->lay.frac ? 2u : 0u)) ||
      h.block_bytes != (uint64_t)p->lay.block_bytes || h.fingerprint != p->fingerprint || h.G < 0 || h.N < 0)
    return TQ_EUNSUPPORTED;
  if (G) *G = h.G;
  if (N) *N = h.N;
  return TQ_OK;
}

tq_status tq_encode(const tq_plan* p, const void* keys, tq_dtype dtype, int64_t G, int64_t N, void* packed,
                    void* stream) {
  if (!p || G < 0 || N < 0) return TQ_EINVAL;
  if (dtype != TQ_F32 && dtype != TQ_F16 && dtype != TQ_BF16) return TQ_EINVAL;
  if (G == 0 || N == 0) return TQ_OK;
  if (!keys || !packed) return TQ_EINVAL;
  if (!aligned16(keys) || !aligned16(packed)) return TQ_EALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // both encodes address key rows by 32-bit TMA coordinates: 2^31 keys of the
  // smallest kind (d = 128, 16-bit) would be 512 GiB, beyond the device
  if (G * N >= (int64_t)INT32_MAX - 2 * kTokensPerBlock) return TQ_EUNSUPPORTED;
  if (encode_tc_supported(p, dtype))
    return from_cuda(launch_encode_tc(p, keys, dtype, G, N, static_cast<uint8_t*>(packed), s));
  if (!encode_wide_supported(p, dtype)) return TQ_EUNSUPPORTED;
  return from_cuda(launch_encode_wide(p, keys, dtype, G, N, static_cast<uint8_t*>(packed), s));
}

size_t tq_score_workspace_bytes(const tq_plan* p, int64_t G, int H, int64_t N, int top_k) {
  if (!p || G < 0 || H < 1 || N < 0 || top_k < 0) return 0;
  return score_workspace_bytes(p, G, H, N, top_k);
}

tq_status tq_score(const tq_plan* p, const float* queries, int64_t G, int H, const void* packed, int64_t N,
                   float* logits, int top_k, float* top_scores, int64_t* top_idx, void* workspace,
                   size_t workspace_bytes, void* stream) {
  if (!p || G < 0 || N < 0 || H < 1 || H > 256 || top_k < 0 || top_k > 64) return TQ_EINVAL;
  if (top_k > 0 && (top_k > N || !top_scores || !top_idx)) return TQ_EINVAL;
  if (G == 0 || N == 0) return TQ_OK;
  if (!queries || !packed || !logits || !workspace) return TQ_EINVAL;
  if (workspace_bytes < tq_score_workspace_bytes(p, G, H, N, top_k)) return TQ_EINVAL;
  if (!aligned16(queries) || !aligned16(packed) || !aligned16(logits)) return TQ_EALIGN;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return TQ_EALIGN;
  if (top_k > 0 && (!aligned16(top_scores) || !aligned16(top_idx))) return TQ_EALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return from_cuda(score_run(p, queries, G, H, static_cast<const uint8_t*>(packed), N, logits, top_k, top_scores,
                             top_idx, workspace, s));
}

tq_status tq_encode_values(const tq_plan* p, const void* values, tq_dtype dtype, int64_t G, int64_t N, void* packed,
                           void* stream) {
  if (!p || p->lay.prod) return TQ_EINVAL;
  if (p->lay.frac) return TQ_EUNSUPPORTED;
  const tq_status st = tq_encode(p, values, dtype, G, N, packed, stream);
  if (st != TQ_OK || G == 0 || N == 0) return st;
  const int64_t nb = (N + kTokensPerBlock - 1) / kTokensPerBlock;
  return from_cuda(launch_values_layout(p, static_cast<uint8_t*>(packed), G * nb, reinterpret_cast<cudaStream_t>(stream)));
}

size_t tq_attend_workspace_bytes(const tq_plan* kplan, const tq_plan* vplan, int64_t G, int H, int64_t N) {
  if (!kplan || !vplan || G < 0 || H < 1 || N < 0) return 0;
  return attend_workspace_bytes(kplan, vplan, G, H, N);
}

tq_status tq_attend(const tq_plan* kplan, const tq_plan* vplan, const float* queries, int64_t G, int H,
                    const void* kpacked, const void* vpacked, int64_t N, float scale, float* out, void* workspace,
                    size_t workspace_bytes, void* stream) {
  if (!kplan || !vplan || G < 0 || N < 0 || H < 1 || !std::isfinite(scale)) return TQ_EINVAL;
  if (!attend_supported(kplan, vplan, H)) return TQ_EUNSUPPORTED;
  if (G == 0 || N == 0) return TQ_OK;
  if (!queries || !kpacked || !vpacked || !out || !workspace) return TQ_EINVAL;
  if (workspace_bytes < attend_workspace_bytes(kplan, vplan, G, H, N)) return TQ_EINVAL;
  if (!aligned16(queries) || !aligned16(kpacked) || !aligned16(vpacked) || !aligned16(out)) return TQ_EALIGN;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return TQ_EALIGN;
  return from_cuda(launch_attend(kplan, vplan, queries, G, H, static_cast<const uint8_t*>(kpacked),
                                 static_cast<const uint8_t*>(vpacked), N, scale, out, workspace,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

tq_status tq_decode(const tq_plan* p, const void* packed, int64_t G, int64_t N, float* out, void* stream) {
  if (!p || G < 0 || N < 0) return TQ_EINVAL;
  if (G == 0 || N == 0) return TQ_OK;
  if (!packed || !out) return TQ_EINVAL;
  if (!aligned16(packed) || !aligned16(out)) return TQ_EALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (decode_tc_supported(p)) return from_cuda(launch_decode_tc(p, static_cast<const uint8_t*>(packed), G, N, out, s));
  if (decode_wide_supported(p))
    return from_cuda(launch_decode_wide(p, static_cast<const uint8_t*>(packed), G, N, out, s));
  return TQ_EUNSUPPORTED;  // every plan the library creates takes one of the two
}

tq_status tq_score_fp32(const float* queries, const float* keys, int64_t G, int H, int64_t N, int d, float* logits,
                        void* stream) {
  if (G < 0 || N < 0 || H < 1 || H > 256 || d < 1 || d > 4096 || d % 4 != 0) return TQ_EINVAL;
  if (G == 0 || N == 0) return TQ_OK;
  if (!queries || !keys || !logits) return TQ_EINVAL;
  if (!aligned16(queries) || !aligned16(keys) || !aligned16(logits)) return TQ_EALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return from_cuda(launch_score_fp32(queries, keys, G, H, N, d, logits, s));
}

tq_status tq_plan_status(tq_plan* p) {
  if (!p) return TQ_EINVAL;
  int v = 0;
  if (cudaMemcpy(&v, p->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return TQ_ECUDA;
  if (v != 0) {
    int zero = 0;
    if (cudaMemcpy(p->err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return TQ_ECUDA;
    return TQ_ETIMEOUT;
  }
  return TQ_OK;
}

}  // extern "C"
