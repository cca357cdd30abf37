/*
 * tq.h -- C ABI of libtq.so: TurboQuantProd key encoding and attention-logit
 * scoring on the compressed keys, for one B300 (sm_103a).
 *
 * Sources:
 *  [PT-KR]  "turboquant-pytorch 소개" (discuss.pytorch.kr, PyTorch Korea user
 *           group): "1단계: 랜덤 회전 + Lloyd-Max 양자화", "2단계: QJL 잔차 보정",
 *           the usage listing ("TurboQuant 핵심 알고리즘 사용 예시"), "성능 지표".
 *  [TAMBUR] "Google acelera LLM 8 veces" (tambur.pub): MSE-only quantisers bias
 *           inner products; a 1-bit QJL residual pass removes the bias; 4-bit
 *           keys speed up attention logits versus 32-bit keys.
 *  [P5]     "알고리즘보다 커널이 성패를 가른다" (tistory27), section 3: the
 *           bit-packed format with QJL metadata needs a dedicated kernel;
 *           section 4: structured (Walsh-Hadamard) rotations as an
 *           acceleration (turboquant_plus).
 *
 * Notation: d = head dimension (a multiple of 128), m = d rows of S,
 * b = total bits per coordinate, k = b-1 Lloyd-Max bits (PROD) or k = b (MSE),
 * L = 2^k centroids, G = groups (batch x layers x KV heads), N = tokens per
 * group, H = query heads per group.
 *
 * Conventions for every entry point:
 *  - Pointers named "device" are CUDA device pointers on the current device;
 *    the caller owns every buffer it passes.  The library allocates device
 *    memory only in tq_plan_create (freed by tq_plan_destroy).
 *  - Keys, queries, logits and packed buffers must be 16-byte aligned and
 *    contiguous in the stated layout; otherwise TQ_EALIGN.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream).  Argument errors are returned synchronously and
 *    nothing is enqueued.  A failed launch returns TQ_ECUDA.  Device-side errors
 *    (a bounded wait that ran out) are reported by tq_plan_status after the
 *    caller synchronises.
 *  - No entry point prints, throws, or falls back to the CPU.
 *  - A plan is immutable after creation: calls on different streams may share
 *    it concurrently.
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TQ_OK = 0,
  TQ_EINVAL = -1,        /* bad size, null pointer, unsupported combination */
  TQ_EALIGN = -2,        /* a pointer is not 16-byte aligned */
  TQ_EUNSUPPORTED = -3,  /* valid request that no kernel of the library handles */
  TQ_ECUDA = -4,         /* a CUDA call failed (launch, copy, allocation) */
  TQ_ETIMEOUT = -5,      /* a bounded device wait ran out (see tq_plan_status) */
  TQ_ENOMEM = -6         /* device allocation failed in tq_plan_create */
} tq_status;

typedef enum { TQ_F32 = 0, TQ_F16 = 1, TQ_BF16 = 2 } tq_dtype;

/* TQ_PROD: TurboQuantProd, (b-1)-bit Lloyd-Max codes + 1-bit QJL signs of
 * S r + ||x|| and ||r||  ([PT-KR] 1단계 and 2단계).
 * TQ_MSE:  TurboQuantMSE, b-bit Lloyd-Max codes + ||x|| ([PT-KR] 1단계). */
typedef enum { TQ_PROD = 0, TQ_MSE = 1 } tq_mode;

typedef struct tq_plan tq_plan;

/* ---------------------------------------------------------------- plan inputs
 * Host-side helpers that build the plan's inputs from random draws the caller
 * makes.  They run on the CPU once per plan (they are set-up, not the path). */

/* Lloyd-Max codebook for one rotated coordinate, treated as N(0, 1/d)
 * ([PT-KR] 1단계: the optimal quantiser for the bell-shaped coordinate
 * distribution, precomputed).  Writes `levels` ascending fp32 centroids
 * (the N(0,1) quantiser scaled by 1/sqrt(d)) to the HOST array `out`.
 * levels in {2,4,8,16}; d >= 1.  Errors: TQ_EINVAL. */
tq_status tq_lloyd_max_codebook(int levels, int d, float* out);

/* Parity (Walsh) expansion of a codebook of `levels` entries (HOST array,
 * ascending, levels in {2,4,8,16}) over the bits of its index:
 *   codebook[idx] = c0 + sum_t coefs[t] * parity(idx & masks[t]),
 * parity(x) = popcount(x) mod 2.  This is how the tensor-core scorer writes
 * the MSE term <Pi q, c[idx]> ([PT-KR] usage listing, ``inner_product``) as
 * dot products with XOR planes of the packed code bits.  Only terms with a
 * non-zero coefficient are returned, in increasing mask order (an exactly
 * odd-symmetric codebook has none on even-weight masks).  Writes *n_terms
 * (<= levels - 1) and that many HOST masks/coefs, and *c0 = codebook[0].
 * Errors: TQ_EINVAL. */
tq_status tq_codebook_parity_expansion(int levels, const float* codebook, int* n_terms, unsigned* masks,
                                       double* coefs, double* c0);

/* Random orthogonal rotation from a d x d Gaussian matrix ([PT-KR] 1단계):
 * Pi = Q diag(sign R_ii) for the Householder QR  gaussian = Q R  (fp64),
 * written as fp32 row-major to the HOST array `Pi_out` (y = Pi u).
 * `gaussian` is a HOST fp64 row-major d x d array.  Errors: TQ_EINVAL
 * (d < 1, d > 8192, null pointer, rank-deficient input). */
tq_status tq_haar_rotation(int d, const double* gaussian, float* Pi_out);

/* ---------------------------------------------------------------- plan */

/* Create a plan for head dimension d and b total bits.
 *   Pi        device fp32 d x d row-major, y = Pi u (orthogonal).
 *   S         device fp32 d x d row-major (m = d rows); NULL for TQ_MSE.
 *   codebook  device fp32, L ascending centroids already scaled for N(0,1/d)
 *             (L = 2^(bits-1) for TQ_PROD, 2^bits for TQ_MSE).
 * The plan copies Pi, S and the codebook and derives M = S Pi^T (fp64
 * accumulation) plus the half-precision operand splits the kernels use; the
 * caller may free its buffers once the plan exists.  Runs on `stream` and
 * synchronises it before returning.
 * Constraints: d % 128 == 0, 128 <= d <= 2048; TQ_PROD bits in {2,3,4};
 * TQ_MSE bits in {1,2,3,4}.  Errors: TQ_EINVAL, TQ_ENOMEM, TQ_ECUDA. */
tq_status tq_plan_create(int d, int bits, tq_mode mode, const float* Pi, const float* S,
                         const float* codebook, void* stream, tq_plan** out);

/* Create a plan whose rotation is the randomised Walsh-Hadamard transform
 * ("알고리즘보다 커널이 성패를 가른다" section 4: a structured WHT rotation in
 * place of the dense random one, as turboquant_plus does):
 *   Pi = H_d diag(signs) / sqrt(d),
 * H_d the Sylvester Hadamard matrix ((-1)^popcount(i & j)).  Each entry of Pi
 * is +-c with c = (float)(1 / sqrt(d)) computed in double, so Pi is
 * determined exactly by the signs.
 *   signs     device fp32, d entries, each +1 or -1.
 *   S, codebook, mode, bits: as tq_plan_create.
 * Everything tq_plan_create documents holds for the resulting plan (every
 * kernel computes with this Pi).  In addition, the d = 128 tensor-core encode
 * forms the rotation with one exact product of the keys and the +-1 matrix
 * H diag(signs), the scale c being folded into the plan's thresholds,
 * centroids and M, instead of the two-product split a dense Pi needs.
 * Constraints: d a power of two, 128 <= d <= 2048.  Errors: TQ_EINVAL (also
 * for a sign that is not +-1), TQ_ENOMEM, TQ_ECUDA. */
tq_status tq_plan_create_hadamard(int d, int bits, tq_mode mode, const float* signs, const float* S,
                                  const float* codebook, void* stream, tq_plan** out);
/* Create a plan at a fractional width ([TAMBUR]: KV caches at 3.5 bits per
 * channel are quality-neutral, at 2.5 bits slightly degraded).  The pages do
 * not say how the channels are split; this library's reading: the first d/2
 * coordinates of the rotated vector take one more Lloyd-Max bit than the
 * last d/2 (after the random rotation every coordinate has the same
 * distribution), so the average is b + 1/2 bits per channel:
 *   TQ_PROD: half_bits 5 (2.5) or 7 (3.5): 1/2 or 2/3 code bits + 1 QJL bit;
 *   TQ_MSE:  half_bits 3 (1.5) or 5 (2.5): 1/2 or 2/3 code bits.
 *   codebook_hi  device fp32, 2^k_hi ascending centroids (coordinates < d/2);
 *   codebook_lo  device fp32, 2^(k_hi-1) ascending centroids (the others);
 *   Pi, S: as tq_plan_create.
 * Packed layout: as tq_packed_bytes describes, except that code plane k_hi - 1
 * holds the first d/2 coordinates only: per 128 coordinates 8 bytes per token
 * (coordinate 64 c + 32 w + i at bit i of little-endian word w of half chunk
 * c), the 128 tokens' 8-byte half chunks in token order; the sign plane and
 * the norms follow.  Bytes per key: 48 (2.5, Prod), 64 (3.5, Prod).
 * Supported: d = 128; encode of fp16/bf16 keys, score with H <= 16, decode,
 * all on the d = 128 tensor-core kernels (other calls: TQ_EUNSUPPORTED).
 * Errors: TQ_EINVAL, TQ_ENOMEM, TQ_ECUDA. */
tq_status tq_plan_create_fractional(int d, int half_bits, tq_mode mode, const float* Pi, const float* S,
                                    const float* codebook_hi, const float* codebook_lo, void* stream,
                                    tq_plan** out);
tq_status tq_plan_destroy(tq_plan* plan);

/* Bytes of the packed buffer for G groups of N tokens.  Layout ([P5] §3):
 * per group, blocks of 128 tokens; per block, for each plane p (the k code
 * bits, LSB first, then the sign plane in TQ_PROD), for each 128-coordinate
 * chunk c, the 128 tokens' 16-byte chunks in token order; then 128 norm pairs
 * {float ||x||, float ||r||} (||r|| = 0 in TQ_MSE).  In a chunk, coordinate
 * 128c + 32w + i is bit i of little-endian uint32 word w.  Tokens past N in the
 * last block are zero.  Bytes per key: (planes*d)/8 + 8, planes = b.
 * Returns 0 for a null plan or negative sizes. */
size_t tq_packed_bytes(const tq_plan* plan, int64_t n_groups, int64_t n_tokens);

/* Packed-cache header, so that a packed buffer can be stored and reloaded as
 * plain bytes.  64 bytes, little-endian: uint32 magic "TQPK", uint32
 * tq_format_version(), uint32 d, bits, mode, kind flags (1: Walsh-Hadamard
 * plan, 2: fractional width), int64 n_groups, n_tokens, uint64 bytes per
 * 128-token block, uint64 plan fingerprint (a hash of d, bits, mode, kind and
 * the bytes of Pi, S and the codebooks given at plan creation), uint64
 * checksum of the preceding 56 bytes.  The header is HOST memory owned by the
 * caller; no GPU work.  tq_packed_header_write fills `header`
 * (TQ_EINVAL for a null plan or pointer, negative sizes).
 * tq_packed_header_read checks `header` against `plan` and returns the sizes
 * it describes: TQ_EINVAL for a null plan or pointer, a wrong magic or a
 * damaged header; TQ_EUNSUPPORTED for a header written for another format
 * version, layout or plan (the bytes would decode to other keys). */
#define TQ_PACKED_HEADER_BYTES 64
tq_status tq_packed_header_write(const tq_plan* plan, int64_t n_groups, int64_t n_tokens, void* header);
tq_status tq_packed_header_read(const tq_plan* plan, const void* header, int64_t* n_groups, int64_t* n_tokens);

/* ---------------------------------------------------------------- the path */

/* Encode keys ([PT-KR] 1단계 + 2단계; usage listing: ``tq.compress``):
 * for each key x: n = ||x||, u = x/n, y = Pi u, idx_j = #{i : t_i < y_j}
 * with t_i = (c_i + c_{i+1})/2; r = x - n Pi^T c[idx]; rho = ||r||;
 * z = [S r >= 0].  A zero key stores idx = #{t_i < 0}, z = 1, rho = 0.
 *   keys    device [G][N][d] row-major in `dtype` (fp32, fp16 or bf16).
 *   packed  device, tq_packed_bytes(plan, G, N) bytes, fully overwritten.
 * G >= 0, N >= 0 (G*N == 0 is a no-op).  Errors: TQ_EINVAL, TQ_EALIGN, TQ_ECUDA;
 * TQ_EUNSUPPORTED for G*N >= 2^31 - 256 keys (key rows are 32-bit copy
 * coordinates; such a call would hold at least 512 GiB of keys). */
tq_status tq_encode(const tq_plan* plan, const void* keys, tq_dtype dtype, int64_t n_groups,
                    int64_t n_tokens, void* packed, void* stream);

/* Bytes of scratch tq_score needs (rotated queries Pi q, projected queries
 * S q and the top-k candidates); the caller allocates it. */
size_t tq_score_workspace_bytes(const tq_plan* plan, int64_t n_groups, int n_heads,
                                int64_t n_tokens, int top_k);

/* Attention logits on the compressed keys ([PT-KR] usage listing:
 * ``tq.inner_product(query, compressed)``; [TAMBUR]: the unbiased estimate):
 *   logit = n <Pi q, c[idx]> + rho * sqrt(pi/2)/m * <S q, 2z - 1>
 * (TQ_MSE: the first term only), which equals <q, x_mse> + the QJL term.
 *   queries    device fp32 [G][H][d].
 *   packed     device, as written by tq_encode for (G, N).
 *   logits     device fp32 [G][H][N], fully overwritten.
 *   top_k      0 for none, else 1..64: also writes, per (g, h), the top_k
 *              logits in descending order (ties: lower token first) to
 *              top_scores fp32 [G][H][top_k] and their token indices to
 *              top_idx int64 [G][H][top_k]; needs top_k <= N.
 *   workspace  device, >= tq_score_workspace_bytes(...), 256-byte aligned.
 * 1 <= H <= 256.  Errors: TQ_EINVAL, TQ_EALIGN, TQ_ECUDA. */
tq_status tq_score(const tq_plan* plan, const float* queries, int64_t n_groups, int n_heads,
                   const void* packed, int64_t n_tokens, float* logits, int top_k,
                   float* top_scores, int64_t* top_idx, void* workspace,
                   size_t workspace_bytes, void* stream);

/* The pages have no counterpart to this entry point: it is a variant of
 * tq_score for callers that cannot allocate device memory -- for example a
 * plugin running inside a runtime that owns all device memory through its own
 * pool (allocating behind the host's back would break its budget), or a
 * latency-critical caller that cannot afford cudaMalloc's device
 * synchronisation.  It computes exactly what tq_score computes, with the same
 * arguments minus the workspace: the scratch comes from one fixed array of
 * TQ_SCORE_NOALLOC_MAX_BYTES in the library's device image, which every GPU
 * that loads the library holds until the process exits.  The call allocates
 * nothing (no cudaMalloc, no cudaFree).
 *  - Requests whose tq_score_workspace_bytes(...) exceeds the maximum return
 *    TQ_EUNSUPPORTED and enqueue nothing.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.  The address is kept per CUDA context: after
 *    cudaDeviceReset (which frees the array with the context; plans made
 *    before it are invalid too) or under another context, the next call looks
 *    it up again, so that call should likewise come before any capture.
 *  - Every call shares the one array: calls whose work overlaps on the GPU
 *    (several streams or threads) race and must be serialised by the caller.
 *    The array keeps the last call's contents; nothing in it needs clearing.
 * Errors: as tq_score, plus TQ_EUNSUPPORTED. */
#define TQ_SCORE_NOALLOC_MAX_BYTES (32u << 20)
tq_status tq_score_noalloc(const tq_plan* plan, const float* queries, int64_t n_groups, int n_heads,
                           const void* packed, int64_t n_tokens, float* logits, int top_k,
                           float* top_scores, int64_t* top_idx, void* stream);

/* Encode value vectors for attention: the TurboQuantMSE encode of tq_encode
 * ([PT-KR] 1단계; the pages' 3-bit KV figure compresses values too) written in
 * the coordinate-major value layout that tq_attend reads: per 128-token block,
 * for each code plane p (LSB first) and coordinate j, 16 bytes hold bit p of
 * coordinate j of the block's 128 tokens (token t = bit t % 32 of
 * little-endian word t / 32); then the 128 pairs {float ||v||, float 0}.  The
 * same bytes per vector as tq_encode (tq_packed_bytes); the same bits,
 * transposed within each block.
 *   plan  a TQ_MSE plan.  values: device [G][N][d] fp32/fp16/bf16.
 * Errors: as tq_encode; TQ_EINVAL for a TQ_PROD plan. */
tq_status tq_encode_values(const tq_plan* plan, const void* values, tq_dtype dtype, int64_t n_groups,
                           int64_t n_tokens, void* packed, void* stream);

/* One decode step of attention on the compressed cache ([TAMBUR]: attention
 * logits computed directly on the compressed keys; [P5] section 3: a dedicated
 * kernel for the packed format):
 *   out[g][h] = sum_t softmax_t(scale * logit[g][h][t]) v_hat[g][t],
 * logit as tq_score computes it from the keys (kplan, TQ_PROD, packed by
 * tq_encode), v_hat = ||v|| Pi_v^T c_v[idx] from the values (vplan, TQ_MSE,
 * packed by tq_encode_values).  The pages name no scale: pass 1/sqrt(d) for
 * the usual scaled dot-product attention.
 *   queries device fp32 [G][H][d]; out device fp32 [G][H][d];
 *   workspace device, >= tq_attend_workspace_bytes(...), 256-byte aligned
 *   (it holds the logits on their way to the softmax: G*H*N*4 bytes and the
 *   per-split partial sums).
 * Supported: d = 128 for both plans; the key plan as tq_score's tensor-core
 * path takes it; a value codebook of 2, 4 or 8 levels, odd-symmetric; H <= 8,
 * or H <= 16 with at most 4 value levels.  Otherwise TQ_EUNSUPPORTED.
 * Device errors go to the key plan's (score) and the value plan's
 * (value contraction) error words.  Errors: TQ_EINVAL, TQ_EALIGN,
 * TQ_EUNSUPPORTED, TQ_ECUDA. */
size_t tq_attend_workspace_bytes(const tq_plan* kplan, const tq_plan* vplan, int64_t n_groups, int n_heads,
                                 int64_t n_tokens);
tq_status tq_attend(const tq_plan* kplan, const tq_plan* vplan, const float* queries, int64_t n_groups,
                    int n_heads, const void* kpacked, const void* vpacked, int64_t n_tokens, float scale,
                    float* out, void* workspace, size_t workspace_bytes, void* stream);

/* Reconstruct keys ([PT-KR] usage listing: ``tq.decompress``):
 * x_hat = n Pi^T c[idx] + rho sqrt(pi/2)/m S^T (2z - 1)  (TQ_MSE: first term),
 * so that <q, x_hat> equals tq_score's logit.  out: device fp32 [G][N][d].
 * Runs on tensor cores at every d (tq_decode_path).  Errors: TQ_EINVAL,
 * TQ_EALIGN, TQ_ECUDA. */
tq_status tq_decode(const tq_plan* plan, const void* packed, int64_t n_groups, int64_t n_tokens,
                    float* out, void* stream);

/* The uncompressed baseline ([TAMBUR]: "32-bit unquantized keys"):
 * logits[g][h][t] = <queries[g][h], keys[g][t]>, all fp32.
 *   queries device [G][H][d]; keys device [G][N][d]; logits device [G][H][N].
 * d % 4 == 0, 1 <= d <= 4096, 1 <= H <= 256. */
tq_status tq_score_fp32(const float* queries, const float* keys, int64_t n_groups, int n_heads,
                        int64_t n_tokens, int d, float* logits, void* stream);

/* Device-side status of the plan's last work (TQ_OK or TQ_ETIMEOUT), read
 * with a synchronous copy; call after synchronising the streams that used it.
 * Reading clears it. */
tq_status tq_plan_status(tq_plan* plan);

const char* tq_status_string(tq_status status);

/* Self-test of the device error path (no GPU fault is involved): launches one
 * small kernel whose mbarrier waits are never satisfied; both bounded-wait
 * forms the tensor-core kernels use give up after their poll limit (about a
 * second), raise the plan's error word and return normally.  After the caller
 * synchronises, tq_plan_status reports TQ_ETIMEOUT (and clears the word); the
 * context and the plan stay usable.  Errors: TQ_EINVAL (null plan), TQ_ECUDA. */
tq_status tq_selftest_wait_expiry(tq_plan* plan, void* stream);

/* Self-test of the error path of a real kernel (no GPU fault is involved):
 * runs tq_encode's tensor-core encode (d = 128, fp16/bf16 keys) on the given
 * keys, except that the producer of CTA 0 withholds the copy of its first key
 * tile.  The waits on that tile give up after their poll limit (about a
 * second) and raise the plan's error word; every role of that CTA then stops,
 * waits for the copies and MMAs it issued and frees its TMEM; the other CTAs
 * finish normally.  After the caller synchronises, tq_plan_status reports
 * TQ_ETIMEOUT (and clears the word); `packed` holds no usable result, and the
 * context and the plan stay usable.  Arguments and layout as tq_encode.
 * Errors: TQ_EINVAL (null plan or pointer, G or N < 1, other dtypes),
 * TQ_EALIGN, TQ_EUNSUPPORTED (a plan or size the d = 128 encode does not
 * take), TQ_ECUDA. */
tq_status tq_selftest_encode_drain(tq_plan* plan, const void* keys, tq_dtype dtype, int64_t n_groups,
                                   int64_t n_tokens, void* packed, void* stream);

/* Version of the packed layout described above (bumped on any change). */
int tq_format_version(void);

/* Which kernel family a call takes, for reports and tests (no GPU work):
 *   TQ_PATH_TENSOR_D128  tcgen05 kernels specialised for d = 128 (encode: fp16/bf16
 *                        keys, either mode; score: H <= 16, odd-symmetric
 *                        codebook, k <= 3);
 *   TQ_PATH_TENSOR_WIDE  tcgen05 kernels for any d (multiple of 128): encode of
 *                        every other plan and key dtype, score up to 256 heads,
 *                        decode for d > 128;
 *   TQ_PATH_CUDA_CORE    CUDA-core kernels (no current path takes one; the value
 *                        stays reserved).
 * Returns the path, or TQ_EINVAL for a null plan or an out-of-range argument
 * (TQ_EUNSUPPORTED if no kernel takes the shape; none of the shapes the entry
 * points accept). */
typedef enum { TQ_PATH_TENSOR_D128 = 0, TQ_PATH_TENSOR_WIDE = 1, TQ_PATH_CUDA_CORE = 2 } tq_path;
int tq_score_path(const tq_plan* plan, int n_heads);
int tq_encode_path(const tq_plan* plan, tq_dtype dtype);
int tq_decode_path(const tq_plan* plan);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H_ */
