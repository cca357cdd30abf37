"""CPU oracle for TurboQuantProd / TurboQuantMSE: plain, slow, fp64.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The CUDA library never calls it, and it never calls the CUDA library:
the two share no code.

Sources (each function cites the passage it follows):

* [PT-KR] "turboquant-pytorch 소개" (discuss.pytorch.kr, PyTorch Korea user
  group), sections "1단계: 랜덤 회전(Random Rotation) + Lloyd-Max 양자화",
  "2단계: QJL 잔차 보정(Residual Correction)", the usage listing "TurboQuant 핵심
  알고리즘 사용 예시 (synthetic validation)" and "turboquant-pytorch의 성능 지표".
* [TAMBUR] "Google acelera LLM 8 veces" (tambur.pub), the paragraph on the
  bias of MSE-only quantisers for inner products and the 1-bit QJL correction.
* [P5] "알고리즘보다 커널이 성패를 가른다" (tistory27), section 3: a bit-packed
  format plus QJL metadata.

Everything is computed in fp64 from the exact values the GPU consumes (fp32,
fp16 and bf16 all convert exactly to fp64).  Readings where the pages are
silent are marked READING and listed in the design notes; they are:

* the codebook is Lloyd-Max for N(0, 1/d): the N(0,1) quantiser scaled by
  1/sqrt(d);
* "b bits" for TurboQuantProd means (b-1) Lloyd-Max bits + 1 QJL bit;
* the residual is r = x - ||x|| Pi^T c[idx] in the original frame;
  S has m = d rows; the estimator constant is sqrt(pi/2)/m;
* a coordinate on a decision boundary takes the lower index
  (idx = #{i : t_i < y}); sign(0) counts as +, i.e. z = [p >= 0];
* a zero vector has u = 0, rho = 0 and z = 1 everywhere.

Parity pins: every function here is pinned by ``tests/test_oracle.py`` to
closed forms, textbook values, brute force or the pages' printed numbers,
except the attention-fidelity sanity numbers, which nothing here computes.
"""
from __future__ import annotations

import math

import numpy as np

KAPPA_NUM = math.sqrt(math.pi / 2.0)   # the QJL estimator uses sqrt(pi/2)/m
TOKENS_PER_BLOCK = 128                 # packed layout: tokens per block
CHUNK_COORDS = 128                     # packed layout: coordinates per 16-byte chunk


# ----------------------------------------------------------------------------
# Stage 1 ingredients: the Lloyd-Max codebook and the random rotation
# ----------------------------------------------------------------------------

def _phi(x: float) -> float:
    """Standard normal density (0 at +-inf)."""
    if math.isinf(x):
        return 0.0
    return math.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)


def _mass(a: float, b: float) -> float:
    """P(a < Z <= b) for Z ~ N(0,1), written with erfc on the tail side so
    that far cells keep their relative precision."""
    if a >= 0.0:
        return 0.5 * (math.erfc(a / math.sqrt(2.0)) - math.erfc(b / math.sqrt(2.0)))
    if b <= 0.0:
        return 0.5 * (math.erfc(-b / math.sqrt(2.0)) - math.erfc(-a / math.sqrt(2.0)))
    return 1.0 - 0.5 * math.erfc(-a / math.sqrt(2.0)) - 0.5 * math.erfc(b / math.sqrt(2.0))


def _inv_normal_cdf(p: float) -> float:
    """Phi^{-1}(p) by bisection on the cdf (only used to start Lloyd-Max)."""
    lo, hi = -40.0, 40.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if 0.5 * math.erfc(-mid / math.sqrt(2.0)) < p:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def lloyd_max_normal(levels: int, tol: float = 1e-15, max_iter: int = 200000) -> np.ndarray:
    """Lloyd-Max scalar quantiser for N(0,1), ``levels`` ascending centroids.

    [PT-KR] "1단계": the codebook is optimal for the bell-shaped distribution
    the rotation produces and is precomputed once.  Lloyd's iteration: the
    boundaries are the midpoints of neighbouring centroids; each centroid is
    the conditional mean E[Z | cell] = (phi(a) - phi(b)) / (Phi(b) - Phi(a)).
    Started from the quantiles Phi^{-1}((i + 1/2) / L).
    """
    c = np.array([_inv_normal_cdf((i + 0.5) / levels) for i in range(levels)], dtype=np.float64)
    for _ in range(max_iter):
        edges = [-math.inf] + [0.5 * (c[i] + c[i + 1]) for i in range(levels - 1)] + [math.inf]
        new = np.array([(_phi(edges[i]) - _phi(edges[i + 1])) / _mass(edges[i], edges[i + 1])
                        for i in range(levels)], dtype=np.float64)
        delta = float(np.max(np.abs(new - c)))
        c = new
        if delta < tol:
            break
    return c


def codebook(levels: int, d: int) -> np.ndarray:
    """Centroids for one rotated coordinate, which is treated as N(0, 1/d)
    (READING): the N(0,1) Lloyd-Max centroids scaled by 1/sqrt(d), fp64."""
    return lloyd_max_normal(levels) / math.sqrt(d)


def codebook_f32(levels: int, d: int) -> np.ndarray:
    """The codebook as the fp32 values both sides consume."""
    return codebook(levels, d).astype(np.float32)


def haar_rotation(gaussian: np.ndarray) -> np.ndarray:
    """Random orthogonal Pi from a d x d Gaussian matrix ([PT-KR] "1단계": the
    input is rotated by a random orthogonal matrix).  Pi = Q diag(sign R_ii)
    for G = QR (Householder QR from LAPACK); the sign fix makes Pi Haar
    distributed and unique for a given G.  Returned in fp64."""
    q, r = np.linalg.qr(np.asarray(gaussian, dtype=np.float64))
    s = np.sign(np.diag(r))
    s[s == 0] = 1.0
    return q * s[None, :]


def hadamard_matrix(d: int) -> np.ndarray:
    """Sylvester's Walsh-Hadamard matrix of order d (a power of two), entries
    +-1, built by its recursive definition H_1 = [1], H_2n = [[H_n, H_n],
    [H_n, -H_n]]."""
    if d < 1 or d & (d - 1):
        raise ValueError("the Walsh-Hadamard matrix needs d a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def hadamard_rotation(signs) -> np.ndarray:
    """Randomised Walsh-Hadamard rotation Pi = H_d diag(signs) / sqrt(d), the
    structured rotation of "알고리즘보다 커널이 성패를 가른다" section 4 (WHT
    rotation, turboquant_plus).  READING: the pages name the transform only;
    the random sign flip before it is the usual way to randomise a fixed
    orthogonal transform (without it every key would see the same H).  The
    signs are an input (+-1, seeded by the caller).  fp64."""
    signs = np.asarray(signs, dtype=np.float64)
    if not np.all(np.abs(signs) == 1.0):
        raise ValueError("signs must be +-1")
    d = signs.size
    return hadamard_matrix(d) * signs[None, :] / math.sqrt(d)


def fwht(v) -> np.ndarray:
    """Fast Walsh-Hadamard transform (unnormalised) of the last axis by
    butterflies: returns H_d v for each row, in O(d log d)."""
    v = np.array(v, dtype=np.float64, copy=True)
    d = v.shape[-1]
    if d & (d - 1):
        raise ValueError("the Walsh-Hadamard transform needs d a power of two")
    h = 1
    while h < d:
        w = v.reshape(v.shape[:-1] + (d // (2 * h), 2, h))
        a, b = w[..., 0, :].copy(), w[..., 1, :].copy()
        w[..., 0, :] = a + b
        w[..., 1, :] = a - b
        h *= 2
    return v


def boundaries(c: np.ndarray) -> np.ndarray:
    """Decision boundaries t_i = (c_i + c_{i+1}) / 2, in fp64."""
    c = np.asarray(c, dtype=np.float64)
    return 0.5 * (c[:-1] + c[1:])


def quantize(y: np.ndarray, t: np.ndarray) -> np.ndarray:
    """Nearest-centroid index per coordinate: idx = #{i : t_i < y}
    (a value exactly on a boundary takes the lower index -- READING)."""
    return (np.asarray(y)[..., None] > np.asarray(t)).sum(axis=-1).astype(np.int64)


# ----------------------------------------------------------------------------
# Encode
# ----------------------------------------------------------------------------

def _as64(a) -> np.ndarray:
    if hasattr(a, "detach"):                     # a torch tensor
        a = a.detach().cpu().double().numpy()
    return np.asarray(a, dtype=np.float64)


def encode_mse(x, Pi, c) -> dict:
    """TurboQuantMSE ([PT-KR] "1단계"): normalise, rotate, quantise every
    coordinate independently with the Lloyd-Max codebook, keep ||x||.

    x: [N][d]; Pi: [d][d] (y = Pi u); c: ascending centroids (fp32 values).
    Returns idx [N][d], n [N], y [N][d] (rotated unit vector) and the
    exemption mask of coordinates within 1e-5 of a boundary.
    """
    x = _as64(x)
    Pi = _as64(Pi)
    c = _as64(c)
    t = boundaries(c)
    n = np.sqrt(np.sum(x * x, axis=1))
    u = np.zeros_like(x)
    nz = n > 0
    u[nz] = x[nz] / n[nz, None]
    y = u @ Pi.T                                  # y = Pi u, one key per row
    idx = quantize(y, t)
    near = np.any(np.abs(y[..., None] - t) <= 1e-5, axis=-1)
    return dict(idx=idx, n=n, y=y, code_exempt=near)


def mse_reconstruct(idx, n, Pi, c) -> np.ndarray:
    """x_mse = ||x|| Pi^T c[idx] for every key (rows)."""
    Pi = _as64(Pi)
    c = _as64(c)
    ytil = c[np.asarray(idx)]
    return _as64(n)[:, None] * (ytil @ Pi)       # (Pi^T ytil)^T = ytil^T Pi


def encode_prod(x, Pi, S, c) -> dict:
    """TurboQuantProd: the MSE stage at (b-1) bits, then QJL on the residual
    ([PT-KR] "2단계": project the quantisation residual with a random Gaussian
    matrix and keep only the sign of every projection; [TAMBUR]: the 1-bit
    QJL pass removes the bias of the MSE-only quantiser).

    r = x - ||x|| Pi^T c[idx]; rho = ||r||; p = S r; z_i = [p_i >= 0].
    Also returns the exemption masks the parity checker uses: codes within
    1e-5 (unit scale) of a boundary and signs with |p_i| <= 1e-5 ||x||.
    """
    out = encode_mse(x, Pi, c)
    out.update(qjl_stage(x, out["idx"], out["n"], Pi, S, c))
    return out


def qjl_stage(x, idx, n, Pi, S, c) -> dict:
    """The second stage for given first-stage codes ([PT-KR] "2단계"):
    r = x - n Pi^T c[idx], rho = ||r||, p = S r, z = [p >= 0], plus the sign
    exemption mask |p_i| <= 1e-5 n.  Also used to form the alternative
    encoding of a key whose coordinate sits on a code boundary (either code
    is then acceptable, and the signs follow the code taken)."""
    x = _as64(x)
    S = _as64(S)
    n = _as64(n)
    r = x - mse_reconstruct(idx, n, Pi, c)
    rho = np.sqrt(np.sum(r * r, axis=1))
    p = r @ S.T                                   # p = S r, one key per row
    z = p >= 0.0
    return dict(r=r, rho=rho, p=p, z=z, sign_exempt=np.abs(p) <= 1e-5 * n[:, None])


# ----------------------------------------------------------------------------
# Score and decode (inner products on the compressed keys)
# ----------------------------------------------------------------------------

def qjl_vector(z) -> np.ndarray:
    """The stored sign bits as +-1 (sign(S r) with sign(0) = +1)."""
    return np.where(np.asarray(z, dtype=bool), 1.0, -1.0)


def score_prod(q, idx, z, n, rho, Pi, S, c) -> np.ndarray:
    """Approximate inner products <q, x> from the compressed keys
    ([PT-KR] usage listing: ``tq.inner_product(query, compressed)``):

        <q, x_mse> + rho * sqrt(pi/2)/m * <S q, sign(S r)>.

    q: [H][d]; idx [N][d]; z [N][m]; n, rho [N] (the stored fp32 values).
    Returns logits [H][N].
    """
    q = _as64(q)
    S = _as64(S)
    m = S.shape[0]
    xm = mse_reconstruct(idx, n, Pi, c)           # [N][d]
    sq = q @ S.T                                  # [H][m]: S q per query
    qjl = sq @ qjl_vector(z).T                    # [H][N]
    return q @ xm.T + (_as64(rho)[None, :] * (KAPPA_NUM / m)) * qjl


def score_mse(q, idx, n, Pi, c) -> np.ndarray:
    """<q, x_mse> for MSE-only codes: [H][N]."""
    return _as64(q) @ mse_reconstruct(idx, n, Pi, c).T


def decode_prod(idx, z, n, rho, Pi, S, c) -> np.ndarray:
    """x_hat = x_mse + rho * sqrt(pi/2)/m * S^T sign(S r): the vector whose
    inner product with any q equals ``score_prod`` ([PT-KR] listing:
    ``tq.decompress(compressed)``)."""
    S = _as64(S)
    m = S.shape[0]
    xm = mse_reconstruct(idx, n, Pi, c)
    return xm + (_as64(rho)[:, None] * (KAPPA_NUM / m)) * (qjl_vector(z) @ S)


# ----------------------------------------------------------------------------
# Packed layout ([P5] section 3: bit-packed codes + QJL metadata)
#
# Keys are stored per group in blocks of 128 tokens.  In a block, for every
# plane p (the k code bits LSB first, then the sign plane when there is one),
# for every 128-coordinate chunk c, the 128 tokens' 16-byte chunks follow one
# another; then the 128 tokens' norm pairs (float ||x||, float ||r||).  In a
# 16-byte chunk, coordinate 128c + 32w + i is bit i of little-endian uint32
# word w.  Tokens past N in the last block are all-zero.
# ----------------------------------------------------------------------------

def plane_count(bits: int, mode: str) -> tuple[int, int]:
    """(code planes k, total planes) for a mode: 'prod' keeps bits-1 code
    planes and a sign plane, 'mse' keeps bits code planes."""
    if mode == "prod":
        return bits - 1, bits
    return bits, bits


def block_bytes(d: int, bits: int, mode: str) -> int:
    _, planes = plane_count(bits, mode)
    return TOKENS_PER_BLOCK * (planes * d // 8 + 8)


def packed_bytes(G: int, N: int, d: int, bits: int, mode: str) -> int:
    nb = -(-N // TOKENS_PER_BLOCK)
    return G * nb * block_bytes(d, bits, mode)


def pack(idx, z, n, rho, d: int, bits: int, mode: str, G: int, N: int) -> np.ndarray:
    """Pack codes [G*N][d], signs [G*N][d] (or None), norms [G*N] into bytes."""
    k, planes = plane_count(bits, mode)
    T = TOKENS_PER_BLOCK
    C = d // CHUNK_COORDS
    nb = -(-N // T)
    npad = nb * T
    bitplanes = np.zeros((G, npad, planes, d), dtype=np.uint64)
    idx = np.asarray(idx).reshape(G, N, d)
    for p in range(k):
        bitplanes[:, :N, p, :] = (idx >> p) & 1
    if mode == "prod":
        bitplanes[:, :N, k, :] = np.asarray(z).reshape(G, N, d).astype(np.uint64)
    # coordinate j = 128c + 32w + i -> bit i of word w of chunk c
    b = bitplanes.reshape(G, nb, T, planes, C, 4, 32)
    words = (b << np.arange(32, dtype=np.uint64)).sum(axis=-1).astype(np.uint32)  # [G][nb][T][planes][C][4]
    words = words.transpose(0, 1, 3, 4, 2, 5)                                        # [G][nb][planes][C][T][4]
    norms = np.zeros((G, npad, 2), dtype=np.float32)
    norms[:, :N, 0] = np.asarray(n, dtype=np.float32).reshape(G, N)
    if mode == "prod":
        norms[:, :N, 1] = np.asarray(rho, dtype=np.float32).reshape(G, N)
    out = bytearray()
    for g in range(G):
        for blk in range(nb):
            out += words[g, blk].astype("<u4").tobytes()
            out += norms[g, blk * T:(blk + 1) * T].astype("<f4").tobytes()
    return np.frombuffer(bytes(out), dtype=np.uint8)


def unpack(buf, d: int, bits: int, mode: str, G: int, N: int) -> dict:
    """Inverse of ``pack``: idx [G*N][d], z [G*N][d] (prod), n, rho [G*N]
    (the stored fp32 values, returned as fp64)."""
    k, planes = plane_count(bits, mode)
    T = TOKENS_PER_BLOCK
    C = d // CHUNK_COORDS
    nb = -(-N // T)
    bb = block_bytes(d, bits, mode)
    buf = np.asarray(buf, dtype=np.uint8)
    assert buf.size == G * nb * bb
    plane_bytes = planes * C * T * 16
    idx = np.zeros((G, nb * T, d), dtype=np.int64)
    z = np.zeros((G, nb * T, d), dtype=bool)
    n = np.zeros((G, nb * T))
    rho = np.zeros((G, nb * T))
    for g in range(G):
        for blk in range(nb):
            base = (g * nb + blk) * bb
            w = np.frombuffer(buf[base:base + plane_bytes].tobytes(), dtype="<u4")
            w = w.reshape(planes, C, T, 4)
            bits_arr = (w[..., None] >> np.arange(32, dtype=np.uint32)) & 1   # [planes][C][T][4][32]
            bits_arr = bits_arr.transpose(2, 0, 1, 3, 4).reshape(T, planes, d)
            rows = slice(blk * T, (blk + 1) * T)
            for p in range(k):
                idx[g, rows] |= bits_arr[:, p, :].astype(np.int64) << p
            if mode == "prod":
                z[g, rows] = bits_arr[:, k, :].astype(bool)
            nr = np.frombuffer(buf[base + plane_bytes:base + bb].tobytes(), dtype="<f4").reshape(T, 2)
            n[g, rows] = nr[:, 0]
            rho[g, rows] = nr[:, 1]
    return dict(idx=idx[:, :N].reshape(G * N, d), z=z[:, :N].reshape(G * N, d),
                n=n[:, :N].reshape(G * N), rho=rho[:, :N].reshape(G * N))


def unpack_blocks(buf, d: int, bits: int, mode: str, n_blocks: int) -> dict:
    """The same layout as ``unpack``, read for whole 128-token blocks at once
    (numpy's little-endian bit order within each 16-byte chunk is exactly
    "coordinate 128c + 32w + i is bit i of little-endian word w").  Returns
    idx [n_blocks*128][d] (uint8), z [n_blocks*128][d] (bool), n, rho (fp64);
    padded tokens included.  Used where ``unpack``'s per-block loop is too
    slow (a million keys)."""
    k, planes = plane_count(bits, mode)
    T = TOKENS_PER_BLOCK
    C = d // CHUNK_COORDS
    bb = block_bytes(d, bits, mode)
    buf = np.asarray(buf, dtype=np.uint8).reshape(n_blocks, bb)
    plane_bytes = planes * C * T * 16
    chunks = buf[:, :plane_bytes].reshape(n_blocks, planes, C, T, 16)
    bits_arr = np.unpackbits(chunks, axis=-1, bitorder="little")            # [B][planes][C][T][128]
    bits_arr = bits_arr.transpose(0, 3, 1, 2, 4).reshape(n_blocks * T, planes, d)
    idx = np.zeros((n_blocks * T, d), dtype=np.uint8)
    for p in range(k):
        idx |= bits_arr[:, p, :] << p
    z = bits_arr[:, k, :].astype(bool) if mode == "prod" else np.zeros((n_blocks * T, d), dtype=bool)
    nr = np.ascontiguousarray(buf[:, plane_bytes:]).view("<f4").reshape(n_blocks * T, 2).astype(np.float64)
    return dict(idx=idx, z=z, n=nr[:, 0], rho=nr[:, 1])


def score_prod_rotated(q, idx, z, n, rho, Pi, S, c) -> np.ndarray:
    """The estimator of ``score_prod`` evaluated in the rotated frame,
    n <Pi q, c[idx]> + rho sqrt(pi/2)/m <S q, 2z - 1>, which equals it for an
    orthogonal Pi (<q, n Pi^T c[idx]> = n <Pi q, c[idx]>).  With the fp32 Pi
    the two differ by Pi's non-orthogonality (about 1e-7 relative).  It costs
    O(H d) per key instead of O(d^2), for scoring a million keys.
    q [H][d] -> logits [H][N]."""
    q = _as64(q)
    S = _as64(S)
    m = S.shape[0]
    qr = q @ _as64(Pi).T                          # [H][d]: Pi q per query
    sq = q @ S.T                                  # [H][m]: S q per query
    ytil = _as64(c)[np.asarray(idx)]              # [N][d]
    return (_as64(n)[None, :] * (qr @ ytil.T) +
            (_as64(rho)[None, :] * (KAPPA_NUM / m)) * (sq @ qjl_vector(z).T))


def score_mse_rotated(q, idx, n, Pi, c) -> np.ndarray:
    """``score_mse`` in the rotated frame, n <Pi q, c[idx]> (see
    ``score_prod_rotated``).  q [H][d] -> logits [H][N]."""
    qr = _as64(q) @ _as64(Pi).T
    return _as64(n)[None, :] * (qr @ _as64(c)[np.asarray(idx)].T)


# ----------------------------------------------------------------------------
# Fractional bit widths (2.5 / 3.5 bits per channel)
#
# [TAMBUR] reports quality-neutral KV caches at 3.5 bits per channel and a
# small degradation at 2.5.  READING (the pages do not say how the channels
# are split): b + 1/2 bits per channel on average, with the first d/2
# coordinates of the rotated vector quantised with one more Lloyd-Max bit
# than the other d/2.  After the random rotation every coordinate has the same
# distribution, so which half gets the extra bit does not matter; the first
# half is taken.  For TurboQuantProd the MSE stage is the mixed quantiser and
# the QJL stage is unchanged (b + 1/2 = (b - 1/2) MSE bits + 1 QJL bit).
# Parity of this reading is unpinned: only what the mathematics fixes is
# pinned (uniform special cases, nearest centroid per coordinate, the
# distortion as the mean of the two codebooks', unbiasedness).
# ----------------------------------------------------------------------------

def mixed_split(d: int) -> int:
    """Rotated coordinates [0, d_hi) take the larger codebook (READING: d/2)."""
    return d // 2


def centroids_mixed(idx, c_hi, c_lo, d_hi: int) -> np.ndarray:
    """c[idx] per coordinate: c_hi for coordinates < d_hi, c_lo for the rest."""
    idx = np.asarray(idx)
    out = np.empty(idx.shape, dtype=np.float64)
    out[..., :d_hi] = _as64(c_hi)[idx[..., :d_hi]]
    out[..., d_hi:] = _as64(c_lo)[idx[..., d_hi:]]
    return out


def encode_mse_mixed(x, Pi, c_hi, c_lo, d_hi: int) -> dict:
    """TurboQuantMSE with two codebooks: normalise, rotate, quantise
    coordinate j < d_hi with c_hi and the others with c_lo (nearest centroid,
    ties to the lower index).  Returns idx, n, y and the boundary-band mask."""
    x = _as64(x)
    n = np.sqrt(np.sum(x * x, axis=1))
    u = np.zeros_like(x)
    nz = n > 0
    u[nz] = x[nz] / n[nz, None]
    y = u @ _as64(Pi).T
    t_hi, t_lo = boundaries(c_hi), boundaries(c_lo)
    idx = np.empty(y.shape, dtype=np.int64)
    idx[:, :d_hi] = quantize(y[:, :d_hi], t_hi)
    idx[:, d_hi:] = quantize(y[:, d_hi:], t_lo)
    near = np.zeros(y.shape, dtype=bool)
    near[:, :d_hi] = np.any(np.abs(y[:, :d_hi, None] - t_hi) <= 1e-5, axis=-1)
    near[:, d_hi:] = np.any(np.abs(y[:, d_hi:, None] - t_lo) <= 1e-5, axis=-1)
    return dict(idx=idx, n=n, y=y, code_exempt=near)


def mse_reconstruct_mixed(idx, n, Pi, c_hi, c_lo, d_hi: int) -> np.ndarray:
    """x_mse = ||x|| Pi^T c[idx] with the per-coordinate codebooks."""
    return _as64(n)[:, None] * (centroids_mixed(idx, c_hi, c_lo, d_hi) @ _as64(Pi))


def encode_prod_mixed(x, Pi, S, c_hi, c_lo, d_hi: int) -> dict:
    """TurboQuantProd at a fractional width: the mixed MSE stage, then the QJL
    stage of ``qjl_stage`` on its residual."""
    out = encode_mse_mixed(x, Pi, c_hi, c_lo, d_hi)
    out.update(qjl_stage_mixed(x, out["idx"], out["n"], Pi, S, c_hi, c_lo, d_hi))
    return out


def qjl_stage_mixed(x, idx, n, Pi, S, c_hi, c_lo, d_hi: int) -> dict:
    """``qjl_stage`` with the mixed reconstruction."""
    x = _as64(x)
    S = _as64(S)
    n = _as64(n)
    r = x - mse_reconstruct_mixed(idx, n, Pi, c_hi, c_lo, d_hi)
    rho = np.sqrt(np.sum(r * r, axis=1))
    p = r @ S.T
    z = p >= 0.0
    return dict(r=r, rho=rho, p=p, z=z, sign_exempt=np.abs(p) <= 1e-5 * n[:, None])


def score_prod_mixed(q, idx, z, n, rho, Pi, S, c_hi, c_lo, d_hi: int) -> np.ndarray:
    """``score_prod`` with the mixed reconstruction: [H][N]."""
    q = _as64(q)
    S = _as64(S)
    m = S.shape[0]
    xm = mse_reconstruct_mixed(idx, n, Pi, c_hi, c_lo, d_hi)
    return q @ xm.T + (_as64(rho)[None, :] * (KAPPA_NUM / m)) * ((q @ S.T) @ qjl_vector(z).T)


def frac_block_bytes(d: int, k_lo: int, prod: bool) -> int:
    """Bytes of a 128-token block at a fractional width: k_lo full code planes
    (16 bytes per 128 coordinates per token), the extra bit of the first d/2
    coordinates (8 bytes per 128 coordinates per token), the sign plane
    (Prod) and the norm pairs."""
    return TOKENS_PER_BLOCK * ((k_lo + (1 if prod else 0)) * d // 8 + d // 16 + 8)


def pack_mixed(idx, z, n, rho, d: int, k_lo: int, prod: bool, G: int, N: int) -> np.ndarray:
    """Packed layout at a fractional width: per 128-token block, the k_lo full
    code planes as ``pack`` writes them (bit p of every coordinate's code),
    then the extra plane (bit k_lo of the codes of coordinates < d/2; 8 bytes
    per 128 coordinates per token, token-major, coordinate 64 c' + 32 w + i at
    bit i of word w of chunk c'), then the sign plane (Prod), then the norm
    pairs {||x||, ||r||} (||r|| = 0 for MSE).  Padded tokens are zero."""
    T = TOKENS_PER_BLOCK
    nb = -(-N // T)
    d_hi = mixed_split(d)
    idx = np.asarray(idx).reshape(G, N, d)
    full = [((idx >> p) & 1).astype(np.uint64) for p in range(k_lo)]
    if prod:
        full.append(np.asarray(z).reshape(G, N, d).astype(np.uint64))
    extra = ((idx[:, :, :d_hi] >> k_lo) & 1).astype(np.uint64)

    def words(bits, width):  # [G][N][width] bits -> [G][nb*T][width // 32] uint32
        b = np.zeros((G, nb * T, width), dtype=np.uint64)
        b[:, :N] = bits
        b = b.reshape(G, nb * T, width // 32, 32)
        return (b << np.arange(32, dtype=np.uint64)).sum(axis=-1).astype(np.uint32)

    out = bytearray()
    fw = [words(f, d) for f in full]
    ew = words(extra, d_hi)
    norms = np.zeros((G, nb * T, 2), dtype=np.float32)
    norms[:, :N, 0] = np.asarray(n, dtype=np.float32).reshape(G, N)
    if prod:
        norms[:, :N, 1] = np.asarray(rho, dtype=np.float32).reshape(G, N)
    C = d // CHUNK_COORDS
    for g in range(G):
        for blk in range(nb):
            rows = slice(blk * T, (blk + 1) * T)
            for p in range(k_lo):                       # full code planes: [C][T][4]
                out += fw[p][g, rows].reshape(T, C, 4).transpose(1, 0, 2).astype("<u4").tobytes()
            out += ew[g, rows].reshape(T, C, 2).transpose(1, 0, 2).astype("<u4").tobytes()
            if prod:
                out += fw[k_lo][g, rows].reshape(T, C, 4).transpose(1, 0, 2).astype("<u4").tobytes()
            out += norms[g, rows].astype("<f4").tobytes()
    return np.frombuffer(bytes(out), dtype=np.uint8)


def unpack_mixed(buf, d: int, k_lo: int, prod: bool, G: int, N: int) -> dict:
    """Inverse of ``pack_mixed``: idx [G*N][d], z (Prod), n, rho."""
    T = TOKENS_PER_BLOCK
    C = d // CHUNK_COORDS
    nb = -(-N // T)
    d_hi = mixed_split(d)
    bb = frac_block_bytes(d, k_lo, prod)
    buf = np.asarray(buf, dtype=np.uint8).reshape(G * nb, bb)
    full_bytes = T * C * 16

    def bits_of(section, width):  # [B][C'][T][w] words -> [B][T][width]
        w = np.ascontiguousarray(section).view("<u4")
        per = width // 32 // C
        w = w.reshape(G * nb, C, T, per).transpose(0, 2, 1, 3).reshape(G * nb, T, width // 32)
        return ((w[..., None] >> np.arange(32, dtype=np.uint32)) & 1).reshape(G * nb, T, width)

    off = 0
    idx = np.zeros((G * nb, T, d), dtype=np.int64)
    for p in range(k_lo):
        idx |= bits_of(buf[:, off:off + full_bytes], d).astype(np.int64) << p
        off += full_bytes
    ext = bits_of(buf[:, off:off + full_bytes // 2], d_hi)
    idx[:, :, :d_hi] |= ext.astype(np.int64) << k_lo
    off += full_bytes // 2
    z = np.zeros((G * nb, T, d), dtype=bool)
    if prod:
        z = bits_of(buf[:, off:off + full_bytes], d).astype(bool)
        off += full_bytes
    nr = np.ascontiguousarray(buf[:, off:off + T * 8]).view("<f4").reshape(G, nb * T, 2).astype(np.float64)
    idx = idx.reshape(G, nb * T, d)[:, :N].reshape(G * N, d)
    z = z.reshape(G, nb * T, d)[:, :N].reshape(G * N, d)
    return dict(idx=idx, z=z, n=nr[:, :N, 0].reshape(G * N), rho=nr[:, :N, 1].reshape(G * N))


# ----------------------------------------------------------------------------
# Values and the attention output of one decode step
#
# The value cache holds TurboQuantMSE codes ([PT-KR] "1단계"; the pages' 58 MB
# figure compresses K and V at 3 bits) in a coordinate-major layout: per group,
# blocks of 128 tokens; per block, for every code plane p (LSB first) and every
# coordinate j, 16 bytes holding bit p of the code of coordinate j of the
# block's 128 tokens, token t at bit t % 32 of little-endian word t // 32;
# then the 128 tokens' {float ||v||, float 0}.  It holds the same bits as
# ``pack`` in MSE mode, transposed within each block (READING: the pages fix
# no layout; this one lets a kernel read one coordinate across a block's
# tokens as one 16-byte chunk).
# ----------------------------------------------------------------------------

def pack_values(idx, n, d: int, bits: int, G: int, N: int) -> np.ndarray:
    """Pack MSE value codes [G*N][d] (bits-bit) and norms [G*N] in the
    coordinate-major value layout."""
    T = TOKENS_PER_BLOCK
    nb = -(-N // T)
    idx = np.asarray(idx).reshape(G, N, d)
    planes = np.zeros((G, nb * T, bits, d), dtype=np.uint64)
    for p in range(bits):
        planes[:, :N, p, :] = (idx >> p) & 1
    b = planes.reshape(G, nb, 4, 32, bits, d)                          # token t = 32 w + i
    words = (b << np.arange(32, dtype=np.uint64)[None, None, None, :, None, None]).sum(axis=3)
    words = words.astype(np.uint32).transpose(0, 1, 3, 4, 2)           # [G][nb][bits][d][4]
    norms = np.zeros((G, nb * T, 2), dtype=np.float32)
    norms[:, :N, 0] = np.asarray(n, dtype=np.float32).reshape(G, N)
    out = bytearray()
    for g in range(G):
        for blk in range(nb):
            out += words[g, blk].astype("<u4").tobytes()
            out += norms[g, blk * T:(blk + 1) * T].astype("<f4").tobytes()
    return np.frombuffer(bytes(out), dtype=np.uint8)


def unpack_values(buf, d: int, bits: int, G: int, N: int) -> dict:
    """Inverse of ``pack_values``: idx [G*N][d], n [G*N] (fp64 of the stored fp32)."""
    T = TOKENS_PER_BLOCK
    nb = -(-N // T)
    bb = block_bytes(d, bits, "mse")
    buf = np.asarray(buf, dtype=np.uint8).reshape(G * nb, bb)
    plane_bytes = bits * d * 16
    w = np.ascontiguousarray(buf[:, :plane_bytes]).view("<u4").reshape(G * nb, bits, d, 4)
    tbits = (w[..., None] >> np.arange(32, dtype=np.uint32)) & 1      # [B][bits][d][4][32]
    tbits = tbits.reshape(G * nb, bits, d, T).transpose(0, 3, 1, 2)    # [B][T][bits][d]
    idx = np.zeros((G * nb, T, d), dtype=np.int64)
    for p in range(bits):
        idx |= tbits[:, :, p, :].astype(np.int64) << p
    nr = np.ascontiguousarray(buf[:, plane_bytes:]).view("<f4").reshape(G, nb * T, 2)
    idx = idx.reshape(G, nb * T, d)
    return dict(idx=idx[:, :N].reshape(G * N, d), n=nr[:, :N, 0].astype(np.float64).reshape(G * N))


def attend(q, kidx, kz, kn, krho, Pi_k, S, c_k, vidx, vn, Pi_v, c_v, scale: float) -> np.ndarray:
    """One decode step of attention on the compressed cache, for one group:
    logits from the compressed keys ([PT-KR] usage listing ``inner_product``;
    [TAMBUR]: attention logits computed directly on the compressed keys),
    softmax over the tokens of scale * logit, and the probability-weighted sum
    of the values reconstructed from their MSE codes (``mse_reconstruct``,
    [PT-KR] ``decompress``):
        out_h = sum_t softmax_t(scale * l_h)_t * v_hat_t.
    READING: the pages name no scale; the caller passes it (1/sqrt(d) for the
    usual scaled dot-product attention).  q [H][d] -> [H][d]."""
    logits = score_prod(q, kidx, kz, kn, krho, Pi_k, S, c_k)           # [H][N]
    z = scale * logits
    z = z - np.max(z, axis=1, keepdims=True)
    e = np.exp(z)
    p = e / np.sum(e, axis=1, keepdims=True)
    return p @ mse_reconstruct(vidx, vn, Pi_v, c_v)


def attend_packed(q, kbuf, vbuf, Pi_k, S, c_k, kbits: int, Pi_v, c_v, vbits: int, G: int, N: int,
                  scale: float) -> np.ndarray:
    """``attend`` for every group: q [G][H][d], keys packed by ``pack`` (Prod),
    values by ``pack_values`` -> [G][H][d]."""
    q = _as64(q)
    d = q.shape[-1]
    ku = unpack(kbuf, d, kbits, "prod", G, N)
    vu = unpack_values(vbuf, d, vbits, G, N)
    out = np.zeros(q.shape)
    for g in range(G):
        r = slice(g * N, (g + 1) * N)
        out[g] = attend(q[g], ku["idx"][r], ku["z"][r], ku["n"][r], ku["rho"][r], Pi_k, S, c_k,
                        vu["idx"][r], vu["n"][r], Pi_v, c_v, scale)
    return out


# ----------------------------------------------------------------------------
# Whole-path helpers the tests and the CPU baseline use
# ----------------------------------------------------------------------------

def encode_pack(x, Pi, S, c, bits: int, mode: str, G: int, N: int):
    """Encode keys [G][N][d] and pack them; returns (bytes, encode dict)."""
    x = _as64(x)
    d = x.shape[-1]
    flat = x.reshape(G * N, d)
    if mode == "prod":
        e = encode_prod(flat, Pi, S, c)
        # stored norms are fp32
        buf = pack(e["idx"], e["z"], e["n"].astype(np.float32), e["rho"].astype(np.float32),
                   d, bits, mode, G, N)
    else:
        e = encode_mse(flat, Pi, c)
        buf = pack(e["idx"], None, e["n"].astype(np.float32), None, d, bits, mode, G, N)
    return buf, e


def score_packed(q, buf, Pi, S, c, bits: int, mode: str, G: int, N: int) -> np.ndarray:
    """Logits [G][H][N] from packed keys and queries [G][H][d]."""
    q = _as64(q)
    d = q.shape[-1]
    u = unpack(buf, d, bits, mode, G, N)
    out = np.zeros((G, q.shape[1], N))
    for g in range(G):
        rows = slice(g * N, (g + 1) * N)
        if mode == "prod":
            out[g] = score_prod(q[g], u["idx"][rows], u["z"][rows], u["n"][rows], u["rho"][rows], Pi, S, c)
        else:
            out[g] = score_mse(q[g], u["idx"][rows], u["n"][rows], Pi, c)
    return out


def decode_packed(buf, Pi, S, c, d: int, bits: int, mode: str, G: int, N: int) -> np.ndarray:
    u = unpack(buf, d, bits, mode, G, N)
    if mode == "prod":
        x = decode_prod(u["idx"], u["z"], u["n"], u["rho"], Pi, S, c)
    else:
        x = mse_reconstruct(u["idx"], u["n"], Pi, c)
    return x.reshape(G, N, d)


def score_fp32(q, x) -> np.ndarray:
    """The uncompressed baseline: exact <q, x> for every (head, key); q [G][H][d], x [G][N][d]."""
    return np.einsum("ghd,gnd->ghn", _as64(q), _as64(x))


def topk(scores, k: int):
    """Top-k per row: descending score, ties to the lower index."""
    s = np.asarray(scores)
    order = np.lexsort((np.broadcast_to(np.arange(s.shape[-1]), s.shape), -s), axis=-1)[..., :k]
    return np.take_along_axis(s, order, axis=-1), order
