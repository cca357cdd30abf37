"""Pins for the CPU oracle: closed forms, textbook values, brute force,
special cases and the numbers the pages print.  CPU only (not gpu).

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, a transposed operand, a wrong constant, a wrong bit offset) fails
at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy import integrate

from oracle import tq_oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


def _haar(d, seed):
    return o.haar_rotation(_rng(seed).standard_normal((d, d)))


# ---------------------------------------------------------------- codebook

@pytest.mark.parametrize("d", [1, 128, 1536])
def test_lloyd_max_one_bit_closed_form(d):
    # 1-bit Lloyd-Max for N(0,1/d): +-E|Z|/sqrt(d) = +-sqrt(2/pi)/sqrt(d)
    c = o.codebook(2, d)
    want = math.sqrt(2.0 / math.pi) / math.sqrt(d)
    assert np.allclose(c, [-want, want], rtol=0, atol=1e-12 / math.sqrt(d))


@pytest.mark.parametrize("levels", [2, 4, 8, 16])
def test_lloyd_max_textbook_tables(levels):
    tab = _golden("lloyd_max_textbook.json")["levels"][str(levels)]
    c = o.lloyd_max_normal(levels)
    pos = c[levels // 2:]
    for got, want in zip(pos, tab["outputs"]):
        assert abs(got - want) <= 6e-4 * max(1.0, want), (got, want)
    # symmetric about 0
    assert np.allclose(c, -c[::-1], atol=1e-13)
    # distortion E[(Z - Q(Z))^2] by numerical integration, independent of the
    # erf-based update the solver uses
    t = o.boundaries(c)
    edges = [-np.inf] + list(t) + [np.inf]
    pdf = lambda z: math.exp(-0.5 * z * z) / math.sqrt(2 * math.pi)
    mse = sum(integrate.quad(lambda z, ci=ci: (z - ci) ** 2 * pdf(z), a, b, epsabs=1e-14)[0]
              for ci, a, b in zip(c, edges[:-1], edges[1:]))
    assert abs(mse - tab["mse"]) <= 2e-4 * tab["mse"] + 5e-6


@pytest.mark.parametrize("levels", [2, 4, 8, 16])
def test_lloyd_max_stationarity(levels):
    # every centroid is the conditional mean of its cell (numerical quadrature)
    c = o.lloyd_max_normal(levels)
    t = o.boundaries(c)
    edges = [-np.inf] + list(t) + [np.inf]
    pdf = lambda z: math.exp(-0.5 * z * z) / math.sqrt(2 * math.pi)
    for ci, a, b in zip(c, edges[:-1], edges[1:]):
        mass = integrate.quad(pdf, a, b, epsabs=1e-15, epsrel=1e-13)[0]
        mean = integrate.quad(lambda z: z * pdf(z), a, b, epsabs=1e-15, epsrel=1e-13)[0] / mass
        assert abs(mean - ci) < 1e-10


def test_boundaries_are_nearest_centroid_decisions():
    # brute force: the threshold rule picks the nearest centroid
    c = o.codebook_f32(8, 128).astype(np.float64)
    t = o.boundaries(c)
    y = _rng(1).standard_normal(20000) / math.sqrt(128) * 1.5
    idx = o.quantize(y, t)
    nearest = np.argmin(np.abs(y[:, None] - c[None, :]), axis=1)
    assert np.array_equal(idx, nearest)


def test_quantize_tie_takes_lower_index():
    c = np.array([-3.0, -1.0, 1.0, 3.0])
    t = o.boundaries(c)                     # -2, 0, 2
    assert list(o.quantize(np.array([-2.0, 0.0, 2.0, 2.0000001, -10.0, 10.0]), t)) == [0, 1, 2, 3, 0, 3]


# ---------------------------------------------------------------- rotation

@pytest.mark.parametrize("d", [16, 128])
def test_rotation_orthogonal_and_norm_preserving(d):
    Pi = _haar(d, 3)
    assert np.max(np.abs(Pi.T @ Pi - np.eye(d))) <= 1e-12
    Pi32 = Pi.astype(np.float32).astype(np.float64)
    x = _rng(4).standard_normal((10000, d))
    ratio = np.linalg.norm(x @ Pi32.T, axis=1) / np.linalg.norm(x, axis=1)
    assert np.max(np.abs(ratio - 1.0)) <= 1e-6


@pytest.mark.parametrize("d", [8, 48])
def test_rotation_matches_gram_schmidt(d):
    # Gram-Schmidt on G's columns gives the QR factor with positive R diagonal,
    # which is what the Haar sign fix must produce
    G = _rng(5).standard_normal((d, d))
    Q = np.zeros_like(G)
    for j in range(d):
        v = G[:, j].copy()
        for _ in range(2):                   # re-orthogonalise once
            for i in range(j):
                v -= (Q[:, i] @ v) * Q[:, i]
        Q[:, j] = v / np.linalg.norm(v)
    assert np.max(np.abs(o.haar_rotation(G) - Q)) <= 1e-9


def test_rotation_of_upper_triangular_is_identity():
    G = np.triu(_rng(6).standard_normal((12, 12)))
    G[np.diag_indices(12)] = np.abs(G[np.diag_indices(12)]) + 0.1
    assert np.allclose(o.haar_rotation(G), np.eye(12), atol=1e-12)
    # with a negative diagonal entry the QR factor with positive R diagonal is
    # diag(sign G_ii)
    G[3, 3] *= -1
    want = np.eye(12)
    want[3, 3] = -1.0
    assert np.allclose(o.haar_rotation(G), want, atol=1e-12)


# ---------------------------------------------------------------- encode special cases

def _signed_perm(d, seed):
    rng = _rng(seed)
    perm = rng.permutation(d)
    sgn = rng.choice([-1.0, 1.0], size=d)
    P = np.zeros((d, d))
    P[np.arange(d), perm] = sgn                # (P u)_j = sgn_j * u_perm[j]
    return P, perm, sgn


def test_encode_with_signed_permutation_rotation():
    # Pi a signed permutation: y_j = sgn_j u_{perm(j)} exactly, so the codes are
    # the scalar quantisation of the permuted unit vector, and the MSE
    # reconstruction is n * Pi^T c[idx] = n * (sgn * c[idx]) scattered back
    d = 32
    Pi, perm, sgn = _signed_perm(d, 11)
    c = o.codebook_f32(4, d)
    x = _rng(12).standard_normal((50, d)) * 3.0
    e = o.encode_mse(x, Pi, c)
    u = x / np.linalg.norm(x, axis=1, keepdims=True)
    want_idx = o.quantize(sgn[None, :] * u[:, perm], o.boundaries(c))
    assert np.array_equal(e["idx"], want_idx)
    xm = o.mse_reconstruct(e["idx"], e["n"], Pi, c)
    want = np.zeros_like(x)
    want[:, perm] = np.linalg.norm(x, axis=1)[:, None] * sgn[None, :] * c[e["idx"]]
    assert np.allclose(xm, want, atol=1e-12)


def test_encode_with_identity_rotation_and_projection():
    # Pi = I: codes quantise u itself.  S = I: p = r, so z = [r >= 0] and the
    # estimator is rho sqrt(pi/2)/d * sum_j q_j sign(r_j)
    d = 64
    I = np.eye(d)
    c = o.codebook_f32(4, d)
    x = _rng(13).standard_normal((40, d))
    e = o.encode_prod(x, I, I, c)
    u = x / np.linalg.norm(x, axis=1, keepdims=True)
    assert np.array_equal(e["idx"], o.quantize(u, o.boundaries(c)))
    r = x - np.linalg.norm(x, axis=1, keepdims=True) * c[e["idx"]]
    assert np.allclose(e["r"], r, atol=1e-12)
    assert np.array_equal(e["z"], r >= 0)
    q = _rng(14).standard_normal((3, d))
    got = o.score_prod(q, e["idx"], e["z"], e["n"], e["rho"], I, I, c)
    want = q @ (x - r).T + np.linalg.norm(r, axis=1)[None, :] * math.sqrt(math.pi / 2) / d * (q @ np.sign(r).T)
    assert np.allclose(got, want, atol=1e-10)


def test_encode_projection_is_S_times_residual():
    # S a signed permutation (not symmetric): p_i = sgn_i r_{perm(i)}
    d = 32
    S, perm, sgn = _signed_perm(d, 15)
    Pi = _haar(d, 16)
    c = o.codebook_f32(2, d)
    x = _rng(17).standard_normal((30, d))
    e = o.encode_prod(x, Pi, S, c)
    assert np.allclose(e["p"], sgn[None, :] * e["r"][:, perm], atol=1e-13)
    assert np.array_equal(e["z"], sgn[None, :] * e["r"][:, perm] >= 0)


def test_encode_scaled_basis_vectors():
    # x = a e_j: n = |a|, y = sign(a) * column j of Pi
    d = 16
    Pi = _haar(d, 18)
    c = o.codebook_f32(4, d)
    for j, a in [(0, 2.5), (5, -0.75), (15, 1e-3)]:
        x = np.zeros((1, d))
        x[0, j] = a
        e = o.encode_mse(x, Pi, c)
        assert abs(e["n"][0] - abs(a)) < 1e-15
        assert np.allclose(e["y"][0], np.sign(a) * Pi[:, j], atol=1e-15)


def test_zero_vector():
    d = 32
    Pi = _haar(d, 19)
    S = _rng(20).standard_normal((d, d))
    c = o.codebook_f32(4, d)
    e = o.encode_prod(np.zeros((1, d)), Pi, S, c)
    t = o.boundaries(c)
    assert e["n"][0] == 0.0 and e["rho"][0] == 0.0
    assert np.all(e["idx"][0] == np.sum(t < 0))
    assert np.all(e["z"][0])
    q = _rng(21).standard_normal((2, d))
    assert np.all(o.score_prod(q, e["idx"], e["z"], e["n"], e["rho"], Pi, S, c) == 0.0)


def test_brute_force_d4():
    # every coordinate's code minimises ||y - c[idx]|| over all L^4 codewords;
    # the sign vector maximises <2z - 1, p> over all 2^4 sign vectors
    d = 4
    Pi = _haar(d, 22)
    S = _rng(23).standard_normal((d, d))
    c = o.codebook_f32(4, d).astype(np.float64)
    x = _rng(24).standard_normal((25, d))
    e = o.encode_prod(x, Pi, S, c)
    words = np.array(list(itertools.product(range(4), repeat=d)))
    signs = np.array(list(itertools.product([-1.0, 1.0], repeat=d)))
    for k in range(x.shape[0]):
        dist = np.sum((e["y"][k][None, :] - c[words]) ** 2, axis=1)
        assert np.array_equal(words[np.argmin(dist)], e["idx"][k])
        best = signs[np.argmax(signs @ e["p"][k])]
        assert np.array_equal(best > 0, e["z"][k])


# ---------------------------------------------------------------- estimator

def test_unbiased_inner_product_over_projections():
    # [PT-KR] '2단계' / [TAMBUR]: the QJL correction makes <q, x> unbiased.
    # Over T draws of S (Pi fixed), the estimate's mean is <q, x> within 4
    # standard errors, and its variance matches the closed form
    #   Var = [(pi/2) rho^2 ||q||^2 - <q, r>^2] / m
    d, T = 64, 3000
    rng = _rng(25)
    Pi = _haar(d, 26)
    c = o.codebook_f32(2, d)
    x = rng.standard_normal((1, d))
    q = rng.standard_normal((1, d))
    base = o.encode_mse(x, Pi, c)
    r = x - o.mse_reconstruct(base["idx"], base["n"], Pi, c)
    rho = np.linalg.norm(r)
    est = np.empty(T)
    for s in range(T):
        S = rng.standard_normal((d, d))
        e = o.encode_prod(x, Pi, S, c)
        est[s] = o.score_prod(q, e["idx"], e["z"], e["n"], e["rho"], Pi, S, c)[0, 0]
    truth = (q @ x.T).item()
    var = ((math.pi / 2) * rho ** 2 * (q @ q.T).item() - (q @ r.T).item() ** 2) / d
    assert abs(est.mean() - truth) <= 4 * math.sqrt(var / T)
    assert abs(est.var() / var - 1.0) <= 0.1


def test_mse_only_is_biased_prod_is_not():
    # [TAMBUR]: an MSE-optimal quantiser gives a biased inner-product estimate
    # (it shrinks); the 1-bit QJL pass removes the bias.  1-bit codebook:
    # E <q, x_mse> ~= (2/pi) <q, x> for large d
    d, T = 64, 1500
    rng = _rng(27)
    x = rng.standard_normal((1, d))
    q = x + 0.3 * rng.standard_normal((1, d))
    truth = (q @ x.T).item()
    c1 = o.codebook_f32(2, d)
    mse, prod = [], []
    for s in range(T):
        Pi = o.haar_rotation(rng.standard_normal((d, d)))
        S = rng.standard_normal((d, d))
        e = o.encode_prod(x, Pi, S, c1)
        mse.append(o.score_mse(q, e["idx"], e["n"], Pi, c1)[0, 0])
        prod.append(o.score_prod(q, e["idx"], e["z"], e["n"], e["rho"], Pi, S, c1)[0, 0])
    bias_mse = np.mean(mse) - truth
    bias_prod = np.mean(prod) - truth
    assert bias_mse < 0 and abs(np.mean(mse) / truth - 2 / math.pi) < 0.05
    assert abs(bias_prod) < abs(bias_mse) / 10


def test_mse_distortion_3bit_matches_the_pages():
    # turboquant-pytorch 소개, '성능 지표': 3-bit MSE distortion measured 0.034,
    # theoretical bound 0.043 (unit vectors; READING: a 3-bit TurboQuantMSE codebook)
    g = _golden("pages_printed_values.json")
    d, n = 128, 40000
    rng = _rng(28)
    Pi = _haar(d, 29)
    c = o.codebook_f32(8, d)
    u = rng.standard_normal((n, d))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    e = o.encode_mse(u, Pi, c)
    D = np.mean(np.sum((u - o.mse_reconstruct(e["idx"], e["n"], Pi, c)) ** 2, axis=1))
    assert D <= g["mse_distortion_3bit_bound"]
    assert abs(D - g["mse_distortion_3bit_measured"]) <= 0.002


def test_decode_and_score_agree():
    d = 128
    rng = _rng(30)
    Pi = _haar(d, 31)
    S = rng.standard_normal((d, d)).astype(np.float32)
    c = o.codebook_f32(4, d)
    x = rng.standard_normal((64, d))
    q = rng.standard_normal((5, d))
    e = o.encode_prod(x, Pi.astype(np.float32), S, c)
    xh = o.decode_prod(e["idx"], e["z"], e["n"], e["rho"], Pi.astype(np.float32), S, c)
    s = o.score_prod(q, e["idx"], e["z"], e["n"], e["rho"], Pi.astype(np.float32), S, c)
    assert np.max(np.abs(q @ xh.T - s)) <= 1e-12 * np.max(np.abs(s))


@pytest.mark.parametrize("m", [32, 48])
def test_decode_prod_is_unbiased_over_projections(m):
    # The QJL stage reconstructs the residual without bias: for S with i.i.d.
    # N(0, 1) entries (m rows), E[s sign(s . r)] = sqrt(2/pi) r / ||r|| per row,
    # so E[sqrt(pi/2)/m * rho * S^T sign(S r)] = r and E_S[x_hat] = x exactly
    # (Pi fixed).  Per coordinate, Var[x_hat_j] = ((pi/2) rho^2 - r_j^2) / m.
    # Independent of score_prod: a wrong constant, a missing rho, S in place
    # of S^T (m = d, where the shapes allow it) or a flipped sign moves the
    # mean; dividing by d instead of m (m != d) moves it too.
    d, T = 32, 4000
    rng = _rng(33 + m)
    Pi = _haar(d, 34)
    c = o.codebook_f32(4, d)
    x = rng.standard_normal((1, d))
    base = o.encode_mse(x, Pi, c)
    r = (x - o.mse_reconstruct(base["idx"], base["n"], Pi, c))[0]
    rho = np.linalg.norm(r)
    xh = np.empty((T, d))
    for s in range(T):
        S = rng.standard_normal((m, d))
        e = o.encode_prod(x, Pi, S, c)
        xh[s] = o.decode_prod(e["idx"], e["z"], e["n"], e["rho"], Pi, S, c)[0]
    var = ((math.pi / 2) * rho ** 2 - r ** 2) / m
    z = (xh.mean(axis=0) - x[0]) / np.sqrt(var / T)
    assert np.all(np.abs(z) <= 4.5), np.abs(z).max()
    assert np.all(np.abs(xh.var(axis=0) / var - 1.0) <= 0.15)


def test_score_fp32_is_the_plain_dot_product():
    rng = _rng(32)
    q = rng.standard_normal((2, 3, 8))
    x = rng.standard_normal((2, 5, 8))
    got = o.score_fp32(q, x)
    for g in range(2):
        for h in range(3):
            for t in range(5):
                assert abs(got[g, h, t] - sum(q[g, h, i] * x[g, t, i] for i in range(8))) < 1e-12


def test_topk_order_and_ties():
    s = np.array([[1.0, 5.0, 3.0, 5.0, 2.0]])
    v, i = o.topk(s, 3)
    assert list(i[0]) == [1, 3, 2] and list(v[0]) == [5.0, 5.0, 3.0]


# ---------------------------------------------------------------- packed layout

@pytest.mark.parametrize("bits,mode", [(2, "prod"), (3, "prod"), (4, "prod"), (3, "mse")])
def test_pack_roundtrip_and_bit_addresses(bits, mode):
    G, N, d = 2, 300, 256
    rng = _rng(33)
    k, planes = o.plane_count(bits, mode)
    idx = rng.integers(0, 1 << k, size=(G * N, d))
    z = rng.integers(0, 2, size=(G * N, d)).astype(bool)
    n = rng.random(G * N).astype(np.float32)
    rho = rng.random(G * N).astype(np.float32)
    buf = o.pack(idx, z, n, rho, d, bits, mode, G, N)
    assert buf.size == o.packed_bytes(G, N, d, bits, mode)
    u = o.unpack(buf, d, bits, mode, G, N)
    assert np.array_equal(u["idx"], idx)
    if mode == "prod":
        assert np.array_equal(u["z"], z)
        assert np.array_equal(u["rho"], rho.astype(np.float64))
    assert np.array_equal(u["n"], n.astype(np.float64))
    # hand-computed addresses: block bytes = 128 * (planes * d / 8 + 8)
    bb = 128 * (planes * d // 8 + 8)
    nb = 3                                  # ceil(300 / 128)
    for (g, tok, p, j) in [(0, 0, 0, 0), (1, 299, planes - 1, d - 1), (1, 130, 0, 37), (0, 257, planes - 1, 129)]:
        blk, t = divmod(tok, 128)
        cch, rem = divmod(j, 128)
        w, i = divmod(rem, 32)
        off = (g * nb + blk) * bb + ((p * (d // 128) + cch) * 128 + t) * 16 + 4 * w
        word = int.from_bytes(bytes(buf[off:off + 4]), "little")
        if p < k:
            want = (idx[g * N + tok, j] >> p) & 1
        else:
            want = int(z[g * N + tok, j])
        assert (word >> i) & 1 == want
        noff = (g * nb + blk) * bb + planes * (d // 128) * 128 * 16 + t * 8
        assert np.frombuffer(bytes(buf[noff:noff + 4]), "<f4")[0] == n[g * N + tok]
    # padded tokens are all zero
    pad_t = 300 - 256
    last = (1 * nb + 2) * bb
    for p in range(planes):
        off = last + ((p * (d // 128)) * 128 + pad_t) * 16
        assert not np.any(buf[off:off + 16])


def test_packed_bytes_per_key_and_footprint():
    # bytes per key: (k d + m)/8 + 8 for Prod
    assert o.block_bytes(128, 2, "prod") // 128 == 40
    assert o.block_bytes(128, 3, "prod") // 128 == 56
    assert o.block_bytes(128, 4, "prod") // 128 == 72
    assert o.block_bytes(1536, 4, "prod") // 128 == 776
    # the pages' KV figure: fp16 K+V of a 36-layer, 2-KV-head, head_dim-128
    # model at 8K context is 289 MB (MiB); 3 bits cut it to 58 MB
    g = _golden("pages_printed_values.json")
    vectors = 36 * 2 * 2 * 8192                        # layers x KV heads x {K,V} x tokens
    fp16_mib = vectors * 128 * 2 / 2 ** 20
    assert abs(fp16_mib - g["kv_cache_fp16_mb_qwen25_3b_8k"]) / 289 < 0.01
    # 3-bit payload (48 B) + two fp16 norms (4 B) per vector reproduces 58 MB
    assert abs(vectors * (3 * 128 / 8 + 4) / 2 ** 20 - g["kv_cache_3bit_mb_qwen25_3b_8k"]) / 58 < 0.02


@pytest.mark.parametrize("bits,mode,d", [(3, "prod", 128), (4, "prod", 256), (4, "mse", 128)])
def test_unpack_blocks_reads_the_same_layout(bits, mode, d):
    # the vectorised reader agrees with unpack (itself pinned to hand-computed
    # bit addresses above) on every token, padding included
    G, N = 2, 300
    rng = _rng(34)
    k, _ = o.plane_count(bits, mode)
    idx = rng.integers(0, 1 << k, size=(G * N, d))
    z = rng.integers(0, 2, size=(G * N, d)).astype(bool)
    n = rng.random(G * N).astype(np.float32)
    rho = rng.random(G * N).astype(np.float32)
    buf = o.pack(idx, z, n, rho, d, bits, mode, G, N)
    nb = 3
    b = o.unpack_blocks(buf, d, bits, mode, G * nb)
    u = o.unpack(buf, d, bits, mode, G, N)
    rows = np.concatenate([g * nb * 128 + np.arange(N) for g in range(G)])
    assert np.array_equal(b["idx"][rows].astype(np.int64), u["idx"])
    assert np.array_equal(b["n"][rows], u["n"])
    if mode == "prod":
        assert np.array_equal(b["z"][rows], u["z"])
        assert np.array_equal(b["rho"][rows], u["rho"])
    pad = np.setdiff1d(np.arange(G * nb * 128), rows)
    assert not b["idx"][pad].any() and not b["z"][pad].any() and not b["n"][pad].any()


def test_score_in_the_rotated_frame_equals_score_prod():
    d = 128
    rng = _rng(35)
    S = rng.standard_normal((d, d)).astype(np.float32)
    c = o.codebook_f32(4, d)
    x = rng.standard_normal((50, d))
    q = rng.standard_normal((3, d))
    # fp64 Haar rotation: the identity <q, n Pi^T c> = n <Pi q, c> holds to rounding
    Pi = _haar(d, 36)
    e = o.encode_prod(x, Pi, S, c)
    a = o.score_prod(q, e["idx"], e["z"], e["n"], e["rho"], Pi, S, c)
    b = o.score_prod_rotated(q, e["idx"], e["z"], e["n"], e["rho"], Pi, S, c)
    assert np.max(np.abs(a - b)) <= 1e-12 * np.max(np.abs(a))
    # fp32 rotation: within its non-orthogonality
    Pi32 = Pi.astype(np.float32)
    e = o.encode_prod(x, Pi32, S, c)
    a = o.score_prod(q, e["idx"], e["z"], e["n"], e["rho"], Pi32, S, c)
    b = o.score_prod_rotated(q, e["idx"], e["z"], e["n"], e["rho"], Pi32, S, c)
    bound = 1e-6 * np.linalg.norm(q, axis=1)[:, None] * e["n"][None, :]
    assert np.all(np.abs(a - b) <= bound)
    # the MSE-only estimate likewise
    m = o.encode_mse(x, Pi, c)
    a = o.score_mse(q, m["idx"], m["n"], Pi, c)
    b = o.score_mse_rotated(q, m["idx"], m["n"], Pi, c)
    assert np.max(np.abs(a - b)) <= 1e-12 * np.max(np.abs(a))


# ---------------------------------------------------------------- Walsh-Hadamard rotation

def test_hadamard_small_orders_by_hand():
    assert np.array_equal(o.hadamard_matrix(1), [[1.0]])
    assert np.array_equal(o.hadamard_matrix(2), [[1, 1], [1, -1]])
    assert np.array_equal(o.hadamard_matrix(4), [[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]])
    with pytest.raises(ValueError):
        o.hadamard_matrix(12)


@pytest.mark.parametrize("d", [8, 128, 1024])
def test_hadamard_rotation_orthogonal_and_matches_the_butterflies(d):
    rng = _rng(40)
    signs = np.where(rng.standard_normal(d) >= 0, 1.0, -1.0)
    Pi = o.hadamard_rotation(signs)
    # H H^T = d I, so Pi is orthogonal (symmetric H, diagonal signs)
    assert np.max(np.abs(Pi @ Pi.T - np.eye(d))) <= 1e-12
    assert np.array_equal(o.hadamard_matrix(d), o.hadamard_matrix(d).T)
    # the matrix and the O(d log d) transform agree: Pi u = H (signs * u) / sqrt(d)
    u = rng.standard_normal((5, d))
    assert np.max(np.abs(u @ Pi.T - o.fwht(u * signs) / math.sqrt(d))) <= 1e-12
    # entry (i, j) is (-1)^popcount(i & j) * signs[j] / sqrt(d)
    for i, j in [(0, 0), (1, 1), (3, 5), (d - 1, d - 1), (d // 2, 1)]:
        want = (-1.0) ** bin(i & j).count("1") * signs[j] / math.sqrt(d)
        assert Pi[i, j] == pytest.approx(want, abs=1e-15)


def test_hadamard_rotation_spreads_a_basis_vector():
    # every rotated coordinate of e_j has magnitude 1/sqrt(d): the structured
    # rotation flattens a spike, as a random rotation does on average
    d = 128
    signs = np.where(_rng(41).standard_normal(d) >= 0, 1.0, -1.0)
    Pi = o.hadamard_rotation(signs)
    for j in (0, 7, 127):
        assert np.allclose(np.abs(Pi[:, j]), 1 / math.sqrt(d), atol=1e-15)
    with pytest.raises(ValueError):
        o.hadamard_rotation(np.array([1.0, 0.5]))


def test_mse_distortion_3bit_with_the_hadamard_rotation():
    # the structured rotation keeps the pages' 3-bit distortion on random unit
    # vectors (the same bound as the dense Haar rotation)
    d, n = 128, 20000
    rng = _rng(42)
    signs = np.where(rng.standard_normal(d) >= 0, 1.0, -1.0)
    Pi = o.hadamard_rotation(signs).astype(np.float32)
    x = rng.standard_normal((n, d))
    x /= np.linalg.norm(x, axis=1, keepdims=True)
    c = o.codebook_f32(8, d)
    e = o.encode_mse(x, Pi, c)
    D = np.mean(np.sum((x - o.mse_reconstruct(e["idx"], e["n"], Pi, c)) ** 2, axis=1))
    g = _golden("pages_printed_values.json")
    assert D <= g["mse_distortion_3bit_bound"]
    assert abs(D - g["mse_distortion_3bit_measured"]) <= 0.002


# ---------------------------------------------------------------- value layout and attention

@pytest.mark.parametrize("bits", [1, 3, 4])
def test_value_layout_roundtrip_and_bit_addresses(bits):
    G, N, d = 2, 300, 256
    rng = _rng(50)
    idx = rng.integers(0, 1 << bits, size=(G * N, d))
    n = rng.random(G * N).astype(np.float32)
    buf = o.pack_values(idx, n, d, bits, G, N)
    # the same number of bytes per key as the MSE layout
    assert buf.size == o.packed_bytes(G, N, d, bits, "mse")
    u = o.unpack_values(buf, d, bits, G, N)
    assert np.array_equal(u["idx"], idx) and np.array_equal(u["n"], n.astype(np.float64))
    # hand-computed addresses: plane p, coordinate j, token t of a block is bit
    # t % 32 of word t // 32 of the 16 bytes at ((p d + j) 16) in the block
    bb = 128 * (bits * d // 8 + 8)
    nb = 3
    for (g, tok, p, j) in [(0, 0, 0, 0), (1, 299, bits - 1, d - 1), (1, 130, 0, 37), (0, 257, bits - 1, 129),
                           (0, 31, 0, 5), (1, 33, bits - 1, 200)]:
        blk, t = divmod(tok, 128)
        w, i = divmod(t, 32)
        off = (g * nb + blk) * bb + (p * d + j) * 16 + 4 * w
        word = int.from_bytes(bytes(buf[off:off + 4]), "little")
        assert (word >> i) & 1 == (idx[g * N + tok, j] >> p) & 1
        noff = (g * nb + blk) * bb + bits * d * 16 + t * 8
        assert np.frombuffer(bytes(buf[noff:noff + 8]), "<f4").tolist() == [n[g * N + tok], 0.0]
    # the same codes as the token-major MSE layout
    m = o.unpack(o.pack(idx, None, n, None, d, bits, "mse", G, N), d, bits, "mse", G, N)
    assert np.array_equal(m["idx"], u["idx"])


def _attention_case(N, seed, d=16, H=3):
    rng = _rng(seed)
    Pi_k, Pi_v = _haar(d, seed + 1), _haar(d, seed + 2)
    S = rng.standard_normal((d, d))
    c_k, c_v = o.codebook_f32(4, d), o.codebook_f32(8, d)
    x = rng.standard_normal((N, d))
    v = rng.standard_normal((N, d))
    q = rng.standard_normal((H, d))
    ke = o.encode_prod(x, Pi_k, S, c_k)
    ve = o.encode_mse(v, Pi_v, c_v)
    kf = (ke["idx"], ke["z"], ke["n"], ke["rho"], Pi_k, S, c_k)
    return q, kf, ve, Pi_v, c_v


def test_attention_two_tokens_is_the_logistic_weighting():
    q, kf, ve, Pi_v, c_v = _attention_case(2, 51)
    scale = 0.3
    out = o.attend(q, *kf, ve["idx"], ve["n"], Pi_v, c_v, scale)
    l = o.score_prod(q, *kf)
    vh = o.mse_reconstruct(ve["idx"], ve["n"], Pi_v, c_v)
    p1 = 1.0 / (1.0 + np.exp(-scale * (l[:, 1] - l[:, 0])))
    want = (1 - p1)[:, None] * vh[0] + p1[:, None] * vh[1]
    assert np.max(np.abs(out - want)) <= 1e-12 * np.max(np.abs(want))


def test_attention_invariants():
    q, kf, ve, Pi_v, c_v = _attention_case(40, 52)
    vh = o.mse_reconstruct(ve["idx"], ve["n"], Pi_v, c_v)
    # scale 0: the plain mean of the reconstructed values, for every head
    out0 = o.attend(q, *kf, ve["idx"], ve["n"], Pi_v, c_v, 0.0)
    assert np.allclose(out0, vh.mean(axis=0)[None, :], atol=1e-12)
    # every value equal: the output is that value whatever the logits
    same_idx = np.repeat(ve["idx"][:1], 40, axis=0)
    same_n = np.repeat(ve["n"][:1], 40)
    outs = o.attend(q, *kf, same_idx, same_n, Pi_v, c_v, 0.7)
    assert np.allclose(outs, o.mse_reconstruct(same_idx[:1], same_n[:1], Pi_v, c_v), atol=1e-12)
    # a large scale selects the value of each head's largest logit
    l = o.score_prod(q, *kf)
    outb = o.attend(q, *kf, ve["idx"], ve["n"], Pi_v, c_v, 1e4)
    assert np.allclose(outb, vh[np.argmax(l, axis=1)], atol=1e-9)
    # permuting the tokens (keys and values together) changes nothing
    perm = _rng(53).permutation(40)
    kp = (kf[0][perm], kf[1][perm], kf[2][perm], kf[3][perm]) + kf[4:]
    outp = o.attend(q, *kp, ve["idx"][perm], ve["n"][perm], Pi_v, c_v, 0.7)
    assert np.allclose(outp, o.attend(q, *kf, ve["idx"], ve["n"], Pi_v, c_v, 0.7), atol=1e-12)
    # the weights are a softmax over tokens (rows sum to one): a value of zero
    # norm at every token but one gives p_t v_t at that token
    n1 = np.zeros(40)
    n1[7] = ve["n"][7]
    out1 = o.attend(q, *kf, ve["idx"], n1, Pi_v, c_v, 0.7)
    z = 0.7 * l
    p7 = np.exp(z[:, 7] - z.max(axis=1)) / np.exp(z - z.max(axis=1, keepdims=True)).sum(axis=1)
    assert np.allclose(out1, p7[:, None] * vh[7][None, :], atol=1e-12)


def test_attend_packed_matches_per_group_attend():
    d, G, N, H = 128, 2, 200, 4
    rng = _rng(54)
    Pi_k, Pi_v = _haar(d, 55).astype(np.float32), _haar(d, 56).astype(np.float32)
    S = rng.standard_normal((d, d)).astype(np.float32)
    c_k, c_v = o.codebook_f32(4, d), o.codebook_f32(8, d)
    x = rng.standard_normal((G, N, d))
    v = rng.standard_normal((G, N, d))
    q = rng.standard_normal((G, H, d))
    kbuf, ke = o.encode_pack(x, Pi_k, S, c_k, 3, "prod", G, N)
    ve = o.encode_mse(v.reshape(G * N, d), Pi_v, c_v)
    vbuf = o.pack_values(ve["idx"], ve["n"].astype(np.float32), d, 3, G, N)
    out = o.attend_packed(q, kbuf, vbuf, Pi_k, S, c_k, 3, Pi_v, c_v, 3, G, N, 1 / math.sqrt(d))
    for g in range(G):
        r = slice(g * N, (g + 1) * N)
        want = o.attend(q[g], ke["idx"][r], ke["z"][r], ke["n"][r].astype(np.float32), ke["rho"][r].astype(np.float32),
                        Pi_k, S, c_k, ve["idx"][r], ve["n"][r].astype(np.float32), Pi_v, c_v, 1 / math.sqrt(d))
        assert np.allclose(out[g], want, rtol=0, atol=1e-12 * np.max(np.abs(want)))


# ---------------------------------------------------------------- fractional bit widths (reading; parity unpinned)

def test_mixed_quantiser_with_one_codebook_is_the_uniform_one():
    d = 64
    rng = _rng(60)
    Pi = _haar(d, 61)
    S = rng.standard_normal((d, d))
    c = o.codebook_f32(4, d)
    x = rng.standard_normal((30, d))
    q = rng.standard_normal((3, d))
    for d_hi in (0, 17, d):
        m = o.encode_prod_mixed(x, Pi, S, c, c, d_hi)
        u = o.encode_prod(x, Pi, S, c)
        assert np.array_equal(m["idx"], u["idx"]) and np.array_equal(m["z"], u["z"])
        assert np.allclose(m["rho"], u["rho"], rtol=0, atol=1e-13)
        a = o.score_prod_mixed(q, m["idx"], m["z"], m["n"], m["rho"], Pi, S, c, c, d_hi)
        b = o.score_prod(q, u["idx"], u["z"], u["n"], u["rho"], Pi, S, c)
        assert np.allclose(a, b, rtol=0, atol=1e-12 * np.max(np.abs(b)))


def test_mixed_quantiser_is_nearest_centroid_per_coordinate():
    d = 8
    rng = _rng(62)
    Pi = _haar(d, 63)
    c_hi, c_lo = o.codebook_f32(8, d), o.codebook_f32(4, d)
    x = rng.standard_normal((200, d))
    e = o.encode_mse_mixed(x, Pi, c_hi, c_lo, 4)
    for j in range(d):
        cb = c_hi if j < 4 else c_lo
        want = np.argmin(np.abs(e["y"][:, j, None] - cb.astype(np.float64)[None, :]), axis=1)
        assert np.array_equal(e["idx"][:, j], want)
    assert e["idx"][:, :4].max() <= 7 and e["idx"][:, 4:].max() <= 3


@pytest.mark.parametrize("k_lo", [1, 2, 3])
def test_mixed_distortion_is_the_mean_of_the_two_codebooks(k_lo):
    # rotated coordinates of random unit vectors are ~N(0, 1/d): the distortion
    # of the split quantiser is the mean of the two Lloyd-Max distortions
    # (Max's table values, not the oracle's)
    d, n = 128, 20000
    tab = _golden("lloyd_max_textbook.json")["levels"]
    rng = _rng(64 + k_lo)
    Pi = _haar(d, 70)
    x = rng.standard_normal((n, d))
    x /= np.linalg.norm(x, axis=1, keepdims=True)
    c_hi, c_lo = o.codebook_f32(2 << k_lo, d), o.codebook_f32(1 << k_lo, d)
    e = o.encode_mse_mixed(x, Pi, c_hi, c_lo, o.mixed_split(d))
    D = np.mean(np.sum((x - o.mse_reconstruct_mixed(e["idx"], e["n"], Pi, c_hi, c_lo, d // 2)) ** 2, axis=1))
    want = 0.5 * (tab[str(2 << k_lo)]["mse"] + tab[str(1 << k_lo)]["mse"])
    assert abs(D - want) <= 0.03 * want


def test_mixed_prod_estimator_is_unbiased():
    d, T = 32, 3000
    rng = _rng(66)
    Pi = _haar(d, 67)
    c_hi, c_lo = o.codebook_f32(4, d), o.codebook_f32(2, d)
    x = rng.standard_normal((1, d))
    q = rng.standard_normal((1, d))
    truth = (q @ x.T).item()
    est = np.empty(T)
    for t in range(T):
        S = _rng(1000 + t).standard_normal((d, d))
        e = o.encode_prod_mixed(x, Pi, S, c_hi, c_lo, d // 2)
        est[t] = o.score_prod_mixed(q, e["idx"], e["z"], e["n"], e["rho"], Pi, S, c_hi, c_lo, d // 2)[0, 0]
    r = e["r"][0]
    var = ((math.pi / 2) * (r @ r).item() * (q @ q.T).item() - (q[0] @ r).item() ** 2) / d
    assert abs(est.mean() - truth) <= 4 * math.sqrt(var / T)
    assert abs(est.var() / var - 1.0) <= 0.1


@pytest.mark.parametrize("k_lo,prod", [(2, True), (1, True), (3, False)])
def test_fractional_layout_roundtrip_and_bit_addresses(k_lo, prod):
    G, N, d = 2, 300, 256
    rng = _rng(68)
    d_hi = o.mixed_split(d)
    idx = rng.integers(0, 1 << k_lo, size=(G * N, d))
    idx[:, :d_hi] = rng.integers(0, 2 << k_lo, size=(G * N, d_hi))
    z = rng.integers(0, 2, size=(G * N, d)).astype(bool)
    n = rng.random(G * N).astype(np.float32)
    rho = rng.random(G * N).astype(np.float32)
    buf = o.pack_mixed(idx, z, n, rho, d, k_lo, prod, G, N)
    nb = 3
    bb = o.frac_block_bytes(d, k_lo, prod)
    assert buf.size == G * nb * bb
    u = o.unpack_mixed(buf, d, k_lo, prod, G, N)
    assert np.array_equal(u["idx"], idx) and np.array_equal(u["n"], n.astype(np.float64))
    if prod:
        assert np.array_equal(u["z"], z) and np.array_equal(u["rho"], rho.astype(np.float64))
    # the extra plane: bit k_lo of coordinate j < d/2 of token t is bit i of
    # word w of the 8 bytes at ((c' 128 + t) 8) after the full planes, j = 64 c' + 32 w + i
    C = d // 128
    for (g, tok, j) in [(0, 0, 0), (1, 299, d_hi - 1), (0, 130, 70), (1, 257, 33)]:
        blk, t = divmod(tok, 128)
        c2, rem = divmod(j, 64)
        w, i = divmod(rem, 32)
        off = (g * nb + blk) * bb + k_lo * C * 128 * 16 + (c2 * 128 + t) * 8 + 4 * w
        word = int.from_bytes(bytes(buf[off:off + 4]), "little")
        assert (word >> i) & 1 == (idx[g * N + tok, j] >> k_lo) & 1
