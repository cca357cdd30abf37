"""Comparison rules between the CUDA path and the oracle (shared by the GPU tests).

Tolerances (from the target the build is held to):
* codes and sign bits are bit-identical, except coordinates within 1e-5 (unit
  scale) of a decision boundary, or signs with |p_i| <= 1e-5 ||x||; the
  mismatch rate over all coordinates is <= 1e-5 and no mismatch lies outside
  those bands;
* norms: |dn| <= 1e-6 n; |drho| <= 1e-5 n (rho is continuous across a code
  flip at a boundary);
* logits from identical packed input: |d logit| <= 1e-4 ||q|| n.
The oracle decides codes and signs in fp64, the kernels in fp32 (exact fp32
products, fp32 accumulation); the bands absorb the difference.
"""
from __future__ import annotations

import numpy as np
import torch

import tq_synth
import vector_quantization_02_b300 as tq
from oracle import tq_oracle as o


class Inputs:
    """Plan inputs for both sides from one set of seeded draws.

    The oracle builds the rotation (LAPACK QR of the seeded Gaussian) and the
    fp32 codebook; the GPU plan is built from exactly those fp32 values, so
    both sides compute on identical Pi, S and centroids.  The library's own
    host helpers (tq_haar_rotation, tq_lloyd_max_codebook) are pinned against
    the oracle separately, on the CPU."""

    def __init__(self, d, bits, mode, rot_seed, proj_seed):
        self.d, self.bits, self.mode = d, bits, mode
        self.k = bits - 1 if mode == "prod" else bits
        self.G_rot = tq_synth.rotation_gaussian(d, rot_seed)
        self.S = tq_synth.projection(d, proj_seed)
        self.Pi_o = np.ascontiguousarray(o.haar_rotation(self.G_rot.numpy()).astype(np.float32))
        self.c_o = o.codebook_f32(1 << self.k, d)
        self.S_o = self.S.numpy()

    def plan(self):
        return tq.Plan(self.d, self.bits, torch.from_numpy(self.Pi_o), self.S if self.mode == "prod" else None,
                       torch.from_numpy(self.c_o.copy()), mode=self.mode)


class HadamardInputs(Inputs):
    """Plan inputs with the randomised Walsh-Hadamard rotation: the oracle's
    Pi = H diag(signs) / sqrt(d) in fp32 (each entry +-fl32(1/sqrt(d)), the
    value the library computes from the same signs), the GPU plan from the
    signs."""

    def __init__(self, d, bits, mode, sign_seed, proj_seed):
        self.d, self.bits, self.mode = d, bits, mode
        self.k = bits - 1 if mode == "prod" else bits
        self.signs = tq_synth.hadamard_signs(d, sign_seed)
        self.S = tq_synth.projection(d, proj_seed)
        self.Pi_o = np.ascontiguousarray(o.hadamard_rotation(self.signs.double().numpy()).astype(np.float32))
        self.c_o = o.codebook_f32(1 << self.k, d)
        self.S_o = self.S.numpy()

    def plan(self):
        return tq.Plan.hadamard(self.d, self.bits, self.signs, self.S if self.mode == "prod" else None,
                                torch.from_numpy(self.c_o.copy()), mode=self.mode)


def oracle_encode(inp: Inputs, keys: torch.Tensor):
    """Oracle encode of keys [G][N][d] (any dtype) -> (bytes, encode dict)."""
    G, N, d = keys.shape
    return o.encode_pack(keys.detach().cpu().double().numpy(), inp.Pi_o, inp.S_o, inp.c_o, inp.bits, inp.mode, G, N)


def compare_fields(inp: Inputs, got: dict, e: dict, x: np.ndarray, pool: dict | None = None) -> dict:
    """Assert the GPU's per-key fields (idx, z, n, rho of keys ``x`` [n][d],
    fp64) agree with the oracle's encoding ``e`` of the same keys.

    A coordinate within 1e-5 of a boundary may take either neighbouring code;
    the key's residual, rho and signs then follow the code taken, so such a key
    is compared against the oracle's own encoding with that boundary resolved
    the other way (``qjl_stage`` on the alternative codes).

    The mismatch rate is over every compared value (code coordinates, and sign
    bits in Prod).  With ``pool`` given, the counts are added to it and the
    rate is asserted later on the pooled total (``assert_pooled_rate``);
    otherwise it is asserted here."""
    total = x.size * (2 if inp.mode == "prod" else 1)
    code_bad = got["idx"] != e["idx"]
    assert not np.any(code_bad & ~e["code_exempt"]), "code mismatch outside the boundary band"
    # a flipped code must be the neighbour across the near boundary
    assert np.all(np.abs(got["idx"][code_bad] - e["idx"][code_bad]) == 1), "flip to a non-neighbour code"
    stats = dict(code_mismatch=int(code_bad.sum()), coords=total)
    mism = int(code_bad.sum())
    n = e["n"]
    assert np.all(np.abs(got["n"] - n) <= 1e-6 * n + 1e-30), "norm mismatch"
    if inp.mode == "prod":
        z_ref, rho_ref, band = e["z"].copy(), e["rho"].copy(), e["sign_exempt"].copy()
        flipped = np.where(code_bad.any(axis=1))[0]
        if flipped.size:
            alt_idx = e["idx"][flipped].copy()
            alt_idx[code_bad[flipped]] = got["idx"][flipped][code_bad[flipped]]
            alt = o.qjl_stage(x[flipped], alt_idx, n[flipped], inp.Pi_o, inp.S_o, inp.c_o)
            z_ref[flipped], rho_ref[flipped], band[flipped] = alt["z"], alt["rho"], alt["sign_exempt"]
        sign_bad = got["z"] != z_ref
        bad_rows = np.where((sign_bad & ~band).any(axis=1))[0]
        assert bad_rows.size == 0, (f"sign mismatch outside the zero band at keys {bad_rows[:8]} "
                                    f"({int((sign_bad & ~band).sum())} signs)")
        mism += int(sign_bad.sum())
        stats["sign_mismatch"] = int(sign_bad.sum())
        stats["boundary_flipped_keys"] = int(flipped.size)
        assert np.all(np.abs(got["rho"] - rho_ref.astype(np.float32)) <= 1e-5 * n + 1e-30), "residual norm mismatch"
    else:
        assert np.all(got["rho"] == 0)
    stats["mismatches"] = mism
    stats["compared"] = total
    if pool is not None:
        pool["mismatches"] = pool.get("mismatches", 0) + mism
        pool["compared"] = pool.get("compared", 0) + total
        return stats
    # the rate can only be resolved on large samples: below 10^6 compared
    # values a couple of band-exempt flips are allowed, above it the rate must
    # be <= 1e-5
    assert mism <= max(1e-5 * total, 2 if total < 10 ** 6 else 0), \
        f"mismatch rate {mism / total:.2e} above 1e-5 ({mism} of {total})"
    return stats


def assert_pooled_rate(pool: dict, min_compared: int = 10 ** 6) -> float:
    """The band-exempt mismatch rate over a pooled sample of at least
    ``min_compared`` values is at most 1e-5."""
    total, mism = pool["compared"], pool["mismatches"]
    assert total >= min_compared, f"pooled sample too small to resolve a 1e-5 rate ({total})"
    assert mism <= 1e-5 * total, f"pooled mismatch rate {mism / total:.2e} above 1e-5 ({mism} of {total})"
    return mism / total


def compare_encode(inp: Inputs, gpu_bytes: np.ndarray, keys: torch.Tensor, check_bytes=True) -> dict:
    """Assert the GPU's packed bytes agree with the oracle's encode of ``keys``
    (all keys; see compare_fields for the rules)."""
    G, N, d = keys.shape
    want_bytes, e = oracle_encode(inp, keys)
    got = o.unpack(gpu_bytes, d, inp.bits, inp.mode, G, N)
    x = keys.detach().cpu().double().numpy().reshape(G * N, d)
    stats = compare_fields(inp, got, e, x)
    if check_bytes and stats["mismatches"] == 0:
        # every code and sign bit agrees: the plane bytes, including the zero
        # padding of the last block, are identical
        nb = -(-N // 128)
        bb = o.block_bytes(d, inp.bits, inp.mode)
        plane = bb - 128 * 8
        gb = gpu_bytes.reshape(G * nb, bb)
        wb = want_bytes.reshape(G * nb, bb)
        assert np.array_equal(gb[:, :plane], wb[:, :plane])
        pad = np.arange(nb * 128) >= N
        norms_g = gb[:, plane:].reshape(G, nb * 128, 8)
        assert not np.any(norms_g[:, pad]), "padded tokens' norms are not zero"
    return stats


def qnorms(q: torch.Tensor) -> np.ndarray:
    return torch.linalg.vector_norm(q.double(), dim=-1).cpu().numpy()          # [G][H]


def compare_logits(got: np.ndarray, want: np.ndarray, q: torch.Tensor, n: np.ndarray, tol=1e-4) -> float:
    """|got - want| <= tol ||q|| n elementwise; got/want [G][H][N], n [G][N]."""
    bound = tol * qnorms(q)[:, :, None] * n[:, None, :]
    err = np.abs(got.astype(np.float64) - want)
    assert np.all(err <= bound + 1e-30), f"max err/bound {np.max(err / (bound + 1e-30)):.3g}"
    return float(np.max(err / (bound + 1e-30)))


def oracle_logits_of_packed(inp: Inputs, packed: np.ndarray, q: np.ndarray, G: int, N: int) -> np.ndarray:
    """The oracle's logits [G][H][N] (fp64) for packed bytes (identical packed
    input: whatever the bytes hold is scored), through ``score_prod`` /
    ``score_mse`` on the fields ``unpack_blocks`` reads."""
    nb = -(-N // 128)
    u = o.unpack_blocks(packed, inp.d, inp.bits, inp.mode, G * nb)
    out = np.empty((G, q.shape[1], N))
    for g in range(G):
        r = slice(g * nb * 128, g * nb * 128 + N)
        if inp.mode == "prod":
            out[g] = o.score_prod(q[g], u["idx"][r], u["z"][r], u["n"][r], u["rho"][r], inp.Pi_o, inp.S_o, inp.c_o)
        else:
            out[g] = o.score_mse(q[g], u["idx"][r], u["n"][r], inp.Pi_o, inp.c_o)
    return out


def check_topk_against_oracle(top_s: np.ndarray, top_i: np.ndarray, oracle_at: np.ndarray, kth_best: np.ndarray,
                              qn: np.ndarray, n_at: np.ndarray, tol=1e-4):
    """Top-k validity: every returned key's oracle score is at least the
    oracle's k-th best score minus tol ||q|| n, and the returned score is the
    oracle's within tol ||q|| n.  Rows are (group, head); ``oracle_at`` holds
    the oracle's scores at the returned indices, ``n_at`` those keys' norms."""
    bound = tol * qn[:, None] * n_at
    assert np.all(oracle_at >= kth_best[:, None] - bound), "a returned key is not among the oracle's top k"
    assert np.all(np.abs(top_s.astype(np.float64) - oracle_at) <= bound), "returned scores disagree with the oracle"
    assert np.all(np.diff(top_s, axis=-1) <= 0), "top-k scores not in descending order"
    for r in range(top_i.shape[0]):
        assert np.unique(top_i[r]).size == top_i.shape[1], "repeated index in a top-k row"
