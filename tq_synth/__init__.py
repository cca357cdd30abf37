"""Seeded synthetic inputs for the TurboQuantProd encode/score path.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no rotation, no codebook, no quantisation, no
projection).  Both the CUDA path (through the package binding) and the CPU
oracle consume what it produces, so it is the only code the two share.

Every tensor is drawn from torch's counter-based Philox generator with an
explicit seed: on the CPU for the small shapes the oracle checks in full, on
the GPU for the full-size workloads (whose sampled rows are copied back to the
host for the oracle).  The two devices give different numbers for one seed;
each workload states which device draws it.

Workloads (keys are ``[G][N][d]`` row-major, queries ``[G][H][d]`` fp32):

* ``single_head_3bit``  -- the synthetic example of the turboquant-pytorch
  introduction ("TurboQuant 핵심 알고리즘 사용 예시"): 4,096 fp32 N(0,1) keys,
  d=128, 16 N(0,1) queries, 3 bits.
* ``qwen25_3b_decode`` -- shaped like Qwen2.5-3B-Instruct (36 layers x 2 KV
  heads, 16 query heads, head_dim 128, 8K context; the model the same
  introduction validates on): fp16 keys N(0,1) x a per-channel lognormal(0,0.5)
  scale per (layer, KV head) with 4 outlier channels x8; 3 bits.
* ``llama31_8b_prefill`` -- shaped like Llama-3.1-8B-Instruct (32 layers x 8 KV
  heads, 32 query heads, context 32,768, batch 16): bf16 keys from the same
  generator, scales per (layer, KV head) shared over the batch; 2/3/4 bits.
* ``long_context_131k`` -- one layer, 8 KV heads x 32 query heads, 131,072 bf16
  keys per head, batch 4; 4 bits.
* ``vector_search_1m`` -- 1,000,000 fp32 N(0,1) vectors, d=1,536, then scaled
  to unit length; 256 N(0,1) queries; 4 bits; top-10 per query.

The random draws the method itself makes -- the Gaussian matrix whose QR
factor is the rotation, and the Gaussian projection S -- are drawn here too
and passed to both sides as inputs.
"""
from __future__ import annotations

import dataclasses

import torch

__all__ = ["Workload", "WORKLOADS", "gaussian", "rotation_gaussian", "hadamard_signs", "projection",
           "channel_scales", "keys", "key_chunk", "queries", "small_case"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    G: int            # KV groups (batch x layers x KV heads)
    N: int            # tokens (keys) per group
    H: int            # query heads per KV group
    d: int            # head dimension
    bits: tuple       # total bits per coordinate (Lloyd-Max bits + 1 QJL bit)
    key_dtype: torch.dtype
    layers: int       # layers represented in G (scale sharing)
    kv_heads: int     # KV heads per layer
    batch: int
    seeds: dict       # rotation, projection, keys, scales, queries
    unit_keys: bool = False
    outliers: bool = True
    top_k: int = 0

    @property
    def n_keys(self) -> int:
        return self.G * self.N


WORKLOADS = {
    "single_head_3bit": Workload(
        "single_head_3bit", G=1, N=4096, H=16, d=128, bits=(3,), key_dtype=torch.float32,
        layers=1, kv_heads=1, batch=1, outliers=False,
        seeds=dict(rotation=101, projection=102, keys=103, scales=0, queries=104)),
    "qwen25_3b_decode": Workload(
        "qwen25_3b_decode", G=72, N=8192, H=8, d=128, bits=(3,), key_dtype=torch.float16,
        layers=36, kv_heads=2, batch=1,
        seeds=dict(rotation=201, projection=202, keys=203, scales=204, queries=205)),
    "llama31_8b_prefill": Workload(
        "llama31_8b_prefill", G=4096, N=32768, H=4, d=128, bits=(2, 3, 4), key_dtype=torch.bfloat16,
        layers=32, kv_heads=8, batch=16,
        seeds=dict(rotation=301, projection=302, keys=303, scales=304, queries=305)),
    "long_context_131k": Workload(
        "long_context_131k", G=32, N=131072, H=4, d=128, bits=(4,), key_dtype=torch.bfloat16,
        layers=1, kv_heads=8, batch=4,
        seeds=dict(rotation=401, projection=402, keys=403, scales=404, queries=405)),
    "vector_search_1m": Workload(
        "vector_search_1m", G=1, N=1_000_000, H=256, d=1536, bits=(4,), key_dtype=torch.float32,
        layers=1, kv_heads=1, batch=1, unit_keys=True, outliers=False, top_k=10,
        seeds=dict(rotation=501, projection=502, keys=503, scales=0, queries=504)),
}


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def gaussian(shape, seed: int, dtype=torch.float64, device="cpu") -> torch.Tensor:
    """i.i.d. N(0,1) samples, seeded."""
    return torch.randn(tuple(shape), generator=_gen(seed, device), dtype=dtype, device=device)


def rotation_gaussian(d: int, seed: int) -> torch.Tensor:
    """The d x d fp64 Gaussian matrix whose (sign-fixed) QR factor is the rotation."""
    return gaussian((d, d), seed, torch.float64)


def hadamard_signs(d: int, seed: int) -> torch.Tensor:
    """d random signs (+1 or -1, fp32) for a randomised Walsh-Hadamard
    rotation: the signs of seeded N(0,1) draws (a draw of exactly 0 counts as
    +1)."""
    g = gaussian((d,), seed, torch.float64)
    return torch.where(g >= 0, 1.0, -1.0).to(torch.float32)


def projection(d: int, seed: int, m: int | None = None) -> torch.Tensor:
    """The m x d Gaussian projection S of the QJL stage, fp32 (m = d by default)."""
    m = d if m is None else m
    return gaussian((m, d), seed, torch.float64).to(torch.float32)


def channel_scales(w: Workload) -> torch.Tensor:
    """Per-(layer, KV head) channel scales, shape [layers * kv_heads, d], fp32.

    s_c = exp(0.5 * g_c) with g_c ~ N(0,1) (lognormal with sigma 0.5); four
    distinct channels per (layer, head), picked by a seeded permutation, are
    multiplied by 8.
    """
    n_lh = w.layers * w.kv_heads
    if not w.outliers:
        return torch.ones(n_lh, w.d, dtype=torch.float32)
    g = gaussian((n_lh, w.d), w.seeds["scales"], torch.float64)
    s = torch.exp(0.5 * g)
    gen = _gen(w.seeds["scales"] + 7919)
    for i in range(n_lh):
        perm = torch.randperm(w.d, generator=gen)[:4]
        s[i, perm] *= 8.0
    return s.to(torch.float32)


def _group_scale_index(w: Workload, G: int) -> torch.Tensor:
    """(layer, KV head) index of every group; groups are ordered batch-major,
    then layer, then KV head, and scales are shared over the batch."""
    g = torch.arange(G)
    return g % (w.layers * w.kv_heads)


KEY_CHUNK_GROUPS = 64   # keys are drawn 64 groups at a time (bounded temporaries)


def keys(w: Workload, G: int | None = None, N: int | None = None, device="cpu",
         seed_offset: int = 0) -> torch.Tensor:
    """Keys [G][N][d] in the workload's dtype, drawn on ``device``.

    Groups [64c, 64c + 64) are drawn with seed 1,000,003 * keys_seed + c
    (+ seed_offset), so that no temporary exceeds 64 groups.
    """
    G = w.G if G is None else G
    N = w.N if N is None else N
    out = torch.empty((G, N, w.d), dtype=w.key_dtype, device=device)
    for c0 in range(0, G, KEY_CHUNK_GROUPS):
        c1 = min(G, c0 + KEY_CHUNK_GROUPS)
        out[c0:c1] = key_chunk(w, c0 // KEY_CHUNK_GROUPS, G, N, device, seed_offset)
    return out


def key_chunk(w: Workload, chunk: int, G: int | None = None, N: int | None = None, device="cpu",
              seed_offset: int = 0) -> torch.Tensor:
    """Groups [64 chunk, 64 chunk + 64) of ``keys(w, G, N)``, drawn alone (the
    same values), so that a large workload can be produced chunk by chunk."""
    G = w.G if G is None else G
    N = w.N if N is None else N
    c0 = chunk * KEY_CHUNK_GROUPS
    c1 = min(G, c0 + KEY_CHUNK_GROUPS)
    seed = 1_000_003 * w.seeds["keys"] + chunk + seed_offset
    z = gaussian((c1 - c0, N, w.d), seed, torch.float32, device)
    if w.unit_keys:
        z /= torch.linalg.vector_norm(z, dim=-1, keepdim=True)
    elif w.outliers:
        sc = channel_scales(w).to(device)[_group_scale_index(w, G)[c0:c1].to(device)]
        z *= sc[:, None, :]
    return z.to(w.key_dtype)


def queries(w: Workload, G: int | None = None, H: int | None = None, device="cpu",
            seed_offset: int = 0) -> torch.Tensor:
    """Queries [G][H][d], fp32 N(0,1)."""
    G = w.G if G is None else G
    H = w.H if H is None else H
    return gaussian((G, H, w.d), w.seeds["queries"] + seed_offset, torch.float32, device)


def small_case(d=128, G=2, N=300, H=4, dtype=torch.float32, seed=7, outliers=False):
    """A small workload for tests: several token blocks and a ragged tail."""
    return Workload(f"small_d{d}", G=G, N=N, H=H, d=d, bits=(2, 3, 4), key_dtype=dtype,
                    layers=G, kv_heads=1, batch=1, outliers=outliers,
                    seeds=dict(rotation=seed, projection=seed + 1, keys=seed + 2,
                               scales=seed + 3, queries=seed + 4))
