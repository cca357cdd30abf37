"""GPU parity at the workloads' full sizes, in the launch configuration bench.py
times: every key of the workload is encoded and every (group, head, token)
logit is scored in one call each, then sampled keys are checked against the
oracle one by one.

Samples per workload: the first, middle and last group and up to five more
seeded groups; in each, the first and last 64 tokens and seeded random tokens,
enough that the pooled sample holds at least 10^6 compared values (code
coordinates, plus sign bits in Prod).  For those keys the codes, sign bits and
norms must agree with the oracle's encoding of the same key bytes
(compare_fields), with the band-exempt mismatch rate asserted on the pooled
sample, and the logits must agree with the oracle's score of the GPU's own
fields (identical packed input) within 1e-4 ||q|| ||x||.

The vector-search workload checks its top-10 per query against the oracle:
the oracle scores all 10^6 packed keys for all 256 queries (in the rotated
frame, ``score_prod_rotated`` / ``score_mse_rotated``: n <Pi q, c[idx]>
+ rho sqrt(pi/2)/m <Sq, 2z-1>, equal to ``score_prod`` up to the fp32
rotation's non-orthogonality, ~1e-7),
and every returned key must score at least the oracle's 10th best minus
1e-4 ||q|| n, with its returned score within 1e-4 ||q|| n of the oracle's.
The long-context workload checks the fp32-key baseline on the sampled keys.
"""
import numpy as np
import pytest
import torch

import tq_synth
import vector_quantization_02_b300 as tq
from oracle import tq_oracle as o

from parity import Inputs, assert_pooled_rate, check_topk_against_oracle, compare_fields, compare_logits

pytestmark = pytest.mark.gpu

MIN_COMPARED = 10 ** 6


def _groups(G: int, seed: int) -> list:
    base = {0, G // 2, G - 1}
    rng = np.random.default_rng(seed)
    extra = rng.choice(G, size=min(G, 5), replace=False)
    return sorted(base | set(int(g) for g in extra))


def _samples(N: int, n_random: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    edge = np.concatenate([np.arange(min(64, N)), np.arange(max(0, N - 64), N)])
    return np.unique(np.concatenate([edge, rng.choice(N, size=min(n_random, N), replace=False)]))


def _group_fields(packed: torch.Tensor, plan, g: int, N: int, d: int, bits: int, mode: str) -> dict:
    per_group = plan.packed_bytes(1, N)
    buf = packed[g * per_group:(g + 1) * per_group].cpu().numpy()
    return o.unpack(buf, d, bits, mode, 1, N)


def _exact_topk(L: np.ndarray, k: int):
    """Top-k of each row by descending value, ties to the lower index."""
    out_s = np.empty((L.shape[0], k), dtype=L.dtype)
    out_i = np.empty((L.shape[0], k), dtype=np.int64)
    for r in range(L.shape[0]):
        row = L[r]
        cand = np.argpartition(-row, k - 1)[:k]
        thr = row[cand].min()
        cand = np.nonzero(row >= thr)[0]
        order = np.lexsort((cand, -row[cand]))[:k]
        out_i[r] = cand[order]
        out_s[r] = row[cand[order]]
    return out_s, out_i


def _oracle_topk_over_all_keys(inp: Inputs, packed: torch.Tensor, q: np.ndarray, N: int, k: int,
                               top_i: np.ndarray, chunk_blocks: int = 128):
    """The oracle's k-th best score per query over every packed key (one
    group), and its scores and norms at the GPU's returned indices."""
    H = q.shape[0]
    bb = o.block_bytes(inp.d, inp.bits, inp.mode)
    nb = -(-N // 128)
    best = np.full((H, k), -np.inf)
    at = np.full(top_i.shape, np.nan)
    n_at = np.full(top_i.shape, np.nan)
    for b0 in range(0, nb, chunk_blocks):
        b1 = min(nb, b0 + chunk_blocks)
        buf = packed[b0 * bb:b1 * bb].cpu().numpy()
        u = o.unpack_blocks(buf, inp.d, inp.bits, inp.mode, b1 - b0)
        t0, t1 = b0 * 128, min(N, b1 * 128)
        r = slice(0, t1 - t0)
        if inp.mode == "prod":
            s = o.score_prod_rotated(q, u["idx"][r], u["z"][r], u["n"][r], u["rho"][r], inp.Pi_o, inp.S_o, inp.c_o)
        else:
            s = o.score_mse_rotated(q, u["idx"][r], u["n"][r], inp.Pi_o, inp.c_o)
        kk = min(k, s.shape[1])
        part = np.partition(s, s.shape[1] - kk, axis=1)[:, s.shape[1] - kk:]
        best = np.sort(np.concatenate([best, part], axis=1), axis=1)[:, -k:]
        inside = (top_i >= t0) & (top_i < t1)
        rows, cols = np.nonzero(inside)
        at[rows, cols] = s[rows, top_i[rows, cols] - t0]
        n_at[rows, cols] = u["n"][top_i[rows, cols] - t0]
    assert not np.isnan(at).any()
    return best[:, 0], at, n_at


CASES = [("single_head_3bit", 3, "prod"), ("qwen25_3b_decode", 3, "prod"), ("llama31_8b_prefill", 2, "prod"),
         ("llama31_8b_prefill", 3, "prod"), ("llama31_8b_prefill", 4, "prod"), ("long_context_131k", 4, "prod"),
         ("vector_search_1m", 4, "prod"),
         # the MSE codec on the same shapes (many tiles per CTA: d = 128 has a
         # single K slice per tile, d = 1536 a 16-level codebook)
         ("qwen25_3b_decode", 3, "mse"), ("vector_search_1m", 4, "mse")]


@pytest.mark.parametrize("name,bits,mode", CASES)
def test_full_size_sampled(cuda, name, bits, mode):
    w = tq_synth.WORKLOADS[name]
    G, N, H, d = w.G, w.N, w.H, w.d
    inp = Inputs(d, bits, mode, w.seeds["rotation"], w.seeds["projection"])
    plan = inp.plan()
    keys = tq_synth.keys(w, device=cuda)
    q = tq_synth.queries(w, device=cuda)
    # the bench's calls: one encode of every key, one score of every query
    packed = tq.tq_encode(plan, keys)
    if w.top_k:
        logits, top_s, top_i = tq.tq_score(plan, q, packed, N, top_k=w.top_k)
    else:
        logits = tq.tq_score(plan, q, packed, N)
    torch.cuda.synchronize()
    assert plan.status() == 0

    groups = _groups(G, seed=bits)
    per_key = d * (2 if mode == "prod" else 1)
    n_random = -(-11 * MIN_COMPARED // (10 * per_key * len(groups)))
    pool = {}
    for g in groups:
        toks = _samples(N, n_random, seed=1000 * g + bits)
        x = keys[g, torch.from_numpy(toks).to(cuda)].double().cpu().numpy()
        e = o.encode_prod(x, inp.Pi_o, inp.S_o, inp.c_o) if mode == "prod" else o.encode_mse(x, inp.Pi_o, inp.c_o)
        f = _group_fields(packed, plan, g, N, d, bits, mode)
        got = {k: v[toks] for k, v in f.items()}
        compare_fields(inp, got, e, x, pool=pool)
        # logits from identical packed input: the oracle scores the GPU's fields
        qg = q[g].cpu()
        if mode == "prod":
            want = o.score_prod(qg.numpy(), got["idx"], got["z"], got["n"], got["rho"], inp.Pi_o, inp.S_o, inp.c_o)
        else:
            want = o.score_mse(qg.numpy(), got["idx"], got["n"], inp.Pi_o, inp.c_o)
        gl = logits[g][:, torch.from_numpy(toks).to(cuda)].cpu().numpy()
        compare_logits(gl[None], want[None], qg[None], got["n"].astype(np.float64)[None])
        if name == "long_context_131k":
            base = tq.tq_score_fp32(q[g:g + 1], keys[g:g + 1].float())
            bw = o.score_fp32(qg[None].numpy(), x[None])
            bg = base[0][:, torch.from_numpy(toks).to(cuda)].cpu().numpy()
            bound = 1e-5 * np.linalg.norm(qg.double().numpy(), axis=-1)[:, None] * np.linalg.norm(x, axis=-1)[None]
            assert np.all(np.abs(bg - bw[0]) <= bound)
    assert_pooled_rate(pool, MIN_COMPARED)
    if w.top_k:
        ts, ti = top_s[0].cpu().numpy(), top_i[0].cpu().numpy()
        # the selection is exact on the GPU's own logits
        want_s, want_i = _exact_topk(logits[0].cpu().numpy(), w.top_k)
        assert np.array_equal(ti, want_i) and np.array_equal(ts, want_s)
        # and valid against the oracle's scores of every key
        qh = q[0].cpu().double().numpy()
        kth, at, n_at = _oracle_topk_over_all_keys(inp, packed, qh, N, w.top_k, ti)
        check_topk_against_oracle(ts, ti, at, kth, np.linalg.norm(qh, axis=-1), n_at)
