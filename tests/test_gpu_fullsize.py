"""GPU parity at the workloads' full sizes, in the launch configuration bench.py
times: every key of the workload is encoded and every (group, head, token)
logit is scored in one call each, then sampled keys are checked against the
oracle one by one.

Samples per workload: the first, middle and last group; in each, the first and
last 64 tokens and 256 seeded random tokens.  For those keys the codes, sign
bits and norms must agree with the oracle's encoding of the same key bytes
(compare_fields), and the logits must agree with the oracle's score of the
GPU's own fields (identical packed input) within 1e-4 ||q|| ||x||.  The
vector-search workload also checks its top-10 per query against the exact
top-10 of the GPU's logits (descending, ties to the lower index), and the
long-context workload the fp32-key baseline on the sampled keys.
"""
import numpy as np
import pytest
import torch

import tq_synth
import vector_quantization_02_b300 as tq
from oracle import tq_oracle as o

from parity import Inputs, compare_fields, compare_logits

pytestmark = pytest.mark.gpu


def _samples(N: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    edge = np.concatenate([np.arange(min(64, N)), np.arange(max(0, N - 64), N)])
    return np.unique(np.concatenate([edge, rng.choice(N, size=min(256, N), replace=False)]))


def _groups(G: int) -> list:
    return sorted({0, G // 2, G - 1})


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

    total_coords = 0
    for g in _groups(G):
        toks = _samples(N, seed=1000 * g + bits)
        x = keys[g, torch.from_numpy(toks).to(cuda)].double().cpu().numpy()
        e = o.encode_prod(x, inp.Pi_o, inp.S_o, inp.c_o) if mode == "prod" else o.encode_mse(x, inp.Pi_o, inp.c_o)
        f = _group_fields(packed, plan, g, N, d, bits, mode)
        got = {k: v[toks] for k, v in f.items()}
        compare_fields(inp, got, e, x)
        total_coords += x.size
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
    assert total_coords > 0
    if w.top_k:
        L = logits[0].cpu().numpy()
        want_s, want_i = _exact_topk(L, w.top_k)
        assert np.array_equal(top_i[0].cpu().numpy(), want_i)
        assert np.array_equal(top_s[0].cpu().numpy(), want_s)
