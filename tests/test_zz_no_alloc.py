"""tq_score_noalloc: scoring for callers that may not allocate device memory.

Some callers cannot call cudaMalloc -- a plugin inside a runtime that owns all
device memory through its own pool, or a latency-critical loop that cannot
afford an allocation's device synchronisation.  For them the library offers a
variant of tq_score that takes its scratch from a fixed array compiled into
the library.  This file checks, through the C ABI, that two calls in a row
give the same logits and top-k as tq_score (the entry point that takes a
caller-allocated workspace), and that oversized requests are refused.  It is
named so that pytest collects it last; it passes run alone in a fresh
process and after the other tests.
"""
import gc

import numpy as np
import pytest
import torch

import tq_synth
import vector_quantization_02_b300 as tq
from parity import Inputs, compare_logits

pytestmark = pytest.mark.gpu


def test_noalloc_score_matches_tq_score_twice(cuda):
    d, G, N, H, bits = 128, 3, 1000, 8, 3
    w = tq_synth.small_case(d=d, G=G, N=N, H=H, dtype=torch.float16, seed=61, outliers=True)
    inp = Inputs(d, bits, "prod", w.seeds["rotation"], w.seeds["projection"])
    plan = inp.plan()
    keys = tq_synth.keys(w).to(cuda)
    packed = tq.tq_encode(plan, keys)
    n = torch.linalg.vector_norm(keys.double(), dim=-1).cpu().numpy()
    for call, top_k in enumerate((0, 10)):
        q = tq_synth.queries(w, seed_offset=call).to(cuda)
        want = tq.tq_score(plan, q, packed, N, top_k=top_k)
        got = tq.tq_score_noalloc(plan, q, packed, N, top_k=top_k)
        torch.cuda.synchronize()
        if top_k:
            want, want_s, want_i = want
            got, got_s, got_i = got
            assert torch.equal(got_i, want_i)
            compare_logits(got_s.cpu().numpy(), want_s.cpu().double().numpy(), q.cpu(),
                           np.take_along_axis(n[:, None, :].repeat(H, 1), want_i.cpu().numpy(), -1)[:, 0, :])
        compare_logits(got.cpu().numpy(), want.cpu().double().numpy(), q.cpu(), n)


def test_noalloc_rejects_requests_beyond_its_scratch(cuda):
    d, bits = 128, 3
    inp = Inputs(d, bits, "prod", 5, 6)
    plan = inp.plan()
    G, H, N = 4096, 16, 1        # rotated + projected queries alone need 64 MiB
    assert tq.score_workspace_bytes(plan, G, H, N) > tq.TQ_SCORE_NOALLOC_MAX_BYTES
    q = torch.zeros(G, H, d, device=cuda)
    packed = torch.zeros(plan.packed_bytes(G, N), dtype=torch.uint8, device=cuda)
    with pytest.raises(tq.TQError) as ei:
        tq.tq_score_noalloc(plan, q, packed, N)
    assert ei.value.status == -3


def test_noalloc_wide_score_with_top_k_twice(cuda):
    # the tensor path for any d (here d = 1536, 40 heads, top-10) keeps a
    # different scratch layout (fp32 Pi q and S q, split operands); two calls
    # in a row through the shared array give tq_score's results
    d, G, N, H, bits, k = 1536, 1, 700, 40, 4, 10
    w = tq_synth.small_case(d=d, G=G, N=N, H=H, seed=63)
    inp = Inputs(d, bits, "prod", w.seeds["rotation"], w.seeds["projection"])
    plan = inp.plan()
    assert plan.score_path(H) == "tensor_wide"
    assert tq.score_workspace_bytes(plan, G, H, N, k) <= tq.TQ_SCORE_NOALLOC_MAX_BYTES
    keys = tq_synth.keys(w).to(cuda)
    packed = tq.tq_encode(plan, keys)
    n = torch.linalg.vector_norm(keys.double(), dim=-1).cpu().numpy()
    for call in range(2):
        q = tq_synth.queries(w, seed_offset=call).to(cuda)
        want, want_s, want_i = tq.tq_score(plan, q, packed, N, top_k=k)
        got, got_s, got_i = tq.tq_score_noalloc(plan, q, packed, N, top_k=k)
        torch.cuda.synchronize()
        assert torch.equal(got_i, want_i)
        compare_logits(got_s.cpu().numpy(), want_s.cpu().double().numpy(), q.cpu(),
                       np.take_along_axis(n[:, None, :].repeat(H, 1), want_i.cpu().numpy(), -1)[:, 0, :])
        compare_logits(got.cpu().numpy(), want.cpu().double().numpy(), q.cpu(), n)


def test_noalloc_call_allocates_nothing(cuda):
    # with the outputs passed in, a call (after a first one has loaded the
    # kernels) changes neither torch's allocated bytes nor the device's free memory
    d, G, N, H, bits, k = 128, 2, 3000, 8, 3, 10
    w = tq_synth.small_case(d=d, G=G, N=N, H=H, dtype=torch.float16, seed=65, outliers=True)
    inp = Inputs(d, bits, "prod", w.seeds["rotation"], w.seeds["projection"])
    plan = inp.plan()
    keys = tq_synth.keys(w).to(cuda)
    packed = tq.tq_encode(plan, keys)
    q = tq_synth.queries(w).to(cuda)
    logits = torch.empty(G, H, N, dtype=torch.float32, device=cuda)
    ts = torch.empty(G, H, k, dtype=torch.float32, device=cuda)
    ti = torch.empty(G, H, k, dtype=torch.int64, device=cuda)
    tq.tq_score_noalloc(plan, q, packed, N, top_k=k, logits=logits, top_scores=ts, top_idx=ti)
    torch.cuda.synchronize()
    gc.collect()  # tensors of earlier tests freed now, not during the measured call
    before = (torch.cuda.memory_allocated(cuda), torch.cuda.mem_get_info(cuda)[0])
    tq.tq_score_noalloc(plan, q, packed, N, top_k=k, logits=logits, top_scores=ts, top_idx=ti)
    torch.cuda.synchronize()
    after = (torch.cuda.memory_allocated(cuda), torch.cuda.mem_get_info(cuda)[0])
    assert after[0] <= before[0]   # nothing allocated through torch
    assert after[1] == before[1]   # nor through the driver: the device's free memory is unchanged
    want, want_s, want_i = tq.tq_score(plan, q, packed, N, top_k=k)
    torch.cuda.synchronize()
    assert torch.equal(ti, want_i)
