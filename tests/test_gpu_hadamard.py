"""GPU parity of plans with the randomised Walsh-Hadamard rotation
(tq_plan_create_hadamard; "알고리즘보다 커널이 성패를 가른다" section 4, the WHT
rotation of turboquant_plus) against the oracle's ``hadamard_rotation``, through
the C ABI.  The d = 128 fp16/bf16 encode forms the rotation with one exact
product of the keys and the +-1 matrix; every other kernel computes with the
dense fp32 Pi the plan holds.  The comparison rules are those of parity.py."""
import numpy as np
import pytest
import torch

import tq_synth
import vector_quantization_02_b300 as tq
from oracle import tq_oracle as o

from parity import HadamardInputs, compare_encode, compare_logits, oracle_encode

pytestmark = pytest.mark.gpu

ENCODE_CASES = [
    # d, G, N, dtype, bits, mode, outliers
    (128, 2, 300, torch.float16, 3, "prod", True),
    (128, 1, 1000, torch.bfloat16, 4, "prod", True),
    (128, 3, 129, torch.bfloat16, 2, "prod", False),
    (128, 2, 40000, torch.float16, 3, "prod", True),
    (128, 2, 300, torch.float16, 3, "mse", True),
    (128, 1, 300, torch.bfloat16, 4, "mse", False),
    (128, 2, 300, torch.float32, 3, "prod", False),
    (256, 1, 200, torch.float32, 4, "prod", False),
    (1024, 1, 130, torch.bfloat16, 3, "prod", True),
]


def _inputs(d, G, N, H, dtype, bits, mode, outliers, seed):
    w = tq_synth.small_case(d=d, G=G, N=N, H=H, dtype=dtype, seed=seed, outliers=outliers)
    return w, HadamardInputs(d, bits, mode, w.seeds["rotation"], w.seeds["projection"])


@pytest.mark.parametrize("d,G,N,dtype,bits,mode,outliers", ENCODE_CASES)
def test_hadamard_encode_matches_oracle(cuda, d, G, N, dtype, bits, mode, outliers):
    w, inp = _inputs(d, G, N, 4, dtype, bits, mode, outliers, seed=71)
    keys = tq_synth.keys(w)
    plan = inp.plan()
    want_path = "tensor_d128" if d == 128 and dtype != torch.float32 else "tensor_wide"
    assert plan.encode_path(dtype) == want_path
    packed = tq.tq_encode(plan, keys.to(cuda))
    torch.cuda.synchronize()
    assert plan.status() == 0
    compare_encode(inp, packed.cpu().numpy(), keys)


@pytest.mark.parametrize("d,G,N,H,bits,mode", [(128, 2, 300, 8, 3, "prod"), (128, 3, 200, 4, 4, "prod"),
                                               (128, 1, 129, 16, 3, "mse"), (256, 1, 300, 20, 3, "prod"),
                                               (128, 1, 257, 40, 2, "prod")])
def test_hadamard_score_from_oracle_packed_keys(cuda, d, G, N, H, bits, mode):
    w, inp = _inputs(d, G, N, H, torch.float32, bits, mode, False, seed=73)
    keys = tq_synth.keys(w)
    q = tq_synth.queries(w)
    buf, e = oracle_encode(inp, keys)
    want = o.score_packed(q.numpy(), buf, inp.Pi_o, inp.S_o, inp.c_o, bits, mode, G, N)
    plan = inp.plan()
    got = tq.tq_score(plan, q.to(cuda), torch.from_numpy(buf.copy()).to(cuda), N)
    torch.cuda.synchronize()
    assert plan.status() == 0
    compare_logits(got.cpu().numpy(), want, q, e["n"].astype(np.float32).astype(np.float64).reshape(G, N))


@pytest.mark.parametrize("d,bits,mode", [(128, 3, "prod"), (128, 4, "mse"), (256, 3, "prod")])
def test_hadamard_decode_matches_oracle(cuda, d, bits, mode):
    G, N = 2, 300
    w, inp = _inputs(d, G, N, 4, torch.float32, bits, mode, False, seed=75)
    keys = tq_synth.keys(w)
    buf, e = oracle_encode(inp, keys)
    want = o.decode_packed(buf, inp.Pi_o, inp.S_o, inp.c_o, d, bits, mode, G, N)
    plan = inp.plan()
    got = tq.tq_decode(plan, torch.from_numpy(buf.copy()).to(cuda), G, N)
    torch.cuda.synchronize()
    assert np.all(np.abs(got.cpu().numpy() - want) <= 1e-5 * e["n"].reshape(G, N, 1) + 1e-30)


def test_hadamard_plan_rejects_bad_signs_and_dims(cuda):
    S = tq_synth.projection(128, 1)
    c = torch.from_numpy(o.codebook_f32(4, 128))
    bad = torch.ones(128)
    bad[5] = 0.5
    with pytest.raises(tq.TQError) as ei:
        tq.Plan.hadamard(128, 3, bad, S, c)
    assert ei.value.status == -1
    with pytest.raises(tq.TQError):
        tq.Plan.hadamard(384, 3, torch.ones(384), tq_synth.projection(384, 1), torch.from_numpy(o.codebook_f32(4, 384)))
