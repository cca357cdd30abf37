"""GPU parity of the CUDA path against the oracle, through the C ABI, on small
seeded inputs that span several token blocks and a ragged tail."""
import numpy as np
import pytest
import torch

import tq_synth
import vector_quantization_02_b300 as tq
from oracle import tq_oracle as o

from parity import (Inputs, check_topk_against_oracle, compare_encode, compare_logits, oracle_encode,
                    oracle_logits_of_packed)

pytestmark = pytest.mark.gpu

ENCODE_CASES = [
    # d, G, N, dtype, bits, mode, outliers
    (128, 1, 1, torch.float32, 3, "prod", False),
    (128, 2, 127, torch.float16, 3, "prod", True),
    (128, 1, 128, torch.bfloat16, 2, "prod", True),
    (128, 3, 129, torch.float32, 4, "prod", False),
    (128, 2, 300, torch.bfloat16, 3, "prod", True),
    (128, 1, 4097, torch.float16, 4, "prod", True),
    (256, 2, 300, torch.float32, 3, "prod", False),
    (256, 1, 200, torch.bfloat16, 4, "prod", True),
    (1536, 1, 130, torch.float32, 4, "prod", False),
    (128, 2, 300, torch.float32, 1, "mse", False),
    (128, 2, 300, torch.float16, 3, "mse", True),
    (256, 1, 150, torch.bfloat16, 4, "mse", True),
    # wide tensor-core encode: fp16 keys at d = 256, three 128-column jobs per
    # phase at d = 384, 2-bit bf16 at d = 512, fp32 d = 1536 over a ragged tail
    (256, 2, 200, torch.float16, 3, "prod", True),
    (384, 1, 300, torch.float32, 3, "prod", True),
    (512, 1, 129, torch.bfloat16, 2, "prod", False),
    (1536, 1, 300, torch.float32, 4, "prod", False),
    # MSE codec: the d = 128 kernel with 16 levels (select path) and with
    # several tiles per CTA; the wide kernel at d = 128 (fp32, several tiles
    # per CTA), d = 384 and fp32 d = 1536
    (128, 1, 300, torch.bfloat16, 4, "mse", True),
    (128, 2, 40000, torch.float16, 3, "mse", False),
    (128, 1, 40000, torch.float32, 4, "mse", True),
    (384, 1, 200, torch.float16, 2, "mse", False),
    (1536, 1, 130, torch.float32, 3, "mse", False),
    # the wide kernel's clusters over many tiles each: four CTAs per tile at
    # d = 512 (about ten tiles per cluster), two at d = 256
    (512, 2, 20000, torch.bfloat16, 3, "prod", False),
    (256, 1, 40000, torch.float16, 4, "prod", True),
]


def _case_inputs(d, G, N, dtype, bits, mode, outliers, seed=11):
    w = tq_synth.small_case(d=d, G=G, N=N, H=4, dtype=dtype, seed=seed, outliers=outliers)
    inp = Inputs(d, bits, mode, w.seeds["rotation"], w.seeds["projection"])
    return w, inp


@pytest.mark.parametrize("d,G,N,dtype,bits,mode,outliers", ENCODE_CASES)
def test_encode_matches_oracle(cuda, d, G, N, dtype, bits, mode, outliers):
    w, inp = _case_inputs(d, G, N, dtype, bits, mode, outliers)
    keys = tq_synth.keys(w)
    plan = inp.plan()
    packed = tq.tq_encode(plan, keys.to(cuda))
    torch.cuda.synchronize()
    assert plan.status() == 0
    compare_encode(inp, packed.cpu().numpy(), keys)


def test_wide_encode_concurrent_streams(cuda):
    """One plan, two streams, two wide encodes at once (fp32, d = 1536, 150 tiles
    each): the residual scratch is chosen per SM, so concurrent launches of the
    kernel never share a slot and each result equals the same call alone."""
    w, inp = _case_inputs(1536, 1, 19200, torch.float32, 4, "prod", False)
    plan = inp.plan()
    ka = tq_synth.keys(w, device=cuda)
    kb = tq_synth.keys(w, device=cuda, seed_offset=5)
    want_a = tq.tq_encode(plan, ka)
    want_b = tq.tq_encode(plan, kb)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    pa, pb = torch.empty_like(want_a), torch.empty_like(want_b)
    for _ in range(3):
        pa.zero_()
        pb.zero_()
        torch.cuda.synchronize()
        tq.tq_encode(plan, ka, packed=pa, stream=sa)
        tq.tq_encode(plan, kb, packed=pb, stream=sb)
        torch.cuda.synchronize()
        assert plan.status() == 0
        assert torch.equal(pa, want_a) and torch.equal(pb, want_b)


def test_encode_special_keys(cuda):
    # zero key, a huge and a tiny key, a basis vector, ties at exact zero
    d, G, N = 128, 1, 6
    _, inp = _case_inputs(d, G, N, torch.float32, 3, "prod", False)
    keys = torch.zeros(G, N, d)
    keys[0, 1] = torch.randn(d) * 1e6
    keys[0, 2] = torch.randn(d) * 1e-6
    keys[0, 3, 5] = 2.0
    keys[0, 4] = torch.randn(d)
    keys[0, 5, :] = 1.0
    plan = inp.plan()
    packed = tq.tq_encode(plan, keys.to(cuda))
    torch.cuda.synchronize()
    compare_encode(inp, packed.cpu().numpy(), keys)
    u = o.unpack(packed.cpu().numpy(), d, 3, "prod", G, N)
    assert u["n"][0] == 0 and u["rho"][0] == 0 and np.all(u["z"][0])


SCORE_CASES = [
    # d, G, N, H, bits, mode
    # wide tensor-core path (d != 128 or H > 16): heads padded to 16, all 256
    # heads, d = 384, MSE with 16 levels, d = 1536 over a ragged tail
    (128, 2, 300, 40, 3, "prod"),
    (128, 1, 257, 256, 4, "prod"),
    (384, 2, 129, 17, 2, "prod"),
    (256, 1, 300, 20, 4, "mse"),
    (1536, 1, 385, 64, 4, "prod"),
    (128, 1, 1, 1, 3, "prod"),
    (128, 2, 300, 4, 2, "prod"),
    (128, 3, 129, 8, 3, "prod"),
    (128, 1, 4096, 16, 3, "prod"),
    (128, 2, 257, 4, 4, "prod"),
    (256, 2, 200, 5, 3, "prod"),
    (1536, 1, 130, 3, 4, "prod"),
    (128, 2, 300, 8, 3, "mse"),
    (256, 1, 140, 4, 1, "mse"),
    # tensor-core path: many groups per CTA (query images change mid-range),
    # padded heads, ragged tails, MSE with one and three code bits
    (128, 300, 200, 4, 3, "prod"),
    (128, 5, 1000, 12, 3, "prod"),
    (128, 3, 129, 16, 2, "prod"),
    (128, 4, 700, 2, 4, "prod"),
    (128, 2, 260, 7, 1, "mse"),
    (128, 1, 385, 16, 4, "mse"),
]


@pytest.mark.parametrize("d,G,N,H,bits,mode", SCORE_CASES)
def test_score_from_oracle_packed_keys(cuda, d, G, N, H, bits, mode):
    # identical packed input: the oracle encodes, both sides score its bytes
    w, inp = _case_inputs(d, G, N, torch.float32, bits, mode, False, seed=23)
    w = tq_synth.small_case(d=d, G=G, N=N, H=H, seed=23)
    keys = tq_synth.keys(w)
    q = tq_synth.queries(w)
    buf, e = oracle_encode(inp, keys)
    want = o.score_packed(q.numpy(), buf, inp.Pi_o, inp.S_o, inp.c_o, bits, mode, G, N)
    plan = inp.plan()
    got = tq.tq_score(plan, q.to(cuda), torch.from_numpy(buf.copy()).to(cuda), N)
    torch.cuda.synchronize()
    assert plan.status() == 0
    n = e["n"].astype(np.float32).astype(np.float64).reshape(G, N)
    compare_logits(got.cpu().numpy(), want, q, n)


@pytest.mark.parametrize("d,G,N,H,k", [(128, 2, 1000, 4, 10), (128, 1, 300, 3, 64), (256, 1, 129, 2, 1),
                                       (128, 3, 70000, 2, 10)])
def test_score_top_k(cuda, d, G, N, H, k):
    w, inp = _case_inputs(d, G, N, torch.float32, 4, "prod", False, seed=31)
    w = tq_synth.small_case(d=d, G=G, N=N, H=H, seed=31)
    keys = tq_synth.keys(w)
    q = tq_synth.queries(w)
    plan = inp.plan()
    packed = tq.tq_encode(plan, keys.to(cuda))
    logits, ts, ti = tq.tq_score(plan, q.to(cuda), packed, N, top_k=k)
    torch.cuda.synchronize()
    L = logits.cpu().numpy()
    ts, ti = ts.cpu().numpy(), ti.cpu().numpy()
    # exact selection on the GPU's own logits
    want_s, want_i = o.topk(L, k)
    assert np.array_equal(ti, want_i)
    assert np.array_equal(ts, want_s)
    # valid against the oracle's scores of the same packed keys
    ol = oracle_logits_of_packed(inp, packed.cpu().numpy(), q.numpy().astype(np.float64), G, N).reshape(G * H, N)
    kth = np.sort(ol, axis=1)[:, -k]
    ti2, ts2 = ti.reshape(G * H, k), ts.reshape(G * H, k)
    at = np.take_along_axis(ol, ti2, axis=1)
    n_all = np.repeat(o.unpack(packed.cpu().numpy(), d, 4, "prod", G, N)["n"].reshape(G, 1, N), H, axis=1)
    n_at = np.take_along_axis(n_all.reshape(G * H, N), ti2, axis=1)
    check_topk_against_oracle(ts2, ti2, at, kth, np.linalg.norm(q.double().numpy(), axis=-1).reshape(-1), n_at)


@pytest.mark.parametrize("d,G,N,bits,mode", [
    (128, 2, 300, 3, "prod"), (256, 1, 129, 4, "prod"), (128, 1, 200, 2, "mse"),
    # the d = 128 tensor-core decode: one key, several tiles per CTA (both
    # modes, 16 levels), 1-bit codes over a ragged tail
    (128, 1, 1, 2, "prod"), (128, 1, 40000, 4, "prod"), (128, 2, 20000, 4, "mse"), (128, 3, 129, 1, "mse"),
    # the wide tensor-core decode: every code width of both modes (register
    # levels for k <= 2, the pair table for k >= 3), the vector-search d, a
    # ragged tail and several tiles per CTA
    (256, 2, 300, 2, "prod"), (384, 1, 77, 3, "prod"), (256, 1, 130, 1, "mse"), (512, 1, 260, 3, "mse"),
    (256, 1, 129, 4, "mse"), (1536, 1, 200, 4, "prod"), (256, 1, 40000, 3, "prod")])
def test_decode_matches_oracle(cuda, d, G, N, bits, mode):
    w, inp = _case_inputs(d, G, N, torch.float32, bits, mode, False, seed=41)
    keys = tq_synth.keys(w)
    buf, e = oracle_encode(inp, keys)
    want = o.decode_packed(buf, inp.Pi_o, inp.S_o, inp.c_o, d, bits, mode, G, N)
    plan = inp.plan()
    assert plan.decode_path() == ("tensor_d128" if d == 128 else "tensor_wide")
    got = tq.tq_decode(plan, torch.from_numpy(buf.copy()).to(cuda), G, N)
    torch.cuda.synchronize()
    assert plan.status() == 0
    n = e["n"].reshape(G, N, 1)
    assert np.all(np.abs(got.cpu().numpy() - want) <= 1e-5 * n + 1e-30)


def test_decode_score_consistency_on_gpu(cuda):
    # <q, tq_decode(packed)> == tq_score(q, packed) within 1e-4 ||q|| n
    d, G, N, H = 128, 2, 300, 4
    w, inp = _case_inputs(d, G, N, torch.bfloat16, 3, "prod", True, seed=43)
    w = tq_synth.small_case(d=d, G=G, N=N, H=H, dtype=torch.bfloat16, seed=43, outliers=True)
    keys = tq_synth.keys(w).to(cuda)
    q = tq_synth.queries(w).to(cuda)
    plan = inp.plan()
    packed = tq.tq_encode(plan, keys)
    s = tq.tq_score(plan, q, packed, N)
    x = tq.tq_decode(plan, packed, G, N)
    torch.cuda.synchronize()
    via_decode = torch.einsum("ghd,gnd->ghn", q.double(), x.double()).cpu().numpy()
    n = torch.linalg.vector_norm(keys.double(), dim=-1).cpu().numpy()
    compare_logits(s.cpu().numpy(), via_decode, q.cpu(), n)


@pytest.mark.parametrize("G,N,H,d", [(1, 1, 1, 128), (2, 300, 4, 128), (1, 100, 256, 128), (1, 50, 3, 1536),
                                     (3, 1000, 12, 128), (2, 129, 9, 64), (1, 257, 16, 132), (2, 5, 2, 8),
                                     (1, 515, 17, 128), (4, 33, 1, 128)])
def test_fp32_baseline(cuda, G, N, H, d):
    g = torch.Generator().manual_seed(5)
    q = torch.randn(G, H, d, generator=g)
    x = torch.randn(G, N, d, generator=g)
    got = tq.tq_score_fp32(q.to(cuda), x.to(cuda))
    torch.cuda.synchronize()
    want = o.score_fp32(q.numpy(), x.numpy())
    bound = 1e-5 * (torch.linalg.vector_norm(q.double(), dim=-1)[:, :, None] *
                    torch.linalg.vector_norm(x.double(), dim=-1)[:, None, :]).numpy()
    assert np.all(np.abs(got.cpu().numpy() - want) <= bound)


def test_fp32_baseline_rejects_ragged_rows(cuda):
    """Rows must be a whole number of 16-byte chunks (d % 4 == 0)."""
    q = torch.zeros(1, 2, 6, device=cuda)
    x = torch.zeros(1, 5, 6, device=cuda)
    with pytest.raises(tq.TQError):
        tq.tq_score_fp32(q, x)


def test_end_to_end_gpu_encode_then_score(cuda):
    # GPU encode -> GPU score against oracle encode -> oracle score, on the keys
    # whose codes and signs agree bit for bit (all of them, barring boundary cases)
    d, G, N, H, bits = 128, 3, 500, 8, 3
    w, inp = _case_inputs(d, G, N, torch.float16, bits, "prod", True, seed=47)
    w = tq_synth.small_case(d=d, G=G, N=N, H=H, dtype=torch.float16, seed=47, outliers=True)
    keys = tq_synth.keys(w)
    q = tq_synth.queries(w)
    plan = inp.plan()
    packed = tq.tq_encode(plan, keys.to(cuda))
    got = tq.tq_score(plan, q.to(cuda), packed, N)
    torch.cuda.synchronize()
    buf, e = oracle_encode(inp, keys)
    want = o.score_packed(q.numpy(), buf, inp.Pi_o, inp.S_o, inp.c_o, bits, "prod", G, N)
    gu = o.unpack(packed.cpu().numpy(), d, bits, "prod", G, N)
    same = (np.all(gu["idx"] == o.unpack(buf, d, bits, "prod", G, N)["idx"], axis=1) &
            np.all(gu["z"] == e["z"], axis=1)).reshape(G, N)
    assert same.mean() > 0.99
    n = e["n"].reshape(G, N)
    gl = got.cpu().numpy()
    gl = np.where(same[:, None, :], gl, want)
    compare_logits(gl, want, q, n)


def test_argument_errors_on_gpu(cuda):
    _, inp = _case_inputs(128, 1, 10, torch.float32, 3, "prod", False)
    plan = inp.plan()
    keys = torch.randn(1, 10, 128, device=cuda)
    packed = tq.tq_encode(plan, keys)
    bad = torch.empty(plan.packed_bytes(1, 10) + 16, dtype=torch.uint8, device=cuda)[1:]
    with pytest.raises(tq.TQError) as ei:
        tq.tq_encode(plan, keys, packed=bad)
    assert ei.value.status == -2
    with pytest.raises(tq.TQError):
        tq.tq_score(plan, torch.randn(1, 300, 128, device=cuda), packed, 10)
    with pytest.raises(tq.TQError):
        tq.tq_score(plan, torch.randn(1, 2, 128, device=cuda), packed, 10, top_k=11)


@pytest.mark.parametrize("d,bits,mode,H,dtype,score_path,encode_path", [
    (128, 3, "prod", 8, torch.float16, "tensor_d128", "tensor_d128"),     # decode cache
    (128, 4, "prod", 4, torch.bfloat16, "tensor_d128", "tensor_d128"),    # long context
    (128, 3, "prod", 16, torch.float32, "tensor_d128", "tensor_wide"),    # single head, fp32 keys
    (1536, 4, "prod", 256, torch.float32, "tensor_wide", "tensor_wide"),  # vector search
    (128, 3, "prod", 40, torch.float16, "tensor_wide", "tensor_d128"),
    (256, 4, "mse", 20, torch.bfloat16, "tensor_wide", "tensor_wide"),
    (128, 3, "mse", 8, torch.float16, "tensor_d128", "tensor_d128"),
    (128, 4, "mse", 8, torch.float32, "tensor_wide", "tensor_wide"),
])
def test_dispatch_paths(cuda, d, bits, mode, H, dtype, score_path, encode_path):
    """The kernel family each workload's shape takes (so bench labels and
    rooflines name the kernel that ran)."""
    plan = Inputs(d, bits, mode, 11, 12).plan()
    assert plan.score_path(H) == score_path
    assert plan.encode_path(dtype) == encode_path


@pytest.mark.parametrize("G,N", [(1, 300), (8, 12000)])
def test_encode_drain_is_reported(cuda, G, N):
    """A real kernel's error path: the d = 128 encode runs with one key tile's
    copy withheld; the waits on it give up, the CTA drains what it issued and
    frees its TMEM, the plan's error word reads TQ_ETIMEOUT once, and the next
    encode on the same context and plan matches the oracle."""
    d = 128
    w, inp = _case_inputs(d, G, N, torch.float16, 3, "prod", True)
    plan = inp.plan()
    keys = tq_synth.keys(w).to(cuda)
    plan.selftest_encode_drain(keys)
    torch.cuda.synchronize()
    assert plan.status() == -5
    assert plan.status() == 0
    packed = tq.tq_encode(plan, keys)
    torch.cuda.synchronize()
    assert plan.status() == 0
    compare_encode(inp, packed.cpu().numpy(), keys.cpu())


def test_packed_header_round_trip(cuda):
    """A packed cache stored as header + bytes reloads under the plan that wrote
    it and is refused under any other: another rotation, bit width, mode or
    format, or a damaged header."""
    d, G, N = 128, 2, 300
    w, inp = _case_inputs(d, G, N, torch.float16, 3, "prod", False)
    plan = inp.plan()
    keys = tq_synth.keys(w).to(cuda)
    packed = tq.tq_encode(plan, keys)
    header = plan.packed_header(G, N)
    assert len(header) == 64 and header[:4] == b"TQPK"
    stored = header + packed.cpu().numpy().tobytes()
    # reload: the header gives the sizes, the bytes decode to the same keys
    g2, n2 = plan.read_packed_header(stored[:64])
    assert (g2, n2) == (G, N)
    again = torch.frombuffer(bytearray(stored[64:]), dtype=torch.uint8).to(cuda)
    torch.cuda.synchronize()
    assert torch.equal(tq.tq_decode(plan, again, g2, n2), tq.tq_decode(plan, packed, G, N))
    # a damaged header
    bad = bytearray(header)
    bad[33] ^= 1
    with pytest.raises(tq.TQError):
        plan.read_packed_header(bytes(bad))
    # the same shape under other plans
    others = [Inputs(d, 3, "prod", 99, 98).plan(), Inputs(d, 4, "prod", 11, 12).plan(),
              Inputs(d, 3, "mse", 11, 12).plan()]
    for other in others:
        with pytest.raises(tq.TQError):
            other.read_packed_header(header)
    # the plan's own fingerprint does not depend on when it was built
    assert inp.plan().read_packed_header(header) == (G, N)


def test_bounded_wait_expiry_is_reported(cuda):
    """A device wait that nothing satisfies gives up after its poll limit and
    raises the plan's error word (TQ_ETIMEOUT once); nothing faults, and the
    context and the plan keep working."""
    d, G, N = 128, 1, 300
    w, inp = _case_inputs(d, G, N, torch.float16, 3, "prod", True)
    plan = inp.plan()
    plan.selftest_wait_expiry()
    torch.cuda.synchronize()
    assert plan.status() == -5
    assert plan.status() == 0
    keys = tq_synth.keys(w)
    packed = tq.tq_encode(plan, keys.to(cuda))
    torch.cuda.synchronize()
    assert plan.status() == 0
    compare_encode(inp, packed.cpu().numpy(), keys)
