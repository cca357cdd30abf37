"""The operand splits of the tensor-core decode, replayed in numpy on the CPU.

The d = 128 decode computes x_hat = n Pi^T c[idx] + rho sqrt(pi/2)/m S^T (2z - 1)
as fp16 tensor-core products: A = 2^8 c[idx] split into fp16 hi + lo (one
16-entry table per plan, its two halves packed into one 32-bit word), the
signs as +-1 fp16 bit patterns, and B = 2^8 Pi^T, 2^8 S^T split hi + lo; three
products for the first term, two for the second, and the scales undone at
the end.  These tests replay exactly that operand construction (the same
bit packing and the same dropped lo x lo product) with fp64 accumulation, and
require the result to sit far inside the 1e-5 n tolerance the GPU decode is
held to against the oracle.  A change of scale that pushes the lo parts into
fp16's subnormal range, or a packing with the halves swapped, fails here
without a GPU.
"""
import numpy as np
import pytest
import torch

import tq_synth
from oracle import tq_oracle as o

from parity import Inputs, oracle_encode


def _f16_split(v):
    h = v.astype(np.float16)
    return h, (v - h.astype(np.float32)).astype(np.float16)


def _pairs_to_f64(p, rows, d):
    """uint32 words holding (coordinate 2m in the low half, 2m + 1 in the high
    half) -> [rows][d] values."""
    halves = np.stack([(p & 0xFFFF).astype(np.uint16), (p >> 16).astype(np.uint16)], -1)
    return halves.reshape(rows, d).view(np.float16).astype(np.float64)


def _replay_decode(inp, f, G, N, d):
    c = inp.c_o.astype(np.float32)
    ch, cl = _f16_split(np.float32(256.0) * c)
    table = ch.view(np.uint16).astype(np.uint32) | (cl.view(np.uint16).astype(np.uint32) << 16)
    idx = f["idx"].reshape(G * N, d)
    t0, t1 = table[idx[:, 0::2]], table[idx[:, 1::2]]
    a_hi = _pairs_to_f64((t0 & 0xFFFF) | ((t1 & 0xFFFF) << 16), G * N, d)
    a_lo = _pairs_to_f64((t0 >> 16) | ((t1 >> 16) << 16), G * N, d)
    b_hi, b_lo = [x.astype(np.float64) for x in _f16_split((np.float32(256.0) * inp.Pi_o.T).astype(np.float32))]
    d1 = a_hi @ b_hi.T + a_hi @ b_lo.T + a_lo @ b_hi.T
    n = f["n"].reshape(G * N).astype(np.float32)
    out = (n * np.float32(1.0 / 65536.0))[:, None] * d1
    if inp.mode == "prod":
        z = f["z"].reshape(G * N, d).astype(np.uint32)
        word = lambda b: 0x3C00 | ((~b & 1) << 15)           # fp16 +1 for z = 1, -1 for z = 0
        sg = _pairs_to_f64((word(z[:, 0::2]) | (word(z[:, 1::2]) << 16)).astype(np.uint32), G * N, d)
        assert np.array_equal(sg, 2.0 * f["z"].reshape(G * N, d) - 1.0)
        s_hi, s_lo = [x.astype(np.float64) for x in _f16_split((np.float32(256.0) * inp.S_o.T).astype(np.float32))]
        d2 = sg @ s_hi.T + sg @ s_lo.T
        kappa = np.float32(np.sqrt(np.pi / 2) / d)
        out = out + (f["rho"].reshape(G * N).astype(np.float32) * kappa * np.float32(1.0 / 256.0))[:, None] * d2
    return out.reshape(G, N, d)


@pytest.mark.parametrize("bits,mode", [(2, "prod"), (3, "prod"), (4, "prod"), (1, "mse"), (3, "mse"), (4, "mse")])
def test_decode_operand_splits_stay_far_inside_the_tolerance(bits, mode):
    d, G, N = 128, 2, 160
    w = tq_synth.small_case(d=d, G=G, N=N, H=4, dtype=torch.float32, seed=47, outliers=True)
    inp = Inputs(d, bits, mode, w.seeds["rotation"], w.seeds["projection"])
    buf, e = oracle_encode(inp, tq_synth.keys(w))
    want = o.decode_packed(buf, inp.Pi_o, inp.S_o, inp.c_o, d, bits, mode, G, N)
    got = _replay_decode(inp, o.unpack(buf, d, bits, mode, G, N), G, N, d)
    rel = np.abs(got - want) / (e["n"].reshape(G, N, 1) + 1e-30)
    assert rel.max() < 1e-6, rel.max()


def test_fp16_splits_are_needed():
    # the reason for fp16: the same three products with bf16 halves (16 bits
    # per pair instead of 22) land over ten times further from the oracle,
    # within an order of magnitude of the 1e-5 n bound
    d, G, N, bits = 128, 1, 160, 3
    w = tq_synth.small_case(d=d, G=G, N=N, H=4, dtype=torch.float32, seed=47, outliers=True)
    inp = Inputs(d, bits, "mse", w.seeds["rotation"], w.seeds["projection"])
    buf, e = oracle_encode(inp, tq_synth.keys(w))
    want = o.decode_packed(buf, inp.Pi_o, inp.S_o, inp.c_o, d, bits, "mse", G, N)
    f = o.unpack(buf, d, bits, "mse", G, N)
    n = e["n"].reshape(G, N, 1) + 1e-30
    fp16_err = (np.abs(_replay_decode(inp, f, G, N, d) - want) / n).max()
    bf = lambda v: torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).bfloat16().float().numpy()
    split = lambda v: (bf(v), bf(v - bf(v)))
    a_hi, a_lo = split(inp.c_o.astype(np.float32)[f["idx"].reshape(G * N, d)])
    b_hi, b_lo = split(inp.Pi_o.T.astype(np.float32))
    a_hi, a_lo, b_hi, b_lo = (x.astype(np.float64) for x in (a_hi, a_lo, b_hi, b_lo))
    got = f["n"].reshape(G * N, 1) * (a_hi @ b_hi.T + a_hi @ b_lo.T + a_lo @ b_hi.T)
    bf16_err = (np.abs(got.reshape(G, N, d) - want) / n).max()
    assert bf16_err > 10 * fp16_err and bf16_err > 1e-6, (bf16_err, fp16_err)
