"""GPU parity of the value layout (tq_encode_values) and of one decode step of
attention on the compressed cache (tq_attend) against the oracle's
``pack_values`` and ``attend_packed``, through the C ABI.

Attention is compared on identical packed input: the oracle encodes the keys
(TurboQuantProd) and the values (TurboQuantMSE, coordinate-major layout) and
both sides attend over the same bytes.  Tolerance, per output element of head
h (derived, not fitted):
* the logits agree within 1e-4 ||q|| n (the scoring bound), so each softmax
  argument scale * logit moves by at most e = scale 1e-4 ||q_h|| max_t n_t and
  the output, a convex combination of the values, by at most 2 e max_t |v_t|;
* the softmax weights enter the tensor cores as four e4m3 slices (about 2^-16
  relative; 2^-14 is allowed) and the values' rotation back is fp32: 1e-5
  max_t ||v_t|| covers both.
"""
import math

import numpy as np
import pytest
import torch

import tq_synth
import vector_quantization_02_b300 as tq
from oracle import tq_oracle as o

from parity import Inputs, compare_fields

pytestmark = pytest.mark.gpu


def _value_inputs(d, bits, seed):
    return Inputs(d, bits, "mse", seed, seed + 1)


@pytest.mark.parametrize("G,N,dtype,bits", [(2, 300, torch.float16, 3), (1, 129, torch.bfloat16, 2),
                                            (3, 1000, torch.float32, 3), (1, 1, torch.float16, 1),
                                            (2, 4097, torch.bfloat16, 4)])
def test_value_layout_matches_oracle(cuda, G, N, dtype, bits):
    d = 128
    w = tq_synth.small_case(d=d, G=G, N=N, H=1, dtype=dtype, seed=81, outliers=True)
    vin = _value_inputs(d, bits, 83)
    vals = tq_synth.keys(w)
    plan = vin.plan()
    packed = tq.tq_encode_values(plan, vals.to(cuda))
    torch.cuda.synchronize()
    assert plan.status() == 0
    x = vals.double().numpy().reshape(G * N, d)
    e = o.encode_mse(x, vin.Pi_o, vin.c_o)
    got = o.unpack_values(packed.cpu().numpy(), d, bits, G, N)
    got["z"] = np.zeros_like(got["idx"], dtype=bool)
    got["rho"] = np.zeros(G * N)
    stats = compare_fields(vin, got, e, x)
    if stats["mismatches"] == 0:
        # every code agrees: the plane bytes, including the zero padding of the
        # last block, are identical (norms are compared within 1e-6 n above)
        want = o.pack_values(e["idx"], e["n"].astype(np.float32), d, bits, G, N)
        nb = -(-N // 128)
        bb = o.block_bytes(d, bits, "mse")
        plane = bits * d * 16
        assert np.array_equal(packed.cpu().numpy().reshape(G * nb, bb)[:, :plane], want.reshape(G * nb, bb)[:, :plane])


ATT_CASES = [
    # G, N, H, key bits, value bits
    (2, 300, 4, 3, 3),
    (3, 1000, 8, 3, 3),
    (1, 4097, 8, 3, 2),
    (2, 129, 2, 2, 3),
    (1, 1, 4, 3, 3),
    (1, 2000, 16, 4, 2),
    (5, 700, 7, 3, 1),
    (72, 256, 8, 3, 3),
]


@pytest.mark.parametrize("G,N,H,kbits,vbits", ATT_CASES)
def test_attend_matches_oracle(cuda, G, N, H, kbits, vbits):
    d = 128
    kin = Inputs(d, kbits, "prod", 91, 92)
    vin = _value_inputs(d, vbits, 93)
    wk = tq_synth.small_case(d=d, G=G, N=N, H=H, dtype=torch.float16, seed=95, outliers=True)
    wv = tq_synth.small_case(d=d, G=G, N=N, H=H, dtype=torch.float16, seed=97, outliers=True)
    keys, vals, q = tq_synth.keys(wk), tq_synth.keys(wv), tq_synth.queries(wk)
    kbuf, ke = o.encode_pack(keys.double().numpy(), kin.Pi_o, kin.S_o, kin.c_o, kbits, "prod", G, N)
    ve = o.encode_mse(vals.double().numpy().reshape(G * N, d), vin.Pi_o, vin.c_o)
    vbuf = o.pack_values(ve["idx"], ve["n"].astype(np.float32), d, vbits, G, N)
    scale = 1.0 / math.sqrt(d)
    kplan, vplan = kin.plan(), vin.plan()
    got = tq.tq_attend(kplan, vplan, q.to(cuda), torch.from_numpy(kbuf.copy()).to(cuda),
                       torch.from_numpy(vbuf.copy()).to(cuda), N, scale)
    torch.cuda.synchronize()
    assert kplan.status() == 0 and vplan.status() == 0
    want = o.attend_packed(q.numpy(), kbuf, vbuf, kin.Pi_o, kin.S_o, kin.c_o, kbits, vin.Pi_o, vin.c_o, vbits,
                           G, N, scale)
    vu = o.unpack_values(vbuf, d, vbits, G, N)
    vhat = o.mse_reconstruct(vu["idx"], vu["n"], vin.Pi_o, vin.c_o).reshape(G, N, d)
    vmax = np.abs(vhat).max(axis=(1, 2))                                  # [G]
    nmax = ke["n"].reshape(G, N).max(axis=1)                              # [G]
    qn = np.linalg.norm(q.double().numpy(), axis=-1)                      # [G][H]
    bound = (2 * scale * 1e-4 * qn * nmax[:, None] + 1e-5)[:, :, None] * vmax[:, None, None]
    err = np.abs(got.cpu().numpy().astype(np.float64) - want)
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound):.3g}"


def test_attend_rejects_unsupported_plans(cuda):
    d = 128
    kin = Inputs(d, 3, "prod", 91, 92)
    kplan = kin.plan()
    q = torch.zeros(1, 4, d, device=cuda)
    kp = torch.zeros(kplan.packed_bytes(1, 10), dtype=torch.uint8, device=cuda)
    with pytest.raises(tq.TQError) as ei:   # values must be an MSE plan
        tq.tq_attend(kplan, kplan, q, kp, kp, 10, 0.1)
    assert ei.value.status == -3
    vplan = _value_inputs(d, 4, 93).plan()  # 16 value levels: no odd-symmetric expansion of that size
    vp = torch.zeros(vplan.packed_bytes(1, 10), dtype=torch.uint8, device=cuda)
    with pytest.raises(tq.TQError) as ei:
        tq.tq_attend(kplan, vplan, q, kp, vp, 10, 0.1)
    assert ei.value.status == -3
