"""GPU parity of fractional widths (tq_plan_create_fractional; "Google acelera
LLM 8 veces": 3.5 and 2.5 bits per channel) against the oracle's mixed
quantiser, through the C ABI.

The split of the channels is this library's reading (the first d/2 rotated
coordinates take one more Lloyd-Max bit), so parity with the pages is
unpinned; these tests hold the CUDA path to the oracle's restatement of that
reading, with the comparison rules of parity.py: codes and sign bits
identical outside the 1e-5 bands, norms within 1e-6 n and 1e-5 n, logits from
identical packed input within 1e-4 ||q|| n, decoded keys within 1e-5 n."""
import numpy as np
import pytest
import torch

import tq_synth
import vector_quantization_02_b300 as tq
from oracle import tq_oracle as o

pytestmark = pytest.mark.gpu


class FracInputs:
    def __init__(self, d, half_bits, mode, rot_seed, proj_seed):
        self.d, self.half_bits, self.mode = d, half_bits, mode
        self.prod = mode == "prod"
        self.k_hi = (half_bits + 1) // 2 - (1 if self.prod else 0)
        self.k_lo = self.k_hi - 1
        self.d_hi = o.mixed_split(d)
        self.Pi_o = np.ascontiguousarray(o.haar_rotation(tq_synth.rotation_gaussian(d, rot_seed).numpy()).astype(np.float32))
        self.S = tq_synth.projection(d, proj_seed)
        self.S_o = self.S.numpy()
        self.c_hi = o.codebook_f32(1 << self.k_hi, d)
        self.c_lo = o.codebook_f32(1 << self.k_lo, d)

    def plan(self):
        return tq.Plan.fractional(self.d, self.half_bits, torch.from_numpy(self.Pi_o), self.S if self.prod else None,
                                  torch.from_numpy(self.c_hi.copy()), torch.from_numpy(self.c_lo.copy()), self.mode)

    def encode(self, x):
        if self.prod:
            return o.encode_prod_mixed(x, self.Pi_o, self.S_o, self.c_hi, self.c_lo, self.d_hi)
        return o.encode_mse_mixed(x, self.Pi_o, self.c_hi, self.c_lo, self.d_hi)


CASES = [(7, "prod", torch.float16), (7, "prod", torch.bfloat16), (5, "prod", torch.float16), (5, "mse", torch.bfloat16),
         (3, "mse", torch.float16)]


@pytest.mark.parametrize("half_bits,mode,dtype", CASES)
def test_fractional_encode_matches_oracle(cuda, half_bits, mode, dtype):
    d, G, N = 128, 2, 1000
    inp = FracInputs(d, half_bits, mode, 111, 112)
    w = tq_synth.small_case(d=d, G=G, N=N, H=4, dtype=dtype, seed=113, outliers=True)
    keys = tq_synth.keys(w)
    plan = inp.plan()
    assert plan.packed_bytes(1, 128) == o.frac_block_bytes(d, inp.k_lo, inp.prod)
    assert plan.encode_path(dtype) == "tensor_d128"
    packed = tq.tq_encode(plan, keys.to(cuda))
    torch.cuda.synchronize()
    assert plan.status() == 0
    x = keys.double().numpy().reshape(G * N, d)
    e = inp.encode(x)
    got = o.unpack_mixed(packed.cpu().numpy(), d, inp.k_lo, inp.prod, G, N)
    code_bad = got["idx"] != e["idx"]
    assert not np.any(code_bad & ~e["code_exempt"]), "code mismatch outside the boundary band"
    assert np.all(np.abs(got["n"] - e["n"]) <= 1e-6 * e["n"] + 1e-30)
    mism = int(code_bad.sum())
    if inp.prod:
        z_ref, rho_ref, band = e["z"].copy(), e["rho"].copy(), e["sign_exempt"].copy()
        flipped = np.where(code_bad.any(axis=1))[0]
        if flipped.size:
            alt_idx = e["idx"][flipped].copy()
            alt_idx[code_bad[flipped]] = got["idx"][flipped][code_bad[flipped]]
            alt = o.qjl_stage_mixed(x[flipped], alt_idx, e["n"][flipped], inp.Pi_o, inp.S_o, inp.c_hi, inp.c_lo, inp.d_hi)
            z_ref[flipped], rho_ref[flipped], band[flipped] = alt["z"], alt["rho"], alt["sign_exempt"]
        sign_bad = got["z"] != z_ref
        assert not np.any(sign_bad & ~band), "sign mismatch outside the zero band"
        assert np.all(np.abs(got["rho"] - rho_ref.astype(np.float32)) <= 1e-5 * e["n"] + 1e-30)
        mism += int(sign_bad.sum())
    else:
        assert np.all(got["rho"] == 0)
    assert mism <= 2
    if mism == 0:
        want = o.pack_mixed(e["idx"], e.get("z"), e["n"].astype(np.float32),
                            e["rho"].astype(np.float32) if inp.prod else None, d, inp.k_lo, inp.prod, G, N)
        nb = -(-N // 128)
        bb = o.frac_block_bytes(d, inp.k_lo, inp.prod)
        planes = bb - 128 * 8
        assert np.array_equal(packed.cpu().numpy().reshape(G * nb, bb)[:, :planes], want.reshape(G * nb, bb)[:, :planes])


@pytest.mark.parametrize("half_bits,mode,H", [(7, "prod", 8), (5, "prod", 4), (5, "mse", 16), (7, "prod", 1)])
def test_fractional_score_from_oracle_packed_keys(cuda, half_bits, mode, H):
    d, G, N = 128, 3, 700
    inp = FracInputs(d, half_bits, mode, 121, 122)
    w = tq_synth.small_case(d=d, G=G, N=N, H=H, seed=123)
    keys, q = tq_synth.keys(w), tq_synth.queries(w)
    x = keys.double().numpy().reshape(G * N, d)
    e = inp.encode(x)
    buf = o.pack_mixed(e["idx"], e.get("z"), e["n"].astype(np.float32),
                       e["rho"].astype(np.float32) if inp.prod else None, d, inp.k_lo, inp.prod, G, N)
    u = o.unpack_mixed(buf, d, inp.k_lo, inp.prod, G, N)
    want = np.empty((G, H, N))
    for g in range(G):
        r = slice(g * N, (g + 1) * N)
        if inp.prod:
            want[g] = o.score_prod_mixed(q[g].numpy(), u["idx"][r], u["z"][r], u["n"][r], u["rho"][r], inp.Pi_o, inp.S_o,
                                         inp.c_hi, inp.c_lo, inp.d_hi)
        else:
            want[g] = q[g].double().numpy() @ o.mse_reconstruct_mixed(u["idx"][r], u["n"][r], inp.Pi_o, inp.c_hi,
                                                                      inp.c_lo, inp.d_hi).T
    plan = inp.plan()
    assert plan.score_path(H) == "tensor_d128"
    got = tq.tq_score(plan, q.to(cuda), torch.from_numpy(buf.copy()).to(cuda), N)
    torch.cuda.synchronize()
    assert plan.status() == 0
    bound = 1e-4 * np.linalg.norm(q.double().numpy(), axis=-1)[:, :, None] * u["n"].reshape(G, 1, N)
    err = np.abs(got.cpu().numpy().astype(np.float64) - want)
    assert np.all(err <= bound + 1e-30), f"max err/bound {np.max(err / (bound + 1e-30)):.3g}"


@pytest.mark.parametrize("half_bits,mode", [(7, "prod"), (5, "prod"), (5, "mse")])
def test_fractional_decode_matches_oracle(cuda, half_bits, mode):
    d, G, N = 128, 2, 300
    inp = FracInputs(d, half_bits, mode, 131, 132)
    w = tq_synth.small_case(d=d, G=G, N=N, H=4, seed=133)
    x = tq_synth.keys(w).double().numpy().reshape(G * N, d)
    e = inp.encode(x)
    buf = o.pack_mixed(e["idx"], e.get("z"), e["n"].astype(np.float32),
                       e["rho"].astype(np.float32) if inp.prod else None, d, inp.k_lo, inp.prod, G, N)
    u = o.unpack_mixed(buf, d, inp.k_lo, inp.prod, G, N)
    want = o.mse_reconstruct_mixed(u["idx"], u["n"], inp.Pi_o, inp.c_hi, inp.c_lo, inp.d_hi)
    if inp.prod:
        want = want + (u["rho"][:, None] * (o.KAPPA_NUM / d)) * (o.qjl_vector(u["z"]) @ inp.S_o.astype(np.float64))
    plan = inp.plan()
    assert plan.decode_path() == "tensor_d128"
    got = tq.tq_decode(plan, torch.from_numpy(buf.copy()).to(cuda), G, N)
    torch.cuda.synchronize()
    assert plan.status() == 0
    err = np.abs(got.cpu().numpy().reshape(G * N, d) - want)
    assert np.all(err <= 1e-5 * u["n"][:, None] + 1e-30)


def test_fractional_plan_bytes_and_refusals(cuda):
    d = 128
    for half_bits, mode, per_key in [(7, "prod", 64), (5, "prod", 48), (5, "mse", 48), (3, "mse", 32)]:
        plan = FracInputs(d, half_bits, mode, 141, 142).plan()
        assert plan.packed_bytes(1, 128) == 128 * per_key
        # fp32 keys take the wide encode, which has no fractional layout
        with pytest.raises(tq.TQError) as ei:
            tq.tq_encode(plan, torch.zeros(1, 5, d, device=cuda))
        assert ei.value.status == -3
    with pytest.raises(tq.TQError):   # 4.5 bits is not a fractional width of this library
        FracInputs(d, 9, "prod", 1, 2).plan()
