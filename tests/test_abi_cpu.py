"""CPU checks of the C-ABI library: it loads, exports every symbol the header
declares, rejects bad arguments without touching a GPU, and its host-side
set-up helpers (Lloyd-Max codebook, Haar rotation) agree with the oracle."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest
import torch

import vector_quantization_02_b300 as tq
from oracle import tq_oracle as o

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(tq_\w+)\s*\(", src))
    return names


def test_library_exports_every_declared_symbol():
    declared = _declared()
    assert declared, "no declarations found"
    for name in declared:
        assert hasattr(tq.lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", tq.lib._name], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (tq_\w+)", out))
    assert declared <= exported, declared - exported
    assert set(tq.EXPORTED) == declared


def test_status_strings_and_version():
    assert tq.lib.tq_status_string(0) == b"ok"
    assert tq.lib.tq_status_string(-2).startswith(b"pointer")
    assert tq.lib.tq_format_version() == 1


def test_argument_errors_need_no_gpu():
    lib = tq.lib
    vp = ctypes.c_void_p
    h = vp()
    # bad d, bad bits, null out: rejected before any CUDA call
    assert lib.tq_plan_create(100, 3, 0, vp(16), vp(16), vp(16), None, ctypes.byref(h)) == -1
    assert lib.tq_plan_create(128, 5, 0, vp(16), vp(16), vp(16), None, ctypes.byref(h)) == -1
    assert lib.tq_plan_create(128, 1, 0, vp(16), vp(16), vp(16), None, ctypes.byref(h)) == -1
    assert lib.tq_plan_create(128, 3, 0, vp(16), None, vp(16), None, ctypes.byref(h)) == -1
    assert lib.tq_plan_create(128, 3, 0, vp(16), vp(16), vp(16), None, None) == -1
    # the Walsh-Hadamard rotation needs d a power of two (128..2048) and signs
    assert lib.tq_plan_create_hadamard(384, 3, 0, vp(16), vp(16), vp(16), None, ctypes.byref(h)) == -1
    assert lib.tq_plan_create_hadamard(64, 3, 0, vp(16), vp(16), vp(16), None, ctypes.byref(h)) == -1
    assert lib.tq_plan_create_hadamard(4096, 3, 0, vp(16), vp(16), vp(16), None, ctypes.byref(h)) == -1
    assert lib.tq_plan_create_hadamard(128, 3, 0, None, vp(16), vp(16), None, ctypes.byref(h)) == -1
    assert lib.tq_plan_create_hadamard(128, 3, 0, vp(16), vp(16), vp(16), None, None) == -1
    assert lib.tq_packed_bytes(None, 1, 1) == 0
    assert lib.tq_encode(None, vp(16), 0, 1, 1, vp(16), None) == -1
    assert lib.tq_score(None, vp(16), 1, 1, vp(16), 1, vp(16), 0, None, None, vp(256), 1 << 20, None) == -1
    assert lib.tq_decode(None, vp(16), 1, 1, vp(16), None) == -1
    assert lib.tq_score_fp32(vp(16), vp(16), 1, 0, 1, 128, vp(16), None) == -1      # H = 0
    assert lib.tq_score_fp32(vp(16), vp(16), 1, 300, 1, 128, vp(16), None) == -1    # H > 256
    assert lib.tq_score_fp32(vp(16), vp(16), 1, 4, 1, 130, vp(16), None) == -1      # d % 4
    assert lib.tq_score_fp32(vp(8), vp(16), 1, 4, 1, 128, vp(16), None) == -2       # misaligned
    assert lib.tq_score_fp32(vp(16), vp(16), 1, 4, 0, 128, vp(16), None) == 0       # empty: no-op
    assert lib.tq_lloyd_max_codebook(3, 128, vp(16)) == -1
    assert lib.tq_haar_rotation(0, vp(16), vp(16)) == -1
    assert lib.tq_plan_status(None) == -1
    # path queries and the self-test reject a null plan
    assert lib.tq_score_path(None, 8) == -1
    assert lib.tq_encode_path(None, 1) == -1
    assert lib.tq_decode_path(None) == -1
    assert lib.tq_selftest_wait_expiry(None, None) == -1
    assert lib.tq_selftest_encode_drain(None, None, 1, 1, 1, None, None) == -1
    assert lib.tq_packed_header_write(None, 1, 1, None) == -1
    assert lib.tq_packed_header_read(None, None, None, None) == -1


@pytest.mark.parametrize("levels", [2, 4, 8, 16])
@pytest.mark.parametrize("d", [128, 1536])
def test_library_codebook_matches_oracle(levels, d):
    got = tq.tq_lloyd_max_codebook(levels, d).numpy()
    want = o.codebook(levels, d)
    assert np.all(np.diff(got) > 0)
    # both are fp64 solutions rounded to fp32: within one fp32 ulp
    assert np.max(np.abs(got.astype(np.float64) - want) / np.abs(want)) <= 2 ** -23


@pytest.mark.parametrize("d", [128, 256])
def test_library_rotation_matches_oracle(d):
    g = torch.randn(d, d, dtype=torch.float64, generator=torch.Generator().manual_seed(d))
    got = tq.tq_haar_rotation(g).numpy().astype(np.float64)
    want = o.haar_rotation(g.numpy())
    assert np.max(np.abs(got - want)) <= 1e-6
    assert np.max(np.abs(got.T @ got - np.eye(d))) <= 1e-5


def test_library_rotation_rejects_rank_deficient():
    g = torch.zeros(8, 8, dtype=torch.float64)
    with pytest.raises(tq.TQError):
        tq.tq_haar_rotation(g)


def _reconstruct(levels, masks, coefs, c0):
    return np.array([c0 + sum(cf * (bin(i & m).count("1") & 1) for m, cf in zip(masks, coefs))
                     for i in range(levels)])


@pytest.mark.parametrize("levels", [2, 4, 8, 16])
def test_parity_expansion_of_the_lloyd_max_codebook(levels):
    # the odd-symmetric codebook has weight only on odd-weight masks: k planes
    # for k <= 2, k + 1 for k = 3 (the triple product), 8 for k = 4
    c = tq.tq_lloyd_max_codebook(levels, 128)
    masks, coefs, c0 = tq.tq_codebook_parity_expansion(c)
    assert all(bin(m).count("1") % 2 == 1 for m in masks)
    assert len(masks) == {2: 1, 4: 2, 8: 4, 16: 8}[levels]
    assert np.max(np.abs(_reconstruct(levels, masks, coefs, c0) - c.numpy().astype(np.float64))) <= 1e-15
    # k = 1 (two levels, -a and a): one plane with weight 2a
    if levels == 2:
        assert masks == [1] and coefs[0] == 2 * float(c[1]) and c0 == float(c[0])


def test_parity_expansion_of_an_asymmetric_codebook():
    # a codebook with no symmetry needs every mask; the expansion is still exact
    c = torch.tensor([-1.5, -0.25, 0.125, 2.0, 2.5, 3.0, 7.0, 7.5])
    masks, coefs, c0 = tq.tq_codebook_parity_expansion(c)
    assert masks == list(range(1, 8))
    assert np.array_equal(_reconstruct(8, masks, coefs, c0), c.numpy().astype(np.float64))
    # a uniform (affine) codebook is linear in the bits: only the single-bit masks
    u = torch.tensor([0.0, 1.0, 2.0, 3.0]) * 0.5 - 0.75
    masks, coefs, c0 = tq.tq_codebook_parity_expansion(u)
    assert masks == [1, 2] and coefs == [0.5, 1.0] and c0 == -0.75
    with pytest.raises(tq.TQError):
        tq.tq_codebook_parity_expansion(torch.zeros(3))
