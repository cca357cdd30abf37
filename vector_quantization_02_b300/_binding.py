"""ctypes binding of libtq.so: argument marshalling only.

Every function here checks that tensors have the shape, dtype, device and
contiguity the C ABI documents (include/tq.h) and passes their pointers; all
computation happens in the library's CUDA kernels.  There is no CPU path: if
libtq.so is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtq.so")

TQ_OK, TQ_EINVAL, TQ_EALIGN, TQ_EUNSUPPORTED, TQ_ECUDA, TQ_ETIMEOUT, TQ_ENOMEM = 0, -1, -2, -3, -4, -5, -6
TQ_F32, TQ_F16, TQ_BF16 = 0, 1, 2
TQ_PROD, TQ_MSE = 0, 1

_DTYPES = {torch.float32: TQ_F32, torch.float16: TQ_F16, torch.bfloat16: TQ_BF16}
_MODES = {"prod": TQ_PROD, "mse": TQ_MSE}


def _load() -> ctypes.CDLL:
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libtq.so not built ({_LIB_PATH}); run `python vector_quantization_02_b300/build.py`")
    lib = ctypes.CDLL(_LIB_PATH)
    c_int, c_i64, c_sz, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p
    sig = {
        "tq_lloyd_max_codebook": (c_int, [c_int, c_int, vp]),
        "tq_haar_rotation": (c_int, [c_int, vp, vp]),
        "tq_plan_create": (c_int, [c_int, c_int, c_int, vp, vp, vp, vp, ctypes.POINTER(vp)]),
        "tq_plan_create_hadamard": (c_int, [c_int, c_int, c_int, vp, vp, vp, vp, ctypes.POINTER(vp)]),
        "tq_plan_create_fractional": (c_int, [c_int, c_int, c_int, vp, vp, vp, vp, vp, ctypes.POINTER(vp)]),
        "tq_plan_destroy": (c_int, [vp]),
        "tq_packed_bytes": (c_sz, [vp, c_i64, c_i64]),
        "tq_encode": (c_int, [vp, vp, c_int, c_i64, c_i64, vp, vp]),
        "tq_score_workspace_bytes": (c_sz, [vp, c_i64, c_int, c_i64, c_int]),
        "tq_score": (c_int, [vp, vp, c_i64, c_int, vp, c_i64, vp, c_int, vp, vp, vp, c_sz, vp]),
        "tq_decode": (c_int, [vp, vp, c_i64, c_i64, vp, vp]),
        "tq_score_fp32": (c_int, [vp, vp, c_i64, c_int, c_i64, c_int, vp, vp]),
        "tq_plan_status": (c_int, [vp]),
        "tq_status_string": (ctypes.c_char_p, [c_int]),
        "tq_format_version": (c_int, []),
        "tq_score_noalloc": (c_int, [vp, vp, c_i64, c_int, vp, c_i64, vp, c_int, vp, vp, vp]),
        "tq_codebook_parity_expansion": (c_int, [c_int, vp, vp, vp, vp, vp]),
        "tq_score_path": (c_int, [vp, c_int]),
        "tq_encode_path": (c_int, [vp, c_int]),
        "tq_decode_path": (c_int, [vp]),
        "tq_selftest_wait_expiry": (c_int, [vp, vp]),
        "tq_packed_header_write": (c_int, [vp, c_i64, c_i64, vp]),
        "tq_packed_header_read": (c_int, [vp, vp, vp, vp]),
        "tq_selftest_encode_drain": (c_int, [vp, vp, c_int, c_i64, c_i64, vp, vp]),
        "tq_encode_values": (c_int, [vp, vp, c_int, c_i64, c_i64, vp, vp]),
        "tq_attend_workspace_bytes": (c_sz, [vp, vp, c_i64, c_int, c_i64]),
        "tq_attend": (c_int, [vp, vp, vp, c_i64, c_int, vp, vp, c_i64, ctypes.c_float, vp, vp, c_sz, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = _load()
EXPORTED = ("tq_lloyd_max_codebook", "tq_haar_rotation", "tq_plan_create", "tq_plan_create_hadamard",
            "tq_plan_create_fractional",
            "tq_plan_destroy",
            "tq_packed_bytes", "tq_encode", "tq_score_workspace_bytes", "tq_score", "tq_decode",
            "tq_score_fp32", "tq_plan_status", "tq_status_string", "tq_format_version", "tq_score_noalloc",
            "tq_codebook_parity_expansion", "tq_score_path", "tq_encode_path", "tq_decode_path",
            "tq_selftest_wait_expiry", "tq_selftest_encode_drain", "tq_packed_header_write",
            "tq_packed_header_read", "tq_encode_values", "tq_attend_workspace_bytes",
            "tq_attend")
PATHS = {0: "tensor_d128", 1: "tensor_wide", 2: "cuda_core"}
TQ_SCORE_NOALLOC_MAX_BYTES = 32 << 20
TQ_PACKED_HEADER_BYTES = 64


class TQError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {lib.tq_status_string(status).decode()} ({status})")
        self.status = status


def _check(status: int, what: str):
    if status != TQ_OK:
        raise TQError(status, what)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr())


# ---------------------------------------------------------------- plan inputs (host)

def tq_lloyd_max_codebook(levels: int, d: int) -> torch.Tensor:
    """Lloyd-Max centroids for N(0, 1/d), fp32 on the host (library's own solver)."""
    out = torch.empty(levels, dtype=torch.float32)
    _check(lib.tq_lloyd_max_codebook(levels, d, ctypes.c_void_p(out.data_ptr())), "tq_lloyd_max_codebook")
    return out


def tq_haar_rotation(gaussian: torch.Tensor) -> torch.Tensor:
    """Haar rotation from a host fp64 d x d Gaussian matrix, fp32 on the host."""
    g = gaussian.detach().to("cpu", torch.float64).contiguous()
    d = g.shape[0]
    assert g.shape == (d, d)
    out = torch.empty(d, d, dtype=torch.float32)
    _check(lib.tq_haar_rotation(d, ctypes.c_void_p(g.data_ptr()), ctypes.c_void_p(out.data_ptr())),
           "tq_haar_rotation")
    return out


def tq_codebook_parity_expansion(codebook: torch.Tensor):
    """Parity expansion of a host codebook: (masks, coefs, c0) with
    codebook[idx] = c0 + sum_t coefs[t] * parity(idx & masks[t])."""
    c = codebook.detach().to("cpu", torch.float32).contiguous()
    L = c.numel()
    n = ctypes.c_int(0)
    masks = (ctypes.c_uint * max(1, L - 1))()
    coefs = (ctypes.c_double * max(1, L - 1))()
    c0 = ctypes.c_double(0.0)
    _check(lib.tq_codebook_parity_expansion(L, ctypes.c_void_p(c.data_ptr()), ctypes.byref(n), masks, coefs,
                                            ctypes.byref(c0)), "tq_codebook_parity_expansion")
    return [int(masks[i]) for i in range(n.value)], [float(coefs[i]) for i in range(n.value)], c0.value


# ---------------------------------------------------------------- plan

class Plan:
    """A TurboQuant plan: rotation Pi, projection S and codebook on the GPU."""

    def __init__(self, d: int, bits: int, Pi: torch.Tensor | None, S: torch.Tensor | None,
                 codebook: torch.Tensor, mode: str = "prod", stream=None, signs: torch.Tensor | None = None):
        """A plan with a dense rotation Pi, or (``signs`` given, Pi None) the
        randomised Walsh-Hadamard rotation Pi = H diag(signs) / sqrt(d)."""
        self.d, self.bits, self.mode = d, bits, mode
        self.hadamard = signs is not None
        dev = torch.device("cuda", torch.cuda.current_device())
        if self.hadamard:
            rot_d = signs.to(dev, torch.float32).contiguous()
            if rot_d.numel() != d:
                raise ValueError("signs must hold d entries")
        else:
            rot_d = Pi.to(dev, torch.float32).contiguous()
        S_d = S.to(dev, torch.float32).contiguous() if S is not None else None
        cb_d = codebook.to(dev, torch.float32).contiguous()
        k = bits - 1 if mode == "prod" else bits
        if cb_d.numel() != 1 << k:
            raise ValueError(f"codebook must have {1 << k} centroids for {bits} bits ({mode})")
        if (S_d is None) != (mode == "mse"):
            raise ValueError("S is required for mode 'prod' and unused for 'mse'")
        h = ctypes.c_void_p()
        create = lib.tq_plan_create_hadamard if self.hadamard else lib.tq_plan_create
        st = create(d, bits, _MODES[mode],
                    _dev(rot_d, "signs", shape=(d,)) if self.hadamard else _dev(rot_d, "Pi", shape=(d, d)),
                    _dev(S_d, "S", shape=(d, d)) if S_d is not None else None,
                    _dev(cb_d, "codebook"), ctypes.c_void_p(_stream(stream)), ctypes.byref(h))
        _check(st, "tq_plan_create_hadamard" if self.hadamard else "tq_plan_create")
        self.handle = h
        self.levels = cb_d.numel()

    @classmethod
    def from_seeds(cls, d: int, bits: int, rotation_gaussian: torch.Tensor, S: torch.Tensor | None,
                   mode: str = "prod"):
        """Build Pi and the codebook with the library's host helpers."""
        k = bits - 1 if mode == "prod" else bits
        return cls(d, bits, tq_haar_rotation(rotation_gaussian), S, tq_lloyd_max_codebook(1 << k, d), mode)

    @classmethod
    def fractional(cls, d: int, half_bits: int, Pi: torch.Tensor, S: torch.Tensor | None, codebook_hi: torch.Tensor,
                   codebook_lo: torch.Tensor, mode: str = "prod", stream=None):
        """A plan at b + 1/2 bits per channel (half_bits = 2b + 1): the first
        d/2 rotated coordinates take codebook_hi, the others codebook_lo
        (tq_plan_create_fractional)."""
        self = cls.__new__(cls)
        self.d, self.mode, self.hadamard, self.half_bits = d, mode, False, half_bits
        dev = torch.device("cuda", torch.cuda.current_device())
        Pi_d = Pi.to(dev, torch.float32).contiguous()
        S_d = S.to(dev, torch.float32).contiguous() if S is not None else None
        hi = codebook_hi.to(dev, torch.float32).contiguous()
        lo = codebook_lo.to(dev, torch.float32).contiguous()
        k_hi = (half_bits + 1) // 2 - (1 if mode == "prod" else 0)
        self.bits = k_hi + 1 if mode == "prod" else k_hi
        if hi.numel() != 1 << k_hi or lo.numel() != 1 << (k_hi - 1):
            raise ValueError(f"codebooks must have {1 << k_hi} and {1 << (k_hi - 1)} centroids")
        h = ctypes.c_void_p()
        st = lib.tq_plan_create_fractional(d, half_bits, _MODES[mode], _dev(Pi_d, "Pi", shape=(d, d)),
                                           _dev(S_d, "S", shape=(d, d)) if S_d is not None else None,
                                           _dev(hi, "codebook_hi"), _dev(lo, "codebook_lo"),
                                           ctypes.c_void_p(_stream(stream)), ctypes.byref(h))
        _check(st, "tq_plan_create_fractional")
        self.handle = h
        self.levels = hi.numel()
        return self

    @classmethod
    def hadamard(cls, d: int, bits: int, signs: torch.Tensor, S: torch.Tensor | None, codebook: torch.Tensor,
                 mode: str = "prod"):
        """The randomised Walsh-Hadamard rotation (tq_plan_create_hadamard)."""
        return cls(d, bits, None, S, codebook, mode, signs=signs)

    def close(self):
        if getattr(self, "handle", None):
            lib.tq_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def packed_bytes(self, G: int, N: int) -> int:
        return int(lib.tq_packed_bytes(self.handle, G, N))

    def status(self) -> int:
        return int(lib.tq_plan_status(self.handle))

    def selftest_wait_expiry(self, stream=None) -> None:
        """Enqueue the bounded-wait self-test; after a sync, status() reports TQ_ETIMEOUT once."""
        _check(lib.tq_selftest_wait_expiry(self.handle, ctypes.c_void_p(_stream(stream))), "tq_selftest_wait_expiry")

    def selftest_encode_drain(self, keys: torch.Tensor, stream=None) -> None:
        """Enqueue the d = 128 encode of keys [G][N][128] (fp16/bf16) with CTA 0's
        first key tile withheld; after a sync, status() reports TQ_ETIMEOUT once."""
        G, N, d = keys.shape
        if d != self.d or keys.dtype not in (torch.float16, torch.bfloat16):
            raise ValueError("the self-test takes fp16/bf16 keys of the plan's d")
        packed = torch.empty(self.packed_bytes(G, N), dtype=torch.uint8, device=keys.device)
        _check(lib.tq_selftest_encode_drain(self.handle, _dev(keys, "keys"), _DTYPES[keys.dtype], G, N,
                                            _dev(packed, "packed"), ctypes.c_void_p(_stream(stream))),
               "tq_selftest_encode_drain")
        self._drain_buffers = (keys, packed)  # alive until the caller synchronises

    def packed_header(self, G: int, N: int) -> bytes:
        """The 64-byte header describing a packed buffer of G x N keys of this plan."""
        buf = ctypes.create_string_buffer(TQ_PACKED_HEADER_BYTES)
        _check(lib.tq_packed_header_write(self.handle, G, N, buf), "tq_packed_header_write")
        return buf.raw

    def read_packed_header(self, header: bytes) -> tuple[int, int]:
        """(G, N) of a header written for this plan; raises TQError otherwise."""
        if len(header) != TQ_PACKED_HEADER_BYTES:
            raise ValueError("a packed header is 64 bytes")
        G, N = ctypes.c_int64(), ctypes.c_int64()
        _check(lib.tq_packed_header_read(self.handle, header, ctypes.byref(G), ctypes.byref(N)),
               "tq_packed_header_read")
        return G.value, N.value

    def score_path(self, H: int) -> str:
        """Kernel family tq_score takes for H heads: tensor_d128 or tensor_wide."""
        r = int(lib.tq_score_path(self.handle, H))
        _check(min(r, 0), "tq_score_path")
        return PATHS[r]

    def encode_path(self, dtype: torch.dtype) -> str:
        """Kernel family tq_encode takes for keys of this dtype."""
        r = int(lib.tq_encode_path(self.handle, _DTYPES[dtype]))
        _check(min(r, 0), "tq_encode_path")
        return PATHS[r]

    def decode_path(self) -> str:
        """Kernel family tq_decode takes: tensor_d128 or cuda_core."""
        r = int(lib.tq_decode_path(self.handle))
        _check(min(r, 0), "tq_decode_path")
        return PATHS[r]


# ---------------------------------------------------------------- the path

def tq_encode(plan: Plan, keys: torch.Tensor, packed: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """keys [G][N][d] (fp32/fp16/bf16, CUDA) -> packed uint8 buffer."""
    G, N, d = keys.shape
    if d != plan.d:
        raise ValueError("keys' last dimension must equal the plan's d")
    nbytes = plan.packed_bytes(G, N)
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=keys.device)
    elif packed.numel() < nbytes or packed.dtype != torch.uint8:
        raise ValueError("packed buffer too small")
    if keys.dtype not in _DTYPES:
        raise ValueError(f"unsupported key dtype {keys.dtype}")
    _check(lib.tq_encode(plan.handle, _dev(keys, "keys"), _DTYPES[keys.dtype], G, N,
                         _dev(packed, "packed"), ctypes.c_void_p(_stream(stream))), "tq_encode")
    return packed


def score_workspace_bytes(plan: Plan, G: int, H: int, N: int, top_k: int = 0) -> int:
    return int(lib.tq_score_workspace_bytes(plan.handle, G, H, N, top_k))


def tq_score(plan: Plan, queries: torch.Tensor, packed: torch.Tensor, N: int, top_k: int = 0,
             logits: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None):
    """queries [G][H][d] fp32 + packed keys -> logits [G][H][N] (and top-k)."""
    G, H, d = queries.shape
    dev = queries.device
    if packed.numel() < plan.packed_bytes(G, N):
        raise ValueError("packed buffer too small for (G, N)")
    if logits is None:
        logits = torch.empty(G, H, N, dtype=torch.float32, device=dev)
    wsb = score_workspace_bytes(plan, G, H, N, top_k)
    if workspace is None:
        workspace = torch.empty(wsb, dtype=torch.uint8, device=dev)
    ts = ti = None
    if top_k:
        ts = torch.empty(G, H, top_k, dtype=torch.float32, device=dev)
        ti = torch.empty(G, H, top_k, dtype=torch.int64, device=dev)
    st = lib.tq_score(plan.handle, _dev(queries, "queries", torch.float32), G, H, _dev(packed, "packed"), N,
                      _dev(logits, "logits", torch.float32, (G, H, N)), top_k,
                      _dev(ts, "top_scores") if top_k else None, _dev(ti, "top_idx") if top_k else None,
                      _dev(workspace, "workspace"), workspace.numel(), ctypes.c_void_p(_stream(stream)))
    _check(st, "tq_score")
    return (logits, ts, ti) if top_k else logits


def tq_decode(plan: Plan, packed: torch.Tensor, G: int, N: int, out: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    if packed.numel() < plan.packed_bytes(G, N):
        raise ValueError("packed buffer too small for (G, N)")
    if out is None:
        out = torch.empty(G, N, plan.d, dtype=torch.float32, device=packed.device)
    _check(lib.tq_decode(plan.handle, _dev(packed, "packed"), G, N, _dev(out, "out", torch.float32, (G, N, plan.d)),
                         ctypes.c_void_p(_stream(stream))), "tq_decode")
    return out


def tq_score_fp32(queries: torch.Tensor, keys: torch.Tensor, logits: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    G, H, d = queries.shape
    G2, N, d2 = keys.shape
    if G2 != G or d2 != d:
        raise ValueError("queries and keys disagree on G or d")
    if logits is None:
        logits = torch.empty(G, H, N, dtype=torch.float32, device=queries.device)
    _check(lib.tq_score_fp32(_dev(queries, "queries", torch.float32), _dev(keys, "keys", torch.float32), G, H, N, d,
                             _dev(logits, "logits", torch.float32, (G, H, N)), ctypes.c_void_p(_stream(stream))),
           "tq_score_fp32")
    return logits


def tq_score_noalloc(plan: Plan, queries: torch.Tensor, packed: torch.Tensor, N: int, top_k: int = 0,
                     logits: torch.Tensor | None = None, top_scores: torch.Tensor | None = None,
                     top_idx: torch.Tensor | None = None, stream=None):
    """tq_score without a workspace argument, for callers that may not allocate
    device memory: the library takes its scratch from a fixed device array
    (TQ_SCORE_NOALLOC_MAX_BYTES).  Outputs must be passed in by such callers;
    when they are omitted this wrapper creates them (the C entry point itself
    never allocates)."""
    G, H, d = queries.shape
    dev = queries.device
    if packed.numel() < plan.packed_bytes(G, N):
        raise ValueError("packed buffer too small for (G, N)")
    if logits is None:
        logits = torch.empty(G, H, N, dtype=torch.float32, device=dev)
    if top_k and top_scores is None:
        top_scores = torch.empty(G, H, top_k, dtype=torch.float32, device=dev)
    if top_k and top_idx is None:
        top_idx = torch.empty(G, H, top_k, dtype=torch.int64, device=dev)
    st = lib.tq_score_noalloc(plan.handle, _dev(queries, "queries", torch.float32), G, H, _dev(packed, "packed"), N,
                              _dev(logits, "logits", torch.float32, (G, H, N)), top_k,
                              _dev(top_scores, "top_scores", torch.float32, (G, H, top_k)) if top_k else None,
                              _dev(top_idx, "top_idx", torch.int64, (G, H, top_k)) if top_k else None,
                              ctypes.c_void_p(_stream(stream)))
    _check(st, "tq_score_noalloc")
    return (logits, top_scores, top_idx) if top_k else logits


def tq_encode_values(plan: Plan, values: torch.Tensor, packed: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """values [G][N][d] (CUDA) -> packed uint8 buffer in the coordinate-major
    value layout (an MSE plan)."""
    G, N, d = values.shape
    if d != plan.d:
        raise ValueError("values' last dimension must equal the plan's d")
    nbytes = plan.packed_bytes(G, N)
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=values.device)
    elif packed.numel() < nbytes or packed.dtype != torch.uint8:
        raise ValueError("packed buffer too small")
    if values.dtype not in _DTYPES:
        raise ValueError(f"unsupported value dtype {values.dtype}")
    _check(lib.tq_encode_values(plan.handle, _dev(values, "values"), _DTYPES[values.dtype], G, N,
                                _dev(packed, "packed"), ctypes.c_void_p(_stream(stream))), "tq_encode_values")
    return packed


def attend_workspace_bytes(kplan: Plan, vplan: Plan, G: int, H: int, N: int) -> int:
    return int(lib.tq_attend_workspace_bytes(kplan.handle, vplan.handle, G, H, N))


def tq_attend(kplan: Plan, vplan: Plan, queries: torch.Tensor, kpacked: torch.Tensor, vpacked: torch.Tensor, N: int,
              scale: float, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    """One decode step of attention on the compressed cache: queries [G][H][d]
    -> out [G][H][d] (softmax of scale * logits over the N tokens, times the
    reconstructed values)."""
    G, H, d = queries.shape
    dev = queries.device
    if kpacked.numel() < kplan.packed_bytes(G, N) or vpacked.numel() < vplan.packed_bytes(G, N):
        raise ValueError("packed buffers too small for (G, N)")
    if out is None:
        out = torch.empty(G, H, d, dtype=torch.float32, device=dev)
    wsb = attend_workspace_bytes(kplan, vplan, G, H, N)
    if workspace is None:
        workspace = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
    st = lib.tq_attend(kplan.handle, vplan.handle, _dev(queries, "queries", torch.float32), G, H,
                       _dev(kpacked, "kpacked"), _dev(vpacked, "vpacked"), N, ctypes.c_float(scale),
                       _dev(out, "out", torch.float32, (G, H, d)), _dev(workspace, "workspace"), workspace.numel(),
                       ctypes.c_void_p(_stream(stream)))
    _check(st, "tq_attend")
    return out
