"""TurboQuantProd key encoding and compressed-key attention scoring on B300.

The compute lives in libtq.so (hand-written CUDA for sm_103a, C ABI in
include/tq.h); this package is its thin binding.  Importing it fails if the
library has not been built (``python vector_quantization_02_b300/build.py``).
"""
from ._binding import (  # noqa: F401
    EXPORTED, TQ_BF16, TQ_F16, TQ_F32, TQ_MSE, TQ_PROD, Plan, TQError, lib, score_workspace_bytes,
    tq_codebook_parity_expansion, tq_decode, tq_encode, tq_haar_rotation, tq_lloyd_max_codebook, tq_score, tq_score_fp32,
    tq_score_noalloc, TQ_SCORE_NOALLOC_MAX_BYTES, attend_workspace_bytes, tq_attend, tq_encode_values)
