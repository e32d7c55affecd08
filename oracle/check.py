"""Consumer-side check (oracle; test infrastructure only).

The block_scaled_quantization module page lists a naive reference matmul
(naive_block_scaled_matmul) that reproduces in plain code how the tensor
cores apply the block scales; the idea is to check quantized operands by
dequantising them through the 5D scale layout and taking a plain dot
product.  Here that is done in float64 on the
CPU, reading the scales through ``scales_from_5d_view`` (a reshape statement
of the layout, independent of the offset formula used to write them).
"""
from __future__ import annotations

import numpy as np

from .layout import scales_from_5d_view
from .blockquant import block_size, dequantize


def naive_block_scaled_matmul(fmt: str, a_packed, a_scales5d, a_tsf,
                              b_packed, b_scales5d, b_tsf, K: int) -> np.ndarray:
    """C = deq(A) @ deq(B)^T in float64; A is (M, K), B is (N, K)."""
    S = K // block_size(fmt)
    M, N = np.asarray(a_packed).shape[0], np.asarray(b_packed).shape[0]
    a = dequantize(fmt, a_packed, scales_from_5d_view(a_scales5d, M, S)[:M, :S], a_tsf)
    b = dequantize(fmt, b_packed, scales_from_5d_view(b_scales5d, N, S)[:N, :S], b_tsf)
    return a @ b.T
