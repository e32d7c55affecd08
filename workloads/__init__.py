"""Seeded synthetic workloads for block-scaled activation quantization.

This module only *draws inputs*: BF16 activation matrices (as uint16 bit
patterns), the FP32 per-tensor / per-expert scale that the workloads pass in
(``tensor_sf = 448*6 / amax``), and mixture-of-experts routing metadata
(``row_offsets``, ``scales_offsets``, ``expert_ids``, ``row_indices``).
It holds none of the quantization arithmetic.  Both the CPU oracle's tests
and the CUDA path's tests and benchmark take their inputs from here, so the
two sides see the same bytes.

Workload shapes follow the activations of the models the grouped block-scaled
matmul dispatch page was tuned on (K = 7168 / 4096 / 2048, 256 experts,
top-8 routing; "grouped_block_scaled_1d1d dispatch", NVFP4 routing table).
No dataset is used: every value is drawn from a NumPy PCG64 generator.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "f32_to_bf16_bits", "bf16_bits_to_f32", "tensor_sf_from_amax",
    "dense_activations", "config_dense_nvfp4_small", "config_dense_nvfp4_large",
    "config_dense_mx_wide", "zipf_topk_routing", "grouped_workload",
    "config_grouped_prefill", "config_grouped_decode",
]

NVFP4_TENSOR_SF_NUM = np.float32(448.0 * 6.0)  # E4M3 max x E2M1 max


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round FP32 values to BF16 (nearest, ties to even); return uint16 bits.

    Inputs are finite (the generators never draw NaN/Inf)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((u + bias) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to FP32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def tensor_sf_from_amax(amax) -> np.float32:
    """FP32 ``448*6/amax`` (1.0 for an all-zero tensor): the per-tensor scale
    the workloads hand to NVFP4 quantization."""
    amax = np.float32(amax)
    if amax == 0:
        return np.float32(1.0)
    return np.float32(NVFP4_TENSOR_SF_NUM / amax)


def _amax_bits(x_bits: np.ndarray) -> np.float32:
    if x_bits.size == 0:
        return np.float32(0.0)
    return np.float32(np.abs(bf16_bits_to_f32(x_bits)).max())


def dense_activations(rng: np.random.Generator, M: int, K: int, kind: str) -> np.ndarray:
    """Draw an (M, K) BF16 activation matrix as uint16 bits.

    kind:
      "outliers1pct"   N(0,1); 1% of entries x30; the 16-block (row 0, cols 0..15) zeroed
      "rowlognormal"   N(0,1) x per-row LogNormal(0,1); 0.1% of entries x50
      "blocklognormal" N(0,1) x LogNormal(0,2) drawn per 32-element block
      "normal"         N(0,1)
    """
    x = rng.standard_normal((M, K), dtype=np.float32)
    if kind == "outliers1pct":
        x = np.where(rng.random((M, K)) < 0.01, x * np.float32(30.0), x)
        if M > 0 and K >= 16:
            x[0, :16] = 0.0
    elif kind == "rowlognormal":
        x *= rng.lognormal(0.0, 1.0, size=(M, 1)).astype(np.float32)
        x = np.where(rng.random((M, K)) < 0.001, x * np.float32(50.0), x)
    elif kind == "blocklognormal":
        assert K % 32 == 0
        s = rng.lognormal(0.0, 2.0, size=(M, K // 32, 1)).astype(np.float32)
        x = (x.reshape(M, K // 32, 32) * s).reshape(M, K)
    elif kind != "normal":
        raise ValueError(kind)
    return f32_to_bf16_bits(x)


def config_dense_nvfp4_small(seed: int = 0, M: int = 128, K: int = 256) -> dict:
    """NVFP4 dense, M=128 K=256: N(0,1), 1% outliers x30, one all-zero block,
    tensor_sf = 448*6/global amax."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = dense_activations(rng, M, K, "outliers1pct")
    return dict(name=f"nvfp4_dense_M{M}_K{K}", fmt="nvfp4", x_bits=x, M=M, K=K,
                tensor_sf=tensor_sf_from_amax(_amax_bits(x)))


def config_dense_nvfp4_large(seed: int = 1, M: int = 8192, K: int = 7168) -> dict:
    """NVFP4 dense, M=8192 K=7168: N(0,1) x per-row LogNormal(0,1), 0.1% outliers
    x50, tensor_sf from the global amax."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = dense_activations(rng, M, K, "rowlognormal")
    return dict(name=f"nvfp4_dense_M{M}_K{K}", fmt="nvfp4", x_bits=x, M=M, K=K,
                tensor_sf=tensor_sf_from_amax(_amax_bits(x)))


def config_dense_mx_wide(seed: int = 2, M: int = 16384, K: int = 4096, fmt: str = "mxfp8") -> dict:
    """MXFP8 / MXFP4 dense, M=16384 K=4096: N(0,1) x LogNormal(0,2) per 32-block."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = dense_activations(rng, M, K, "blocklognormal")
    return dict(name=f"{fmt}_dense_M{M}_K{K}", fmt=fmt, x_bits=x, M=M, K=K,
                tensor_sf=np.float32(1.0))


def zipf_topk_routing(rng: np.random.Generator, tokens: int, num_experts: int,
                      top_k: int, zipf_s: float = 1.1) -> np.ndarray:
    """Route each token to ``top_k`` distinct experts, drawn without
    replacement with popularity p(rank r) ~ r^-zipf_s; ranks are mapped to
    expert ids by a random permutation.  Returns int32 (tokens, top_k)."""
    p = np.arange(1, num_experts + 1, dtype=np.float64) ** (-zipf_s)
    p /= p.sum()
    perm = rng.permutation(num_experts)
    out = np.empty((tokens, top_k), dtype=np.int32)
    for t in range(tokens):
        out[t] = perm[rng.choice(num_experts, size=top_k, replace=False, p=p)]
    return out


def grouped_workload(rng: np.random.Generator, x_bits: np.ndarray, routes: np.ndarray,
                     num_experts: int, tile_rows: int = 128) -> dict:
    """Sort routed (token, expert) pairs by expert and build the grouped
    metadata: one group per active expert (increasing id), destination rows
    contiguous per group, ``row_indices[dst] = token``, ``row_offsets`` the
    row prefix sums, ``scales_offsets`` the prefix sums of the counts rounded
    up to ``tile_rows``, and the per-expert ``sf[e] = 448*6/amax`` over the
    expert's gathered rows (1.0 for inactive experts)."""
    tokens, top_k = routes.shape
    flat_e = routes.reshape(-1)
    flat_t = np.repeat(np.arange(tokens, dtype=np.int32), top_k)
    order = np.lexsort((flat_t, flat_e))          # by expert, then token
    e_sorted = flat_e[order]
    row_indices = flat_t[order].astype(np.int32)
    counts = np.bincount(e_sorted, minlength=num_experts)
    active = np.nonzero(counts)[0].astype(np.int32)
    m = counts[active].astype(np.int64)
    row_offsets = np.concatenate([[0], np.cumsum(m)]).astype(np.uint32)
    padded = (m + tile_rows - 1) // tile_rows * tile_rows
    scales_offsets = np.concatenate([[0], np.cumsum(padded)]).astype(np.uint32)
    sf = np.ones(num_experts, dtype=np.float32)
    xf = bf16_bits_to_f32(x_bits)
    for g, e in enumerate(active):
        rows = row_indices[row_offsets[g]:row_offsets[g + 1]]
        sf[e] = tensor_sf_from_amax(np.abs(xf[rows]).max() if rows.size else 0.0)
    return dict(row_indices=row_indices, row_offsets=row_offsets,
                scales_offsets=scales_offsets, expert_ids=active, sf_tensor=sf,
                G=int(active.size), total_rows=int(row_offsets[-1]),
                total_scale_rows=int(scales_offsets[-1]), num_experts=num_experts)


def config_grouped_prefill(seed: int = 3, tokens: int = 4096, K: int = 7168,
                           num_experts: int = 256, top_k: int = 8, fmt: str = "nvfp4") -> dict:
    """Grouped prefill: ``tokens`` x K N(0,1) tokens, top-8 over 256 experts
    with Zipf(1.1) popularity, row_indices gather from the token matrix."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = dense_activations(rng, tokens, K, "normal")
    routes = zipf_topk_routing(rng, tokens, num_experts, top_k)
    d = grouped_workload(rng, x, routes, num_experts)
    d.update(name=f"{fmt}_grouped_prefill_T{tokens}_K{K}", fmt=fmt, x_bits=x,
             in_rows=tokens, K=K, routes=routes)
    return d


def config_grouped_decode(seed: int = 4, tokens: int = 64, K: int = 7168,
                          num_experts: int = 256, top_k: int = 8, fmt: str = "nvfp4") -> dict:
    """Grouped decode: 64 tokens top-8 over 256 experts (average rows per
    active expert <= 8, many 1-row experts), row_indices gather."""
    d = config_grouped_prefill(seed=seed, tokens=tokens, K=K, num_experts=num_experts,
                               top_k=top_k, fmt=fmt)
    d["name"] = f"{fmt}_grouped_decode_T{tokens}_K{K}"
    return d
