"""CPU oracle for block-scaled BF16 -> NVFP4 / MXFP4 / MXFP8 quantization.

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow, obviously correct
CPU statement of what the GPU path computes.  Only the test suite, the
package-level ``smoke()`` check and the benchmark's ``cpu_baseline`` leg may
import it; the product path (the CUDA library and its Python binding) never
does, and shares no code, table or helper with it.  Inputs come from the
separate ``workloads`` module.

Sources.  The method is the one the Modular "block_scaled_quantization" pages
describe: quantization of activations to the NVFP4, MXFP4 and MXFP8 block
formats (module page), the NVFP4 kernel that derives one scale per group of
elements and packs the FP4 codes, with an FP32 ``tensor_sf`` argument
("quantize_dynamic_scaled_async_fp4_kernel", description and signature), the
grouped per-expert kernel driven by ``row_offsets``, ``scales_offsets``,
``expert_ids``, ``sf_tensor`` and an optional ``row_indices``
("grouped_quantize_dynamic_scaled_fp4_async_kernel", signature and parameter
list) and the rank-2 -> 5D TCGEN scale reinterleave
("block_scales_interleave", module index).  The pages never define the
element formats, the block-scale formula, the rounding or the 5D layout;
the readings taken are:

* formats: OCP Microscaling v1.0 E2M1, E4M3 (FN: max 448, no Inf), E8M0;
* encode = nearest representable value, ties to the even code, |v| beyond
  the largest finite magnitude saturates to it, the sign bit is kept
  (also for values that round to zero);
* NVFP4 block (16 elements): s = fl32(fl32(amax/6) * tensor_sf) -> E4M3,
  element scale os = 0 if the decoded scale is 0 else fl32(tensor_sf/ds),
  q_i = E2M1(fl32(x_i * os));
* MX block (32 elements): s = fl32(amax/Qmax) (Qmax 6 for E2M1, 448 for
  E4M3), e = ceil(log2 s) clamped to [-127, 127] (e = -127 for s = 0),
  scale byte e+127, q_i = encode(fl32(x_i * 2^-e));
* FP4 packing: element 2k in the low nibble of byte k, 2k+1 in the high;
* 5D TCGEN scale layout (Mt, Kt, 32, 4, 4): byte of (row m, scale column s)
  at ((m/128)*Kt + s/4)*512 + (m%32)*16 + ((m%128)/32)*4 + s%4, padding
  entries of the dense output 0x00;
* tensor scale (computed on the GPU before quantizing): ``tensor_sf =
  fl32(448*6 / amax)``, amax the exact max |x| (per expert over its gathered
  rows), 1.0 for an all-zero tensor;
* grouped: ``row_offsets``/``scales_offsets`` are uint32 prefix sums of
  length G+1 (``scales_offsets`` in rows, multiples of 128), groups with a
  negative expert id are skipped, padding scale rows are not written.

Floating point decides integers here (scale bytes, element codes), so the
scale arithmetic runs in FP32 exactly as the definitions order it (NumPy
float32 operations are IEEE round-to-nearest), and the encoders decide
"nearest" exactly (see ``formats``).

Parity pins: every function here is pinned by the ``-m "not gpu"`` tests
(exhaustive codec sweeps against exact rational brute force and the
torch float8 conversions, hand-worked blocks under ``tests/golden``,
E8M0/NVFP4 invariants and error bounds, an independent reshape statement of
the 5D layout, dense <-> grouped reductions).  No function is unpinned.
"""
from .formats import (E2M1_MAGNITUDES, E4M3_MAGNITUDES, e2m1_decode, e4m3_decode,
                      e8m0_decode, e2m1_encode, e4m3_encode, e8m0_ceil_exponent)
from .blockquant import (FORMATS, block_size, packed_row_bytes, quantize_rank2,
                         quantize, grouped_quantize, dequantize, nvfp4_block_scale,
                         nvfp4_element_scale, mx_block_exponent)
from .layout import (scales5d_bytes, offset_5d, scales_to_5d, scales_interleave,
                     scales_from_5d_view)
from .check import naive_block_scaled_matmul
from .tensor_scale import tensor_sf, expert_tensor_sf

__all__ = [
    "E2M1_MAGNITUDES", "E4M3_MAGNITUDES", "e2m1_decode", "e4m3_decode", "e8m0_decode",
    "e2m1_encode", "e4m3_encode", "e8m0_ceil_exponent", "FORMATS", "block_size",
    "packed_row_bytes", "quantize_rank2", "quantize", "grouped_quantize", "dequantize",
    "scales5d_bytes", "offset_5d", "scales_to_5d", "scales_interleave",
    "scales_from_5d_view", "naive_block_scaled_matmul", "nvfp4_block_scale",
    "nvfp4_element_scale", "mx_block_exponent", "tensor_sf", "expert_tensor_sf",
]
