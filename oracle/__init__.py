"""Plain CPU oracle for grouped microscaled (MX) and blockwise-FP8 GEMMs.

TEST INFRASTRUCTURE ONLY.  Nothing in the library (``fp8_bf16_mxfp4_gb300``)
imports, links or calls this package; only ``tests/``, the smoke check and the
bench's CPU-baseline leg do.  It shares no code, table or constant generator
with the CUDA path.

Everything here is written for clarity, not speed: NumPy in float64 (float32
where the method itself fixes fp32 arithmetic), one library matmul per expert,
no blocking or fusion.  Each function cites the passage it follows:

* "Triton mxfp4 (and a8w4) grouped GEMM kernel" (ROCm TransformerEngine PR
  #723): the grouped forward / dgrad / variable-K wgrad passes, split checks,
  and the segment-padded columnwise wgrad operand.
* ROCm TransformerEngine PR #745 (MXFP4 / a8w4 GroupedLinear): the a8w4 mix,
  the MXFP8 E4M3 reference quantizer, and the review "Clamp tiny block scales
  to preserve nonzero values" (scale exponent clamped at -127).
* "Add ROCm Triton blockwise FP8 grouped GEMM" (PR #716): 1x128 / 128x128
  blockwise FP8 with amax clamped to 1e-4 and the segment-padded colwise
  operand.
* "Integrate MXFP4 hipblaslt GEMM support" (PR #697): the per-pass shapes
  (forward contracts hidden, dgrad contracts out, wgrad contracts tokens).
* "Integrate MXFP4 hipblaslt GEMM support" (PR #697), Takeaways, and the
  "fused scale packing kernel" commit of "Grouped MXFP8 GEMMs with
  HipKittens" (PR #661): MX scales written in the
  matrix engine's blocked order (``oracle.packed``).
* The OCP Microscaling Formats (MX) v1.0 specification for the E2M1 / E4M3
  element encodings and the shared-exponent rule.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against hand-worked blocks, a second scalar formulation, exhaustive BF16
sweeps, exact rational arithmetic and algebraic invariants.
"""

from .mx import (  # noqa: F401
    E2M1_MAGNITUDES,
    e4m3_magnitudes,
    decode,
    round_to_grid,
    shared_exponent,
    quantize_mx,
    dequantize_mx,
    pack_e2m1,
    unpack_e2m1,
    quantize_mx_rowwise,
    quantize_mx_colwise_segment_padded,
    padded_offsets,
)
from .blockwise import (  # noqa: F401
    quantize_bw_1x128,
    quantize_bw_128x128,
    quantize_bw_colwise_padded,
    dequantize_bw_1x128,
    dequantize_bw_128x128,
    transpose_bw_128x128,
    pow2_scale,
)
from .packed import (  # noqa: F401
    tile_prefix,
    packed_scale_bytes,
    pack_scales_mma,
    pack_scales_mma_by_tiles,
    kseg_chunk_prefix,
    pack_scales_mma_kseg,
    pack_scales_mma_kseg_by_experts,
)
from .gemm import (  # noqa: F401
    check_splits,
    grouped_fwd,
    grouped_dgrad,
    grouped_wgrad,
    tolerance_violation,
    assert_gemm_close,
    fp64_sum_is_exact,
)
