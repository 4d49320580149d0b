"""CPU oracle for the weight-only quantized GEMV / GEMM path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or link
anything in this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code with the CUDA
library and does not import it.

It is plain and slow on purpose: every weight is dequantised to fp32 with
exactly one rounding of its exact real value, dot products are taken in fp64,
and each result is rounded to bf16 once.  Each function cites the passage of
the source pages it follows:

* "TurboEXL3" article (TurboEXL3: Why EXL3 should be the default model formats
  for modern Macs), §2.1 block-scaled formats, §2.2 W4A16, §4.1 prefill chain,
  §4.2 decode chain, §4.4 numerics.
* "Q6_K operand PR" (perf: Q6_K's zero point in the operands of the Apple7/8
  register decode tile, #19), "What changed" and its commit messages (the 5-bit
  nibble operand of Q5_K, Q5_1 and Q5_0).
* The same article, §2.2: the W4A4 mode, activations quantised to NVFP4 on the fly
  (``act_quant``).

Parity pins for every function live in ``tests/test_oracle_pins.py``.
"""
from .formats import (  # noqa: F401
    e2m1_value, e8m0_value, e4m3fn_value, bf16_value, bf16_bits_of, round_to_bf16, dequant, dequant_rows,
    bits_per_weight, q6k_half_operand_bits, q5_half_operand_bits, dequant_operand_bf16,
)
from .gemv import gemv, gemv_rows, row_norms, tolerance  # noqa: F401
from .moe import route, sigmoid, silu, swiglu_bf16, moe_forward, expert_ffn  # noqa: F401
from .layout import unpack, packed_sizes  # noqa: F401
from .act_quant import e2m1_encode, e4m3_encode, quantize_act_nvfp4, gemm_w4a4  # noqa: F401
