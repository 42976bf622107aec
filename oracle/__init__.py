"""CPU oracle for the MXFP8 linear layer: test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library and never imports it.
"""

from .mx_oracle import (BLOCK, block_exponent, dequantize, e4m3_encode, e4m3_value,  # noqa: F401
                        e8m0_value, linear, linear_bf16, quantize, scale_bytes)
from .mx_oracle import (FP6_FORMATS, fp6_emax, fp6_encode, fp6_max, fp6_value,  # noqa: F401,E402
                        quantize_fp6)
