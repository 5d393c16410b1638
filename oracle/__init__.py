"""fp64 CPU oracle of the fused normalization block, its normalize step fed
by per-tile partial statistics, and the row softmax (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares no code with the CUDA
library and imports nothing from ``normalization_fwd_gb300``.
"""

from .norm import (E4M3_MAX, LAYERNORM, RMSNORM, norm_bwd, norm_fwd, quantize_fp8_e4m3,
                   round_to_e4m3_satfinite, round_to_format)
from .partials import (SUM_M2, SUM_SQ, combine_partials, norm_fwd_from_partials,
                       row_tile_partials, tile_widths)
from .softmax import softmax_fwd

__all__ = ["LAYERNORM", "RMSNORM", "norm_fwd", "norm_bwd", "round_to_format",
           "round_to_e4m3_satfinite", "quantize_fp8_e4m3", "E4M3_MAX", "softmax_fwd",
           "SUM_SQ", "SUM_M2", "tile_widths", "row_tile_partials", "combine_partials",
           "norm_fwd_from_partials"]
