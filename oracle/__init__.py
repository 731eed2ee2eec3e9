"""Float64 CPU oracle for the flash-CCE ORPO head.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may call it.  It shares no code with the CUDA library under
``orpo_preference_loss_gb300/``.
"""

from .orpo_oracle import (  # noqa: F401
    bf16_bits_to_f64,
    log1mexp,
    softcap_value,
    softcap_slope,
    head_forward,
    orpo_loss,
    head_backward,
    head_block_max,
    TILE_ROWS,
    TILE_COLS,
    GROUP_ROWS,
    full_chain,
    pref_loss,
    PREF_KINDS,
    dequant_affine,
    OracleError,
)
