"""Oracle package: test infrastructure only (see flce_oracle's docstring)."""
from .flce_oracle import (REDUCTIONS, ce_reference, flce_reference, flce_rows,  # noqa: F401
                          full_logits_bytes, grad_weight_rows, lse_rows, widen)
