"""Parity helpers for the tests: see oracle/parity.py for the tolerances."""
import numpy as np

from oracle.parity import (BF16_REL, FP32_ATOL, bf16_ulp, check_bf16, check_fp32,  # noqa: F401
                           h_norm_allowance, y_allowance, _bits as bits)
