"""Float64 CPU oracle for the Muon step (test infrastructure only; the CUDA
library never imports it)."""
from .muon_ref import *  # noqa: F401,F403
from .muon_ref import (DEFAULT_COEFFS, DEFAULT_EPS, DEFAULT_STEPS,  # noqa: F401
                       SCALE_ONE, SCALE_RMS_0P2_SQRT_MAXDIM,
                       SCALE_SQRT_MAX1_R_OVER_C)
