"""CPU oracle (test infrastructure): plain NumPy float64 restatement of the
owner-local Muon step, AdamW and RMNP. Only tests, the smoke check and the
benchmark's CPU-baseline leg import it; the library never does."""
from .oracle import *  # noqa: F401,F403
from .oracle import (NS_COEFFS, NS_EPS, RMNP_EPS, adamw_step, bf16_round, decoupled_update,
                     frobenius_normalize, momentum, muon_matrix_step, muon_table_step,
                     newton_schulz, newton_schulz_pages_form, rmnp_direction, rmnp_matrix_step,
                     rmnp_row_sharded, rmnp_table_step, shape_scale, rmnp_colcut_direction,
                     rmnp_colcut_matrix_step, RMNP_COLCUT_EPS, match_rms_adamw_scale,
                     nesterov_direction, htrmnp_direction, htrmnp_matrix_step, HTRMNP_POWER)
