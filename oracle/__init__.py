"""CPU float64 oracle of the Muon step -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  It shares no code with the CUDA path.
"""

from .muon_oracle import (  # noqa: F401
    NS5_COEFFS,
    NS5_EPS,
    NS5_STEPS,
    apply_update,
    frobenius_normalise,
    momentum_buffer_update,
    muon_step,
    muon_step_batched,
    nesterov_blend,
    newton_schulz5,
    newton_schulz5_batched,
    rescale_factor,
)
from .adam_oracle import ADAM_BETAS, ADAM_EPS, ADAM_LR, adam_step  # noqa: F401,E402
