"""CPU oracle of the MSA hot path (test infrastructure only; see msa_oracle)."""
from . import msa_oracle  # noqa: F401
