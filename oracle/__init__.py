"""CPU oracle for MSA block-sparse attention (test infrastructure only; see
msa_oracle's header for who may use it)."""
from .msa_oracle import *  # noqa: F401,F403
