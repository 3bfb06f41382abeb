"""fp64 CPU oracle for the Muon step (test infrastructure; see muon_oracle)."""
from .muon_oracle import *  # noqa: F401,F403
