"""CPU oracle for the DSA forward hot path (test infrastructure only; see
dsa_oracle.py).  Imported by the tests, the smoke check and the bench's CPU
baseline, never by the product package."""
from .dsa_oracle import *  # noqa: F401,F403
