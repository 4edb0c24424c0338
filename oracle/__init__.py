"""fp64 CPU oracle for speculative-decoding verification -- test infrastructure only.

Importable by tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg; never by
the product package.
"""
from .specdec_oracle import *  # noqa: F401,F403
from .specdec_oracle import (  # noqa: F401
    GREEDY_T, STATUS_BAD_LOGIT, STATUS_EMPTY_ROW, STATUS_BAD_TOKEN, STATUS_BAD_PROB,
    STATUS_BAD_UNIFORM, STATUS_BAD_TREE, STATUS_BAD_TEMPERATURE, STATUS_ZERO_Q, STATUS_ZERO_RESIDUAL,
    STATUS_ERROR_MASK,
)
