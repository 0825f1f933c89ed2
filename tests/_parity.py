"""The parity rules (oracle/parity.py), under the name the tests import."""
from oracle.parity import (LOGPROB_ATOL, MARGIN, ParityReport, check_structure,  # noqa: F401
                           compare)
