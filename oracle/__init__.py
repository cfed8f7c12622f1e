"""CPU oracle for the TokenGate path: test infrastructure only (see
``oracle/tokengate_oracle.py``).  Imported by ``tests/``, ``__graft_entry__``'s
smoke check and the CPU legs of ``bench.py``, never by the product path."""
from .tokengate_oracle import *  # noqa: F401,F403
from . import model_oracle as model  # noqa: E402,F401
