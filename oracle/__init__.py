"""CPU oracle (test infrastructure only; see exq_oracle's header).

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline and
reference legs may import this package. The product path never does.
"""
from .exq_oracle import *  # noqa: F401,F403
