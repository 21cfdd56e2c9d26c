"""CPU oracle (test infrastructure only): see ``tp_oracle``.  Imported only by
the test suite, the smoke check and the benchmark's CPU baseline leg."""
from .tp_oracle import *  # noqa: F401,F403
