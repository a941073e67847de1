"""fp64 CPU oracle for routing attention -- test infrastructure only.

Imported by the test suite, the package smoke check and the benchmark's CPU
baseline leg; never by the library.
"""

from .routing_oracle import *  # noqa: F401,F403
