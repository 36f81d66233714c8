"""CPU oracle for attention-score-driven KV-cache compression (test infrastructure).

Plain numpy in float64.  Only the test suite, the package smoke check and the benchmark's
CPU-baseline arm import this package; the library's product path never does, and this
package imports nothing from it.  See ``kvc_oracle`` for the definitions and citations.
"""
from .kvc_oracle import *  # noqa: F401,F403
