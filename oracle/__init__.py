"""Float64 CPU oracle of the Moshi/PersonaPlex per-frame decode step.

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the bench's CPU-baseline leg
use it to check and to time against; the library never imports it.
"""
from .oracle import Oracle, OracleStream, build, lib  # noqa: F401
