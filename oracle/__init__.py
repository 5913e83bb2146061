"""Oracle of the multi-tenant LoRA layer: TEST INFRASTRUCTURE ONLY.

A plain float64 CPU restatement of the layer, written from the EpiLoRA and
PreFT pages. The CUDA library never imports it; only tests, the smoke check
and the benchmark's CPU baseline do. Parity pins: see tests/test_oracle_*.py.
"""
from . import epilora_oracle, fpformats  # noqa: F401
from .epilora_oracle import *  # noqa: F401,F403
