"""CPU oracle for the DFlash drafter pass: TEST INFRASTRUCTURE.

Imported only by the tests, the smoke check and the bench's CPU baseline leg.
It shares no code with the CUDA library.
"""
from .dflash_oracle import *  # noqa: F401,F403
from .dflash_oracle import OracleDrafter  # noqa: F401
