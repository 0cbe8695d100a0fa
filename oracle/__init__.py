"""CPU oracle for the AdaHOP MXFP4 linear layer.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference leg of ``bench.py``; never by the product package.
"""
from . import adahop_oracle  # noqa: F401
from .adahop_oracle import *  # noqa: F401,F403
