"""Seeded synthetic inputs shared by the oracle checks and the CUDA path.

Holds input recipes only (noise, planted spikes, cost tables, planted target
argmaxes); none of the method's arithmetic lives here.
"""
from .synth import *  # noqa: F401,F403
