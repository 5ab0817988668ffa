"""GB300 (sm_103a) Mixture-of-Experts decode-layer forward.

The compute is the C-ABI library ``libmoe_gb300.so`` (``include/moe.h``);
``binding`` is its ctypes binding, ``layer.MoeLayer`` a thin holder of weights
and workspace, ``synth`` the seeded synthetic inputs.
"""
from . import binding  # noqa: F401
