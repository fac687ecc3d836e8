"""GB300 (sm_103a) routed-MoE NVFP4 (W4A16) prefill: thin Python binding of the C ABI.

The compute path is the CUDA library built from ``csrc/`` (``build.py``); this package only
marshals torch tensors into its C calls (``_lib``) and offers a small host-side helper to
upload NVFP4 weights (``weights``).
"""

from ._lib import *  # noqa: F401,F403
from ._lib import MoeError, load  # noqa: F401
