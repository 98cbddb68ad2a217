"""libtriattn: triangular (pair-biased, slice-batched) attention forward and
backward on NVIDIA GB300 (sm_103a), behind a C ABI (include/triattn.h).

``triattn`` is the ctypes binding, ``build`` compiles the CUDA library
in-tree, ``synthetic`` draws seeded inputs.
"""
from . import build, synthetic, triattn  # noqa: F401
from .triattn import (TriAttnError, bwd_workspace_bytes, device_status, set_wait_limit_ns,  # noqa: F401
                      tri_attn_bwd, tri_attn_fwd, triangle_attention)
