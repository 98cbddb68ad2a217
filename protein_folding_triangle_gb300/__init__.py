"""libtriattn: triangular (pair-biased, slice-batched) attention forward and
backward on NVIDIA GB300 (sm_103a), behind a C ABI (include/triattn.h), with
the triangle-attention module around it and the triangle multiplicative
update.

``triattn`` is the ctypes binding, ``build`` compiles the CUDA library
in-tree, ``synthetic`` draws seeded inputs, ``sharding`` splits the outer axis
across GPUs or into memory-bounded chunks on one GPU, ``layers`` wraps the
module and the multiplicative update as autograd functions and torch modules.
"""
from . import build, synthetic, triattn  # noqa: F401
from .triattn import (TriAttnError, bwd_workspace_bytes, device_status, set_wait_limit_ns,  # noqa: F401
                      tri_attn_bwd, tri_attn_fwd, tri_attn_module_bwd, tri_attn_module_fwd, triangle_attention,
                      triattn_trimul_bwd, triattn_trimul_fwd)
