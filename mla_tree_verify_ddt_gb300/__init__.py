"""GB300-native DDTree verify step (libddtree) — Python binding.

The hot path lives in libddtree.so (CUDA for sm_103a, C ABI in
include/ddtree.h); ``ddtree`` marshals torch tensors into it.
"""
from . import ddtree  # noqa: F401
from .ddtree import (VerifyStep, ddt_read_device_status, ddt_selftest_bounded_wait,  # noqa: F401
                     ddt_tree_accept, ddt_tree_build, ddt_verify_mla_attn, ddt_workspace_size)
