"""Fusion groups on one GB300: a chain of up to 64 elementwise nodes in one
loop nest, the reduction-rooted softmax region, and the AdamW step over a
parameter tree, each one CUDA launch through a C ABI (include/psk.h).

    from reduction_groups_gb300 import psk_group_run, psk_softmax_region, psk_adamw_tree
"""

from .ops import (  # noqa: F401
    psk_adamw_clip_scale,
    psk_adamw_group_sqsums,
    psk_adamw_lr,
    psk_adamw_scalars,
    psk_adamw_tree,
    psk_adamw_tree_ex,
    psk_adamw_tree_scaled,
    psk_adamw_tree_static,
    psk_adamw_workspace,
    psk_device_status,
    psk_group_check,
    psk_group_prepare,
    psk_group_run,
    psk_group_run_interp,
    psk_norm_region,
    psk_softmax_backward,
    psk_softmax_masked,
    psk_softmax_region,
    psk_test_drop_row,
    psk_test_fast_exp,
)
from ._native import PskError  # noqa: F401
