"""GB300-native hot path of DFlash-style block-diffusion speculative drafting.

Python binding of libdflash (include/dflash.h): argument marshalling only.
Every step of the path runs in the library's sm_103a kernels; PyTorch
provides device memory and streams. There is no CPU fallback: importing this
package fails if the library is not built.

    from block_diffusion_speculative_tap_gb300 import Drafter, topk, verify_greedy
"""
from .drafter import (  # noqa: F401
    Drafter,
    State,
    config_validate,
    draft_stop,
    fused_row_bytes,
    kind,
    launch_count,
    select_path,
    tap_row_bytes,
    topk,
    tree_build,
    tree_size,
    tree_verify,
    verify_greedy,
    verify_sample,
)
from ._abi import DFlashError  # noqa: F401
