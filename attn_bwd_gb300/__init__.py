"""attn_bwd_gb300: exact softmax attention backward for GB300 (sm_103a).

The C ABI lives in ``include/fa.h``; ``_lib`` binds it with the same names,
``torch_api`` wraps it for torch tensors, ``inputs`` draws seeded workloads,
and ``build`` compiles the CUDA library in-tree.  Importing the package does
not load the library; the first call does, and fails loudly if it is missing.
"""
from ._lib import (FA_BF16, FA_F16, FA_OK, fa_bwd, fa_bwd_dq, fa_bwd_main, fa_bwd_preprocess,  # noqa: F401
                   fa_bwd_workspace_size, fa_fwd, fa_last_device_error, fa_selftest_wait_timeout, fa_strerror)
