"""FORGE fused weight-gradient + optimizer step for one GB300 (sm_103a).

The compute lives in ``libforge.so`` (hand-written CUDA kernels behind the
C ABI in ``include/forge.h``); this package is its thin Python binding.
"""

from ._lib import (  # noqa: F401
    BF16, EXPORTED, F32, FLAG_BACKWARD_FUSED, FLAG_BACKWARD_SPLIT, FLAG_DGRAD_ALL_TOKENS, FLAG_DGRAD_TOKENS_128,
    FLAG_TEST_FORCE_TIMEOUT, FLAG_TILE_N_64,
    FLAG_TILE_N_128, FLAG_TILE_N_256, FLAG_TILE_N_AUTO, FLAG_TILE_PAIR_256, I8B128, LIB_PATH, RULES, ForgeError, backward_step,
    backward_accumulate, backward_step_no_alloc, dgrad, lib, sync_status, tensor_desc, version, wgrad_accumulate,
    wgrad_step_accumulated, wgrad_step_adamw, wgrad_step_adagrad, wgrad_step_lion, wgrad_step_nadam,
    wgrad_step_radam, wgrad_step_rmsprop, wgrad_step_sgd, wgrad_step_sgdm, workspace_bytes, selftest_math)
