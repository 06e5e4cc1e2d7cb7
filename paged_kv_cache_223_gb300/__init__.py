"""GB300 (sm_103a) paged-attention decode: a C-ABI CUDA library and its Python binding.

The library (csrc/, built into _lib/libpagedattn.so) implements the cache-write scatter,
the block-table gather, the GQA head-group decode, the causal multi-token verify and the
split-context log-sum-exp merge. `pagedattn` is the ctypes binding.
"""
from .pagedattn import (PA_BF16, PA_FP16, PA_OK, PA_ERR_CUDA, PA_ERR_DEVICE_BOUNDS, PA_ERR_INVALID_ARG,  # noqa: F401
                        PA_ERR_OOM, PA_ERR_TIMEOUT, PA_ERR_UNSUPPORTED, PagedAttnError, Pool, lib, status_string)
