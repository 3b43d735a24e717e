"""8-bit block-scaled paged KV cache for GB300: quantize-and-scatter store and split-K decode.

The compute lives in ``libkvq.so`` (CUDA, sm_103a, built from ``csrc/``); ``kvq`` is its ctypes
binding and ``workloads`` the seeded synthetic inputs.
"""
from . import kvq  # noqa: F401
from .kvq import (Layout, KvqError, alloc_pool, alloc_workspace, kvq_bytes_per_token,  # noqa: F401
                  kvq_decode, kvq_decode_workspace_bytes, kvq_dequant_probe, kvq_device_check,
                  kvq_encode_probe, kvq_num_pages, kvq_pool_bytes, kvq_scale_bytes, kvq_store,
                  kvq_version, kvq_workspace_status)

__version__ = "0.1.0"
