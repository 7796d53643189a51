"""Paged-KV decode attention for GB300 (sm_103a).

The product is the C-ABI library ``libpa.so`` (``include/pa.h``); ``capi``
binds it for torch tensors.  ``workload`` draws seeded synthetic inputs.
"""
from .capi import (PAError, lib, pa_copy_blocks, pa_copy_blocks_workspace_bytes, pa_decode,  # noqa: F401
                   pa_decode_partition_tokens,
                   pa_decode_noalloc, pa_decode_shared_prefix, pa_decode_shared_prefix_workspace_bytes,
                   pa_decode_workspace_bytes, pa_decode_step_host, pa_decode_step_host_staging_bytes,
                   pa_mixed_step, mixed_workspace, pa_prefill_batch, pa_prefill_chunk, pa_prefill_workspace_bytes,
                   prefill_workspace, pa_reshape_and_cache,
                   pa_selftest_bounded_wait,
                   pa_status_string, decode_workspace)
from .block_manager import BlockManager  # noqa: F401,E402
