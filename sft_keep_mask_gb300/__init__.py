"""GB300-native fused LM-head scoring with keep-mask compaction.

The compute path is the CUDA library ``_lib/liblmhead.so`` (sources in
``csrc/``, C ABI in ``include/lmhead.h``); ``lmhead`` is its thin ctypes
binding, ``api`` a small convenience layer that allocates outputs and the
workspace with torch, and ``autograd`` the op ``hidden_to_logprobs`` (forward
and backward through the library under torch autograd).  ``synth`` draws
seeded synthetic inputs.
"""

from .autograd import hidden_to_logprobs  # noqa: F401

from .lmhead import (  # noqa: F401
    DEFAULT_CHUNK_ROWS,
    LmheadError,
    lmhead_build_keep_mask,
    lmhead_bwd,
    lmhead_bwd_blocksparse,
    lmhead_bwd_shard,
    lmhead_compact,
    lmhead_expand,
    lmhead_fwd,
    lmhead_fwd_blocksparse,
    lmhead_fwd_shard,
    lmhead_get_status,
    lmhead_get_timeout_record,
    lmhead_launch_count,
    lmhead_merge_shards,
    lmhead_profile_enable,
    lmhead_profile_read,
    lmhead_selective_log_softmax_bwd,
    lmhead_selective_log_softmax_fwd,
    lmhead_strerror,
    lmhead_version,
    lmhead_workspace_size,
)
