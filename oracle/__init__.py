"""CPU oracle for paged-KV decode: TEST INFRASTRUCTURE.

Plain, slow float64 (and integer) restatements of what the decode path
computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline leg may import it; the CUDA library shares no code with it and never
calls it.  Each function cites the passage of the pages it follows.
"""
from . import fp8  # noqa: F401
from .attention import (  # noqa: F401
    alibi_bias,
    attention_one_head,
    decode_v1,
    gather_kv,
    partition_ranges,
    sequence_block_ids,
    split_chunk_size,
    token_offsets,
    v2_partition,
    v2_reduce,
)
from .metadata import (  # noqa: F401
    cdiv,
    copy_page_indices,
    cu_num_pages,
    decode_set_metadata,
    ext_device_core_count,
    log2_f32,
    num_kv_splits,
    swa_spec_page_table,
    wrap_int32,
)
