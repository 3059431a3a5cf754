"""The C-ABI library builds, loads and exports every symbol its header
declares; host-side argument checks reject bad calls before any launch.
No GPU is needed: every call here fails validation (or has nothing to do)
before the library touches the CUDA runtime."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "paged_kv.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_decode_tables_gb300 import _build
    try:
        _build.nvcc_path()
    except RuntimeError:
        pytest.skip("no CUDA toolkit")
    _build.build()
    import paged_kv_decode_tables_gb300 as pkv
    return pkv.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+char\s*\*|pkv_status_t|size_t)\s*(\w+)\s*\(", text, flags=re.M)
    return names


def test_header_declares_the_five_operations():
    names = declared_functions()
    for n in ("paged_attention_decode", "paged_attention_v2_partition", "paged_attention_v2_reduce",
              "copy_page_indices", "compute_num_kv_splits"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import paged_kv_decode_tables_gb300 as pkv
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", pkv.lib_path()], capture_output=True,
                         text=True)
    if out.returncode == 0:
        exported = set(line.split()[-1] for line in out.stdout.splitlines() if line.strip())
        for n in names:
            assert n in exported, n


def test_struct_layout_matches_binding(lib):
    import paged_kv_decode_tables_gb300 as pkv
    assert lib.pkv_decode_args_size() == ctypes.sizeof(pkv.DecodeArgs)
    assert "sm_103a" in pkv.version()
    assert lib.pkv_status_string(0) == b"ok"
    assert lib.pkv_status_string(2).startswith(b"unsupported")


def _args(**kw):
    import paged_kv_decode_tables_gb300 as pkv
    a = pkv.DecodeArgs()
    a.num_seqs, a.num_heads, a.num_kv_heads, a.head_size = 2, 8, 2, 128
    a.block_size, a.x, a.max_blocks_per_seq, a.num_blocks = 16, 8, 4, 32
    a.dtype, a.scale = 2, 0.1
    a.query = a.key_cache = a.value_cache = 0x1000
    a.block_tables = a.seq_lens = 0x2000
    a.k_stride[:] = [2 * 16 * 16 * 8, 16 * 16 * 8, 16 * 8, 8, 1]
    a.v_stride[:] = [2 * 128 * 16, 128 * 16, 16, 1]
    a.q_stride[:] = [8 * 128, 128, 1]
    a.bt_stride[:] = [4, 1]
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def _decode(lib, a, out=0x3000):
    strides = (ctypes.c_int64 * 3)(8 * 128, 128, 1)
    return lib.paged_attention_decode(out, strides, ctypes.byref(a) if a is not None else None, None)


@pytest.mark.parametrize("field,value,status", [
    ("num_heads", 7, 1),        # not a multiple of num_kv_heads
    ("x", 4, 1),                # x * sizeof(bf16) != 16
    ("head_size", 96, 2),       # not built
    ("block_size", 24, 2),      # not built
    ("num_kv_heads", 1, 1),     # grid limit on kv heads x query-head sub-groups (below)
    ("query", None, 1),         # null pointer
    ("seq_lens", None, 1),
    ("num_blocks", 0, 1),
    ("dtype", 7, 1),
    ("scale", float("nan"), 1),
])
def test_decode_rejects_bad_arguments(lib, field, value, status):
    if field == "num_kv_heads":
        a = _args(num_heads=40000 * 9, num_kv_heads=40000)  # 40000 kv heads x 2 sub-groups
        assert _decode(lib, a) == 2
        return
    a = _args(**{field: value})
    assert _decode(lib, a) == status


def test_decode_rejects_noncontiguous_pages_and_misalignment(lib):
    a = _args()
    a.k_stride[3] = 16  # x-groups not packed
    assert _decode(lib, a) == 2
    a = _args()
    a.v_stride[3] = 2
    assert _decode(lib, a) == 2
    a = _args(key_cache=0x1008)  # not 16-byte aligned
    assert _decode(lib, a) == 1
    a = _args()
    a.k_stride[0] = a.k_stride[0] + 4  # 8-byte block stride
    assert _decode(lib, a) == 1
    assert _decode(lib, None) == 1
    assert _decode(lib, _args(), out=0) == 1


def _fp8_args(**kw):
    """Valid arguments for a bf16-query decode over an fp8 cache (x = 16)."""
    a = _args(kv_cache_dtype=1, k_scale=0.5, v_scale=2.0, x=16)
    a.k_stride[:] = [2 * 8 * 16 * 16, 8 * 16 * 16, 16 * 16, 16, 1]
    a.v_stride[:] = [2 * 128 * 16, 128 * 16, 16, 1]
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_fp8_cache_and_alibi_argument_checks(lib):
    assert _decode(lib, _fp8_args(num_seqs=0)) == 0        # valid, nothing to do
    assert _decode(lib, _fp8_args(kv_cache_dtype=3)) == 1   # unknown cache format
    assert _decode(lib, _fp8_args(dtype=0)) == 2            # fp32 queries over fp8: not built
    assert _decode(lib, _fp8_args(k_scale=float("inf"))) == 1
    assert _decode(lib, _fp8_args(v_scale=float("nan"))) == 1
    assert _decode(lib, _fp8_args(x=8)) == 1                # x * 1 byte != 16
    a = _fp8_args()
    a.k_stride[0] += 8                                      # 8-byte block stride
    assert _decode(lib, a) == 1
    assert _decode(lib, _args(alibi_slopes=0x2002)) == 1    # slopes not 4-byte aligned
    assert _decode(lib, _args(num_seqs=0, alibi_slopes=0x2004)) == 0
    # auto caches ignore the scales, even non-finite ones
    assert _decode(lib, _args(num_seqs=0, k_scale=float("nan"))) == 0


def test_empty_batch_is_a_no_op(lib):
    assert _decode(lib, _args(num_seqs=0)) == 0
    assert lib.copy_page_indices(0, 0, 0, 0, 0, 0, 0, 0, None, None) == 0


def test_partition_rejects_bad_partitioning(lib):
    a = _args()
    p = 0x4000
    # partition size not a multiple of block_size
    assert lib.paged_attention_v2_partition(p, p, p, 4, 24, None, ctypes.byref(a), None) == 1
    # too few partitions for max_blocks_per_seq * block_size = 64 tokens at P = 16
    assert lib.paged_attention_v2_partition(p, p, p, 3, 16, None, ctypes.byref(a), None) == 1
    assert lib.paged_attention_v2_partition(0, p, p, 4, 16, None, ctypes.byref(a), None) == 1
    assert lib.paged_attention_v2_partition(p, p, p, 0, 16, None, ctypes.byref(a), None) == 1


def test_noalloc_scratch_bound_cannot_overflow(lib):
    """The no-allocation entry point refuses a request beyond its fixed array
    before enqueuing anything, however large the head and partition counts:
    32768 seqs x 2^17 heads x 2^30 partitions is 2^62 rows, whose byte count
    wraps to 0 in 64-bit arithmetic."""
    out, s = 0x3000, (ctypes.c_int64 * 3)(1, 1, 1)
    splits = 0x5000  # split counts given: no partition-size rule applies
    a = _args(num_seqs=1 << 15, num_heads=1 << 17, num_kv_heads=1 << 14)
    st = lib.paged_attention_v2_noalloc(out, s, 1 << 30, 0, splits, ctypes.byref(a), None)
    assert st == 4  # PKV_ERR_SCRATCH_TOO_SMALL
    # each factor alone beyond the array
    for kw, parts in (({"num_seqs": 65535}, 1024), ({"num_heads": 65535 * 8, "num_kv_heads": 65535},
                                                    1), ({}, (1 << 31) - 1)):
        st = lib.paged_attention_v2_noalloc(out, s, parts, 0, splits, ctypes.byref(_args(**kw)),
                                            None)
        assert st == 4, kw


def test_noalloc_checks_arguments_before_its_scratch_size(lib):
    """A malformed call gets the partition pass's own status (not a
    scratch-size refusal), even when its sizes would also overflow the array."""
    out, s, splits = 0x3000, (ctypes.c_int64 * 3)(1, 1, 1), 0x5000
    huge = 1 << 30
    assert lib.paged_attention_v2_noalloc(out, s, huge, 0, splits,
                                          ctypes.byref(_args(head_size=96)), None) == 2
    assert lib.paged_attention_v2_noalloc(out, s, huge, 0, splits,
                                          ctypes.byref(_args(num_seqs=70000)), None) == 2
    assert lib.paged_attention_v2_noalloc(out, s, huge, 0, splits,
                                          ctypes.byref(_args(query=None)), None) == 1
    # fixed partitions: partition size not a multiple of block_size
    assert lib.paged_attention_v2_noalloc(out, s, huge, 24, None, ctypes.byref(_args()),
                                          None) == 1
    assert lib.paged_attention_v2_noalloc(out, s, 0, 0, splits, ctypes.byref(_args()), None) == 1
    assert lib.paged_attention_v2_noalloc(0, s, 4, 0, splits, ctypes.byref(_args()), None) == 1
    # an empty batch is a no-op, whatever it would need
    assert lib.paged_attention_v2_noalloc(out, s, huge, 0, splits,
                                          ctypes.byref(_args(num_seqs=0)), None) == 0


def test_reduce_and_metadata_reject_bad_arguments(lib):
    s = (ctypes.c_int64 * 3)(1, 1, 1)
    p = 0x4000
    assert lib.paged_attention_v2_reduce(p, s, p, p, p, p, None, 2, 8, 96, 16, 4, 512, 2, None,
                                         None) == 2
    assert lib.paged_attention_v2_reduce(p, s, p, p, p, p, None, 2, 8, 128, 16, 0, 512, 2, None,
                                         None) == 1
    assert lib.paged_attention_v2_reduce(p, s, p + 4, p, p, p, None, 2, 8, 128, 16, 4, 512, 2,
                                         None, None) == 1
    assert lib.compute_num_kv_splits(p, p, 0, 1, 32, 8, 16, 148, None) == 1
    assert lib.compute_num_kv_splits(p, p, 4, 1, 4, 8, 16, 148, None) == 1
    assert lib.compute_num_kv_splits(p, p, 4, 1, 32, 8, 0, 148, None) == 1
    assert lib.compute_num_kv_splits(p, p, 4, 1, 32, 8, 16, 0, None) == 1
    assert lib.copy_page_indices(0, 10, p, 4, 4, 1, p, 2, None, None) == 1
    assert lib.prepare_decode_metadata(p, 10, p, 4, 4, 1, p, 0, p, p, 1, 32, 8, 16, 148, None,
                                       None) == 1
    assert lib.prepare_decode_metadata(p, 10, p, 4, 4, 1, p, 2, p, p, 1, 8, 32, 16, 148, None,
                                       None) == 1
    import paged_kv_decode_tables_gb300 as pkv
    m = pkv.DecodeMetadataArgs()
    m.batch_size, m.max_seq_pages, m.page_size = 2, 4, 3  # page size not a power of two
    m.seq_lens = m.cache_seqlens = m.cu_seqlens_k = m.req_to_token = p
    m.req_pool_indices = m.page_table = p
    assert lib.normal_decode_set_metadata(ctypes.byref(m), None) == 1
    m.page_size = 16
    m.swa_page_table = p  # without a mapping
    assert lib.normal_decode_set_metadata(ctypes.byref(m), None) == 1
    m.swa_page_table = None
    m.batch_size = 0
    assert lib.normal_decode_set_metadata(ctypes.byref(m), None) == 1
    assert lib.normal_decode_set_metadata(None, None) == 1
    assert lib.pkv_set_wait_limit_ns(61 * 10 ** 9) == 1
    assert lib.pkv_set_wait_limit_ns(0) == 0
    assert lib.pkv_test_set_unarrived_bytes(17) == 1
    assert lib.pkv_test_set_unarrived_bytes(0) == 0
    assert lib.pkv_set_attention_warps(3) == 1
    assert lib.pkv_set_attention_warps(0) == 0
    assert lib.pkv_set_fp8_kernel(2) == 1
    assert lib.pkv_set_fp8_kernel(-1) == 1
    assert lib.pkv_set_fp8_kernel(0) == 0
    assert lib.pkv_set_split_fold(3) == 1
    assert lib.pkv_set_split_fold(-1) == 1
    assert lib.pkv_set_split_fold(0) == 0
    assert lib.pkv_set_split_fold(2) == 0
    assert lib.pkv_set_split_fold(1) == 0
    assert lib.pkv_order_by_length(p, p, -1, None) == 1
    assert lib.pkv_order_by_length(None, p, 4, None) == 1
    assert lib.pkv_order_by_length(p, None, 4, None) == 1
    assert lib.pkv_order_by_length(None, None, 0, None) == 0


def test_binding_refuses_host_tensors():
    import torch

    import paged_kv_decode_tables_gb300 as pkv
    q = torch.zeros(1, 1, 64)
    with pytest.raises(ValueError):
        pkv.paged_attention_decode(q, q, torch.zeros(1, 1, 16, 8, 4), torch.zeros(1, 1, 64, 8),
                                   torch.zeros(1, 1, dtype=torch.int32),
                                   torch.zeros(1, dtype=torch.int32), 0.1)


def test_binding_resolves_the_cache_format():
    """kv_cache_dtype names and float8 tensor types map to pkv_kv_cache_dtype_t;
    contradictions and wrong element types are refused (host-side only)."""
    import torch

    import paged_kv_decode_tables_gb300 as pkv
    q = torch.zeros(1, 1, 16, dtype=torch.bfloat16)
    u8 = torch.zeros(1, 1, 1, 4, 16, dtype=torch.uint8)
    e4 = u8.view(torch.float8_e4m3fn)
    e5 = u8.view(torch.float8_e5m2)
    bf = torch.zeros(1, 1, 2, 4, 8, dtype=torch.bfloat16)
    assert pkv._kv_cache_code(bf, bf, q, "auto") == 0
    assert pkv._kv_cache_code(u8, u8, q, "fp8") == 1
    assert pkv._kv_cache_code(u8, u8, q, "fp8_e4m3") == 1
    assert pkv._kv_cache_code(u8, u8, q, "fp8_e5m2") == 2
    assert pkv._kv_cache_code(e4, e4, q, "auto") == 1
    assert pkv._kv_cache_code(e5, e5, q, "auto") == 2
    assert pkv._kv_cache_code(e5, e5, q, "fp8_e5m2") == 2
    with pytest.raises(ValueError):
        pkv._kv_cache_code(e4, e4, q, "fp8_e5m2")      # contradicts the tensor type
    with pytest.raises(ValueError):
        pkv._kv_cache_code(u8, u8, q, "auto")          # codes need a format name
    with pytest.raises(ValueError):
        pkv._kv_cache_code(bf, bf, q, "fp8")           # fp8 caches are codes
    with pytest.raises(ValueError):
        pkv._kv_cache_code(u8, u8, q, "int8")          # unknown name
    with pytest.raises(ValueError):
        pkv._kv_cache_code(u8, e4, q, "fp8")           # key and value differ
