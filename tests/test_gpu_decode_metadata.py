"""GPU fused decode metadata (sglang normal_decode_set_metadata) against the
oracle, bit-exact: page sizes 1..64, with and without the sliding-window
table, strided outputs, wrap-around of the int32 cast, bad indices flagged."""
import pytest
import torch

import oracle
import paged_kv_decode_tables_gb300 as pkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_kv_decode_tables_gb300 import _build
    _build.build()


def _case(B, page_size, msp, pool_rows=None, swa=False, seed=0, delta=1, strided=False):
    g = torch.Generator().manual_seed(seed)
    pool_rows = pool_rows or B + 3
    cols = max(1, msp * page_size)
    rt = torch.randint(0, 1 << 22, (pool_rows, cols), generator=g, dtype=torch.int32)
    pool = torch.randperm(pool_rows, generator=g)[:B].to(torch.int64)
    lens = torch.randint(0, cols + 1, (B,), generator=g, dtype=torch.int64)
    mapping = torch.randint(0, 1 << 30, (1 << 22,), generator=g, dtype=torch.int64)
    dev = "cuda"
    cache = torch.full((B,), -9, dtype=torch.int32, device=dev)
    cu_store = torch.full((2 * (B + 1),), -9, dtype=torch.int32, device=dev)
    cu = cu_store[::2] if strided else cu_store[:B + 1]
    pt_store = torch.full((B, msp + 5), -9, dtype=torch.int32, device=dev)
    pt = pt_store[:, :msp] if msp else pt_store[:, :1]
    swa_t = torch.full((B, max(msp, 1)), -9, dtype=torch.int32, device=dev) if swa else None
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.normal_decode_set_metadata(cache, cu, pt, rt.to(dev), pool.to(dev), lens.to(dev),
                                   seq_len_delta=delta, page_size=page_size, max_seq_pages=msp,
                                   swa_page_table=swa_t,
                                   full_to_swa_mapping=mapping.to(dev) if swa else None,
                                   err_flag=err)
    want = oracle.decode_set_metadata(lens.tolist(), rt, pool.tolist(), msp, delta, page_size,
                                      full_to_swa_mapping=mapping if swa else None)
    return cache, cu, pt, swa_t, err, want, pt_store


@pytest.mark.parametrize("page_size", [1, 2, 16, 64])
@pytest.mark.parametrize("swa", [False, True])
@pytest.mark.parametrize("B,msp", [(1, 1), (5, 300), (37, 513), (300, 64)])
def test_decode_metadata_bit_exact(page_size, swa, B, msp):
    cache, cu, pt, swa_t, err, want, pt_store = _case(B, page_size, msp, swa=swa,
                                                      seed=B + page_size + msp)
    torch.cuda.synchronize()
    assert cache.cpu().tolist() == want[0]
    assert cu.cpu().tolist() == want[1]
    assert pt.cpu().tolist() == want[2]
    if swa:
        assert swa_t.cpu().tolist() == want[3]
    assert bool((pt_store[:, msp:] == -9).all())  # columns past max_seq_pages untouched
    assert int(err.item()) == 0


def test_decode_metadata_strided_indptr_and_many_rows():
    cache, cu, pt, _, err, want, _ = _case(3000, 16, 40, strided=True, seed=3, delta=0)
    assert cu.cpu().tolist() == want[1]
    assert cache.cpu().tolist() == want[0]
    assert pt.cpu().tolist() == want[2]


def test_decode_metadata_int32_wrap_and_zero_pages():
    dev = "cuda"
    lens = torch.tensor([2 ** 31 - 1, 5, 7], dtype=torch.int64, device=dev)
    cache = torch.empty(3, dtype=torch.int32, device=dev)
    cu = torch.empty(4, dtype=torch.int32, device=dev)
    pt = torch.empty(3, 1, dtype=torch.int32, device=dev)
    rt = torch.zeros(1, 1, dtype=torch.int32, device=dev)
    pool = torch.zeros(3, dtype=torch.int64, device=dev)
    pkv.normal_decode_set_metadata(cache, cu, pt, rt, pool, lens, seq_len_delta=1, page_size=1,
                                   max_seq_pages=0)
    want = oracle.decode_set_metadata(lens.tolist(), [[0]], [0, 0, 0], 0, 1, 1)
    assert cache.cpu().tolist() == want[0]
    assert cu.cpu().tolist() == want[1]


def test_decode_metadata_flags_bad_pool_rows():
    dev = "cuda"
    lens = torch.tensor([10, 20], dtype=torch.int64, device=dev)
    rt = torch.arange(16, dtype=torch.int32, device=dev).view(2, 8)
    pool = torch.tensor([1, 5], dtype=torch.int64, device=dev)  # row 5 does not exist
    cache = torch.empty(2, dtype=torch.int32, device=dev)
    cu = torch.empty(3, dtype=torch.int32, device=dev)
    pt = torch.full((2, 4), -1, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.normal_decode_set_metadata(cache, cu, pt, rt, pool, lens, seq_len_delta=0, page_size=2,
                                   err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.PKV_ERRF_INDPTR
    assert pt[0].cpu().tolist() == [4, 5, 6, 7]  # row 1: tokens 8,10,12,14 >> 1
    assert pt[1].cpu().tolist() == [0, 0, 0, 0]


@pytest.mark.parametrize("B,msp", [(3, 4), (5, 300), (2, 4096), (4, 4099), (3, 8195), (600, 37)])
def test_decode_metadata_row_copy_path(B, msp):
    """Page size 1, no sliding-window table, unit-stride 16-byte aligned rows:
    the 16-byte row copy, including a ragged tail inside a padded row."""
    g = torch.Generator().manual_seed(B * 7 + msp)
    width = -(-msp // 4) * 4
    rt = torch.randint(0, 1 << 30, (B + 4, width + 8), generator=g, dtype=torch.int32)
    pool = torch.randperm(B + 4, generator=g)[:B].to(torch.int64)
    lens = torch.randint(0, msp + 1, (B,), generator=g, dtype=torch.int64)
    dev = "cuda"
    cache = torch.empty(B, dtype=torch.int32, device=dev)
    cu = torch.empty(B + 1, dtype=torch.int32, device=dev)
    pt_store = torch.full((B, width + 4), -9, dtype=torch.int32, device=dev)
    pt = pt_store[:, :msp]
    assert pt.stride(0) % 4 == 0 and pt.stride(1) == 1
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.normal_decode_set_metadata(cache, cu, pt, rt.to(dev), pool.to(dev), lens.to(dev),
                                   seq_len_delta=1, page_size=1, max_seq_pages=msp, err_flag=err)
    want = oracle.decode_set_metadata(lens.tolist(), rt, pool.tolist(), msp, 1, 1)
    torch.cuda.synchronize()
    assert cache.cpu().tolist() == want[0]
    assert cu.cpu().tolist() == want[1]
    assert pt.cpu().tolist() == want[2]
    assert bool((pt_store[:, msp:] == -9).all())
    assert int(err.item()) == 0


def test_decode_metadata_row_copy_short_and_bad_rows():
    """Row copy with pool rows narrower than max_seq_pages (columns past the
    width write 0) and a pool index outside the pool (the row writes 0):
    both flagged."""
    dev = "cuda"
    rt = torch.arange(3 * 100, dtype=torch.int32, device=dev).view(3, 100)
    pool = torch.tensor([2, 7, 0], dtype=torch.int64, device=dev)  # 7 is outside the pool
    lens = torch.tensor([5, 6, 7], dtype=torch.int64, device=dev)
    cache = torch.empty(3, dtype=torch.int32, device=dev)
    cu = torch.empty(4, dtype=torch.int32, device=dev)
    pt = torch.full((3, 132), -1, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.normal_decode_set_metadata(cache, cu, pt, rt, pool, lens, seq_len_delta=0, page_size=1,
                                   max_seq_pages=130, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.PKV_ERRF_INDPTR
    got = pt.cpu()
    assert got[0, :100].tolist() == list(range(200, 300)) and got[0, 100:130].tolist() == [0] * 30
    assert got[1, :130].tolist() == [0] * 130
    assert got[2, :100].tolist() == list(range(0, 100)) and got[2, 100:130].tolist() == [0] * 30
    assert got[:, 130:].tolist() == [[-1, -1]] * 3


@pytest.mark.parametrize("page_size", [1, 16, 64])
@pytest.mark.parametrize("strided", [False, True])
def test_decode_metadata_page_count_indptr(page_size, strided):
    """The optional cu_num_pages output equals the oracle's page-count indptr
    bit for bit: 700 rows (three rounds of the scan), a length that turns
    negative with the delta, strided output; the other outputs unchanged."""
    B, msp = 700, 4
    g = torch.Generator().manual_seed(61 + page_size)
    pool_rows, cols = B + 3, msp * page_size
    rt = torch.randint(0, 1 << 22, (pool_rows, cols), generator=g, dtype=torch.int32)
    pool = torch.randperm(pool_rows, generator=g)[:B].to(torch.int64)
    lens = torch.randint(0, 70000, (B,), generator=g, dtype=torch.int64)
    lens[3], lens[4] = -5, 0
    dev = "cuda"
    cache = torch.empty(B, dtype=torch.int32, device=dev)
    cu = torch.empty(B + 1, dtype=torch.int32, device=dev)
    pt = torch.empty(B, msp, dtype=torch.int32, device=dev)
    store = torch.full((2 * (B + 1),), -9, dtype=torch.int32, device=dev)
    cup = store[::2] if strided else store[:B + 1]
    pkv.normal_decode_set_metadata(cache, cu, pt, rt.to(dev), pool.to(dev), lens.to(dev),
                                   seq_len_delta=1, page_size=page_size, max_seq_pages=msp,
                                   cu_num_pages=cup)
    want_cache, want_cu, want_pt, _ = oracle.decode_set_metadata(lens.tolist(), rt, pool.tolist(),
                                                                 msp, 1, page_size)
    assert cup.tolist() == oracle.cu_num_pages(want_cache, page_size)
    assert cache.tolist() == want_cache and cu.tolist() == want_cu and pt.tolist() == want_pt
    if strided:
        assert bool((store[1::2] == -9).all())


def test_decode_metadata_page_count_indptr_int32_wrap():
    dev = "cuda"
    lens = torch.tensor([2 ** 31 - 1, 5], dtype=torch.int64, device=dev)
    cache = torch.empty(2, dtype=torch.int32, device=dev)
    cu = torch.empty(3, dtype=torch.int32, device=dev)
    cup = torch.empty(3, dtype=torch.int32, device=dev)
    pt = torch.empty(2, 1, dtype=torch.int32, device=dev)
    rt = torch.zeros(1, 1, dtype=torch.int32, device=dev)
    pool = torch.zeros(2, dtype=torch.int64, device=dev)
    pkv.normal_decode_set_metadata(cache, cu, pt, rt, pool, lens, seq_len_delta=1, page_size=1,
                                   max_seq_pages=0, cu_num_pages=cup)
    want_cache = [-(2 ** 31), 6]
    assert cache.tolist() == want_cache
    assert cup.tolist() == oracle.cu_num_pages(want_cache, 1) == [0, 0, 6]
