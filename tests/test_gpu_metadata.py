"""GPU metadata kernels, bit-exact against the oracle: the page-index copy
(any strides, empty rows, untouched tail) and the split-count heuristic
(hand-worked cases and an exhaustive sweep of the float32 step)."""
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_tables_gb300 as pkv

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_kv_decode_tables_gb300 import _build
    _build.build()


@pytest.mark.parametrize("col_step", [1, 2, 3])
@pytest.mark.parametrize("R,W", [(1, 1), (7, 9), (64, 300), (512, 2048)])
def test_copy_page_indices_bit_exact(R, W, col_step):
    g = torch.Generator().manual_seed(R * 31 + W + col_step)
    storage = torch.randint(-2 ** 31, 2 ** 31 - 1, (R, W * col_step), generator=g,
                            dtype=torch.int64).to(torch.int32)
    bt = storage[:, ::col_step]
    n = torch.randint(0, W + 1, (R,), generator=g)
    if R > 2:
        n[1] = 0
        n[-1] = W
    cu = [0]
    for v in n.tolist():
        cu.append(cu[-1] + v)
    cap = cu[-1] + 37
    out = torch.full((cap,), -77, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.copy_page_indices(out, storage.cuda()[:, ::col_step],
                          torch.tensor(cu, dtype=torch.int32, device="cuda"), err_flag=err)
    want = oracle.copy_page_indices(bt, cu, cap, fill=-77)
    assert out.cpu().tolist() == want
    assert int(err.item()) == 0


def test_copy_page_indices_flags_overlong_rows():
    bt = torch.arange(12, dtype=torch.int32, device="cuda").view(3, 4)
    cu = torch.tensor([0, 2, 9, 10], dtype=torch.int32, device="cuda")  # row 1 asks for 7 > 4
    out = torch.full((10,), -1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.copy_page_indices(out, bt, cu, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.PKV_ERRF_INDPTR
    assert out[:6].cpu().tolist() == [0, 1, 4, 5, 6, 7]


def _split_cases():
    cases = []
    for line in open(os.path.join(GOLDEN, "num_kv_splits_cases.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        name, lens, params, expected = [p.strip() for p in line.split("|")]
        cases.append((name, [int(v) for v in lens.split()], [int(v) for v in params.split()],
                      [int(v) for v in expected.split()]))
    return cases


def _gpu_splits(lens, ng, nh, nkv, mx, cores, lens_dev=None):
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda") if lens_dev is None else lens_dev
    out = torch.full((len(lens) * ng,), -1, dtype=torch.int32, device="cuda")
    pkv.compute_num_kv_splits(out, seq, num_group=ng, num_head=nh, num_kv_head=nkv,
                              max_kv_splits=mx, device_core_count=cores)
    return out


@pytest.mark.parametrize("case", _split_cases(), ids=lambda c: c[0])
def test_num_kv_splits_hand_worked(case):
    name, lens, (ng, nh, nkv, mx, cores), want = case
    assert _gpu_splits(lens, ng, nh, nkv, mx, cores).cpu().tolist() == want


def test_num_kv_splits_random_batches():
    g = torch.Generator().manual_seed(1)
    for trial in range(60):
        B = int(torch.randint(1, 3000, (1,), generator=g))
        hi = [64, 4096, 1 << 17][trial % 3]
        lens = torch.randint(0, hi, (B,), generator=g).tolist()
        nh, nkv = [(32, 8), (64, 8), (32, 32), (16, 1), (28, 4), (40, 40)][trial % 6]
        mx = [1, 4, 16, 64][trial % 4]
        ng = 1 + trial % 3
        got = _gpu_splits(lens, ng, nh, nkv, mx, 148).cpu().tolist()
        assert got == oracle.num_kv_splits(lens, ng, nh, nkv, mx, 148), trial


def test_num_kv_splits_float32_step_large_lengths():
    """The float32 step on 20,000 seeded random max_seq_len in [2^18, 2^31)
    and on every length whose float32 intermediate the oracle puts within
    3e-4 of an integer in a further 200,000 draws (where a one-ulp error in
    the log2 would move the truncation), with the same construction as the
    exhaustive test below: token_grid = e and e - 1."""
    gen = torch.Generator().manual_seed(61)
    draws = torch.randint(1 << 18, (1 << 31) - 1, (220_000,), generator=gen).tolist()
    lens = draws[:20_000]
    for L in draws[20_000:]:
        ext_len = np.float32(np.float32(L) / np.float32(64.0))
        lg = np.float32(np.log2(np.float64(ext_len)))
        prod = np.float32(np.float32(148.0) * max(lg, np.float32(1.0)))
        if abs(float(prod) - round(float(prod))) < 3e-4:
            lens.append(L)
    N = len(lens)
    assert N > 20_000
    dl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    lib = pkv.lib()
    out = torch.full((2 * N,), -1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    base_l, base_o = dl.data_ptr(), out.data_ptr()
    want = []
    for i, L in enumerate(lens):
        e = oracle.ext_device_core_count(L, 148)
        for j, tg in enumerate((e, max(e - 1, 1))):
            st = lib.compute_num_kv_splits(base_o + 4 * (2 * i + j), base_l + 4 * i, 1, 1, tg, tg,
                                           1 << 30, 148, stream)
            assert st == 0
            want.append(oracle.num_kv_splits([L], 1, tg, tg, 1 << 30, 148)[0])
    got = out.cpu().tolist()
    bad = [(lens[k // 2], got[k], want[k]) for k in range(2 * N) if got[k] != want[k]]
    assert not bad, bad[:10]


def test_num_kv_splits_float32_step_exhaustive():
    """Every max_seq_len in [1, 2^18]: the GPU's split count equals the
    oracle's in two single-sequence batches whose head counts are chosen
    (from the oracle's float32 intermediate e) so that any difference in that
    intermediate changes the output: token_grid = e gives 1 split iff the
    GPU's value is <= e, token_grid = e - 1 gives 2 iff it is >= e."""
    N = 1 << 18
    lens = torch.arange(1, N + 1, dtype=torch.int32, device="cuda")
    lib = pkv.lib()
    out = torch.full((2 * N,), -1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    base_l, base_o = lens.data_ptr(), out.data_ptr()
    want = []
    for i in range(N):
        L = i + 1
        e = oracle.ext_device_core_count(L, 148)
        for j, tg in enumerate((e, max(e - 1, 1))):
            st = lib.compute_num_kv_splits(base_o + 4 * (2 * i + j), base_l + 4 * i, 1, 1, tg, tg,
                                           1 << 30, 148, stream)
            assert st == 0
            want.append(oracle.num_kv_splits([L], 1, tg, tg, 1 << 30, 148)[0])
    got = out.cpu().tolist()
    bad = [(k // 2 + 1, got[k], want[k]) for k in range(2 * N) if got[k] != want[k]]
    assert not bad, bad[:10]


@pytest.mark.parametrize("W", [300, 2048])
@pytest.mark.parametrize("col_step", [1, 2])
@pytest.mark.parametrize("R", [1, 7, 9, 512, 1000])
def test_fused_metadata_equals_both_steps(R, col_step, W):
    """prepare_decode_metadata == copy_page_indices + compute_num_kv_splits, bit
    for bit (rows of up to 300 and 2048 columns: two and eight 256-column
    segments)."""
    g = torch.Generator().manual_seed(R + 17 * col_step + W)
    storage = torch.randint(0, 1 << 20, (R, W * col_step), generator=g, dtype=torch.int32)
    bt = storage[:, ::col_step]
    lens = torch.randint(0, W * 16 + 1, (R,), generator=g)
    lens[0] = 1
    n = [-(-int(L) // 16) for L in lens]
    cu = [0]
    for v in n:
        cu.append(cu[-1] + v)
    cap = cu[-1] + 5
    pi = torch.full((cap,), -3, dtype=torch.int32, device="cuda")
    splits = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.prepare_decode_metadata(pi, storage.cuda()[:, ::col_step],
                                torch.tensor(cu, dtype=torch.int32, device="cuda"), splits,
                                lens.to(torch.int32).cuda(), num_group=1, num_head=32,
                                num_kv_head=8, max_kv_splits=16, device_core_count=148,
                                err_flag=err)
    assert pi.cpu().tolist() == oracle.copy_page_indices(bt, cu, cap, fill=-3)
    assert splits.cpu().tolist() == oracle.num_kv_splits(lens.tolist(), 1, 32, 8, 16, 148)
    assert int(err.item()) == 0


def test_fused_metadata_flags_bad_indptr_rows():
    """The fused copy applies copy_page_indices' checks: a row longer than the
    table is cut to its width, a negative start skips the row, a row past the
    output capacity is cut to it; each is flagged."""
    W = 600
    bt = torch.arange(4 * W, dtype=torch.int32).view(4, W)
    cu = [0, 700, 710, 720, 760]        # row 0 claims 700 > W columns
    cap = 745                           # row 3 ends past the capacity
    pi = torch.full((cap,), -3, dtype=torch.int32, device="cuda")
    splits = torch.empty(4, dtype=torch.int32, device="cuda")
    lens = torch.tensor([700 * 16, 10 * 16, 10 * 16, 40 * 16], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.prepare_decode_metadata(pi, bt.cuda(), torch.tensor(cu, dtype=torch.int32, device="cuda"),
                                splits, lens, num_group=1, num_head=32, num_kv_head=8,
                                max_kv_splits=16, device_core_count=148, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.PKV_ERRF_INDPTR
    got = pi.cpu().tolist()
    assert got[0:W] == bt[0].tolist()             # row 0 cut to the table width
    assert got[W:700] == [-3] * (700 - W)         # nothing past it
    assert got[700:710] == bt[1, :10].tolist()
    assert got[710:720] == bt[2, :10].tolist()
    assert got[720:745] == bt[3, :25].tolist()    # row 3 cut at the capacity
