"""GPU sliding-window speculative page table (sglang
prepare_swa_spec_page_table_triton) against the oracle, bit-exact."""
import os

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


def test_golden_example():
    d = {"A": {}, "B": {}, "expect": {}}
    for line in open(os.path.join(GOLDEN, "swa_spec_page_table_example.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, val = line.split(":")
        vals = [int(v) for v in val.split()]
        parts = key.split()
        if parts[0] in ("A", "B", "expect"):
            d[parts[0]][int(parts[1])] = vals
        else:
            d[key] = vals
    A = torch.tensor([d["A"][i] for i in range(2)], dtype=torch.int32, device="cuda")
    B = torch.tensor([d["B"][i] for i in range(4)], dtype=torch.int32, device="cuda")
    dst = torch.full((4, 7), -1, dtype=torch.int32, device="cuda")
    pkv.prepare_swa_spec_page_table(dst, A, B,
                                    torch.tensor(d["seq_len_a"], dtype=torch.int32, device="cuda"),
                                    torch.tensor(d["seq_len_b"], dtype=torch.int32, device="cuda"),
                                    d["draft_tokens"][0])
    assert dst.cpu().tolist() == [d["expect"][i] for i in range(4)]


@pytest.mark.parametrize("bs,R,LA,LB", [(1, 1, 1, 1), (3, 4, 100, 7), (16, 2, 2048, 64),
                                        (64, 8, 1500, 300), (2, 3, 0, 5), (2, 3, 5, 0)])
@pytest.mark.parametrize("over", [False, True])
def test_random_tables_bit_exact(bs, R, LA, LB, over):
    g = torch.Generator().manual_seed(bs * 7 + R + LA + LB + over)
    A = torch.randint(-2 ** 31, 2 ** 31 - 1, (bs, max(LA, 1)), generator=g,
                      dtype=torch.int64).to(torch.int32)[:, :LA]
    Bt = torch.randint(-2 ** 31, 2 ** 31 - 1, (bs * R, max(LB, 1)), generator=g,
                       dtype=torch.int64).to(torch.int32)[:, :LB]
    hi_a, hi_b = (LA + 5, LB + 5) if over else (LA, LB)  # lengths past the widths
    la = torch.randint(0, hi_a + 1, (bs,), generator=g, dtype=torch.int32)
    lb = torch.randint(0, hi_b + 1, (bs * R,), generator=g, dtype=torch.int32)
    width = LA + LB + 3
    dst = torch.full((bs * R, width), -77, dtype=torch.int32)
    want = oracle.swa_spec_page_table(dst.tolist(), A.tolist() if LA else [[]] * bs,
                                      Bt.tolist() if LB else [[]] * (bs * R), la.tolist(),
                                      lb.tolist(), R)
    d_dst = dst.cuda()
    pkv.prepare_swa_spec_page_table(d_dst, A.cuda(), Bt.cuda(), la.cuda(), lb.cuda(), R)
    assert d_dst.cpu().tolist() == want


def test_strided_views_and_negative_length_flag():
    A_store = torch.arange(40, dtype=torch.int32, device="cuda").view(4, 10)
    A = A_store[:, ::2]  # [4, 5], column stride 2
    Bt = torch.arange(100, 124, dtype=torch.int32, device="cuda").view(8, 3)
    la = torch.tensor([5, 2, -1, 4], dtype=torch.int32, device="cuda")
    lb = torch.tensor([1, 2, 3, 0, 1, 2, 3, 0], dtype=torch.int32, device="cuda")
    dst_store = torch.full((8, 20), -9, dtype=torch.int32, device="cuda")
    dst = dst_store[:, :8]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.prepare_swa_spec_page_table(dst, A, Bt, la, lb, 2, err_flag=err)
    want = oracle.swa_spec_page_table([[-9] * 8 for _ in range(8)], A.cpu().tolist(),
                                      Bt.cpu().tolist(), [5, 2, 0, 4], lb.cpu().tolist(), 2)
    torch.cuda.synchronize()
    assert dst.cpu().tolist() == want
    assert bool((dst_store[:, 8:] == -9).all())
    assert int(err.item()) & pkv.PKV_ERRF_SEQ_LEN
