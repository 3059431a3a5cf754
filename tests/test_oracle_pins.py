"""Pins of the CPU oracle against values the pages print, closed forms,
invariants and library routines (no GPU).

Each pin is chosen so that a plausible slip in the oracle (a wrong index, a
dropped weight, a transposed operand, float64 where the page computes in
float32) fails at least one of them; ``test_pins_catch_planted_mistakes``
plants such slips in the oracle and checks that they are caught.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import oracle.attention as oatt
import oracle.metadata as ometa
import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- helpers ---

def _read_worked_example():
    table, bs, rows = None, None, []
    with open(os.path.join(GOLDEN, "worked_example_offsets.txt")) as f:
        for line in f:
            line = line.strip()
            if line.startswith("# block_table:"):
                table = [int(v) for v in line.split(":")[1].split()]
            elif line.startswith("# block_size:"):
                bs = int(line.split(":")[1])
            elif line and not line.startswith("#"):
                t, off = line.split()
                rows.append((int(t), int(off)))
    return table, bs, rows


def _read_split_cases():
    cases = []
    with open(os.path.join(GOLDEN, "num_kv_splits_cases.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            name, lens, params, expected = [p.strip() for p in line.split("|")]
            cases.append((name, [int(v) for v in lens.split()],
                          [int(v) for v in params.split()], [int(v) for v in expected.split()]))
    return cases


def _scatter_to_pages(K_log, V_log, rows, seq_lens, num_blocks, bs, x):
    """Write contiguous per-sequence K/V ``[B][L, Hk, D]`` into paged caches,
    element by element from the layout statement
    key_cache[num_blocks, num_kv_heads, head_size/x, block_size, x] and
    value_cache[num_blocks, num_kv_heads, head_size, block_size]."""
    Hk, D = K_log[0].shape[1], K_log[0].shape[2]
    key_cache = torch.zeros(num_blocks, Hk, D // x, bs, x, dtype=torch.float64)
    value_cache = torch.zeros(num_blocks, Hk, D, bs, dtype=torch.float64)
    kc = key_cache.numpy()
    vc = value_cache.numpy()
    for s, L in enumerate(seq_lens):
        Kn, Vn = K_log[s].numpy(), V_log[s].numpy()
        for t in range(L):
            b = rows[s][t // bs]
            slot = t % bs
            for h in range(Hk):
                for d in range(D):
                    kc[b, h, d // x, slot, d % x] = Kn[t, h, d]
                    vc[b, h, d, slot] = Vn[t, h, d]
    return key_cache, value_cache


def _random_paged_problem(seed, B, H, Hk, D, bs, x, lens=None, num_blocks=None):
    g = torch.Generator().manual_seed(seed)
    if lens is None:
        lens = [int(v) for v in torch.randint(1, 5 * bs, (B,), generator=g)]
    nblk = [-(-L // bs) for L in lens]
    num_blocks = num_blocks or sum(nblk) + 5
    perm = torch.randperm(num_blocks, generator=g).tolist()
    rows, off = [], 0
    for n in nblk:
        rows.append(perm[off:off + n])
        off += n
    K_log = [torch.randn(L, Hk, D, generator=g, dtype=torch.float64) for L in lens]
    V_log = [torch.randn(L, Hk, D, generator=g, dtype=torch.float64) for L in lens]
    q = torch.randn(B, H, D, generator=g, dtype=torch.float64)
    kc, vc = _scatter_to_pages(K_log, V_log, rows, lens, num_blocks, bs, x)
    width = max(nblk)
    bt = torch.full((B, width), -1, dtype=torch.int32)
    for s, r in enumerate(rows):
        bt[s, :len(r)] = torch.tensor(r, dtype=torch.int32)
    return dict(q=q, kc=kc, vc=vc, bt=bt, lens=lens, K_log=K_log, V_log=V_log, rows=rows,
                num_blocks=num_blocks)


def _sdpa_reference(q, K_log, V_log, lens, scale):
    """torch's scaled_dot_product_attention (float64, contiguous K/V) per sequence."""
    B, H, D = q.shape
    Hk = K_log[0].shape[1]
    out = torch.zeros(B, H, D, dtype=torch.float64)
    for s in range(B):
        K = K_log[s].permute(1, 0, 2).repeat_interleave(H // Hk, dim=0)  # [H, L, D]
        V = V_log[s].permute(1, 0, 2).repeat_interleave(H // Hk, dim=0)
        o = F.scaled_dot_product_attention(q[s][:, None, :], K, V, scale=scale)
        out[s] = o[:, 0, :]
    return out


# ------------------------------------------------- worked example (page 1) ---

def test_worked_example_offsets():
    table, bs, rows = _read_worked_example()
    assert table == [40, 30] and bs == 8 and len(rows) == 16
    got = oracle.token_offsets(table, bs, len(rows))
    assert got == [off for _, off in rows]


def test_worked_example_through_the_gather():
    """The gather reproduces the page's offsets when the cache stores, at
    (block b, slot s), the value b + s (unit block and slot strides), and the
    strided offsets when it stores b * 8 + s (a real cache)."""
    table, bs, rows = _read_worked_example()
    NB = 64
    b = torch.arange(NB, dtype=torch.float64).view(NB, 1)
    s = torch.arange(bs, dtype=torch.float64).view(1, bs)
    for block_stride in (1, bs):
        val = b * block_stride + s  # [NB, bs]
        key_cache = val.view(NB, 1, 1, bs, 1)  # head_size 1, x 1
        value_cache = val.view(NB, 1, 1, bs)
        K, V = oracle.gather_kv(key_cache, value_cache, torch.tensor(table), len(rows), 0)
        want = oracle.token_offsets(table, bs, len(rows), block_stride=block_stride)
        assert K[:, 0].tolist() == want
        assert V[:, 0].tolist() == want
    assert oracle.token_offsets(table, bs, 16, block_stride=1) == [o for _, o in rows]


def test_tiny_workload_uses_worked_example_row():
    inp = workloads.make_workload("tiny_mha_fp32")
    assert inp["block_tables"][0].tolist() == [40, 30]
    assert inp["seq_lens_list"] == [16, 13]
    r1 = inp["block_tables"][1].tolist()
    assert len(set(r1)) == 2 and not set(r1) & {40, 30}


# ------------------------------------------- attention: brute force + forms ---

@pytest.mark.parametrize("B,H,Hk,D,bs,x", [
    (3, 4, 4, 8, 4, 4),
    (2, 8, 2, 16, 8, 8),
    (4, 6, 3, 8, 2, 2),
    (2, 4, 1, 16, 16, 4),
])
def test_oracle_matches_contiguous_sdpa(B, H, Hk, D, bs, x):
    pr = _random_paged_problem(7 + B + H, B, H, Hk, D, bs, x)
    scale = 1.0 / math.sqrt(D)
    got = oracle.decode_v1(pr["q"], pr["kc"], pr["vc"], pr["bt"], pr["lens"], scale)
    want = _sdpa_reference(pr["q"], pr["K_log"], pr["V_log"], pr["lens"], scale)
    assert torch.allclose(got, want, rtol=0, atol=1e-12)


def test_single_token_returns_its_value_row():
    pr = _random_paged_problem(3, 2, 4, 2, 16, 4, 4, lens=[1, 1])
    got = oracle.decode_v1(pr["q"], pr["kc"], pr["vc"], pr["bt"], pr["lens"], 0.25)
    for s in range(2):
        for h in range(4):
            assert torch.equal(got[s, h], pr["V_log"][s][0, h // 2])


def test_zero_query_gives_mean_of_values():
    pr = _random_paged_problem(4, 2, 2, 2, 8, 4, 4, lens=[11, 6])
    q = torch.zeros_like(pr["q"])
    got = oracle.decode_v1(q, pr["kc"], pr["vc"], pr["bt"], pr["lens"], 0.3)
    for s in range(2):
        for h in range(2):
            mean = pr["V_log"][s][:, h].mean(dim=0)
            assert torch.allclose(got[s, h], mean, rtol=0, atol=1e-14)


def test_two_token_closed_form():
    """k_0 = a*q, k_1 = 0: logits a*scale*|q|^2 and 0, so the output is
    (e^z v_0 + v_1) / (e^z + 1)."""
    D, bs, x = 8, 4, 4
    q = torch.tensor([[[1.0, -2.0, 0.5, 0.0, 3.0, 1.0, -1.0, 2.0]]], dtype=torch.float64)
    a, scale = 0.37, 0.5
    K_log = [torch.stack([a * q[0, 0], torch.zeros(D, dtype=torch.float64)])[:, None, :]]
    V_log = [torch.tensor([[1.0] * D, [-3.0] * D], dtype=torch.float64)[:, None, :]]
    kc, vc = _scatter_to_pages(K_log, V_log, [[2]], [2], 4, bs, x)
    bt = torch.tensor([[2]], dtype=torch.int32)
    got = oracle.decode_v1(q, kc, vc, bt, [2], scale)
    z = a * scale * float((q[0, 0] ** 2).sum())
    want = (math.exp(z) * 1.0 + (-3.0)) / (math.exp(z) + 1.0)
    assert abs(float(got[0, 0, 0]) - want) < 1e-14


def test_gqa_groups_are_contiguous():
    """kv head j serves query heads j*g .. j*g+g-1: with value rows constant
    per kv head, every query head returns its own kv head's constant."""
    B, H, Hk, D, bs, x = 1, 6, 3, 8, 4, 4
    L = 9
    g = torch.Generator().manual_seed(11)
    K_log = [torch.randn(L, Hk, D, generator=g, dtype=torch.float64)]
    V_log = [torch.empty(L, Hk, D, dtype=torch.float64)]
    for j in range(Hk):
        V_log[0][:, j, :] = float(j + 1)
    kc, vc = _scatter_to_pages(K_log, V_log, [[5, 1, 3]], [L], 8, bs, x)
    bt = torch.tensor([[5, 1, 3]], dtype=torch.int32)
    q = torch.randn(B, H, D, generator=g, dtype=torch.float64)
    got = oracle.decode_v1(q, kc, vc, bt, [L], 0.35)
    for h in range(H):
        assert torch.allclose(got[0, h], torch.full((D,), float(h // 2 + 1), dtype=torch.float64),
                              rtol=0, atol=1e-14)


def test_block_permutation_invariance_is_exact():
    """Relabelling physical blocks (moving page contents, rewriting the table)
    leaves the logical K/V, hence the output, bit-identical."""
    pr = _random_paged_problem(21, 3, 4, 2, 16, 4, 4, lens=[13, 4, 9])
    base = oracle.decode_v1(pr["q"], pr["kc"], pr["vc"], pr["bt"], pr["lens"], 0.25)
    NB = pr["num_blocks"]
    relabel = torch.randperm(NB, generator=torch.Generator().manual_seed(5))
    kc2 = torch.empty_like(pr["kc"])
    vc2 = torch.empty_like(pr["vc"])
    kc2[relabel] = pr["kc"]
    vc2[relabel] = pr["vc"]
    bt2 = pr["bt"].clone()
    m = bt2 >= 0
    bt2[m] = relabel[bt2[m].long()].to(torch.int32)
    moved = oracle.decode_v1(pr["q"], kc2, vc2, bt2, pr["lens"], 0.25)
    assert torch.equal(base, moved)


# ------------------------------------------------------------ split-KV v2 ---

def test_v2_equals_v1_for_every_partition_size():
    bs = 4
    pr = _random_paged_problem(31, 3, 4, 2, 8, bs, 4, lens=[23, 1, 16])
    v1 = oracle.decode_v1(pr["q"], pr["kc"], pr["vc"], pr["bt"], pr["lens"], 0.4)
    for P in range(bs, 28, bs):
        maxP = -(-23 // P)
        tmp, es, ml = oracle.v2_partition(pr["q"], pr["kc"], pr["vc"], pr["bt"], pr["lens"], 0.4,
                                          maxP, partition_size=P)
        out = oracle.v2_reduce(tmp, es, ml, pr["lens"], bs, partition_size=P)
        assert torch.allclose(out, v1, rtol=0, atol=1e-12), P


def test_v2_equals_v1_for_every_split_count():
    bs = 4
    pr = _random_paged_problem(32, 3, 2, 1, 8, bs, 4, lens=[29, 3, 12])
    v1 = oracle.decode_v1(pr["q"], pr["kc"], pr["vc"], pr["bt"], pr["lens"], 0.4)
    for n in range(1, 10):
        splits = [n, max(1, n // 2), n]
        tmp, es, ml = oracle.v2_partition(pr["q"], pr["kc"], pr["vc"], pr["bt"], pr["lens"], 0.4,
                                          12, num_kv_splits=splits)
        out = oracle.v2_reduce(tmp, es, ml, pr["lens"], bs, num_kv_splits=splits)
        assert torch.allclose(out, v1, rtol=0, atol=1e-12), n
        for s, L in enumerate(pr["lens"]):
            c = oracle.split_chunk_size(L, splits[s], bs)
            nonempty = [p for p in range(12) if es[s, 0, p] > 0]
            assert nonempty == list(range(-(-L // c)))
            assert len(nonempty) <= splits[s] and c % bs == 0


def test_empty_partitions_carry_neg_inf_and_zero():
    pr = _random_paged_problem(33, 1, 2, 2, 8, 4, 4, lens=[9])
    tmp, es, ml = oracle.v2_partition(pr["q"], pr["kc"], pr["vc"], pr["bt"], pr["lens"], 0.3,
                                      5, partition_size=4)
    assert torch.all(es[0, :, 3:] == 0) and torch.all(ml[0, :, 3:] == float("-inf"))
    assert torch.all(es[0, :, :3] > 0) and torch.all(torch.isfinite(ml[0, :, :3]))
    # exp_sums of the partial partition [8, 9) is exp(z - max z) over one token = 1
    assert torch.allclose(es[0, :, 2], torch.ones(2, dtype=torch.float64))


def test_reduce_closed_form():
    """Two partitions with max logits 0 and ln 2, sums 1 and 1, partial
    outputs a and b: weights e^{-ln2}*1 = 1/2 and 1, output (a/2 + b) / 1.5."""
    a = torch.tensor([1.0, 2.0, -4.0], dtype=torch.float64)
    b = torch.tensor([7.0, 0.0, 2.0], dtype=torch.float64)
    tmp = torch.stack([a, b])[None, None]  # [1, 1, 2, 3]
    es = torch.tensor([[[1.0, 1.0]]], dtype=torch.float64)
    ml = torch.tensor([[[0.0, math.log(2.0)]]], dtype=torch.float64)
    out = oracle.v2_reduce(tmp, es, ml, [2 * 4], 4, partition_size=4)
    assert torch.allclose(out[0, 0], (a / 2 + b) / 1.5, rtol=0, atol=1e-15)
    # exp_sums scale the weights: sums 3 and 1 give weights 3/2 and 1.
    es2 = torch.tensor([[[3.0, 1.0]]], dtype=torch.float64)
    out2 = oracle.v2_reduce(tmp, es2, ml, [8], 4, partition_size=4)
    assert torch.allclose(out2[0, 0], (1.5 * a + b) / 2.5, rtol=0, atol=1e-15)


def test_zero_length_sequence_gives_zero_output():
    pr = _random_paged_problem(34, 2, 2, 2, 8, 4, 4, lens=[5, 3])
    lens = [0, 3]
    v1 = oracle.decode_v1(pr["q"], pr["kc"], pr["vc"], pr["bt"], lens, 0.3)
    assert torch.equal(v1[0], torch.zeros(2, 8, dtype=torch.float64))
    tmp, es, ml = oracle.v2_partition(pr["q"], pr["kc"], pr["vc"], pr["bt"], lens, 0.3, 3,
                                      partition_size=4)
    assert torch.all(es[0] == 0) and torch.all(ml[0] == float("-inf"))
    out = oracle.v2_reduce(tmp, es, ml, lens, 4, partition_size=4)
    assert torch.equal(out[0], torch.zeros(2, 8, dtype=torch.float64))
    assert torch.allclose(out[1], v1[1], rtol=0, atol=1e-12)


def test_csr_page_list_equals_block_table():
    """Reading block ids through (page_indices, indptr) gives the same result
    as the 2-D table they were flattened from."""
    pr = _random_paged_problem(35, 3, 2, 2, 8, 4, 4, lens=[7, 12, 2])
    nblk = [-(-L // 4) for L in pr["lens"]]
    cu = [0]
    for n in nblk:
        cu.append(cu[-1] + n)
    flat = torch.tensor(oracle.copy_page_indices(pr["bt"], cu, cu[-1]), dtype=torch.int32)
    a = oracle.decode_v1(pr["q"], pr["kc"], pr["vc"], pr["bt"], pr["lens"], 0.3)
    b = oracle.decode_v1(pr["q"], pr["kc"], pr["vc"], flat, pr["lens"], 0.3,
                         kv_indptr=torch.tensor(cu))
    assert torch.equal(a, b)


# -------------------------------------------------------- metadata: copy ---

def test_copy_page_indices_equals_boolean_mask_gather():
    """The page-index copy computes what ``block_table[mask]`` (mask[i, j] =
    j < num_blocks_i) computes; vLLM PR 35765 replaces exactly that
    data-dependent indexing.  Covers a stride-2 column view and empty rows."""
    g = torch.Generator().manual_seed(3)
    for col_step in (1, 2, 3):
        B, W = 7, 9
        storage = torch.randint(0, 1000, (B, W * col_step), generator=g, dtype=torch.int32)
        bt = storage[:, ::col_step]
        n = torch.randint(0, W + 1, (B,), generator=g)
        n[2] = 0
        cu = [0]
        for v in n.tolist():
            cu.append(cu[-1] + v)
        mask = torch.arange(W)[None, :] < n[:, None]
        want = bt[mask].tolist()
        got = oracle.copy_page_indices(bt, cu, cu[-1] + 5, fill=-9)
        assert got[:cu[-1]] == want
        assert got[cu[-1]:] == [-9] * 5


# ------------------------------------------------- metadata: split count ---

def test_num_kv_splits_hand_worked_cases():
    cases = _read_split_cases()
    assert len(cases) >= 10
    for name, lens, (ng, nh, nkv, mx, cores), want in cases:
        got = oracle.num_kv_splits(lens, ng, nh, nkv, mx, cores)
        assert got == want, name


def test_ext_core_count_float32_step():
    path = os.path.join(GOLDEN, "ext_core_count_f32.txt")
    rows = [tuple(int(v) for v in line.split()) for line in open(path)
            if line.strip() and not line.startswith("#")]
    assert len(rows) >= 8
    for L, cores, f32_result, exact_trunc in rows:
        assert oracle.ext_device_core_count(L, cores) == f32_result, L
        # the exact real value truncates to the other integer at the
        # sensitive lengths: float64 throughout would have been wrong there
        exact = cores * max(math.log2(L / 64.0), 1.0)
        assert int(exact) in (exact_trunc, exact_trunc + 1)


def _nearest_f32(v, mpmath):
    f = np.float32(float(v))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    return min(cands, key=lambda c: abs(mpmath.mpf(float(c)) - v))


def test_log2_f32_is_correctly_rounded():
    """log2 rounded to float32, against 50-digit arithmetic, on every
    max_seq_len/64 for max_seq_len = 1, 97, 193, ... < 2^18 and the
    float32-sensitive lengths."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    lens = list(range(1, 1 << 18, 97)) + [12084, 30545, 61090, 62831, 103223, 105175,
                                           122180, 125662]
    for L in lens:
        e = np.float32(L) / np.float32(64.0)
        want = _nearest_f32(mpmath.log(mpmath.mpf(float(e)), 2), mpmath)
        assert oracle.log2_f32(e) == want, L


def test_ext_core_count_against_high_precision():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    for L in list(range(1, 1 << 18, 331)) + [12084, 125662, 1 << 18]:
        e = np.float32(L) / np.float32(64.0)
        lg = _nearest_f32(mpmath.log(mpmath.mpf(float(e)), 2), mpmath)
        lg = max(lg, np.float32(1.0))
        prod = _nearest_f32(mpmath.mpf(148) * mpmath.mpf(float(lg)), mpmath)
        assert oracle.ext_device_core_count(L, 148) == int(prod), L


def test_num_kv_splits_bounds():
    g = torch.Generator().manual_seed(9)
    for trial in range(40):
        B = int(torch.randint(1, 40, (1,), generator=g))
        lens = [int(v) for v in torch.randint(1, 1 << 17, (B,), generator=g)]
        nh, nkv = [(32, 8), (64, 8), (32, 32), (16, 1), (28, 4)][trial % 5]
        mx = [1, 4, 16, 64][trial % 4]
        out = oracle.num_kv_splits(lens, 1, nh, nkv, mx, 148)
        assert all(1 <= v <= mx for v in out)
        # longer sequences never get fewer splits than shorter ones in the same batch
        order = sorted(range(B), key=lambda i: lens[i])
        assert all(out[order[i]] <= out[order[i + 1]] for i in range(B - 1))


# ----------------------------------------- the pins catch planted mistakes ---

def test_pins_catch_planted_mistakes(monkeypatch):
    """Plant slips in the oracle (on the CPU) and check a pin fails on each."""
    # 1. kv-head map h % num_kv_heads instead of contiguous groups
    monkeypatch.setattr(oatt, "kv_head_of", lambda h, H, Hk: h % Hk)
    with pytest.raises(AssertionError):
        test_gqa_groups_are_contiguous()
    monkeypatch.undo()

    # 2. block and slot roles swapped in the gather
    def bad_gather(key_cache, value_cache, block_ids, seq_len, kv_head):
        bs = key_cache.shape[3]
        D = value_cache.shape[2]
        t = torch.arange(seq_len)
        blk = block_ids[torch.clamp(t % bs, max=len(block_ids) - 1)]
        slot = (t // bs) % bs
        K = key_cache[blk, kv_head, :, slot, :].to(torch.float64).reshape(seq_len, D)
        V = value_cache[blk, kv_head, :, slot].to(torch.float64)
        return K, V

    monkeypatch.setattr(oatt, "gather_kv", bad_gather)
    monkeypatch.setattr(oracle, "gather_kv", bad_gather)
    with pytest.raises(AssertionError):
        test_worked_example_through_the_gather()
    monkeypatch.undo()

    # 3. x-packed key dims read in the wrong order (d % x and d // x swapped)
    def bad_gather_x(key_cache, value_cache, block_ids, seq_len, kv_head):
        bs = key_cache.shape[3]
        D = value_cache.shape[2]
        t = torch.arange(seq_len)
        blk = block_ids[t // bs]
        slot = t % bs
        K = key_cache[blk, kv_head, :, slot, :].to(torch.float64).transpose(1, 2).reshape(seq_len, D)
        V = value_cache[blk, kv_head, :, slot].to(torch.float64)
        return K, V

    monkeypatch.setattr(oatt, "gather_kv", bad_gather_x)
    with pytest.raises(AssertionError):
        test_oracle_matches_contiguous_sdpa(2, 8, 2, 16, 8, 8)
    monkeypatch.undo()

    # 4. reduce that forgets the exp_sums factor
    orig_reduce = oatt.v2_reduce

    def bad_reduce(tmp_output, exp_sums, max_logits, seq_lens, block_size, partition_size=None,
                   num_kv_splits=None, seqs=None, heads=None):
        return orig_reduce(tmp_output, torch.ones_like(exp_sums), max_logits, seq_lens,
                           block_size, partition_size, num_kv_splits, seqs, heads)

    monkeypatch.setattr(oracle, "v2_reduce", bad_reduce)
    with pytest.raises(AssertionError):
        test_reduce_closed_form()
    monkeypatch.undo()

    # 5. the split heuristic's log2 step in float64 instead of float32
    def ext_f64(max_seq_len, device_core_count):
        return int(device_core_count * max(math.log2(max_seq_len / 64.0), 1.0))

    monkeypatch.setattr(ometa, "ext_device_core_count", ext_f64)
    with pytest.raises(AssertionError):
        test_num_kv_splits_hand_worked_cases()
    monkeypatch.undo()

    # 6. softmax without the max subtraction is still exact here, but a
    #    dropped normalisation is not
    def bad_attention(q, K, V, scale, bias=None):
        z = (K @ q.to(torch.float64)) * scale
        p = torch.exp(z - z.max())
        return p @ V, z

    monkeypatch.setattr(oatt, "attention_one_head", bad_attention)
    with pytest.raises(AssertionError):
        test_zero_query_gives_mean_of_values()
    monkeypatch.undo()


# ------------------------------------------- metadata: fused decode metadata ---

def _read_decode_metadata_example():
    d = {"rt": {}}
    for line in open(os.path.join(GOLDEN, "decode_set_metadata_example.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, val = line.split(":")
        vals = [int(v) for v in val.split()]
        if key.startswith("req_to_token"):
            d["rt"][int(key.split()[1])] = vals
        else:
            d[key] = vals
    return d


def test_decode_set_metadata_golden():
    d = _read_decode_metadata_example()
    rt = [d["rt"][i] for i in range(len(d["rt"]))]
    mapping = [100 + t for t in range(128)]
    cache, cu, pt, swa = oracle.decode_set_metadata(
        d["seq_lens"], rt, d["req_pool_indices"], d["max_seq_pages"][0], d["delta"][0],
        d["page_size"][0], full_to_swa_mapping=mapping)
    assert cache == d["expect cache_seqlens"]
    assert cu == d["expect cu_seqlens_k"]
    assert pt == [d["expect page_table 0"], d["expect page_table 1"]]
    assert swa == [d["expect swa_page_table 0"], d["expect swa_page_table 1"]]


@pytest.mark.parametrize("page_size", [1, 2, 16, 64])
def test_decode_set_metadata_against_library_routines(page_size):
    """cumsum for the indptr, floor division by the page size for the shift
    (the docstring's "page_table = page_indices // page_size"), integer
    indexing for both gathers."""
    g = torch.Generator().manual_seed(page_size)
    pool_rows, cols, B, msp = 9, 64 * page_size, 6, 40
    rt = torch.randint(0, 1 << 20, (pool_rows, cols), generator=g, dtype=torch.int64)
    pool = torch.randint(0, pool_rows, (B,), generator=g)
    lens = torch.randint(0, 5000, (B,), generator=g)
    mapping = torch.randint(0, 1 << 24, (1 << 20,), generator=g, dtype=torch.int64)
    cache, cu, pt, swa = oracle.decode_set_metadata(lens.tolist(), rt.tolist(), pool.tolist(), msp,
                                                    1, page_size, full_to_swa_mapping=mapping)
    want_cache = (lens + 1).tolist()
    assert cache == want_cache
    assert cu == [0] + np.cumsum(want_cache).tolist()
    page_index = rt[pool][:, ::page_size][:, :msp]
    assert pt == torch.div(page_index, page_size, rounding_mode="floor").tolist()
    assert swa == torch.div(mapping[page_index], page_size, rounding_mode="floor").tolist()


def test_decode_set_metadata_int32_cast_wraps():
    cache, cu, _, _ = oracle.decode_set_metadata([2 ** 31 - 1, 5], [[0]], [0, 0], 0, 1, 1)
    want = np.array([2 ** 31 - 1, 5], dtype=np.int64) + 1
    assert cache == want.astype(np.int32).tolist() == [-(2 ** 31), 6]
    assert cu == [0, -(2 ** 31), -(2 ** 31) + 6]


def test_cu_num_pages_pins():
    """The page-count indptr: a hand-worked case (page size 16, an empty and
    a negative length hold no page), page size 1 equals the running sum of
    the lengths, numpy's ceil-division cumsum on random lengths, and the
    ragged workload's indptr (built there from the block rows it allocates,
    not from this function)."""
    assert oracle.cu_num_pages([0, 1, 16, 17, -5, 32], 16) == [0, 0, 1, 2, 4, 4, 6]
    g = torch.Generator().manual_seed(5)
    lens = torch.randint(0, 40000, (300,), generator=g)
    assert oracle.cu_num_pages(lens.tolist(), 1) == [0] + np.cumsum(lens.numpy()).tolist()
    for ps in (2, 16, 64):
        want = [0] + np.cumsum(-(-lens.numpy() // ps)).tolist()
        assert oracle.cu_num_pages(lens.tolist(), ps) == want
    inp = workloads.make_workload("ragged_v2_bf16", seed=0, num_seqs=40)
    assert oracle.cu_num_pages(inp["seq_lens_list"], 16) == inp["cu_num_blocks"].tolist()
    # int32 running sum, as cu_seqlens_k
    assert oracle.cu_num_pages([2 ** 31 - 1, 1], 1) == [0, 2 ** 31 - 1, -(2 ** 31)]


# ------------------------------------------- metadata: SWA speculative table ---

def _read_swa_example():
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
    return d


def test_swa_spec_page_table_golden():
    d = _read_swa_example()
    A = [d["A"][i] for i in range(len(d["A"]))]
    B = [d["B"][i] for i in range(len(d["B"]))]
    dst = [[-1] * 7 for _ in range(4)]
    oracle.swa_spec_page_table(dst, A, B, d["seq_len_a"], d["seq_len_b"], d["draft_tokens"][0])
    assert dst == [d["expect"][i] for i in range(4)]


def test_swa_spec_page_table_is_a_concatenation():
    """Within the tables' widths the row is torch.cat of the two cut rows,
    and nothing past the combined length is written."""
    g = torch.Generator().manual_seed(5)
    bs, R, LA, LB = 5, 3, 40, 9
    A = torch.randint(0, 1000, (bs, LA), generator=g)
    Bt = torch.randint(0, 1000, (bs * R, LB), generator=g)
    la = torch.randint(0, LA + 1, (bs,), generator=g)
    lb = torch.randint(0, LB + 1, (bs * R,), generator=g)
    dst = [[-5] * (LA + LB) for _ in range(bs * R)]
    oracle.swa_spec_page_table(dst, A.tolist(), Bt.tolist(), la.tolist(), lb.tolist(), R)
    for m in range(bs * R):
        a_len, b_len = int(la[m // R]), int(lb[m])
        want = torch.cat([A[m // R, :a_len], Bt[m, :b_len]]).tolist()
        assert dst[m][:a_len + b_len] == want
        assert dst[m][a_len + b_len:] == [-5] * (LA + LB - a_len - b_len)


def test_swa_spec_page_table_pads_past_table_widths_with_zero():
    dst = [[-1] * 6]
    oracle.swa_spec_page_table(dst, [[7, 8]], [[4, 5]], [3], [3], 1)
    # la 3 > LEN_A 2: column 2 is 0; the B part starts at column 3 (k = 0);
    # nothing is written at or past LEN_A + LEN_B = 4 columns
    assert dst == [[7, 8, 0, 4, -1, -1]]
    dst = [[-1] * 4]
    oracle.swa_spec_page_table(dst, [[7, 8]], [[4, 5]], [1], [3], 1)
    # la 1: column 0 from A; k = 0, 1 from B; k = 2 >= LEN_B: 0
    assert dst == [[7, 4, 5, 0]]
