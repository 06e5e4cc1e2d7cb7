"""The host-side block allocator (free pool, reference counts, copy-on-write, append) through the C ABI.

Pure host code: runs without a GPU. A plain Python model of the same bookkeeping is the reference for
randomised operation sequences."""
import numpy as np
import pytest

from paged_kv_cache_223_gb300 import _build

_build.build_cuda()
from paged_kv_cache_223_gb300 import pagedattn as pa  # noqa: E402


def test_reference_count_four_for_four_samples():
    """Four parallel samples share the prompt's blocks: each shared block has reference count 4
    (yangyu.win blog #54, section 5 question 2)."""
    A = pa.BlockAllocator(64, 16)
    table = np.full(8, -1, np.int32)
    slots, L, pair = A.append(table, 0, 40)                 # prompt: 40 tokens -> 3 blocks
    assert L == 40 and pair is None and A.num_free == 61
    assert np.array_equal(slots, table[np.arange(40) // 16].astype(np.int64) * 16 + np.arange(40) % 16)
    for _ in range(3):
        A.fork(table[:3])
    assert [A.ref_count(int(b)) for b in table[:3]] == [4, 4, 4]
    # each sample appends one token: the partly filled block 2 is copied for the first three writers
    rows = [table.copy() for _ in range(4)]
    copies = []
    for r in rows:
        _, L2, pair = A.append(r, 40, 1)
        copies.append(pair)
    assert [c is not None for c in copies] == [True, True, True, False]   # the last writer owns it alone
    assert all(c[0] == table[2] for c in copies[:3])
    assert len({int(r[2]) for r in rows}) == 4
    assert A.ref_count(int(table[0])) == 4 and A.ref_count(int(table[2])) == 1
    assert A.num_free == 61 - 3


def test_append_crosses_block_boundaries():
    A = pa.BlockAllocator(16, 16)
    row = np.full(4, -1, np.int32)
    s1, L, _ = A.append(row, 0, 16)
    assert L == 16 and (row[1:] == -1).all()
    s2, L, _ = A.append(row, 16, 1)                           # token 16 needs block 1
    assert L == 17 and row[1] >= 0 and s2[0] == row[1] * 16
    with pytest.raises(pa.PagedAttnError):
        A.append(row, 17, 64)                                 # beyond the row's capacity (64 tokens)


def test_full_block_is_not_copied_even_if_shared():
    A = pa.BlockAllocator(8, 16)
    row = np.full(4, -1, np.int32)
    A.append(row, 0, 32)
    A.fork(row[:2])
    other = row.copy()
    _, _, pair = A.append(other, 32, 1)                       # next token opens a new block: nothing to copy
    assert pair is None and other[2] not in row[:2]


def test_oom_changes_nothing():
    A = pa.BlockAllocator(4, 16)
    A.alloc(3)
    with pytest.raises(pa.PagedAttnError) as e:
        A.alloc(2)
    assert e.value.status == pa.PA_ERR_OOM and A.num_free == 1
    row = np.full(4, -1, np.int32)
    with pytest.raises(pa.PagedAttnError):
        A.append(row, 0, 33)                                  # needs 3 blocks, 1 free
    assert A.num_free == 1 and (row == -1).all()


def test_bad_frees_and_forks_are_rejected_atomically():
    A = pa.BlockAllocator(8, 16)
    ids = A.alloc(2)
    with pytest.raises(pa.PagedAttnError):
        A.free([ids[0], ids[0]])                              # two drops, one reference
    assert A.ref_count(int(ids[0])) == 1
    with pytest.raises(pa.PagedAttnError):
        A.fork([ids[1], 7])                                   # 7 is free
    assert A.ref_count(int(ids[1])) == 1
    A.free(ids)
    assert A.num_free == 8


def test_random_operations_match_a_plain_model():
    rng = np.random.default_rng(0)
    NB = 40
    A = pa.BlockAllocator(NB, 16)
    ref = {}                                                   # model: block -> count
    for step in range(3000):
        op = rng.integers(0, 4)
        live = [b for b, c in ref.items() if c > 0]
        if op == 0:
            n = int(rng.integers(0, 5))
            if n > NB - len(live):
                with pytest.raises(pa.PagedAttnError):
                    A.alloc(n)
            else:
                got = A.alloc(n)
                assert len(set(got.tolist())) == n and not (set(got.tolist()) & set(live))
                for b in got:
                    ref[int(b)] = 1
        elif op == 1 and live:
            pick = rng.choice(live, size=int(rng.integers(1, 4)))
            A.fork(pick)
            for b in pick:
                ref[int(b)] += 1
        elif op == 2 and live:
            pick = rng.choice(live, size=int(rng.integers(1, 3)), replace=False)
            A.free(pick)
            for b in pick:
                ref[int(b)] -= 1
        elif op == 3 and live:
            b = int(rng.choice(live))
            if ref[b] > 1 and len(live) == NB:
                with pytest.raises(pa.PagedAttnError):
                    A.cow(b)
                continue
            nb, copied = A.cow(b)
            assert copied == (ref[b] > 1)
            if copied:
                ref[b] -= 1
                assert ref.get(nb, 0) == 0
                ref[nb] = 1
            else:
                assert nb == b
        for b in range(NB):
            assert A.ref_count(b) == ref.get(b, 0)
        assert A.num_free == sum(1 for b in range(NB) if ref.get(b, 0) == 0)
