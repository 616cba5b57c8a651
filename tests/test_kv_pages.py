"""Host logic of the paged KV cache: the page pool hands out scattered pages, grows a sequence
page by page, returns pages on release and refuses what it cannot hold."""
import numpy as np
import pytest

from bit_exact_speculative_gb300.model import KvPagePool


def test_pages_follow_the_given_order_and_cover_lengths():
    pool = KvPagePool(8, 64, 2, 4, device="cpu", order=[5, 2, 7, 0, 6, 3, 1, 4])
    pool.ensure(0, 60)          # one page
    pool.ensure(1, 65)          # two pages
    pool.ensure(0, 129)         # two more (three in all)
    assert pool.host.tolist() == [[5, 0, 6, -1], [2, 7, -1, -1]]
    pool.sync()
    assert pool.table.tolist() == pool.host.tolist()
    pool.ensure(0, 100)         # already covered: nothing changes
    assert not pool.dirty


def test_release_returns_pages_for_reuse():
    pool = KvPagePool(4, 128, 2, 2, device="cpu")
    pool.ensure(0, 256)
    pool.ensure(1, 1)
    pool.release(0)
    assert pool.host[0].tolist() == [-1, -1] and pool.held[0] == 0
    pool.ensure(1, 256)
    pool.ensure(0, 200)
    used = sorted(int(x) for x in pool.host.reshape(-1) if x >= 0)
    assert used == [0, 1, 2, 3]                       # every page in use once
    assert len(set(pool.host[0]) & set(pool.host[1])) == 0


def test_limits():
    pool = KvPagePool(3, 64, 2, 2, device="cpu")
    with pytest.raises(ValueError):
        pool.ensure(0, 129)                             # more than max_pages pages
    pool.ensure(0, 128)
    pool.ensure(1, 64)
    with pytest.raises(MemoryError):
        pool.ensure(1, 65)                              # pool empty
    with pytest.raises(ValueError):
        KvPagePool(3, 64, 1, 3, device="cpu", order=[0, 0, 1])


def test_scattered_pages_reproduce_positions():
    """Position p of sequence b, looked up through the table, is the page row the pool wrote."""
    rng = np.random.default_rng(0)
    page, B, maxp = 64, 3, 5
    pool = KvPagePool(B * maxp, page, B, maxp, device="cpu", order=rng.permutation(B * maxp))
    lens = [300, 64, 1]
    for b, n in enumerate(lens):
        pool.ensure(b, n)
    seen = set()
    for b, n in enumerate(lens):
        for p in range(n):
            pg = pool.host[b, p // page]
            assert 0 <= pg < B * maxp
            seen.add((int(pg), p % page))
    assert len(seen) == sum(lens)                      # no two positions share a slot
