"""Host page allocator (the C ABI's w4a16_page_* and w4a16_seq_* calls):
pure host bookkeeping, so these run on the CPU against the built library.

Invariants pinned: a page is never handed out twice while in use, freed
pages are handed out again, failed calls change nothing (all or nothing),
bad frees are refused, and block-table rows grow one page per 16 tokens."""
import ctypes

import numpy as np
import pytest

from w4a16_decode_paged_gb300 import _lib, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def _new(lib, n):
    h = ctypes.c_void_p()
    assert lib.w4a16_page_allocator_create(n, ctypes.byref(h)) == 0
    return h


def _alloc(lib, a, n):
    out = np.full(max(n, 1), -7, np.int32)
    rc = lib.w4a16_page_alloc(a, n, out.ctypes.data)
    return rc, out[:n]


def _free(lib, a, pages):
    pages = np.ascontiguousarray(pages, np.int32)
    return lib.w4a16_page_free(a, pages.ctypes.data if pages.size else None, int(pages.size))


def test_hands_out_every_page_once_then_reports_no_pages(lib):
    a = _new(lib, 37)
    rc, p = _alloc(lib, a, 37)
    assert rc == 0 and sorted(p.tolist()) == list(range(37))
    assert lib.w4a16_page_free_count(a) == 0
    rc, _ = _alloc(lib, a, 1)
    assert rc == 8                                    # W4A16_ERR_NO_PAGES
    lib.w4a16_page_allocator_destroy(a)


def test_failed_alloc_changes_nothing(lib):
    a = _new(lib, 10)
    rc, p = _alloc(lib, a, 7)
    assert rc == 0
    rc, _ = _alloc(lib, a, 4)                         # only 3 free: all or nothing
    assert rc == 8 and lib.w4a16_page_free_count(a) == 3
    rc, q = _alloc(lib, a, 3)
    assert rc == 0 and not (set(q.tolist()) & set(p.tolist()))
    lib.w4a16_page_allocator_destroy(a)


def test_freed_pages_are_reused_and_bad_frees_refused(lib):
    a = _new(lib, 8)
    rc, p = _alloc(lib, a, 8)
    assert _free(lib, a, p[:3]) == 0 and lib.w4a16_page_free_count(a) == 3
    rc, q = _alloc(lib, a, 3)
    assert rc == 0 and sorted(q.tolist()) == sorted(p[:3].tolist())
    assert _free(lib, a, [q[0], q[0]]) == 1           # named twice: refused, nothing freed
    assert lib.w4a16_page_free_count(a) == 0
    assert _free(lib, a, [8]) == 1                    # outside the pool
    assert _free(lib, a, [-1]) == 1
    assert _free(lib, a, [q[1]]) == 0
    assert _free(lib, a, [q[1]]) == 1                 # double free across calls
    assert _free(lib, a, [q[2], q[1]]) == 1           # one bad page: the good one is not freed either
    assert lib.w4a16_page_free_count(a) == 1
    lib.w4a16_page_allocator_destroy(a)


def test_random_alloc_free_sequence_against_a_set(lib):
    rng = np.random.default_rng(123)
    n = 64
    a = _new(lib, n)
    held = set()
    for _ in range(2000):
        if rng.random() < 0.55:
            k = int(rng.integers(0, 9))
            rc, p = _alloc(lib, a, k)
            if k <= n - len(held):
                assert rc == 0 and len(set(p.tolist())) == k and not (set(p.tolist()) & held)
                assert all(0 <= x < n for x in p)
                held |= set(p.tolist())
            else:
                assert rc == 8
        elif held:
            k = int(rng.integers(1, len(held) + 1))
            pick = rng.choice(sorted(held), size=k, replace=False)
            assert _free(lib, a, pick) == 0
            held -= set(int(x) for x in pick)
        assert lib.w4a16_page_free_count(a) == n - len(held)
    lib.w4a16_page_allocator_destroy(a)


def test_sequence_rows_grow_one_page_per_16_tokens(lib):
    a = _new(lib, 6)
    row = np.full(4, -1, np.int32)
    for L, pages in ((0, 0), (1, 1), (16, 1), (17, 2), (32, 2), (33, 3), (64, 4)):
        assert lib.w4a16_seq_reserve(a, row.ctypes.data, 4, L) == 0
        assert int((row >= 0).sum()) == pages, L
    kept = row.copy()
    assert lib.w4a16_seq_reserve(a, row.ctypes.data, 4, 65) == 3     # W4A16_ERR_SHAPE: 5 pages > 4 blocks
    assert np.array_equal(row, kept)
    other = np.full(4, -1, np.int32)
    assert lib.w4a16_seq_reserve(a, other.ctypes.data, 4, 48) == 8   # 3 pages wanted, 2 free: nothing taken
    assert np.all(other == -1) and lib.w4a16_page_free_count(a) == 2
    assert lib.w4a16_seq_release(a, row.ctypes.data, 4) == 0
    assert np.all(row == -1) and lib.w4a16_page_free_count(a) == 6
    assert lib.w4a16_seq_reserve(a, other.ctypes.data, 4, 48) == 0
    assert len(set(other[:3].tolist())) == 3
    lib.w4a16_page_allocator_destroy(a)


def test_concurrent_alloc_and_free_from_several_threads(lib):
    """The allocator serialises its calls (one mutex per pool): threads that
    allocate and free at the same time never receive a page another thread
    still holds, and every page comes back at the end.  ctypes releases the
    GIL around each call, so the calls do overlap."""
    import threading

    n_pages, n_threads, rounds = 64, 4, 400
    a = _new(lib, n_pages)
    held, guard, errors = set(), threading.Lock(), []

    def worker(seed):
        rng = np.random.default_rng(seed)
        mine = []
        for _ in range(rounds):
            if mine and (rng.random() < 0.5 or len(mine) > 24):
                k = int(rng.integers(1, len(mine) + 1))
                give, mine = mine[:k], mine[k:]
                with guard:
                    held.difference_update(give)
                if _free(lib, a, give) != 0:
                    errors.append("free refused")
            else:
                rc, got = _alloc(lib, a, int(rng.integers(1, 6)))
                if rc == 0:
                    with guard:
                        dup = held.intersection(got.tolist())
                        if dup or len(set(got.tolist())) != got.size:
                            errors.append(f"page handed out twice: {sorted(dup)}")
                        held.update(got.tolist())
                    mine += got.tolist()
                elif rc != 8:  # W4A16_ERR_NO_PAGES is the only expected refusal
                    errors.append(f"alloc rc {rc}")
        with guard:
            held.difference_update(mine)
        if mine and _free(lib, a, mine) != 0:
            errors.append("final free refused")

    ts = [threading.Thread(target=worker, args=(100 + i,)) for i in range(n_threads)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors[:3]
    assert not held
    assert lib.w4a16_page_free_count(a) == n_pages
    rc, pages = _alloc(lib, a, n_pages)
    assert rc == 0 and sorted(pages.tolist()) == list(range(n_pages))
    lib.w4a16_page_allocator_destroy(a)
