"""The block-table (paged) cache the oracle reads: a permuted pool read back
through its block table is the contiguous cache again."""
import numpy as np

import oracle


def test_permuted_pool_round_trip():
    rng = np.random.default_rng(3)
    B, Tcap = 3, 40
    kv = rng.integers(0, 1 << 16, size=(B, Tcap, 512), dtype=np.uint16)
    kr = rng.integers(0, 1 << 16, size=(B, Tcap, 64), dtype=np.uint16)
    extra = 17
    perm = rng.permutation(B * Tcap + extra)  # pool row of each (b, p), junk rows in between
    pool_kv = rng.integers(0, 1 << 16, size=(B * Tcap + extra, 512), dtype=np.uint16)
    pool_kr = rng.integers(0, 1 << 16, size=(B * Tcap + extra, 64), dtype=np.uint16)
    kvi = perm[: B * Tcap].reshape(B, Tcap).astype(np.int32)
    pool_kv[kvi.ravel()] = kv.reshape(-1, 512)
    pool_kr[kvi.ravel()] = kr.reshape(-1, 64)
    gkv, gkr = oracle.gather_paged(pool_kv, pool_kr, kvi)
    np.testing.assert_array_equal(gkv, kv)
    np.testing.assert_array_equal(gkr, kr)


def test_out_of_range_entries_read_as_zero():
    pool_kv = np.ones((4, 512), np.uint16)
    pool_kr = np.ones((4, 64), np.uint16)
    kvi = np.array([[0, 3, -1, 4]], np.int32)
    gkv, gkr = oracle.gather_paged(pool_kv, pool_kr, kvi)
    assert gkv[0, :2].min() == 1 and gkv[0, 2:].max() == 0 and gkr[0, 2:].max() == 0
