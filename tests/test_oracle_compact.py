"""Pins of the oracle's accepted-branch KV compaction (SD 20.5, "Keeping the caches
consistent after a rejection"): hand-worked layouts, the chain case (no move, only the
length), paged and contiguous layouts agreeing, and the untouched regions."""
import numpy as np

from oracle import specdec_oracle as so


def test_hand_worked_tree_compaction():
    """Prefix of 3 slots, a 6-node tree; the walk accepted nodes 1 then 4 (a child of 1):
    slot 3 takes node 1's entry and slot 4 node 4's; everything else stays."""
    S, W = 12, 2
    cache = np.arange(S * W, dtype=np.int64).reshape(1, S, W)
    out, new_len, st = so.compact_kv(cache, [3], [[1, 4, -1]], [2])
    want = cache.copy()
    want[0, 3] = cache[0, 3 + 1]
    want[0, 4] = cache[0, 3 + 4]
    np.testing.assert_array_equal(out, want)
    assert list(new_len) == [5] and list(st) == [0]


def test_chain_paths_only_move_the_length():
    rng = np.random.default_rng(0)
    cache = rng.integers(0, 1000, size=(4, 20, 3))
    J = [0, 3, 5, -1]
    paths = [list(range(5)) for _ in J]
    out, new_len, st = so.compact_kv(cache, [2, 4, 6, 1], paths, J)
    np.testing.assert_array_equal(out, cache)
    assert list(new_len) == [2, 7, 11, 1] and not st.any()


def test_paged_layout_matches_the_contiguous_one():
    rng = np.random.default_rng(1)
    B, S, W, bs = 3, 16, 4, 4
    cache = rng.integers(0, 10 ** 6, size=(B, S, W))
    perm = rng.permutation(B * S // bs)
    table = perm.reshape(B, S // bs)
    pool = np.zeros((B * S // bs, bs, W), dtype=cache.dtype)
    for b in range(B):
        for blk in range(S // bs):
            pool[table[b, blk]] = cache[b, blk * bs:(blk + 1) * bs]
    prefix, paths, J = [2, 5, 0], [[0, 3, 7], [2, 4, -1], [1, 5, 9]], [3, 2, 3]
    flat, l1, s1 = so.compact_kv(cache, prefix, paths, J)
    paged, l2, s2 = so.compact_kv(pool, prefix, paths, J, block_table=table, block_size=bs)
    for b in range(B):
        for blk in range(S // bs):
            np.testing.assert_array_equal(paged[table[b, blk]], flat[b, blk * bs:(blk + 1) * bs])
    assert list(l1) == list(l2) == [5, 7, 3]


def test_invalid_paths_leave_the_sequence_alone():
    cache = np.arange(40).reshape(2, 10, 2)
    out, new_len, st = so.compact_kv(cache, [1, 1], [[2, 1], [0, 0]], [2, 2])
    np.testing.assert_array_equal(out, cache)
    assert list(st) == [so.STATUS_BAD_TREE] * 2 and list(new_len) == [1, 1]


def test_sequential_in_place_moves_equal_the_gather():
    """Moving depth by depth in place (what a kernel does) gives the gather's result for
    every climbing path: a source slot is never a destination written earlier."""
    rng = np.random.default_rng(2)
    for _ in range(200):
        S, P0 = 30, int(rng.integers(0, 5))
        J = int(rng.integers(0, 8))
        path = np.sort(rng.choice(np.arange(S - P0 - 1), J, replace=False)) if J else np.zeros(0, int)
        path = np.maximum(path, np.arange(J))
        if J and (np.diff(path) <= 0).any():
            continue
        cache = rng.integers(0, 10 ** 6, size=(1, S, 2))
        want, _, st = so.compact_kv(cache, [P0], [list(path)], [J])
        assert not st.any()
        seq = cache.copy()
        for d in range(J):
            seq[0, P0 + d] = seq[0, P0 + path[d]]
        np.testing.assert_array_equal(seq, want)
