"""Pins for the oracle's paged-KV bookkeeping: packing, block table, slots, append, gather."""

import json
import os

import numpy as np
import pytest

from oracle import allocate_block_table, gather_kv, kv_append, pack_cu_seqlens, slot_mapping

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_pack_matches_page_example():
    g = _golden("packed_cu_seqlens.json")
    cu = pack_cu_seqlens(g["lengths"])
    assert cu.tolist() == g["cu_seqlens"]
    assert int(cu[-1]) == g["total_tokens"]
    assert cu.dtype == np.int32


def test_pack_rejects_empty_sequence():
    with pytest.raises(ValueError):
        pack_cu_seqlens([3, 0, 2])


def test_page_counts_match_pages():
    for c in _golden("page_counts.json")["cases"]:
        bs = c["page_size"]
        need = c["pages"]
        free = np.arange(need + 5, dtype=np.int32)
        bt = allocate_block_table([c["tokens"]], bs, free, max_blocks=need + 3)
        assert int((bt[0] >= 0).sum()) == need
        assert bt[0, need:].tolist() == [-1] * 3


def test_allocator_is_fifo_in_batch_order():
    free = np.array([9, 4, 7, 1, 0, 3, 8, 2, 6, 5], dtype=np.int32)
    bt = allocate_block_table([5, 1, 9, 4], 4, free, max_blocks=3)
    # ceil(5/4)=2, ceil(1/4)=1, ceil(9/4)=3, ceil(4/4)=1 pages, taken from the front in order
    assert bt.tolist() == [[9, 4, -1], [7, -1, -1], [1, 0, 3], [8, -1, -1]]


def test_allocator_raises_when_pool_exhausted():
    with pytest.raises(RuntimeError):
        allocate_block_table([16, 17], 16, np.arange(2, dtype=np.int32), max_blocks=2)
    with pytest.raises(ValueError):
        allocate_block_table([33], 16, np.arange(8, dtype=np.int32), max_blocks=2)


def test_slot_mapping_hand_example():
    # seq 0: L=6, q=2 -> positions 4, 5 -> logical page 1 (physical 2) offsets 0, 1
    # seq 1: L=3, q=3 -> positions 0, 1, 2 -> logical page 0 (physical 7)
    bt = np.array([[5, 2], [7, -1]], dtype=np.int32)
    slots = slot_mapping([0, 2, 5], [6, 3], bt, 4)
    assert slots.tolist() == [8, 9, 28, 29, 30]
    assert slots.dtype == np.int64


def test_append_then_gather_round_trip():
    rng = np.random.default_rng(3)
    P, H, bs, d = 12, 2, 4, 8
    L = [7, 3, 10]
    q = [7, 1, 4]
    free = rng.permutation(P).astype(np.int32)
    bt = allocate_block_table(L, bs, free, max_blocks=3)
    cu = pack_cu_seqlens(q)
    T = int(cu[-1])
    kp = rng.integers(0, 1 << 16, size=(P, H, bs, d), dtype=np.uint16)
    vp = rng.integers(0, 1 << 16, size=(P, H, bs, d), dtype=np.uint16)
    kn = rng.integers(0, 1 << 16, size=(T, H, d), dtype=np.uint16)
    vn = rng.integers(0, 1 << 16, size=(T, H, d), dtype=np.uint16)
    slots = slot_mapping(cu, L, bt, bs)
    kp2, vp2 = kv_append(kp, vp, kn, vn, slots)
    touched = np.zeros((P, bs), dtype=bool)
    for i in range(3):
        for h in range(H):
            K = gather_kv(kp2, bt[i], L[i], h)
            V = gather_kv(vp2, bt[i], L[i], h)
            assert K.shape == (L[i], d)
            # the last q_i rows of the gathered cache are exactly the new tokens
            assert np.array_equal(K[L[i] - q[i]:], kn[cu[i]:cu[i + 1], h])
            assert np.array_equal(V[L[i] - q[i]:], vn[cu[i]:cu[i + 1], h])
            # and the prior rows are what the pages held before
            assert np.array_equal(K[: L[i] - q[i]], gather_kv(kp, bt[i], L[i], h)[: L[i] - q[i]])
        for j in range(q[i]):
            s = int(slots[cu[i] + j])
            touched[s // bs, s % bs] = True
    # untouched slots keep their bits
    for p in range(P):
        for o in range(bs):
            if not touched[p, o]:
                assert np.array_equal(kp2[p, :, o], kp[p, :, o])
                assert np.array_equal(vp2[p, :, o], vp[p, :, o])


def test_append_skips_negative_slots():
    kp = np.zeros((2, 1, 4, 2), np.uint16)
    kn = np.full((2, 1, 2), 7, np.uint16)
    kp2, _ = kv_append(kp, kp, kn, kn, np.array([-1, 5]))
    assert kp2[1, 0, 1].tolist() == [7, 7]
    assert int(kp2.sum()) == 14


def test_gather_contiguous_identity_table():
    P, H, bs, d = 6, 1, 4, 3
    pages = np.arange(P * H * bs * d, dtype=np.float64).reshape(P, H, bs, d)
    bt = np.arange(P, dtype=np.int32)
    K = gather_kv(pages, bt, 22, 0)
    assert np.array_equal(K, pages[:, 0].reshape(P * bs, d)[:22])


def test_gather_rejects_out_of_range_page():
    pages = np.zeros((3, 1, 4, 2))
    with pytest.raises(ValueError):
        gather_kv(pages, np.array([0, 3]), 8, 0)
    with pytest.raises(ValueError):
        gather_kv(pages, np.array([0, -1]), 8, 0)
