"""Pins for the oracle's decomposer + reorder (task table): the pages' 16 x 16 decomposition,
brute-force coverage of every visible (row, key) pair, an independent stable sort and deal,
and the workspace layout of split tiles."""

import numpy as np
import pytest

from oracle import build_task_table, pack_cu_seqlens


def _pages_decompose(q_len, kv_len, blk, heads):
    """The decomposer as the pages describe it: every (q block, kv block) pair of a
    q_len x kv_len problem becomes a task whose load is its actual area times the heads."""
    out = []
    for q0 in range(0, q_len, blk):
        for k0 in range(0, kv_len, blk):
            aq, ak = min(blk, q_len - q0), min(blk, kv_len - k0)
            out.append((q0, aq, k0, k0 + ak, aq * ak * heads))
    return out


def test_matches_pages_16x16_decomposition():
    q_lens, ctx = [7, 40, 1, 16], [7, 40, 33, 100]
    cu = pack_cu_seqlens(q_lens)
    r = build_task_table(cu, ctx, 3, 3, 64, False, 5, 16, 16)
    tasks = r["tasks"]
    for i in range(4):
        for g in range(3):
            mine = sorted((int(t[2]), int(t[3]), int(t[4]), int(t[5])) for t in tasks
                          if t[0] == i and t[1] == g)
            ref = sorted((q0, aq, k0, k1) for (q0, aq, k0, k1, _) in _pages_decompose(q_lens[i], ctx[i], 16, 1))
            assert mine == ref
    expect_loads = sorted((ld for i in range(4) for g in range(3)
                           for *_, ld in _pages_decompose(q_lens[i], ctx[i], 16, 1)), reverse=True)
    assert r["loads"].tolist() == expect_loads
    assert len(tasks) == 3 * sum(-(-q // 16) * -(-L // 16) for q, L in zip(q_lens, ctx))


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("q_tile,kv_chunk,Hq,Hkv", [(3, 5, 4, 2), (1, 7, 2, 2), (4, 4, 6, 3), (128, 4096, 8, 8)])
def test_every_visible_pair_covered_exactly_once(causal, q_tile, kv_chunk, Hq, Hkv):
    q_lens, ctx = [7, 1, 9, 2, 13], [7, 19, 12, 2, 30]
    cu = pack_cu_seqlens(q_lens)
    r = build_task_table(cu, ctx, Hq, Hkv, 16, causal, 3, q_tile, kv_chunk)
    G = Hq // Hkv
    cover = {}
    for t in r["tasks"]:
        i, g, q0, qr, k0, k1, ns, ws = (int(x) for x in t)
        assert 1 <= qr <= q_tile and k0 < k1 and k1 - k0 <= kv_chunk
        assert k0 % kv_chunk == 0
        for j in range(q0, q0 + qr):
            for h in range(g * G, (g + 1) * G):
                for k in range(k0, k1):
                    cover[(i, h, j, k)] = cover.get((i, h, j, k), 0) + 1
    for i, (qn, L) in enumerate(zip(q_lens, ctx)):
        for h in range(Hq):
            for j in range(qn):
                last = (L - qn + j) if causal else L - 1
                for k in range(L):
                    c = cover.get((i, h, j, k), 0)
                    if k <= last:
                        assert c == 1, (i, h, j, k)
                    else:
                        assert c <= 1
    # keys beyond what the tile's last row can see are never scheduled
    for (i, h, j, k) in cover:
        assert k < ctx[i]


def test_sort_is_stable_descending_and_dealt_round_robin():
    rng = np.random.default_rng(0)
    q_lens = rng.integers(1, 40, size=12)
    ctx = q_lens + rng.integers(0, 90, size=12)
    cu = pack_cu_seqlens(q_lens)
    num_ctas = 7
    r = build_task_table(cu, ctx, 4, 2, 32, True, num_ctas, 8, 32)
    # rebuild the enumeration independently and sort with numpy's stable sort
    recs = []
    for i in range(12):
        for g in range(2):
            for q0 in range(0, int(q_lens[i]), 8):
                qr = min(8, int(q_lens[i]) - q0)
                hi = int(ctx[i]) - int(q_lens[i]) + q0 + qr
                for k0 in range(0, hi, 32):
                    recs.append((i, g, q0, qr, k0, min(hi, k0 + 32), qr * 2 * (min(hi, k0 + 32) - k0)))
    loads = np.array([x[-1] for x in recs])
    order = np.argsort(-loads, kind="stable")
    assert [tuple(int(v) for v in r["tasks"][p][:6]) for p in range(len(order))] == [recs[k][:6] for k in order]
    assert r["loads"].tolist() == loads[order].tolist()
    cta = np.zeros(num_ctas, np.int64)
    for p, k in enumerate(order):
        cta[p % num_ctas] += loads[k]
    assert r["cta_loads"].tolist() == cta.tolist()
    assert r["balance"] == cta.min() / cta.max()
    assert np.all(np.diff(r["loads"]) <= 0)


def test_workspace_layout_of_split_tiles():
    q_lens, ctx = [1, 20, 3], [100, 20, 50]
    cu = pack_cu_seqlens(q_lens)
    d, G = 32, 4
    r = build_task_table(cu, ctx, 8, 2, d, True, 4, 8, 16)
    merges = r["merges"]
    used = np.zeros(r["workspace_bytes"] // ((d + 1) * 4), dtype=np.int32)
    for m in merges:
        i, g, q0, qr, ns, base, z0, z1 = (int(x) for x in m)
        assert ns > 1 and z0 == 0 and z1 == 0
        used[base: base + ns * qr * G] += 1
        # the tile's splits point at consecutive slices of its region
        mine = sorted(int(t[7]) for t in r["tasks"] if t[0] == i and t[1] == g and t[2] == q0)
        assert mine == [base + c * qr * G for c in range(ns)]
    assert np.all(used == 1)
    for t in r["tasks"]:
        assert (int(t[6]) == 1) == (int(t[7]) == -1)
    # merges are listed in enumeration order and regions are allocated in that order
    bases = [int(m[5]) for m in merges]
    assert bases == sorted(bases)
    total_rows = sum(int(m[3]) * G * int(m[4]) for m in merges)
    assert r["workspace_bytes"] == total_rows * (d + 1) * 4


def test_decode_tile_and_split_counts():
    # decode: one tile of one token, kv range [0, L) cut into ceil(L / chunk) splits
    r = build_task_table([0, 1, 2], [4096, 4097], 64, 8, 128, True, 152, 16, 4096)
    t = r["tasks"]
    assert len(t) == 8 * (1 + 2)
    assert sorted(set(int(x) for x in t[:, 6])) == [1, 2]
    assert sum(int(x[5]) - int(x[4]) for x in t if x[0] == 1) == 8 * 4097


def test_empty_batch_and_errors():
    r = build_task_table([0], [], 4, 2, 64, True, 3, 8, 64)
    assert r["tasks"].shape == (0, 8) and r["workspace_bytes"] == 0 and r["balance"] == 1.0
    with pytest.raises(ValueError):
        build_task_table([0, 5], [4], 4, 2, 64, True, 3, 8, 64)   # q_len > context
    with pytest.raises(ValueError):
        build_task_table([0, 1], [4], 6, 4, 64, True, 3, 8, 64)   # Hq not a multiple of Hkv


def _area_order(r0):
    return [tuple(int(v) for v in t) for t in r0["tasks"]]


def test_mixed_schedule_equals_serpentine_schedule_without_small_tasks():
    # every task carries >= 128 rows (q_tile 32 x G 4, q_len a multiple of 32): charging
    # max(rows, 128) changes no load and there is nothing to alternate with, so the tables coincide
    cu = pack_cu_seqlens([192, 256, 128])
    ctx = [900, 256, 4000]
    a = build_task_table(cu, ctx, 8, 2, 128, True, 5, 32, 256, schedule=1)
    b = build_task_table(cu, ctx, 8, 2, 128, True, 5, 32, 256, schedule=2)
    assert all(int(t[3]) * 4 >= 128 for t in a["tasks"])
    assert np.array_equal(a["tasks"], b["tasks"]) and a["balance"] == b["balance"]


def test_mixed_schedule_equals_serpentine_schedule_for_pure_decode():
    # all tasks are 1-row decode tasks (G = 1): every load is scaled by the same 128
    rng = np.random.default_rng(3)
    ctx = rng.integers(1, 5000, size=40)
    cu = pack_cu_seqlens(np.ones(40, dtype=np.int64))
    a = build_task_table(cu, ctx, 4, 4, 128, True, 9, 1, 512, schedule=1)
    b = build_task_table(cu, ctx, 4, 4, 128, True, 9, 1, 512, schedule=2)
    assert np.array_equal(a["tasks"], b["tasks"])
    assert b["loads"].tolist() == (a["loads"] * 128).tolist()


def test_mixed_schedule_interleaves_in_proportion_within_each_cta():
    rng = np.random.default_rng(4)
    q_lens = np.concatenate([np.full(6, 300), np.ones(50, dtype=np.int64)])
    ctx = q_lens + rng.integers(0, 3000, size=len(q_lens))
    cu = pack_cu_seqlens(q_lens)
    G, num_ctas, q_tile, chunk = 4, 11, 32, 512
    b = build_task_table(cu, ctx, 8, 2, 128, True, num_ctas, q_tile, chunk, schedule=2)
    # rebuild the charged loads (padded 128-row tiles; small tasks as one tile), sort and deal
    recs = []
    for i in range(len(q_lens)):
        qn, L = int(q_lens[i]), int(ctx[i])
        for g in range(2):
            for q0 in range(0, qn, q_tile):
                qr = min(q_tile, qn - q0)
                hi = L - qn + q0 + qr
                for k0 in range(0, hi, chunk):
                    k1 = min(hi, k0 + chunk)
                    recs.append(((i, g, q0, qr, k0, k1), 128 * (k1 - k0)))
    order = np.argsort(-np.array([x[1] for x in recs]), kind="stable")
    assert len(order) == len(b["tasks"])
    got = [tuple(int(v) for v in t[:6]) for t in b["tasks"]]
    load_of = {x[0]: x[1] for x in recs}
    dealt_to = _serpentine_assignment(len(order), num_ctas)
    both = 0
    for c in range(num_ctas):
        dealt = [recs[order[p]][0] for p in range(len(order)) if dealt_to[p] == c]
        mine = got[c::num_ctas]
        assert sorted(mine) == sorted(dealt)
        assert int(b["cta_loads"][c]) == sum(load_of[x] for x in dealt)
        lists = {}
        for kind in (True, False):
            want = [x for x in dealt if (x[3] * G > 16) == kind]
            seen = [x for x in mine if (x[3] * G > 16) == kind]
            # each kind runs its dealt order, rotated to start at the CTA's phase c / num_ctas
            assert len(seen) == len(want)
            if want:
                r = want.index(seen[0])
                assert seen == want[r:] + want[:r]
                tot = sum(load_of[x] for x in want)
                starts = np.cumsum([0] + [load_of[x] for x in want[:-1]])
                # a task starting at fraction s of its list runs at time (s + c / num_ctas) mod 1:
                # the CTA begins with the first task at s >= 1 - c / num_ctas (else the first one)
                late = [q for q in range(len(want)) if starts[q] * num_ctas >= (num_ctas - c) * tot]
                assert r == (late[0] if late else 0)
            lists[kind] = (want, seen)
        if not lists[True][0] or not lists[False][0]:
            continue
        both += 1
        # proportionality: whenever a task starts, the fraction of each list already run (from
        # the phase on) differs by less than one task's share of that list
        frac = {k: 0.0 for k in (True, False)}
        tot = {k: sum(load_of[x] for x in lists[k][0]) for k in (True, False)}
        biggest = {k: max(load_of[x] for x in lists[k][0]) / tot[k] for k in (True, False)}
        for x in mine:
            k = x[3] * G > 16
            other = not k
            assert frac[k] <= frac[other] + biggest[other] + 1e-12
            frac[k] += load_of[x] / tot[k]
    assert both > 0


def _serpentine_assignment(N, n):
    """CTA of each sorted position under the serpentine reading of "symmetric round-robin":
    complete rounds alternate direction (round 0 forwards), the final partial round forwards."""
    out = []
    for p in range(N):
        r, i = divmod(p, n)
        backwards = r % 2 == 1 and (r + 1) * n <= N
        out.append(n - 1 - i if backwards else i)
    return out


def test_serpentine_schedule_deals_alternate_rounds_backwards():
    rng = np.random.default_rng(9)
    q_lens = rng.integers(1, 60, size=15)
    ctx = q_lens + rng.integers(0, 200, size=15)
    cu = pack_cu_seqlens(q_lens)
    num_ctas = 5
    a = build_task_table(cu, ctx, 4, 2, 32, True, num_ctas, 8, 32, schedule=0)
    s = build_task_table(cu, ctx, 4, 2, 32, True, num_ctas, 8, 32, schedule=1)
    N = len(a["tasks"])
    assert N % num_ctas != 0 and (N // num_ctas) % 2 == 1   # a partial final round after an odd one
    sorted_tasks = [tuple(int(v) for v in t) for t in a["tasks"]]   # schedule 0 = the plain sorted list
    cta = _serpentine_assignment(N, num_ctas)
    for c in range(num_ctas):
        mine = [sorted_tasks[p] for p in range(N) if cta[p] == c]
        assert [tuple(int(v) for v in t) for t in s["tasks"][c::num_ctas]] == mine
    # every CTA of a complete round gets one task of it; the sum of loads is unchanged
    assert int(s["loads"].sum()) == int(a["loads"].sum())
    assert sorted(s["loads"].tolist()) == sorted(a["loads"].tolist())
    # on a sorted list the serpentine deal is never less balanced than the plain one here
    assert s["balance"] >= a["balance"]


def test_unknown_schedule_rejected():
    with pytest.raises(ValueError):
        build_task_table([0, 1], [4], 4, 2, 64, True, 3, 8, 64, schedule=5)


def test_dynamic_schedule_is_the_greedy_loads_sorted_and_undealt():
    # schedule 4 holds exactly the greedy schedule's tasks (no holes) in descending order of the
    # same loads, except that the tasks of a chunk over a long prior context (q > 1 new tokens,
    # L - q >= q) follow the largest task of their (sequence, KV head): the group leaders and the
    # other tasks form a descending list, each group is contiguous and descending, and ties keep
    # the enumeration order (sequence, kv head, query tile, chunk) -- which fixes the order
    rng = np.random.default_rng(8)
    q = rng.integers(1, 40, size=9)
    L = q + rng.integers(0, 900, size=9)
    q[0], L[1] = 1, q[1]   # a decode row and a prompt without prior context beside the chunks
    cu = np.concatenate([[0], np.cumsum(q)])
    dyn = build_task_table(cu, L, 8, 2, 128, True, 5, 16, 256, schedule=4)
    gre = build_task_table(cu, L, 8, 2, 128, True, 5, 16, 256, schedule=3)
    real = gre["tasks"][gre["tasks"][:, 0] >= 0]
    assert len(dyn["tasks"]) == len(real) and not np.any(dyn["tasks"][:, 0] < 0)
    key = lambda t: tuple(t)
    assert sorted(map(key, dyn["tasks"])) == sorted(map(key, real))
    tasks, loads = dyn["tasks"], dyn["loads"]
    chunk = {i for i in range(len(q)) if q[i] > 1 and L[i] - q[i] >= q[i]}
    assert 0 < len(chunk) < len(q)
    group = [(int(t[0]), int(t[1])) if int(t[0]) in chunk else None for t in tasks]
    assert any(sum(1 for x in group if x == g) > 1 for g in set(group) if g is not None)

    def enum_order(a, b):
        ta, tb = tasks[a], tasks[b]
        return (ta[0], ta[1], ta[2], ta[4]) < (tb[0], tb[1], tb[2], tb[4])

    heads, seen, pos = [], set(), 0
    while pos < len(tasks):
        heads.append(pos)
        g, end = group[pos], pos
        if g is not None:
            assert g not in seen   # a group is contiguous
            seen.add(g)
            while end + 1 < len(tasks) and group[end + 1] == g:
                end += 1
            for a in range(pos, end):
                assert loads[a] > loads[a + 1] or (loads[a] == loads[a + 1] and enum_order(a, a + 1))
        pos = end + 1
    for a, b in zip(heads, heads[1:]):
        assert loads[a] > loads[b] or (loads[a] == loads[b] and enum_order(a, b))


def test_greedy_schedule_is_longest_processing_time_first():
    rng = np.random.default_rng(12)
    q_lens = np.concatenate([rng.integers(30, 400, size=6), np.ones(30, dtype=np.int64)])
    ctx = q_lens + rng.integers(0, 3000, size=len(q_lens))
    cu = pack_cu_seqlens(q_lens)
    n, G = 7, 4
    g = build_task_table(cu, ctx, 8, 2, 128, True, n, 32, 512, schedule=3)
    a = build_task_table(cu, ctx, 8, 2, 128, True, n, 32, 512, schedule=0)
    real = [tuple(int(v) for v in t) for t in a["tasks"]]
    # the same tasks, plus hole records; the table is num_ctas times the longest list
    got = [tuple(int(v) for v in t) for t in g["tasks"]]
    holes = [t for t in got if t == (-1, 0, 0, 0, 0, 0, 0, -1)]
    assert sorted(t for t in got if t[0] >= 0) == sorted(real)
    assert len(got) % n == 0 and len(got) == len(real) + len(holes)
    # independent restatement: charged load, stable sort, each task to the least loaded CTA
    def charged(t):
        rows = t[3] * G
        return 128 * max(1, -(-rows // 128)) * (t[5] - t[4] + 512)
    real.sort(key=lambda t: (t[0], t[1], t[2], t[4]))       # enumeration order
    order = sorted(range(len(real)), key=lambda k: charged(real[k]), reverse=True)
    load = [0] * n
    lists = [[] for _ in range(n)]
    for k in order:
        c = min(range(n), key=lambda c: (load[c], c))
        lists[c].append(real[k])
        load[c] += charged(real[k])
    for c in range(n):
        mine = [t for t in got[c::n] if t[0] >= 0]
        assert mine == lists[c]
        # a CTA's holes come after its tasks
        seq = [t[0] >= 0 for t in got[c::n]]
        assert seq == sorted(seq, reverse=True)
    assert g["cta_loads"].tolist() == load
    # greedy never balances worse than the plain deal of the same charged loads
    assert g["balance"] >= min(load) / max(load) - 1e-12
