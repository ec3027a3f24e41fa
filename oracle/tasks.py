"""Dynamic decomposer + attention task reorder, restated for the oracle (test infrastructure only).

[XY] §2.2 component 1 / §4.4 ``decompose_attention``: the (q_len x kv_len) work of a
sequence is cut into fixed-size (query block x KV block) tasks that record their ranges,
their actual shape and a compute load equal to the tile area (times the heads).
[XY] §2.2 component 2 ``AttentionTaskReorder.reorder``: tasks are sorted by load,
largest first, and dealt round-robin, task i going to core i mod num_cores; the ratio
min/max of the per-core load sums measures the balance.

Readings taken here (the pages are written for 16 x 16 Ascend blocks):

* The unit of work is one (sequence, KV head, query tile, KV chunk).  A query tile holds
  ``q_tile`` tokens and all G = Hq / Hkv query heads that share the KV head, so a tile
  has q_rows * G score rows.  The KV range of a tile is cut into chunks of ``kv_chunk``
  keys ("split-KV"); with causal attention the range ends at the last visible key of the
  tile's last row (L - q + row_end), otherwise at L.
* load = q_rows * G * (kv_end - kv_start): the tile area times the heads it carries.
* The sort is stable (Python ``sorted`` keeps equal keys in enumeration order, which is
  sequence -> KV head -> query tile -> chunk); the deal is plain ``i % num_ctas``.
* A tile split into n > 1 chunks writes n partial results to a workspace and needs one
  merge; partial rows are numbered in enumeration order: the tile's group starts at
  ws_row and chunk c owns rows ws_row + c * q_rows * G + t * G + h_local.
"""

from fractions import Fraction
import heapq

import numpy as np

TASK_FIELDS = ("seq", "kv_head", "q_start", "q_rows", "kv_start", "kv_end", "num_splits", "ws_row")
MERGE_FIELDS = ("seq", "kv_head", "q_start", "q_rows", "num_splits", "ws_row", "zero0", "zero1")


# Schedules (the pages' reorder is schedule 0):
# * 1 reads "symmetric round-robin" as a serpentine deal: the same stable sort by area, then every
#   complete odd round of num_ctas positions goes to the CTAs in reverse order (CTA num_ctas-1
#   first), so a CTA that took one of the largest tasks of a round takes one of the smallest of the
#   next; the final partial round keeps the plain order, so the table stays dense.
# * 2 is a variant for batches that mix HBM-bound decode tasks with tensor-core tiles:
#   charged load = TILE_ROWS * max(1, ceil(rows / TILE_ROWS)) * keys (a tile costs its padded
#   128-row MMA area; a small task, rows <= SMALL_ROWS, streams its keys' KV in about the time of
#   one 128-row tile over the same keys), the serpentine deal of schedule 1, then each CTA
#   interleaves its small and large tasks in proportion to their charged loads, starting at phase
#   c / num_ctas of its timeline, so that at any moment about the small tasks' share of the CTAs
#   streams KV while the others keep the tensor cores busy.
# * 3 deals greedily (longest processing time first): tasks sorted by a load that also charges
#   a fixed per-task cost, TILE_ROWS * max(1, ceil(rows / TILE_ROWS)) * (keys + TASK_KEYS), each to
#   the CTA with the smallest load so far (the lowest index on ties).  CTAs then hold different
#   numbers of tasks; the table keeps the layout "CTA c runs positions c, c + num_ctas, ..." and
#   fills the positions a CTA does not use with HOLE records, which the kernels skip.
SMALL_ROWS = 16
TILE_ROWS = 128
TASK_KEYS = 512
MAX_TOTAL_LOAD = 1 << 55
MAX_CTAS = 1 << 16
SCHEDULES = (0, 1, 2, 3, 4)
HOLE = (-1, 0, 0, 0, 0, 0, 0, -1)


def _serpentine(order, num_ctas):
    """Reverse every complete odd round of the dealt order (see schedule 1)."""
    out = list(order)
    for r in range(1, len(order) // num_ctas, 2):
        out[r * num_ctas:(r + 1) * num_ctas] = order[r * num_ctas:(r + 1) * num_ctas][::-1]
    return out


def _charged_rows(rows):
    return TILE_ROWS * max(1, -(-rows // TILE_ROWS))


def _interleave(big, small, c, num_ctas):
    """Order one CTA's tasks.  big / small: lists of (task, load) in dealt order.  Each task gets
    the key (start of the task within its own list + phase) mod 1, where start = loads before it /
    the list's total and phase = c / num_ctas; tasks run by increasing key, a large task first
    on a tie.  Exact rational arithmetic (Python integers)."""
    if not big or not small:
        return [t for t, _ in big] + [t for t, _ in small]
    keyed = []
    for kind, lst in ((0, big), (1, small)):
        tot = sum(ld for _, ld in lst)
        done = 0
        for t, ld in lst:
            keyed.append(((Fraction(done, tot) + Fraction(c, num_ctas)) % 1, kind, t))
            done += ld
    keyed.sort(key=lambda x: (x[0], x[1]))
    return [t for _, _, t in keyed]


def _group_chunk_tasks(order, records, cu, context_lens):
    """Schedule 4's order after the sort: the tasks of one (sequence, KV head) whose sequence is a
    chunk over a long prior context (more than one new token, prior context L - q >= q) follow the
    first of them in the sorted order, keeping their own order; every other task keeps its place.
    Written as its definition: a stable sort by (position of the group's first task, position)."""
    first = {}
    keyed = []
    for pos, k in enumerate(order):
        i, g = records[k][0], records[k][1]
        qn = cu[i + 1] - cu[i]
        if qn > 1 and int(context_lens[i]) - qn >= qn:
            first.setdefault((i, g), pos)
            keyed.append((first[(i, g)], pos, k))
        else:
            keyed.append((pos, pos, k))
    keyed.sort(key=lambda x: (x[0], x[1]))
    return [k for _, _, k in keyed]


def build_task_table(cu_seqlens_q, context_lens, num_heads_q, num_heads_kv, head_dim, causal,
                     num_ctas, q_tile, kv_chunk, schedule=0):
    """Return dict(tasks=int32 [n, 8] in dealt order, merges=int32 [m, 8], loads=int64 [n],
    cta_loads=int64 [num_ctas], balance=min/max, workspace_bytes=int).

    CTA c runs tasks c, c + num_ctas, c + 2*num_ctas, ... of ``tasks``.
    schedule 0: the pages' reorder (load = area, stable sort descending, round-robin deal).
    schedule 1: the same sort, serpentine deal.  schedule 2: charged load, serpentine deal and
    per-CTA proportional interleave.  schedule 3: greedy deal with HOLE records (see above).
    schedule 4: schedule 3's loads, sorted, not dealt: the CTAs claim tasks in this order at run
    time (the cta_loads reported are those of positions mod num_ctas); the tasks of a chunk over a
    long prior context are then brought together (_group_chunk_tasks).
    """
    if schedule not in SCHEDULES:
        raise ValueError("schedule must be 0, 1, 2, 3 or 4")
    if num_heads_q % num_heads_kv:
        raise ValueError("Hq must be a multiple of Hkv")
    if q_tile < 1 or kv_chunk < 1 or num_ctas < 1:
        raise ValueError("q_tile, kv_chunk and num_ctas must be positive")
    G = num_heads_q // num_heads_kv
    cu = [int(x) for x in cu_seqlens_q]
    S = len(cu) - 1

    records, loads, merges = [], [], []
    ws_rows = 0
    for i in range(S):
        qn = cu[i + 1] - cu[i]
        L = int(context_lens[i])
        if qn < 1 or qn > L:
            raise ValueError(f"sequence {i}: need 1 <= q_len <= context_len")
        for g in range(num_heads_kv):
            for t0 in range(0, qn, q_tile):
                rows = min(q_tile, qn - t0)
                kv_hi = (L - qn + t0 + rows) if causal else L
                nsplit = -(-kv_hi // kv_chunk)
                base = -1
                if nsplit > 1:
                    base = ws_rows
                    merges.append((i, g, t0, rows, nsplit, base, 0, 0))
                    ws_rows += nsplit * rows * G
                for c in range(nsplit):
                    k0 = c * kv_chunk
                    k1 = min(kv_hi, k0 + kv_chunk)
                    row = -1 if nsplit == 1 else base + c * rows * G
                    records.append((i, g, t0, rows, k0, k1, nsplit, row))
                    r = rows * G
                    if schedule == 2:
                        r = _charged_rows(r)
                    if schedule in (3, 4):
                        loads.append(_charged_rows(r) * (k1 - k0 + TASK_KEYS))
                    else:
                        loads.append(r * (k1 - k0))

    order = sorted(range(len(records)), key=lambda k: loads[k], reverse=True)
    if schedule == 4:
        order = _group_chunk_tasks(order, records, cu, context_lens)
    if schedule in (1, 2):
        order = _serpentine(order, num_ctas)
    if schedule == 2:
        if sum(loads) >= MAX_TOTAL_LOAD or num_ctas > MAX_CTAS:
            raise ValueError("total load or num_ctas too large for schedule 1")
        # positions c, c + num_ctas, ... belong to CTA c; reorder each CTA's tasks among them
        for c in range(min(num_ctas, len(order))):
            pos = list(range(c, len(order), num_ctas))
            big = [(k, loads[k]) for k in (order[q] for q in pos) if records[k][3] * G > SMALL_ROWS]
            small = [(k, loads[k]) for k in (order[q] for q in pos) if records[k][3] * G <= SMALL_ROWS]
            for q, k in zip(pos, _interleave(big, small, c, num_ctas)):
                order[q] = k
    if schedule == 3:
        if sum(loads) >= MAX_TOTAL_LOAD:
            raise ValueError("total load too large for schedule 3")
        heap = [(0, c) for c in range(num_ctas)]
        lists = [[] for _ in range(num_ctas)]
        for k in order:
            ld, c = heapq.heappop(heap)
            lists[c].append(k)
            heapq.heappush(heap, (ld + loads[k], c))
        depth = max((len(x) for x in lists), default=0)
        order = [None] * (depth * num_ctas)
        for c, lst in enumerate(lists):
            for pos, k in enumerate(lst):
                order[pos * num_ctas + c] = k
    tasks = np.array([records[k] if k is not None else HOLE for k in order], dtype=np.int32).reshape(-1, 8)
    sorted_loads = np.array([loads[k] if k is not None else 0 for k in order], dtype=np.int64)

    cta_loads = np.zeros(num_ctas, dtype=np.int64)
    for pos, ld in enumerate(sorted_loads):
        cta_loads[pos % num_ctas] += ld
    mx = int(cta_loads.max()) if num_ctas else 0
    balance = (int(cta_loads.min()) / mx) if mx > 0 else 1.0

    return dict(
        tasks=tasks,
        merges=np.array(merges, dtype=np.int32).reshape(-1, 8),
        loads=sorted_loads,
        cta_loads=cta_loads,
        balance=balance,
        workspace_bytes=ws_rows * (head_dim + 1) * 4,
    )
