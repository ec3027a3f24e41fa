"""Paged KV cache bookkeeping for the oracle (test infrastructure only).

Covers: packing variable-length queries into cu_seqlens, the page (block) table
built from a FIFO free list, the slot mapping of new tokens, the KV append into
pages, and the gather of a sequence's keys/values through its block table.
"""

import numpy as np


def pack_cu_seqlens(lengths):
    """cu_seqlens for a packed batch: [0, l0, l0+l1, ...] (int32).

    [CANN] §2.3: a batch of lengths [128, 64, 256] is packed into one buffer of 448 tokens
    with cu_seqlens = [0, 128, 192, 448].  [CANN] §4.4 requires cu_seqlens[0] == 0 and
    strictly increasing entries, i.e. every length >= 1.
    """
    lengths = [int(x) for x in lengths]
    if any(x < 1 for x in lengths):
        raise ValueError("every packed sequence needs at least one token")
    cu = [0]
    for x in lengths:
        cu.append(cu[-1] + x)
    return np.array(cu, dtype=np.int32)


def allocate_block_table(context_lens, block_size, free_list, max_blocks):
    """Block table [S, max_blocks] (int32, -1 = unallocated) from a FIFO free list.

    [CANN] §2.2: a sequence of L tokens takes ceil(L / page_size) pages (327 tokens at 16
    per page -> 21 pages); page_table[i][j] is the physical page of logical page j of
    sequence i, and unallocated entries are -1 ([CANN] §3.1).  [CANN] §3.2 takes the pages
    from the front of the free list; [XY] §4.2 ``KVCacheAllocator.allocate`` pops from the
    front and raises when the list is empty.  Sequences are served in batch order.
    """
    free = [int(p) for p in free_list]
    S = len(context_lens)
    table = np.full((S, max_blocks), -1, dtype=np.int32)
    pos = 0
    for i in range(S):
        L = int(context_lens[i])
        n = -(-L // block_size)  # ceil
        if n > max_blocks:
            raise ValueError(f"sequence {i} needs {n} blocks > max_blocks {max_blocks}")
        if pos + n > len(free):
            raise RuntimeError("KV page pool exhausted")
        for j in range(n):
            table[i, j] = free[pos + j]
        pos += n
    return table


def slot_mapping(cu_seqlens_q, context_lens, block_table, block_size):
    """Physical slot of every new (packed) token, int64 [T].

    Reading (pages silent; [ATB] "KV缓存复用" and [MindIE] "Prefill Chunking" only say new
    tokens are appended after the existing cache): context_lens[i] counts the tokens of
    sequence i *including* its q_i new ones, so new token j sits at absolute position
    p = L_i - q_i + j, in logical page p // bs at offset p % bs, and its slot is
    block_table[i][p // bs] * bs + p % bs.
    """
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    S = len(cu) - 1
    slots = np.empty(int(cu[-1]), dtype=np.int64)
    for i in range(S):
        q = int(cu[i + 1] - cu[i])
        L = int(context_lens[i])
        if q > L:
            raise ValueError(f"sequence {i}: q_len {q} > context_len {L}")
        for j in range(q):
            p = L - q + j
            page = int(block_table[i, p // block_size])
            if page < 0:
                raise ValueError(f"sequence {i}: position {p} has no page")
            slots[int(cu[i]) + j] = page * block_size + p % block_size
    return slots


def kv_append(k_pages_bits, v_pages_bits, k_new_bits, v_new_bits, slots):
    """Write new K/V rows into their slots; returns new page arrays (uint16 bf16 bits).

    Pages are [P, Hkv, bs, d] ([CANN] §3.1 lays a page out as [num_heads, page_size,
    head_dim]); new rows are [T, Hkv, d].  Token t goes to page slot // bs, offset
    slot % bs, for every KV head.  A negative slot marks a padding token and is skipped.
    The copy is of bit patterns, so it is exact.
    """
    kp = np.array(k_pages_bits, dtype=np.uint16, copy=True)
    vp = np.array(v_pages_bits, dtype=np.uint16, copy=True)
    P, H, bs, d = kp.shape
    for t in range(len(slots)):
        s = int(slots[t])
        if s < 0:
            continue
        page, off = s // bs, s % bs
        if page >= P:
            raise ValueError(f"slot {s} outside the pool")
        for h in range(H):
            kp[page, h, off, :] = k_new_bits[t, h, :]
            vp[page, h, off, :] = v_new_bits[t, h, :]
    return kp, vp


def gather_kv(pages, block_table_row, context_len, kv_head):
    """The first context_len rows of one sequence's keys (or values) for one KV head.

    [CANN] §3.3: the operator finds a sequence's K/V pages through its page table; logical
    page j is physical page block_table_row[j].  Concatenating the pages in logical order
    and cutting at the context length gives the contiguous cache.
    """
    P, H, bs, d = pages.shape
    n = -(-int(context_len) // bs)
    rows = []
    for j in range(n):
        page = int(block_table_row[j])
        if not (0 <= page < P):
            raise ValueError(f"page index {page} out of range [0, {P})")
        rows.append(pages[page, kv_head])
    if not rows:
        return pages[:0, 0, 0, :]
    return np.concatenate(rows, axis=0)[: int(context_len)]
