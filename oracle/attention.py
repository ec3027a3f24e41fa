"""Attention over the paged KV cache, in float64 (test infrastructure only).

What is computed is the definition of attention ([XY] §1.1: a query is scored against
every key it may see, the scores are normalised with a softmax, and the values are
averaged with those weights), over the keys gathered through the block table
([CANN] §3.3), with the causal mask of the packed operator ([CANN] §3.3,
``is_causal=True``) and the virtual mask of ragged tiles ([XY] §2.3 technique 1).
"""

import math

import numpy as np

from .paged import gather_kv


def virtual_mask(q_rows, kv_cols, tile_q=16, tile_kv=16):
    """Boolean [tile_q, tile_kv] mask of the valid cells of a ragged tile.

    [XY] §2.3 technique 1: a [7, 13] block in a 16 x 16 tile keeps 7*13 = 91 valid cells; the
    other cells are masked on chip instead of padded in memory.
    """
    m = np.zeros((tile_q, tile_kv), dtype=bool)
    m[:q_rows, :kv_cols] = True
    return m


def attention_row(q, K, V, n_valid, scale):
    """One output row: softmax(scale * K[:n] q) weighted sum of V[:n], in float64.

    n_valid >= 1 keys are visible (every row sees at least its own key).  The maximum is
    subtracted before exp, which does not change the softmax.
    """
    if n_valid < 1:
        raise ValueError("a row must see at least one key")
    s = scale * (K[:n_valid] @ q)
    s = s - s.max()
    w = np.exp(s)
    w = w / w.sum()
    return w @ V[:n_valid]


def _visible_keys(context_len, q_len, j, causal):
    """Keys visible to new token j of a sequence: all L keys, or (causal) the keys up to
    its absolute position L - q + j (bottom-right alignment with the prior context)."""
    if causal:
        return context_len - q_len + j + 1
    return context_len


def paged_attention(q, cu_seqlens_q, context_lens, block_table, k_pages, v_pages, scale, causal):
    """Output [T, Hq, d] float64 of attention for a packed batch over a paged cache.

    q: float64 [T, Hq, d]; k_pages/v_pages: float64 [P, Hkv, bs, d].  Query head h reads KV
    head h // (Hq / Hkv) (contiguous GQA groups; the pages only show equal head counts).
    Sequence i owns packed rows cu[i]..cu[i+1]-1 ([CANN] §2.3) and sees context_lens[i]
    keys, which include its own new tokens.
    """
    T, Hq, d = q.shape
    Hkv = k_pages.shape[1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    out = np.zeros((T, Hq, d), dtype=np.float64)
    S = len(cu_seqlens_q) - 1
    for i in range(S):
        t0, t1 = int(cu_seqlens_q[i]), int(cu_seqlens_q[i + 1])
        qn, L = t1 - t0, int(context_lens[i])
        if qn > L:
            raise ValueError(f"sequence {i}: q_len {qn} > context_len {L}")
        for g in range(Hkv):
            K = gather_kv(k_pages, block_table[i], L, g)
            V = gather_kv(v_pages, block_table[i], L, g)
            for h in range(g * G, (g + 1) * G):
                for j in range(qn):
                    n = _visible_keys(L, qn, j, causal)
                    out[t0 + j, h] = attention_row(q[t0 + j, h], K, V, n, scale)
    return out


def attention_rows(rows, q, cu_seqlens_q, context_lens, block_table, k_pages, v_pages, scale, causal):
    """Selected output rows: ``rows`` is a list of (packed token t, query head h).

    Same definition as ``paged_attention`` for the listed rows only, so that full-size
    batches can be checked on a sample.
    """
    Hq = q.shape[1]
    Hkv = k_pages.shape[1]
    G = Hq // Hkv
    cu = np.asarray(cu_seqlens_q)
    res = []
    gathered = {}           # (sequence, kv head) -> (K, V), gathered once per call
    for (t, h) in rows:
        i = int(np.searchsorted(cu, t, side="right") - 1)
        qn, L = int(cu[i + 1] - cu[i]), int(context_lens[i])
        j = t - int(cu[i])
        key = (i, h // G)
        if key not in gathered:
            gathered[key] = (gather_kv(k_pages, block_table[i], L, h // G),
                             gather_kv(v_pages, block_table[i], L, h // G))
        K, V = gathered[key]
        res.append(attention_row(q[t, h], K, V, _visible_keys(L, qn, j, causal), scale))
    return np.array(res, dtype=np.float64).reshape(len(rows), q.shape[2])


def split_row_partials(q, K, V, n_valid, scale, chunk):
    """Split-KV partials of one row: for keys [c, c+chunk) ∩ [0, n_valid), the normalised
    partial output O_c and its log-sum-exp lse_c = log Σ exp(scale * K q).

    The pages give no exact cross-block merge (their module averages or overwrites the
    per-block results, [XY] §4.3, and says a real kernel needs a cross-block softmax);
    the exact one follows from the softmax definition: with Z_c = Σ_{k in c} exp(s_k),
    O = Σ_c Z_c O_c / Σ_c Z_c.  ``combine_partials`` applies it.
    """
    outs, lses = [], []
    for c in range(0, n_valid, chunk):
        e = min(n_valid, c + chunk)
        s = scale * (K[c:e] @ q)
        m = s.max()
        w = np.exp(s - m)
        Z = w.sum()
        outs.append((w / Z) @ V[c:e])
        lses.append(m + math.log(Z))
    return np.array(outs), np.array(lses)


def combine_partials(outs, lses):
    """Merge split partials (O_c, lse_c): O = Σ_c exp(lse_c - LSE) O_c, LSE = log Σ_c exp(lse_c)."""
    lses = np.asarray(lses, dtype=np.float64)
    M = lses.max()
    w = np.exp(lses - M)
    return (w[:, None] * np.asarray(outs)).sum(axis=0) / w.sum()
