"""Pins for the oracle's attention: brute force against a textbook routine, invariants the pages
fix, closed forms, and the pages' own wrong merges as cases the oracle must not match."""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import (allocate_block_table, attention_row, attention_rows, bf16_bits_to_f64,
                    combine_partials, f64_to_bf16_bits, pack_cu_seqlens, paged_attention,
                    split_row_partials, virtual_mask)
from oracle import attention as oracle_attention

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _pages_from_contiguous(Ks, Vs, bs, free, max_blocks):
    """Lay out per-sequence contiguous K/V [L, Hkv, d] into a page pool through the allocator."""
    Hkv, d = Ks[0].shape[1], Ks[0].shape[2]
    P = len(free)
    L = [k.shape[0] for k in Ks]
    bt = allocate_block_table(L, bs, free, max_blocks)
    kp = np.zeros((P, Hkv, bs, d))
    vp = np.zeros((P, Hkv, bs, d))
    for i, (K, V) in enumerate(zip(Ks, Vs)):
        for p in range(L[i]):
            kp[bt[i, p // bs], :, p % bs] = K[p]
            vp[bt[i, p // bs], :, p % bs] = V[p]
    return bt, kp, vp


def _sdpa_reference(q_seq, K, V, Hq, causal, scale):
    """torch SDPA in float64 on one sequence with an explicit boolean mask."""
    qn, L = q_seq.shape[0], K.shape[0]
    Hkv = K.shape[1]
    G = Hq // Hkv
    Kx = np.repeat(K, G, axis=1)
    Vx = np.repeat(V, G, axis=1)
    qt = torch.from_numpy(q_seq).permute(1, 0, 2)[None]
    kt = torch.from_numpy(Kx).permute(1, 0, 2)[None]
    vt = torch.from_numpy(Vx).permute(1, 0, 2)[None]
    j = torch.arange(qn)[:, None]
    k = torch.arange(L)[None, :]
    mask = (k <= (L - qn + j)) if causal else torch.ones(qn, L, dtype=torch.bool)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


def _random_batch(rng, q_lens, ctx, Hq, Hkv, d, bs, P=None):
    Ks = [rng.standard_normal((L, Hkv, d)) for L in ctx]
    Vs = [rng.standard_normal((L, Hkv, d)) for L in ctx]
    need = sum(-(-L // bs) for L in ctx)
    P = P or need + 5
    free = rng.permutation(P).astype(np.int32)
    bt, kp, vp = _pages_from_contiguous(Ks, Vs, bs, free, max(-(-L // bs) for L in ctx))
    cu = pack_cu_seqlens(q_lens)
    q = rng.standard_normal((int(cu[-1]), Hq, d))
    return dict(Ks=Ks, Vs=Vs, bt=bt, kp=kp, vp=vp, cu=cu, q=q, ctx=ctx, free=free)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (3, 3), (8, 1)])
def test_brute_force_against_sdpa(causal, Hq, Hkv):
    rng = np.random.default_rng(11 + Hq + 7 * Hkv + int(causal))
    q_lens, ctx = [7, 16, 1, 1, 5], [7, 16, 33, 50, 21]
    b = _random_batch(rng, q_lens, ctx, Hq, Hkv, 16, 4)
    scale = 1 / math.sqrt(16)
    out = paged_attention(b["q"], b["cu"], ctx, b["bt"], b["kp"], b["vp"], scale, causal)
    for i in range(len(q_lens)):
        ref = _sdpa_reference(b["q"][b["cu"][i]:b["cu"][i + 1]], b["Ks"][i], b["Vs"][i], Hq, causal, scale)
        assert np.max(np.abs(out[b["cu"][i]:b["cu"][i + 1]] - ref)) < 1e-12


def test_rows_api_matches_full():
    rng = np.random.default_rng(5)
    q_lens, ctx = [3, 1, 9], [10, 40, 9]
    b = _random_batch(rng, q_lens, ctx, 6, 2, 8, 8)
    full = paged_attention(b["q"], b["cu"], ctx, b["bt"], b["kp"], b["vp"], 0.3, True)
    rows = [(0, 0), (2, 5), (3, 1), (12, 4), (5, 3)]
    part = attention_rows(rows, b["q"], b["cu"], ctx, b["bt"], b["kp"], b["vp"], 0.3, True)
    for r, (t, h) in enumerate(rows):
        assert np.array_equal(part[r], full[t, h])


def test_physical_page_permutation_invariance():
    rng = np.random.default_rng(1)
    q_lens, ctx = [5, 1, 12], [20, 37, 12]
    b = _random_batch(rng, q_lens, ctx, 4, 2, 8, 4, P=40)
    out = paged_attention(b["q"], b["cu"], ctx, b["bt"], b["kp"], b["vp"], 0.35, True)
    perm = rng.permutation(40)          # physical page p moves to perm[p]
    kp2 = np.empty_like(b["kp"])
    vp2 = np.empty_like(b["vp"])
    kp2[perm] = b["kp"]
    vp2[perm] = b["vp"]
    bt2 = np.where(b["bt"] >= 0, perm[np.maximum(b["bt"], 0)], -1).astype(np.int32)
    out2 = paged_attention(b["q"], b["cu"], ctx, bt2, kp2, vp2, 0.35, True)
    assert np.array_equal(out, out2)


def test_packed_equals_padded_on_page_example():
    g = json.load(open(os.path.join(GOLDEN, "packed_cu_seqlens.json")))
    lens = g["lengths"]
    rng = np.random.default_rng(2)
    Hq = Hkv = 2
    d = 8
    b = _random_batch(rng, lens, lens, Hq, Hkv, d, 16)
    assert b["cu"].tolist() == g["cu_seqlens"]
    out = paged_attention(b["q"], b["cu"], lens, b["bt"], b["kp"], b["vp"], 0.3, True)
    # padded layout: [batch, max_len, H, d] with a key-padding mask, via SDPA
    Lm = max(lens)
    qpad = np.zeros((3, Lm, Hq, d))
    kpad = np.zeros((3, Lm, Hkv, d))
    vpad = np.zeros((3, Lm, Hkv, d))
    for i, L in enumerate(lens):
        qpad[i, :L] = b["q"][b["cu"][i]:b["cu"][i + 1]]
        kpad[i, :L] = b["Ks"][i]
        vpad[i, :L] = b["Vs"][i]
    j = torch.arange(Lm)[:, None]
    k = torch.arange(Lm)[None, :]
    mask = torch.stack([(k <= j) & (k < L) | (j >= L) & (k == 0) for L in lens])[:, None]
    o = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qpad).permute(0, 2, 1, 3), torch.from_numpy(kpad).permute(0, 2, 1, 3),
        torch.from_numpy(vpad).permute(0, 2, 1, 3), attn_mask=mask, scale=0.3).permute(0, 2, 1, 3).numpy()
    for i, L in enumerate(lens):
        assert np.max(np.abs(out[b["cu"][i]:b["cu"][i + 1]] - o[i, :L])) < 1e-12


def test_chunked_prefill_equals_whole_prefill():
    rng = np.random.default_rng(4)
    L, Hq, Hkv, d, bs = 45, 4, 2, 8, 8
    K = rng.standard_normal((L, Hkv, d))
    V = rng.standard_normal((L, Hkv, d))
    q_all = rng.standard_normal((L, Hq, d))
    P = 8
    free = rng.permutation(P).astype(np.int32)
    bt, kp, vp = _pages_from_contiguous([K], [V], bs, free, 6)
    whole = paged_attention(q_all, [0, L], [L], bt, kp, vp, 0.4, True)
    done = 0
    for chunk in (16, 16, 13):          # chunks appended one after another
        piece = paged_attention(q_all[done:done + chunk], [0, chunk], [done + chunk], bt, kp, vp, 0.4, True)
        assert np.max(np.abs(piece - whole[done:done + chunk])) < 1e-13
        done += chunk


def test_decode_equals_last_prefill_row():
    rng = np.random.default_rng(6)
    L, Hq, Hkv, d, bs = 29, 2, 1, 16, 4
    b = _random_batch(rng, [L], [L], Hq, Hkv, d, bs)
    whole = paged_attention(b["q"], b["cu"], [L], b["bt"], b["kp"], b["vp"], 0.25, True)
    dec = paged_attention(b["q"][-1:], [0, 1], [L], b["bt"], b["kp"], b["vp"], 0.25, True)
    assert np.max(np.abs(dec[0] - whole[-1])) < 1e-13


def test_single_key_returns_v_exactly():
    rng = np.random.default_rng(8)
    d = 64
    vbits = rng.integers(0, 0x7F00, size=(1, 1, d), dtype=np.uint16)  # finite positive/negative-free patterns
    kbits = rng.integers(0, 0x3F00, size=(1, 1, d), dtype=np.uint16)
    kp = np.zeros((2, 1, 16, d))
    vp = np.zeros((2, 1, 16, d))
    kp[1, 0, 0] = bf16_bits_to_f64(kbits[0, 0])
    vp[1, 0, 0] = bf16_bits_to_f64(vbits[0, 0])
    q = rng.standard_normal((1, 1, d))
    out = paged_attention(q, [0, 1], [1], np.array([[1]], np.int32), kp, vp, 0.125, True)
    assert np.array_equal(out[0, 0], vp[1, 0, 0])
    assert np.array_equal(f64_to_bf16_bits(out[0, 0]), vbits[0, 0])


def test_equal_keys_give_mean_of_visible_values():
    rng = np.random.default_rng(9)
    L, d, bs = 23, 8, 4
    K = np.tile(rng.standard_normal((1, 1, d)), (L, 1, 1))
    V = rng.standard_normal((L, 1, d))
    bt, kp, vp = _pages_from_contiguous([K], [V], bs, np.arange(6, dtype=np.int32), 6)
    q = rng.standard_normal((5, 1, d))
    out = paged_attention(q, [0, 5], [L], bt, kp, vp, 0.7, True)
    for j in range(5):
        n = L - 5 + j + 1
        assert np.max(np.abs(out[j, 0] - V[:n, 0].mean(axis=0))) < 1e-13


def test_causal_alignment_counts_visible_keys():
    """q = 0 gives uniform weights; with one-hot values the output reads off the visible set."""
    L, q_n, d, bs = 20, 6, 32, 8
    K = np.random.default_rng(0).standard_normal((L, 1, d))
    V = np.zeros((L, 1, d))
    for p in range(L):
        V[p, 0, p] = 1.0
    bt, kp, vp = _pages_from_contiguous([K], [V], bs, np.array([2, 0, 1], np.int32), 3)
    out = paged_attention(np.zeros((q_n, 1, d)), [0, q_n], [L], bt, kp, vp, 1.0, True)
    for j in range(q_n):
        n = L - q_n + j + 1          # new token j sits at absolute position L - q + j
        expect = np.zeros(d)
        expect[:n] = 1.0 / n
        assert np.max(np.abs(out[j, 0] - expect)) < 1e-15
    out_nc = paged_attention(np.zeros((q_n, 1, d)), [0, q_n], [L], bt, kp, vp, 1.0, False)
    assert np.max(np.abs(out_nc[:, 0, :L] - 1.0 / L)) < 1e-15


def test_two_key_closed_form():
    d = 4
    K = np.array([[[1.0, 0, 0, 0]], [[0, 2.0, 0, 0]]])
    V = np.array([[[1.0, 2, 3, 4]], [[-1.0, 0, 5, 1]]])
    bt, kp, vp = _pages_from_contiguous([K], [V], 2, np.array([0], np.int32), 1)
    q = np.array([[[0.5, 1.5, 0, 0]]])
    scale = 0.8
    out = paged_attention(q, [0, 1], [2], bt, kp, vp, scale, True)
    a, b_ = scale * 0.5, scale * 3.0
    w1 = 1.0 / (1.0 + math.exp(a - b_))
    assert np.max(np.abs(out[0, 0] - ((1 - w1) * V[0, 0] + w1 * V[1, 0]))) < 1e-15


def test_session_isolation():
    rng = np.random.default_rng(12)
    q_lens, ctx = [4, 1], [9, 30]
    b = _random_batch(rng, q_lens, ctx, 2, 2, 8, 4)
    out = paged_attention(b["q"], b["cu"], ctx, b["bt"], b["kp"], b["vp"], 0.3, True)
    kp2, vp2 = b["kp"].copy(), b["vp"].copy()
    for p in b["bt"][1]:
        if p >= 0:
            kp2[p] += 5.0
            vp2[p] -= 3.0
    out2 = paged_attention(b["q"], b["cu"], ctx, b["bt"], kp2, vp2, 0.3, True)
    assert np.array_equal(out[:4], out2[:4])
    assert not np.allclose(out[4:], out2[4:])


def _pages_mean_merge(q, K, V, scale, blk):
    """The Meta-Attention module's blocked attention on its printed path: per-block softmax,
    then the block outputs are averaged (a simplification the page itself flags)."""
    outs = []
    for c in range(0, K.shape[0], blk):
        s = scale * (K[c:c + blk] @ q)
        w = np.exp(s - s.max())
        outs.append((w / w.sum()) @ V[c:c + blk])
    return np.mean(outs, axis=0)


def _pages_overwrite_merge(q, K, V, scale, blk):
    """The task-table path as printed: each task overwrites the output, so the last block wins."""
    out = None
    for c in range(0, K.shape[0], blk):
        s = scale * (K[c:c + blk] @ q)
        w = np.exp(s - s.max())
        out = (w / w.sum()) @ V[c:c + blk]
    return out


def test_printed_merges_are_not_attention():
    rng = np.random.default_rng(13)
    K = rng.standard_normal((40, 16))
    V = rng.standard_normal((40, 16))
    q = rng.standard_normal(16)
    exact = attention_row(q, K, V, 40, 0.25)
    assert np.max(np.abs(exact - _pages_mean_merge(q, K, V, 0.25, 16))) > 1e-3
    assert np.max(np.abs(exact - _pages_overwrite_merge(q, K, V, 0.25, 16))) > 1e-3
    # with a single block the printed code is exact
    assert np.max(np.abs(attention_row(q, K, V, 16, 0.25) - _pages_mean_merge(q, K[:16], V[:16], 0.25, 16))) < 1e-14


@pytest.mark.parametrize("chunk", [1, 3, 16, 64, 1000])
def test_split_combine_identity(chunk):
    rng = np.random.default_rng(chunk)
    K = rng.standard_normal((300, 8)) * 3
    V = rng.standard_normal((300, 8))
    q = rng.standard_normal(8)
    outs, lses = split_row_partials(q, K, V, 257, 0.5, chunk)
    assert len(outs) == -(-257 // chunk)
    assert np.max(np.abs(combine_partials(outs, lses) - attention_row(q, K, V, 257, 0.5))) < 1e-12
    # lse of a single chunk is the log-sum-exp of its scores
    s = 0.5 * (K[:min(chunk, 257)] @ q)
    assert abs(lses[0] - np.log(np.exp(s).sum())) < 1e-10


def test_virtual_mask_page_example():
    g = json.load(open(os.path.join(GOLDEN, "virtual_padding.json")))
    m = virtual_mask(*g["actual"], *g["tile"])
    assert int(m.sum()) == g["valid_cells"]
    eb = g["element_bytes"]
    padded = g["tile"][0] * g["tile"][1] * eb * 2     # read + write the padded tile
    virtual = int(m.sum()) * eb
    assert padded == g["padded_bytes"] and virtual == g["virtual_bytes"]
    assert round(padded / virtual, 1) == g["ratio_rounded"]


# ---- planted mistakes: each must be caught by one of the pins above -------------------------

def test_planted_causal_off_by_one_is_caught(monkeypatch):
    monkeypatch.setattr(oracle_attention, "_visible_keys",
                        lambda L, q, j, causal: (L - q + j) if causal else L)
    with pytest.raises(AssertionError):
        test_causal_alignment_counts_visible_keys()


def test_planted_gqa_mapping_is_caught(monkeypatch):
    real = oracle_attention.gather_kv

    def swapped(pages, row, L, g):             # reads the other KV head
        return real(pages, row, L, (g + 1) % pages.shape[1])
    monkeypatch.setattr(oracle_attention, "gather_kv", swapped)
    with pytest.raises(AssertionError):
        test_brute_force_against_sdpa(True, 4, 2)


def test_planted_missing_scale_is_caught(monkeypatch):
    real = oracle_attention.attention_row
    monkeypatch.setattr(oracle_attention, "attention_row", lambda q, K, V, n, scale: real(q, K, V, n, 1.0))
    with pytest.raises(AssertionError):
        test_brute_force_against_sdpa(False, 3, 3)
