"""Prefix-shared pages: several sequences' block tables point at the same physical pages for a
common prefix ([XY] §2.3 technique 2, automatic prefix cache; [ATB] KV缓存复用, multi-turn
sessions reusing a conversation's KV).  The kernels read pages only through the block table, so
sharing needs no new code; these tests pin that on the oracle and on the CUDA path.

The new tokens of every sequence land after the shared prefix, in pages of its own, so the
append never writes a shared page."""

import numpy as np
import pytest
import torch

import oracle

BS = 16
PREFIX_PAGES = 24            # 384 shared tokens


def _batch(rng, q_lens, suffix):
    """Block table whose rows share the first PREFIX_PAGES physical pages, and its private twin in
    which every sequence has its own copy of them (appended after the shared pool).  Returns
    (cu, ctx, bt_shared, bt_private, P_shared, copy_of) with copy_of[p] = the shared page that
    private page p copies."""
    S = len(q_lens)
    ctx = PREFIX_PAGES * BS + np.asarray(suffix, dtype=np.int64)
    assert np.all(np.asarray(suffix) >= np.asarray(q_lens))      # new tokens after the prefix
    pages_per_seq = (ctx + BS - 1) // BS
    own_total = int((pages_per_seq - PREFIX_PAGES).sum())
    P = PREFIX_PAGES + own_total + 8
    perm = rng.permutation(P).astype(np.int32)
    MB = int(pages_per_seq.max())
    bt = -np.ones((S, MB), dtype=np.int32)
    nxt = PREFIX_PAGES
    for i in range(S):
        own = int(pages_per_seq[i]) - PREFIX_PAGES
        row = list(range(PREFIX_PAGES)) + list(range(nxt, nxt + own))
        nxt += own
        bt[i, :len(row)] = perm[row]
    bt_private = bt.copy()
    copy_of = {}
    for i in range(S):
        for k in range(PREFIX_PAGES):
            page = P + i * PREFIX_PAGES + k
            copy_of[page] = int(bt[i, k])
            bt_private[i, k] = page
    return oracle.pack_cu_seqlens(q_lens), ctx.astype(np.int32), bt, bt_private, P, copy_of


def _with_copies(vals, P, copy_of):
    """The pool extended by the private copies of the shared pages."""
    out = dict(vals)
    for name in ("k_pool", "v_pool"):
        idx = torch.tensor([copy_of[p] for p in sorted(copy_of)], dtype=torch.long)
        out[name] = torch.cat([vals[name], vals[name].index_select(0, idx)])
    return out


def _values(seed, T, Hq, Hkv, d, P):
    g = torch.Generator().manual_seed(seed)
    mk = lambda *s: torch.randn(*s, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return dict(q=mk(T, Hq, d), k_new=mk(T, Hkv, d), v_new=mk(T, Hkv, d),
                k_pool=mk(P, Hkv, BS, d), v_pool=mk(P, Hkv, BS, d))


def _bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _oracle_out(cu, ctx, bt, vals, Hq, Hkv, d, scale):
    slots = oracle.slot_mapping(cu, ctx, bt, BS)
    kp, vp = oracle.kv_append(_bits(vals["k_pool"]), _bits(vals["v_pool"]), _bits(vals["k_new"]),
                              _bits(vals["v_new"]), slots)
    out = oracle.paged_attention(oracle.bf16_bits_to_f64(_bits(vals["q"])), cu, ctx, bt,
                                 oracle.bf16_bits_to_f64(kp), oracle.bf16_bits_to_f64(vp), scale, True)
    return slots, kp, vp, out


def test_oracle_shared_prefix_equals_private_copies():
    q_lens, suffix = [1, 3, 1, 20], [40, 50, 17, 33]
    Hq, Hkv, d = 4, 2, 64
    cu, ctx, bt_s, bt_p, P, copy_of = _batch(np.random.default_rng(1), q_lens, suffix)
    vals = _values(5, int(cu[-1]), Hq, Hkv, d, P)
    scale = 1.0 / np.sqrt(d)
    _, _, _, out_s = _oracle_out(cu, ctx, bt_s, vals, Hq, Hkv, d, scale)
    _, _, _, out_p = _oracle_out(cu, ctx, bt_p, _with_copies(vals, P, copy_of), Hq, Hkv, d, scale)
    assert np.array_equal(out_s, out_p)
    # no append writes a shared page
    slots = oracle.slot_mapping(cu, ctx, bt_s, BS)
    assert not set(int(s) // BS for s in slots) & set(int(p) for p in bt_s[0, :PREFIX_PAGES])


@pytest.mark.gpu
@pytest.mark.parametrize("d,G", [(128, 4), (64, 2)])
def test_gpu_shared_prefix_matches_oracle_and_private_copies(d, G):
    from paged_kv_varlen_xy_gb300 import build
    from paged_kv_varlen_xy_gb300 import step as xystep
    from gpu_cases import MAX_ABS, MEAN_ABS
    build.build()
    q_lens, suffix = [1, 1, 5, 1, 64, 1, 8], [30, 200, 41, 700, 90, 16, 8]
    Hkv = 4
    Hq = Hkv * G
    scale = 1.0 / np.sqrt(d)
    cu, ctx, bt_s, bt_p, P, copy_of = _batch(np.random.default_rng(11), q_lens, suffix)
    base = _values(13, int(cu[-1]), Hq, Hkv, d, P)
    outs = {}
    for shared in (True, False):
        bt = bt_s if shared else bt_p
        vals = base if shared else _with_copies(base, P, copy_of)
        ref_slots, ref_kp, ref_vp, ref_out = _oracle_out(cu, ctx, bt, vals, Hq, Hkv, d, scale)
        dev = {k: v.cuda() for k, v in vals.items()}
        need = int(((ctx + BS - 1) // BS).sum())
        batch = xystep.PagedBatch(cu, ctx, np.arange(need, dtype=np.int32), BS, bt.shape[1], Hq, Hkv, d, True)
        batch.block_table.copy_(torch.from_numpy(bt))
        out = xystep.run_step(batch, dev["q"], dev["k_new"], dev["v_new"], dev["k_pool"], dev["v_pool"], scale)
        torch.cuda.synchronize()
        assert int(batch.err.item()) == 0
        assert np.array_equal(batch.slots.cpu().numpy(), ref_slots)
        assert np.array_equal(_bits(dev["k_pool"]), ref_kp) and np.array_equal(_bits(dev["v_pool"]), ref_vp)
        got = oracle.bf16_bits_to_f64(_bits(out))
        diff = np.abs(got - ref_out)
        assert diff.max() <= MAX_ABS and diff.mean() <= MEAN_ABS
        outs[shared] = _bits(out)
    # same lengths, same task table, same page contents: sharing changes nothing
    assert np.array_equal(outs[True], outs[False])


@pytest.mark.gpu
def test_gpu_full_size_prefix_batch_sampled():
    # the bench's prefix-shared batch (64 x 4096 keys, 3584 on row 0's pages) in its launch
    # configuration (dynamic deal); the oracle checks every head of eight sampled sequences, each
    # gathered through the shared block table
    import workloads
    from paged_kv_varlen_xy_gb300 import build
    from paged_kv_varlen_xy_gb300 import step as xystep
    from gpu_cases import MAX_ABS, MEAN_ABS
    build.build()
    wl = workloads.prefix()
    vals = wl.tensors("cuda")
    batch = xystep.PagedBatch(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                              wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.causal, schedule=4)
    bt = workloads.share_prefix(batch.block_table_host, wl.shared_prefix_tokens, wl.block_size)
    batch.block_table.copy_(torch.from_numpy(bt))
    sample = [0, 1, 17, 33, 40, 51, 62, 63]
    pages = np.unique(np.concatenate([bt[i][bt[i] >= 0] for i in sample]))
    idx = torch.from_numpy(pages).long().cuda()
    k_before, v_before = _bits(vals["k_pool"].index_select(0, idx)), _bits(vals["v_pool"].index_select(0, idx))
    out = xystep.run_step(batch, vals["q"], vals["k_new"], vals["v_new"], vals["k_pool"], vals["v_pool"], wl.scale)
    torch.cuda.synchronize()
    assert int(batch.err.item()) == 0
    lut = {int(p): i for i, p in enumerate(pages)}
    local = np.array([[lut.get(int(p), -1) if p >= 0 else -1 for p in row] for row in bt], dtype=np.int32)
    slots = oracle.slot_mapping(wl.cu_seqlens_q, wl.context_lens, bt, wl.block_size)
    assert np.array_equal(batch.slots.cpu().numpy(), slots)
    local_slots = np.array([lut[int(s) // wl.block_size] * wl.block_size + int(s) % wl.block_size
                            if int(s) // wl.block_size in lut else -1 for s in slots], dtype=np.int64)
    kp, vp = oracle.kv_append(k_before, v_before, _bits(vals["k_new"]), _bits(vals["v_new"]), local_slots)
    assert np.array_equal(_bits(vals["k_pool"].index_select(0, idx)), kp)
    assert np.array_equal(_bits(vals["v_pool"].index_select(0, idx)), vp)
    rows = [(int(wl.cu_seqlens_q[i]), h) for i in sample for h in range(wl.num_heads_q)]
    ref = oracle.attention_rows(rows, oracle.bf16_bits_to_f64(_bits(vals["q"])), wl.cu_seqlens_q, wl.context_lens,
                                local, oracle.bf16_bits_to_f64(kp), oracle.bf16_bits_to_f64(vp), wl.scale, True)
    got = oracle.bf16_bits_to_f64(_bits(out))
    got = np.stack([got[t, h] for t, h in rows])
    diff = np.abs(got - ref)
    assert np.isfinite(got).all() and diff.max() <= MAX_ABS and diff.mean() <= MEAN_ABS, (diff.max(), diff.mean())
