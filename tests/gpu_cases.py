"""Helpers for the GPU parity tests: run one step of the CUDA path and the oracle on the same
seeded workload and compare (bit-exact for integer/byte work, the bf16 tolerance for outputs)."""

import numpy as np
import torch

import oracle
from paged_kv_varlen_xy_gb300 import step as xystep

# bf16 output vs the fp64 oracle (fp32 accumulation on the GPU)
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def bits(t):
    """uint16 numpy view of a bf16 tensor (copied to the host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def run(wl, rows=None, sample_seqs=None, q_tile=None, kv_chunk=None, num_ctas=None, pool_fill=None, schedule=3,
        transform=None, per_seq_oracle=False):
    """Run the CUDA step and the oracle step on workload `wl`.

    rows: list of (token, head) to compare, or None for every row.  sample_seqs: sequences whose
    pages the oracle receives (default: all).  pool_fill: value written to the whole pool before
    the step instead of random data (e.g. NaN, to check unused slots never leak into outputs).
    transform: callable applied in place to the device tensors before the step (both sides see
    its result).  per_seq_oracle: run the oracle once per sampled sequence, on that sequence's pages
    only (bounds the oracle's memory for very long contexts; the result is the same).
    Returns dict with both sides' results and error statistics.
    """
    dev = torch.device("cuda")
    vals = wl.tensors(dev)
    if pool_fill is not None:
        vals["k_pool"].fill_(pool_fill)
        vals["v_pool"].fill_(pool_fill)
    if transform is not None:
        transform(vals)
    batch = xystep.PagedBatch(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                              wl.num_heads_q, wl.num_heads_kv, wl.head_dim, wl.causal, device=dev,
                              num_ctas=num_ctas, q_tile=q_tile, kv_chunk=kv_chunk, schedule=schedule)
    bt = batch.block_table_host
    if sample_seqs is None:
        pages = None
    else:
        pages = np.unique(np.concatenate([bt[i][bt[i] >= 0] for i in sample_seqs]))
    pool_idx = torch.arange(wl.num_pages, device=dev) if pages is None else torch.from_numpy(pages).long().to(dev)
    k_before = bits(vals["k_pool"].index_select(0, pool_idx))
    v_before = bits(vals["v_pool"].index_select(0, pool_idx))

    out = xystep.run_step(batch, vals["q"], vals["k_new"], vals["v_new"], vals["k_pool"], vals["v_pool"], wl.scale)
    torch.cuda.synchronize()
    err = int(batch.err.item())

    q_bits, kn_bits, vn_bits = bits(vals["q"]), bits(vals["k_new"]), bits(vals["v_new"])
    if per_seq_oracle:
        cu = wl.cu_seqlens_q
        pos = {int(p): i for i, p in enumerate(pages)}
        k_ref, v_ref, outs = k_before.copy(), v_before.copy(), {}
        for s in sample_seqs:
            sp = np.unique(bt[s][bt[s] >= 0])
            sel = np.array([pos[int(p)] for p in sp])
            srows = [(t, h) for (t, h) in rows if cu[s] <= t < cu[s + 1]]
            r = oracle.step.run_step(cu, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks, q_bits,
                                     kn_bits, vn_bits, k_before[sel], v_before[sel], wl.scale, wl.causal,
                                     pool_pages=sp, rows=srows)
            k_ref[sel], v_ref[sel] = r["k_pages"], r["v_pages"]
            outs.update(zip(srows, r["out"]))
        ref = dict(block_table=r["block_table"], slots=r["slots"], k_pages=k_ref, v_pages=v_ref,
                   out=np.stack([outs[x] for x in rows]))
    else:
        ref = oracle.step.run_step(wl.cu_seqlens_q, wl.context_lens, wl.free_list, wl.block_size, wl.max_blocks,
                                   q_bits, kn_bits, vn_bits, k_before, v_before, wl.scale, wl.causal,
                                   pool_pages=pages, rows=rows)
    gpu_out = oracle.bf16_bits_to_f64(bits(out))
    if rows is not None:
        gpu_out = np.stack([gpu_out[t, h] for (t, h) in rows]) if rows else np.zeros((0, wl.head_dim))
    diff = np.abs(gpu_out - ref["out"])
    return dict(
        err=err,
        batch=batch,
        block_table_gpu=bt,
        slots_gpu=batch.slots.cpu().numpy(),
        k_after=bits(vals["k_pool"].index_select(0, pool_idx)),
        v_after=bits(vals["v_pool"].index_select(0, pool_idx)),
        gpu_out=gpu_out,
        ref=ref,
        max_abs=float(diff.max()) if diff.size else 0.0,
        mean_abs=float(diff.mean()) if diff.size else 0.0,
        finite=bool(np.isfinite(gpu_out).all()),
    )


def assert_parity(r, check_pages=True):
    assert r["err"] == 0, f"device error word {r['err']:#x}"
    assert np.array_equal(r["block_table_gpu"], r["ref"]["block_table"])
    assert np.array_equal(r["slots_gpu"], r["ref"]["slots"])
    if check_pages:
        assert np.array_equal(r["k_after"], r["ref"]["k_pages"])
        assert np.array_equal(r["v_after"], r["ref"]["v_pages"])
    assert r["finite"]
    assert r["max_abs"] <= MAX_ABS, r["max_abs"]
    assert r["mean_abs"] <= MEAN_ABS, r["mean_abs"]


def sample_rows(wl, seqs, rng, per_seq=24, q_tile=None):
    """Rows (token, head) of the given sequences: first and last token, tile edges, random ones."""
    cu = wl.cu_seqlens_q
    rows = []
    for i in seqs:
        t0, t1 = int(cu[i]), int(cu[i + 1])
        toks = {t0, t1 - 1}
        if q_tile:
            for e in range(t0 + q_tile, t1, q_tile):
                toks.update({e - 1, e})
        toks.update(int(x) for x in rng.integers(t0, t1, size=min(per_seq, t1 - t0)))
        for t in sorted(toks):
            if t1 - t0 == 1:   # decode: every head
                rows.extend((t, h) for h in range(wl.num_heads_q))
            else:
                rows.extend((t, int(h)) for h in rng.choice(wl.num_heads_q, size=2, replace=False))
    return rows
