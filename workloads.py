"""Seeded synthetic workloads for the paged-KV varlen attention path.

Shared by the tests, ``bench.py`` and ``__graft_entry__.smoke()``; it feeds both the CUDA
path and the oracle and holds none of the method's arithmetic: it only draws lengths, a
shuffled free-page list and bf16 values.  Random numbers the method uses (the free-list
order) are drawn here and passed to both sides.

Shapes follow the workloads the pages describe: 16-token pages ([CANN] §2.2) and
256-token blocks ([MindIE] block management), ragged prompts from tens to ~20k tokens
([XY] §1.2), 512-token prefill chunks ([MindIE] Prefill Chunking), 128K contexts
([MindIE]), and a mix of chat/code/summary lengths ([XY] §1.2).  No dataset is used.

Values: fp32 N(0, 1) from ``torch.Generator`` rounded to bf16 (round to nearest even).
The page pool is filled with such values before the step, so every slot holds finite
data; the prior context of a sequence is whatever its pages hold.
"""

from dataclasses import dataclass, field
import math

import numpy as np
import torch


@dataclass
class Workload:
    name: str
    q_lens: np.ndarray          # int32 [S]
    context_lens: np.ndarray    # int32 [S], including the new tokens
    num_heads_q: int
    num_heads_kv: int
    head_dim: int
    block_size: int
    num_pages: int
    max_blocks: int
    causal: bool
    seed: int
    free_list: np.ndarray = field(repr=False)   # int32 permutation of range(num_pages)
    shared_prefix_tokens: int = 0               # > 0: rows share their first pages (share_prefix)

    @property
    def num_seqs(self):
        return len(self.q_lens)

    @property
    def num_tokens(self):
        return int(np.sum(self.q_lens, dtype=np.int64))

    @property
    def cu_seqlens_q(self):
        return np.concatenate([[0], np.cumsum(self.q_lens, dtype=np.int64)]).astype(np.int32)

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def group(self):
        return self.num_heads_q // self.num_heads_kv

    def tensors(self, device="cpu", pool=True):
        """bf16 tensors: q [T,Hq,d], k_new/v_new [T,Hkv,d], k_pool/v_pool [P,Hkv,bs,d]."""
        dev = torch.device(device)
        gen = torch.Generator(device=dev)
        T, d = self.num_tokens, self.head_dim
        out = {}

        def draw(shape, offset):
            gen.manual_seed(self.seed * 16 + offset)
            n = int(np.prod(shape))
            flat = torch.empty(n, dtype=torch.bfloat16, device=dev)
            step = 1 << 26
            for s in range(0, n, step):
                e = min(n, s + step)
                flat[s:e] = torch.randn(e - s, generator=gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
            return flat.view(*shape)

        out["q"] = draw((T, self.num_heads_q, d), 1)
        out["k_new"] = draw((T, self.num_heads_kv, d), 2)
        out["v_new"] = draw((T, self.num_heads_kv, d), 3)
        if pool:
            shape = (self.num_pages, self.num_heads_kv, self.block_size, d)
            out["k_pool"] = draw(shape, 4)
            out["v_pool"] = draw(shape, 5)
        return out


def _finish(name, q_lens, ctx, Hq, Hkv, d, bs, causal, seed, rng, num_pages=None, slack=1.25):
    q_lens = np.asarray(q_lens, dtype=np.int32)
    ctx = np.asarray(ctx, dtype=np.int32)
    blocks = -(-ctx.astype(np.int64) // bs)
    need = int(blocks.sum())
    if num_pages is None:
        num_pages = max(1, int(math.ceil(slack * need)))
    free = rng.permutation(num_pages).astype(np.int32)
    return Workload(name=name, q_lens=q_lens, context_lens=ctx, num_heads_q=Hq, num_heads_kv=Hkv,
                    head_dim=d, block_size=bs, num_pages=num_pages,
                    max_blocks=int(blocks.max()) if len(blocks) else 1, causal=causal, seed=seed,
                    free_list=free)


def tiny(seed=1001):
    """4 seqs: prefill q=7 and q=16 without prior context, decode q=1 over contexts 33 and 50;
    Hq=4, Hkv=2 (GQA), d=64, bs=16, 64 physical pages shuffled, causal."""
    rng = np.random.default_rng(seed)
    return _finish("tiny", [7, 16, 1, 1], [7, 16, 33, 50], 4, 2, 64, 16, True, seed, rng, num_pages=64)


def decode(seed=1002, num_seqs=64):
    """64 decode seqs, q=1, context U[128, 4096]; Hq=Hkv=32, d=128, bs=16."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(128, 4096, size=num_seqs, endpoint=True)
    return _finish("decode", np.ones(num_seqs), ctx, 32, 32, 128, 16, True, seed, rng)


def prefill(seed=1003, num_seqs=16):
    """16 packed prompts, lengths lognormal(median 512, sigma 1) clipped to [32, 8192], causal,
    no prior context; Hq=32, Hkv=8, d=128, bs=16."""
    rng = np.random.default_rng(seed)
    lens = np.clip(np.round(rng.lognormal(math.log(512.0), 1.0, size=num_seqs)), 32, 8192).astype(np.int64)
    return _finish("prefill", lens, lens, 32, 8, 128, 16, True, seed, rng)


def mixed(seed=1004, num_chunks=8, num_decodes=120):
    """8 chunked-prefill chunks of 512 tokens after a prior context U[0, 16384], then 120 decode
    seqs with context U[256, 32768]; Hq=32, Hkv=8, d=128, bs=16."""
    rng = np.random.default_rng(seed)
    prior = rng.integers(0, 16384, size=num_chunks, endpoint=True)
    dctx = rng.integers(256, 32768, size=num_decodes, endpoint=True)
    q = np.concatenate([np.full(num_chunks, 512), np.ones(num_decodes)])
    ctx = np.concatenate([prior + 512, dctx])
    return _finish("mixed", q, ctx, 32, 8, 128, 16, True, seed, rng)


def skew(seed=1005, num_long=4, num_short=252, long_len=131072, short_len=512):
    """256 decode seqs: 4 at context 131072 (at shuffled batch positions), 252 at 512;
    Hq=64, Hkv=8, d=128, bs=256."""
    rng = np.random.default_rng(seed)
    ctx = np.full(num_long + num_short, short_len, dtype=np.int64)
    ctx[rng.choice(num_long + num_short, size=num_long, replace=False)] = long_len
    return _finish("skew", np.ones(num_long + num_short), ctx, 64, 8, 128, 256, True, seed, rng)


def verify(seed=1006, num_seqs=64):
    """64 speculative-verify steps: q U{2..8} draft tokens per sequence over a context U[512, 8192]
    (including them); Hq=32, Hkv=8, d=128, bs=16 ([ATB] speculative decoding: the target model
    scores a few draft tokens per sequence in one pass)."""
    rng = np.random.default_rng(seed)
    q = rng.integers(2, 8, size=num_seqs, endpoint=True)
    ctx = rng.integers(512, 8192, size=num_seqs, endpoint=True)
    return _finish("verify", q, ctx, 32, 8, 128, 16, True, seed, rng)


def prefix(seed=1007, num_seqs=64, context=4096, shared=3584):
    """64 decode sequences of context 4096 whose first 3584 tokens (224 pages of 16) are one shared
    prompt prefix ([XY] §2.3 technique 2, prefix cache; [ATB] KV cache reuse): every row of the
    block table points at the same physical pages for it (see share_prefix).  Hq=Hkv=32, d=128."""
    rng = np.random.default_rng(seed)
    wl = _finish("prefix", np.ones(num_seqs), np.full(num_seqs, context), 32, 32, 128, 16, True, seed, rng)
    wl.shared_prefix_tokens = shared
    return wl


def share_prefix(block_table, shared_tokens, block_size):
    """The block table of a prefix-shared batch: the first shared_tokens / block_size entries of
    every row replaced by row 0's (the rows' own pages for those positions go unused).  Batch
    construction only: which physical page each logical page of a sequence is."""
    n = shared_tokens // block_size
    bt = np.array(block_table, copy=True)
    bt[:, :n] = bt[0, :n]
    return bt


def custom(q_lens, context_lens, num_heads_q, num_heads_kv, head_dim, block_size, causal=True,
           seed=7, num_pages=None, name="custom"):
    """Any batch shape (parity tests: ragged tails, several tiles, edge cases)."""
    rng = np.random.default_rng(seed)
    return _finish(name, q_lens, context_lens, num_heads_q, num_heads_kv, head_dim, block_size,
                   causal, seed, rng, num_pages=num_pages)


CONFIGS = {"tiny": tiny, "decode": decode, "prefill": prefill, "mixed": mixed, "skew": skew, "verify": verify,
           "prefix": prefix}


def make(name, **kw):
    return CONFIGS[name](**kw)
