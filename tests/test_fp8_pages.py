"""8-bit (E4M3) KV pages on the GPU against the oracle: the quantizing append bit for bit."""

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("d", [64, 128])
def test_append_fp8_bit_exact(d):
    import paged_kv_varlen_xy_gb300 as xy
    from paged_kv_varlen_xy_gb300 import build
    build.build()
    rng = np.random.default_rng(d)
    P, Hkv, bs, T = 37, 4, 16, 300
    g = torch.Generator().manual_seed(d)
    scale = torch.tensor([1e-3, 1.0, 40.0])[torch.randint(0, 3, (T, Hkv, 1), generator=g)]
    k_new = (torch.randn(T, Hkv, d, generator=g) * scale).to(torch.bfloat16)
    v_new = (torch.randn(T, Hkv, d, generator=g) * scale).to(torch.bfloat16)
    k_new[5, 1] = 0                                    # an all-zero row
    slots = rng.permutation(P * bs)[:T].astype(np.int64)
    slots[7] = -1
    kp = torch.randint(0, 256, (P, Hkv, bs, d), generator=g, dtype=torch.uint8)
    vp = torch.randint(0, 256, (P, Hkv, bs, d), generator=g, dtype=torch.uint8)
    ks = torch.rand(P, Hkv, bs, generator=g)
    vs = torch.rand(P, Hkv, bs, generator=g)
    ref = oracle.kv_append_fp8(kp.numpy(), vp.numpy(), ks.numpy(), vs.numpy(), _bits(k_new), _bits(v_new), slots)
    dev = [t.cuda() for t in (k_new, v_new, kp, vp, ks, vs)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    xy.xy_kv_append_fp8(dev[0], dev[1], torch.from_numpy(slots).cuda(), dev[2], dev[3], dev[4], dev[5], err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(dev[2].cpu().numpy(), ref[0]) and np.array_equal(dev[3].cpu().numpy(), ref[1])
    assert np.array_equal(dev[4].cpu().numpy().view(np.uint32), ref[2].view(np.uint32))
    assert np.array_equal(dev[5].cpu().numpy().view(np.uint32), ref[3].view(np.uint32))
