"""GPU: kvc_append / kvc_append_latent are bit-exact slot writes (oracle: append_to_paged)."""

import numpy as np
import pytest
import torch

from oracle import paged as OP
from paged_kv_cache_157_gb300 import workloads as W

pytestmark = pytest.mark.gpu

INT_VIEW = {torch.float32: torch.int32, torch.float16: torch.int16, torch.bfloat16: torch.int16}


def bits(t):
    return t.detach().cpu().view(INT_VIEW[t.dtype]).numpy()


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("hkv,D,bs", [(8, 128, 16), (1, 64, 32), (4, 32, 16)])
def test_append_bit_exact_with_sentinel(kvc, dtype, hkv, D, bs):
    g = torch.Generator().manual_seed(3)
    nblk = 12
    T = 40
    kc = W.normal((nblk, hkv, bs, D), dtype, g)
    vc = W.normal((nblk, hkv, bs, D), dtype, g)
    k = W.normal((T, hkv, D), dtype, g)
    v = W.normal((T, hkv, D), dtype, g)
    slots = torch.randperm(nblk * bs, generator=g)[:T].to(torch.int64)
    slots[::7] = -1  # padding tokens are skipped
    kd, vd = kc.cuda(), vc.cuda()
    kvc.append(k.cuda(), v.cuda(), slots.cuda(), kd, vd)
    torch.cuda.synchronize()
    ek, ev = OP.append_to_paged(bits(k), bits(v), slots.numpy(), bits(kc), bits(vc))
    assert np.array_equal(bits(kd), ek)
    assert np.array_equal(bits(vd), ev)
    assert kvc.get_error_flags() == 0


def test_append_out_of_range_slot_flags_and_skips(kvc):
    g = torch.Generator().manual_seed(4)
    kc = W.normal((4, 2, 16, 64), "bf16", g)
    vc = W.normal((4, 2, 16, 64), "bf16", g)
    k = W.normal((3, 2, 64), "bf16", g)
    v = W.normal((3, 2, 64), "bf16", g)
    slots = torch.tensor([5, 4 * 16, 63], dtype=torch.int64)
    kd, vd = kc.cuda(), vc.cuda()
    kvc.append(k.cuda(), v.cuda(), slots.cuda(), kd, vd)
    assert kvc.get_error_flags() & kvc.FLAG_BAD_SLOT
    s2 = slots.clone()
    s2[1] = -1
    ek, ev = OP.append_to_paged(bits(k), bits(v), s2.numpy(), bits(kc), bits(vc))
    assert np.array_equal(bits(kd), ek) and np.array_equal(bits(vd), ev)


def test_append_latent_bit_exact(kvc):
    g = torch.Generator().manual_seed(5)
    nblk, bs, W_ = 6, 64, 576
    lc = W.normal((nblk, bs, W_), "bf16", g)
    c = W.normal((50, W_), "bf16", g)
    slots = torch.randperm(nblk * bs, generator=g)[:50].to(torch.int64)
    ld = lc.cuda()
    kvc.append_latent(c.cuda(), slots.cuda(), ld, 512)
    torch.cuda.synchronize()
    # the latent cache is the one-head special case of the paged layout
    e, _ = OP.append_to_paged(bits(c)[:, None, :], bits(c)[:, None, :], slots.numpy(), bits(lc)[:, None],
                              bits(lc)[:, None])
    assert np.array_equal(bits(ld), e[:, 0])


def test_append_large_batch_many_tokens(kvc):
    g = torch.Generator().manual_seed(6)
    nblk, hkv, bs, D = 300, 8, 16, 128
    kc = torch.zeros((nblk, hkv, bs, D), dtype=torch.bfloat16)
    vc = torch.zeros((nblk, hkv, bs, D), dtype=torch.bfloat16)
    T = nblk * bs
    k = W.normal((T, hkv, D), "bf16", g)
    v = W.normal((T, hkv, D), "bf16", g)
    slots = torch.randperm(T, generator=g).to(torch.int64)
    kd, vd = kc.cuda(), vc.cuda()
    kvc.append(k.cuda(), v.cuda(), slots.cuda(), kd, vd)
    torch.cuda.synchronize()
    # every slot written exactly once: cache row at slot s equals token t with slots[t] = s
    inv = torch.empty_like(slots)
    inv[slots] = torch.arange(T)
    got = kd.cpu().permute(0, 2, 1, 3).reshape(T, hkv, D)
    assert torch.equal(got.view(torch.int16), k[inv].view(torch.int16))
