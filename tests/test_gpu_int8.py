"""GPU parity: INT8 KV cache: kvc_append_int8 (bit-exact codes and scales) and
kvc_decode_attention_int8 (against float64 attention over the dequantised pools)."""

import math

import numpy as np
import pytest
import torch

from oracle import paged as OP
from oracle import quant as Q
from paged_kv_cache_157_gb300 import workloads as W

from gpu_helpers import f64, last_position_slots, max_err

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(autouse=True)
def _reset_options(kvc):
    for o in (kvc.OPT_BLOCKS_PER_CTA, kvc.OPT_MAX_CTAS, kvc.OPT_CHECKED):
        kvc.set_option(o, 0)
    yield
    for o in (kvc.OPT_BLOCKS_PER_CTA, kvc.OPT_MAX_CTAS, kvc.OPT_CHECKED):
        kvc.set_option(o, 0)


def _append_both(kvc, case, dev, slots):
    kvc.append_int8(dev["k_new"], dev["v_new"], slots.cuda(), dev["k_cache"], dev["v_cache"], dev["v_scale"],
                    dev["k_scale"])
    return Q.append_int8(case["k_new"].float().numpy(), case["v_new"].float().numpy(), slots.numpy(),
                         case["k_cache"].numpy(), case["v_cache"].numpy(), case["v_scale"].numpy(),
                         case["k_scale"].numpy())


def int8_step(kvc, case, workspace=True, pairs=None):
    """Append every sequence's new token (quantised on the GPU), decode, compare with the oracle."""
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in case.items()}
    slots = last_position_slots(kvc, case)
    kc, vc, vs = _append_both(kvc, case, dev, slots)
    torch.cuda.synchronize()
    bs = case["block_size"]
    for s in slots.tolist():
        b, o = s // bs, s % bs
        assert np.array_equal(dev["k_cache"][b, :, o].cpu().numpy(), kc[b, :, o])
        assert np.array_equal(dev["v_cache"][b, :, o].cpu().numpy(), vc[b, :, o])
        assert np.array_equal(dev["v_scale"][b, :, o].cpu().numpy(), vs[b, :, o])
    B, Hq, D = case["q"].shape
    _, Hkv, _, _ = case["k_cache"].shape
    out = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    ws = kvc.new_decode_workspace(B, Hq, Hkv, D, bs, case["block_tables"].shape[1]) if workspace else None
    scale = 1.0 / math.sqrt(D)
    kvc.decode_attention_int8(dev["q"], dev["k_cache"], dev["v_cache"], dev["k_scale"], dev["v_scale"],
                              dev["block_tables"], dev["context_lens"], scale, out, ws)
    torch.cuda.synchronize()
    K, V = Q.dequantized_pools_int8(kc, vc, vs, case["k_scale"].numpy())
    q = f64(case["q"])
    tables, lens = case["block_tables"].numpy(), case["context_lens"].numpy()
    if pairs is None:
        ref = OP.paged_decode(q, K, V, tables, lens, scale)
        err = max_err(out, ref)
    else:
        g = Hq // Hkv
        got = f64(out)
        err = 0.0
        for (i, h) in pairs:
            r, _ = OP.paged_decode_one(q[i, h], K, V, tables[i], int(lens[i]), h // g, scale)
            err = max(err, float(np.max(np.abs(got[i, h] - r))))
    assert err <= TOL, f"max abs error {err:.3e}"
    assert torch.isfinite(out).all()
    assert kvc.get_error_flags() == 0


@pytest.mark.parametrize("hq,hkv,D", [(32, 8, 128), (8, 8, 64), (16, 2, 128), (16, 2, 256), (64, 8, 128),
                                      (8, 1, 64)])
def test_int8_ragged(kvc, hq, hkv, D):
    lens = [1, 15, 16, 17, 33, 200, 129]
    case = W.int8_case(len(lens), hq, hkv, D, 16, lens, seed=180 + D + hq)
    int8_step(kvc, case)


@pytest.mark.parametrize("blocks_per_cta", [1, 3])
def test_int8_forced_split_k(kvc, blocks_per_cta):
    kvc.set_option(kvc.OPT_BLOCKS_PER_CTA, blocks_per_cta)
    case = W.int8_case(5, 32, 8, 128, 16, [1, 17, 160, 333, 64], seed=190)
    int8_step(kvc, case)


def test_int8_without_workspace_block_64(kvc):
    case = W.int8_case(3, 16, 4, 128, 64, [5, 300, 129], seed=191)
    int8_step(kvc, case, workspace=False)


def test_int8_append_ties_saturation_zero_rows_bit_exact(kvc):
    # K scales of 0.25 and K values on the 0.125 grid put k / s on half-integers (ties to even); K values beyond
    # 127 * s saturate; one all-zero V row takes scale 1; f32, f16 and bf16 inputs.
    for dt in (torch.float32, torch.float16, torch.bfloat16):
        case = W.int8_case(4, 8, 4, 64, 16, [3, 20, 16, 1], seed=192)
        T, hkv, d = case["k_new"].shape
        g = torch.Generator().manual_seed(7)
        grid = torch.randint(-400, 401, (T, hkv, d), generator=g).float() * 0.125  # |k / s| up to 200
        case["k_scale"] = torch.full((hkv, d), 0.25, dtype=torch.float32)
        case["k_new"] = grid.to(dt)
        v = case["v_new"].float() * 37.5
        v[1, 2] = 0.0
        case["v_new"] = v.to(dt)
        dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in case.items()}
        slots = last_position_slots(kvc, case)
        kc, vc, vs = _append_both(kvc, case, dev, slots)
        assert np.array_equal(dev["k_cache"].cpu().numpy(), kc)
        assert np.array_equal(dev["v_cache"].cpu().numpy(), vc)
        assert np.array_equal(dev["v_scale"].cpu().numpy(), vs)
        assert np.abs(kc).max() == 127 and kc.min() >= -127


def test_int8_skipped_slots(kvc):
    case = W.int8_case(4, 8, 4, 64, 16, [3, 20, 16, 1], seed=193)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in case.items()}
    slots = last_position_slots(kvc, case)
    slots[1] = -1
    kc, vc, vs = _append_both(kvc, case, dev, slots)
    assert np.array_equal(dev["k_cache"].cpu().numpy(), kc)
    assert np.array_equal(dev["v_cache"].cpu().numpy(), vc)
    assert np.array_equal(dev["v_scale"].cpu().numpy(), vs)
    assert kvc.get_error_flags() == 0


def test_int8_full_size_sampled(kvc):
    # Llama-3-8B-shaped layer, batch 32, lengths 4096, int8 cache
    case = W.int8_case(32, 32, 8, 128, 16, [4096] * 32, seed=194)
    rng = np.random.default_rng(1)
    pairs = [(int(i), int(h)) for i, h in zip(rng.integers(0, 32, 12), rng.integers(0, 32, 12))] + [(0, 0), (31, 31)]
    int8_step(kvc, case, pairs=pairs)
