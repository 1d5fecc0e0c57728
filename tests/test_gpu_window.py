"""GPU parity: sliding-window decode (kvc_decode_attention_window) against the oracle."""

import math

import numpy as np
import pytest
import torch

from oracle import paged as OP
from paged_kv_cache_157_gb300 import workloads as W

from gpu_helpers import TOL, append_new_tokens, device_case, f64, last_position_slots, max_err

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_options(kvc):
    for o in (kvc.OPT_BLOCKS_PER_CTA, kvc.OPT_MAX_CTAS, kvc.OPT_CHECKED):
        kvc.set_option(o, 0)
    yield
    for o in (kvc.OPT_BLOCKS_PER_CTA, kvc.OPT_MAX_CTAS, kvc.OPT_CHECKED):
        kvc.set_option(o, 0)


def window_step(kvc, case, window, tol, workspace=True, out_dtype=torch.float32, poison_outside=False):
    """Append every sequence's new token, run the windowed decode, compare with the oracle."""
    dev = device_case(case)
    slots = last_position_slots(kvc, case)
    append_new_tokens(kvc, case, dev, slots)
    kc, vc = OP.append_to_paged(f64(case["k_new"]), f64(case["v_new"]), slots.numpy(), f64(case["k_cache"]),
                                f64(case["v_cache"]))
    if poison_outside:
        # rows before the window may hold anything: NaN there must not reach the output
        bs = case["block_size"]
        for i, n in enumerate(case["context_lens"].tolist()):
            for pos in range(max(0, n - window)):
                blk = int(case["block_tables"][i, pos // bs])
                dev["k_cache"][blk, :, pos % bs, :] = float("nan")
                dev["v_cache"][blk, :, pos % bs, :] = float("nan")
    B, Hq, D = case["q"].shape
    _, Hkv, bs, _ = case["k_cache"].shape
    out = torch.empty((B, Hq, D), dtype=out_dtype, device="cuda")
    ws = kvc.new_decode_workspace(B, Hq, Hkv, D, bs, case["block_tables"].shape[1]) if workspace else None
    scale = 1.0 / math.sqrt(D)
    kvc.decode_attention_window(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"],
                                scale, window, out, ws)
    torch.cuda.synchronize()
    ref = OP.paged_decode_window(f64(case["q"]), kc, vc, case["block_tables"].numpy(),
                                 case["context_lens"].numpy(), scale, window)
    err = max_err(out, ref)
    assert err <= tol, f"window {window}: max abs error {err:.3e} > {tol}"
    assert torch.isfinite(out).all()
    assert kvc.get_error_flags() == 0
    return out


@pytest.mark.parametrize("window", [1, 2, 15, 16, 17, 31, 33, 100, 1000])
def test_window_ragged_bf16(kvc, window):
    lens = [1, 15, 16, 17, 31, 32, 33, 47, 200, 129]
    case = W.gqa_case(len(lens), 32, 8, 128, 16, lens, "bf16", seed=61)
    window_step(kvc, case, window, TOL["bf16"])


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("hq,hkv,D", [(8, 8, 64), (16, 2, 128), (8, 4, 32), (16, 2, 256)])
def test_window_dtypes_and_groups(kvc, dtype, hq, hkv, D):
    lens = [3, 40, 77, 130]
    case = W.gqa_case(len(lens), hq, hkv, D, 16, lens, dtype, seed=62)
    window_step(kvc, case, 37, TOL[dtype])


@pytest.mark.parametrize("blocks_per_cta", [1, 2, 5])
def test_window_forced_split_k(kvc, blocks_per_cta):
    kvc.set_option(kvc.OPT_BLOCKS_PER_CTA, blocks_per_cta)
    case = W.gqa_case(5, 32, 8, 128, 16, [1, 17, 160, 333, 64], "bf16", seed=63)
    window_step(kvc, case, 50, TOL["bf16"])


def test_window_without_workspace_and_larger_blocks(kvc):
    case = W.gqa_case(4, 16, 4, 128, 64, [5, 700, 64, 130], "bf16", seed=64)
    window_step(kvc, case, 90, TOL["bf16"], workspace=False)


def test_rows_outside_the_window_are_never_read(kvc):
    case = W.gqa_case(6, 32, 8, 128, 16, [20, 64, 65, 300, 17, 1000], "bf16", seed=65)
    window_step(kvc, case, 33, TOL["bf16"], poison_outside=True)


def test_window_one_returns_the_new_value_exactly(kvc):
    case = W.gqa_case(3, 8, 2, 128, 16, [1, 50, 123], "f32", seed=66)
    out = window_step(kvc, case, 1, 0.0)  # a single weight of 1: the value row itself
    assert out is not None


def test_window_must_be_positive(kvc):
    case = W.gqa_case(1, 8, 8, 64, 16, [10], "bf16", seed=67)
    dev = device_case(case)
    out = torch.empty((1, 8, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(kvc.KvcError) as e:
        kvc.decode_attention_window(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                    dev["context_lens"], 0.125, 0, out, None)
    assert e.value.status == kvc.ERR_INVALID_ARG


def test_window_full_size_sampled(kvc):
    # Llama-3-8B-shaped layer with a Mistral-style window: batch 32, lengths 4096, W = 1024
    case = W.gqa_case(32, 32, 8, 128, 16, [4096] * 32, "bf16", seed=68)
    window_step(kvc, case, 1024, TOL["bf16"])
