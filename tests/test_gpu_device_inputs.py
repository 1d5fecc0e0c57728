"""GPU: decode inputs written on the device by the kernel right before the decode.

The decode kernels start while the previous kernel of the stream still runs
(programmatic stream serialisation, so a step's append and decode overlap).
Every thread of a decode kernel must therefore wait for that kernel before it
reads the lengths, block tables or queries, or writes the output. These tests
make the previous kernel the one that writes those inputs (a torch kernel on
the same stream, no host synchronisation in between) and check the result
against the oracle on the final values.
"""

import math

import numpy as np
import pytest
import torch

from oracle import mla as OM
from oracle import paged as OP
from paged_kv_cache_157_gb300 import workloads as W

from gpu_helpers import f64

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_options(kvc):
    for o in (kvc.OPT_BLOCKS_PER_CTA, kvc.OPT_MAX_CTAS, kvc.OPT_CHECKED, kvc.OPT_GQA_ENGINE):
        kvc.set_option(o, 0)
    yield
    for o in (kvc.OPT_BLOCKS_PER_CTA, kvc.OPT_MAX_CTAS, kvc.OPT_CHECKED, kvc.OPT_GQA_ENGINE):
        kvc.set_option(o, 0)


def _stale_then_fixed(case):
    """Device copies of the lengths and tables with wrong contents (lengths one short of the truth, the table
    rows reversed), plus on-device sources for the right values."""
    lens = case["context_lens"].cuda()
    tables = case["block_tables"].cuda()
    return lens - 1, tables.flip(0).contiguous(), lens, tables


def _fix_on_device(lens_dev, tables_dev, lens_src, tables_src, last):
    """Rewrite lengths and tables with torch kernels on the current stream; `last` says which is written by the
    kernel that runs immediately before the decode."""
    rows = torch.arange(tables_dev.shape[0], device="cuda")
    if last == "lens":
        tables_dev.index_copy_(0, rows, tables_src)
        lens_dev.add_(lens_src - lens_dev)  # one kernel: lens_dev += (lens - stale), i.e. lens
    else:
        lens_dev.add_(lens_src - lens_dev)
        tables_dev.index_copy_(0, rows, tables_src)


@pytest.mark.parametrize("hq,hkv,engine", [(32, 8, 0), (64, 8, 2), (8, 8, 0)])
@pytest.mark.parametrize("last", ["lens", "tables"])
def test_gqa_inputs_written_by_previous_kernel(kvc, hq, hkv, engine, last):
    kvc.set_option(kvc.OPT_GQA_ENGINE, engine)
    D = 128
    scale = 1.0 / math.sqrt(D)
    case = W.gqa_case(6, hq, hkv, D, 16, [700, 1, 33, 2048, 129, 1500], "bf16", seed=71)
    kc, vc, q = case["k_cache"].cuda(), case["v_cache"].cuda(), case["q"].cuda()
    ws = kvc.new_decode_workspace(6, hq, hkv, D, 16, case["block_tables"].shape[1])
    lens_dev, tables_dev, lens_src, tables_src = _stale_then_fixed(case)
    out = torch.full((6, hq, D), float("nan"), device="cuda")
    torch.cuda.synchronize()
    for _ in range(3):  # repeated: the stale values are restored before each call
        lens_dev.sub_(1)
        tables_dev.copy_(tables_src.flip(0))
        _fix_on_device(lens_dev, tables_dev, lens_src, tables_src, last)
        kvc.decode_attention(q, kc, vc, tables_dev, lens_dev, scale, out, ws)
    torch.cuda.synchronize()
    ref = OP.paged_decode(f64(case["q"]), f64(case["k_cache"]), f64(case["v_cache"]), case["block_tables"].numpy(),
                          case["context_lens"].numpy(), scale)
    err = float(np.max(np.abs(f64(out) - ref)))
    assert err <= 2e-3, err
    assert kvc.get_error_flags() == 0


def test_gqa_query_written_by_previous_kernel(kvc):
    # the query rows themselves produced by the kernel just before the decode
    D = 128
    scale = 1.0 / math.sqrt(D)
    case = W.gqa_case(4, 32, 8, D, 16, [900, 17, 4000, 256], "bf16", seed=72)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in case.items()}
    ws = kvc.new_decode_workspace(4, 32, 8, D, 16, case["block_tables"].shape[1])
    q_dev = torch.zeros_like(dev["q"])
    out = torch.empty((4, 32, D), device="cuda")
    torch.cuda.synchronize()
    q_dev.add_(dev["q"])  # the previous kernel writes q
    kvc.decode_attention(q_dev, dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"], scale, out,
                         ws)
    torch.cuda.synchronize()
    ref = OP.paged_decode(f64(case["q"]), f64(case["k_cache"]), f64(case["v_cache"]), case["block_tables"].numpy(),
                          case["context_lens"].numpy(), scale)
    assert float(np.max(np.abs(f64(out) - ref))) <= 2e-3
    assert kvc.get_error_flags() == 0


def test_mla_lengths_written_by_previous_kernel(kvc):
    D_C, D_R, H = 512, 64, 128
    case = W.mla_case(4, H, D_C, D_R, 64, [70, 1, 1200, 300], "bf16", seed=73)
    lat, q = case["latent_cache"].cuda(), case["q"].cuda()
    tables = case["block_tables"].cuda()
    lens_src = case["context_lens"].cuda()
    lens_dev = lens_src - 5
    n = kvc.decode_mla_workspace_size(4, H, D_C, D_R, 64, case["block_tables"].shape[1])
    ws = torch.zeros(max(1, n), dtype=torch.uint8, device="cuda")
    out = torch.empty((4, H, D_C), device="cuda")
    torch.cuda.synchronize()
    lens_dev.add_(5)  # the previous kernel writes the lengths
    kvc.decode_attention_mla(q, lat, tables, lens_dev, 1.0 / 24.0, D_C, out, ws)
    torch.cuda.synchronize()
    ref, _ = OM.mla_absorbed_decode(f64(case["q"]), f64(case["latent_cache"]), case["block_tables"].numpy(),
                                    case["context_lens"].numpy(), 1.0 / 24.0, D_C)
    assert float(np.max(np.abs(f64(out) - ref))) <= 2e-3
    assert kvc.get_error_flags() == 0
