"""GPU parity: the tensor-core decode for kv heads with 8 to 32 queries, against the oracle and against the
CUDA-core kernel. KVC_OPT_GQA_ENGINE = 2 forces the tensor-core kernel at any size (the automatic choice keeps
small caches on the CUDA-core kernel), 1 forces the CUDA-core kernel on the same inputs."""

import math

import numpy as np
import pytest
import torch

from oracle import paged as OP
from paged_kv_cache_157_gb300 import workloads as W

from gpu_helpers import TOL, append_new_tokens, device_case, f64, last_position_slots, max_err, \
    oracle_decode_sampled, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_options(kvc):
    opts = (kvc.OPT_BLOCKS_PER_CTA, kvc.OPT_MAX_CTAS, kvc.OPT_CHECKED, kvc.OPT_GQA_ENGINE)
    for o in opts:
        kvc.set_option(o, 0)
    kvc.set_option(kvc.OPT_GQA_ENGINE, 2)
    yield
    for o in opts:
        kvc.set_option(o, 0)


def decode_and_compare(kvc, case, tol, workspace="auto", engine=2):
    kvc.set_option(kvc.OPT_GQA_ENGINE, engine)
    dev = device_case(case)
    slots = last_position_slots(kvc, case)
    append_new_tokens(kvc, case, dev, slots)
    scale = 1.0 / math.sqrt(case["q"].shape[-1])
    out = run_decode(kvc, dev, scale, torch.float32, workspace)
    kc, vc = OP.append_to_paged(f64(case["k_new"]), f64(case["v_new"]), slots.numpy(), f64(case["k_cache"]),
                                f64(case["v_cache"]))
    ref = OP.paged_decode(f64(case["q"]), kc, vc, case["block_tables"].numpy(), case["context_lens"].numpy(), scale)
    err = max_err(out, ref)
    assert err <= tol, f"engine {engine}: max abs error {err:.3e} > {tol}"
    assert torch.isfinite(out).all()
    assert kvc.get_error_flags() == 0
    return out


LENS = [1, 15, 16, 17, 127, 128, 129, 255, 256, 257, 1000]


@pytest.mark.parametrize("engine", [0, 1, 2])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("hq,hkv", [(64, 8), (32, 2), (32, 1), (24, 2), (8, 1)])
def test_wide_groups_both_engines(kvc, engine, dtype, hq, hkv):
    # 8, 16, 32, 12 and 8 queries per kv head (MQA at 32 and 8)
    case = W.gqa_case(len(LENS), hq, hkv, 128, 16, LENS, dtype, seed=120 + hq + hkv)
    decode_and_compare(kvc, case, TOL[dtype], engine=engine)


def test_engines_agree(kvc):
    case = W.gqa_case(6, 64, 8, 128, 16, (1, 3000), "bf16", seed=121)
    a = decode_and_compare(kvc, case, TOL["bf16"], engine=2)
    b = decode_and_compare(kvc, case, TOL["bf16"], engine=1)
    assert float((a - b).abs().max()) <= 2e-3


@pytest.mark.parametrize("bs", [32, 64, 128])
def test_wide_block_sizes(kvc, bs):
    case = W.gqa_case(5, 64, 8, 128, bs, [1, bs - 1, bs + 1, 700, 129], "bf16", seed=122)
    decode_and_compare(kvc, case, TOL["bf16"])


@pytest.mark.parametrize("blocks_per_cta", [1, 8, 64])
def test_wide_forced_split_k(kvc, blocks_per_cta):
    # many contributors per unit (up to 5000 / 16 with one block per CTA: records merged in chunks of 64)
    kvc.set_option(kvc.OPT_BLOCKS_PER_CTA, blocks_per_cta)
    case = W.gqa_case(4, 32, 2, 128, 16, [5000, 3000, 1, 129], "bf16", seed=123)
    decode_and_compare(kvc, case, TOL["bf16"])


def test_wide_few_ctas_many_segments(kvc):
    kvc.set_option(kvc.OPT_MAX_CTAS, 3)
    case = W.gqa_case(9, 64, 8, 128, 16, (1, 400), "f16", seed=124)
    decode_and_compare(kvc, case, TOL["f16"])


def test_wide_without_workspace(kvc):
    case = W.gqa_case(4, 64, 8, 128, 16, [5, 1700, 64, 1], "bf16", seed=125)
    decode_and_compare(kvc, case, TOL["bf16"], workspace=None)


def test_wide_nan_in_unused_tail_slots(kvc):
    lens = [17, 31, 40, 1, 130]
    case = W.gqa_case(len(lens), 64, 8, 128, 16, lens, "bf16", seed=126)
    for i, n in enumerate(lens):
        blk = int(case["block_tables"][i, (n - 1) // 16])
        for c in ("k_cache", "v_cache"):
            case[c][blk, :, n % 16 if n % 16 else 16:, :] = float("nan")
    dev = device_case(case)
    out = run_decode(kvc, dev, 1.0 / math.sqrt(128))
    assert torch.isfinite(out).all()
    ref = OP.paged_decode(f64(case["q"]), f64(case["k_cache"]), f64(case["v_cache"]), case["block_tables"].numpy(),
                          case["context_lens"].numpy(), 1.0 / math.sqrt(128))
    assert max_err(out, ref) <= TOL["bf16"]


def test_wide_single_row_is_the_value_exactly(kvc):
    case = W.gqa_case(3, 64, 8, 128, 16, [1, 1, 1], "bf16", seed=127)
    dev = device_case(case)
    out = run_decode(kvc, dev, 0.1)
    for i in range(3):
        blk = int(case["block_tables"][i, 0])
        for h in range(64):
            assert torch.equal(out[i, h].cpu(), case["v_cache"][blk, h // 8, 0].float())


@pytest.mark.parametrize("T,hq,hkv", [(2, 64, 8), (8, 32, 8), (3, 32, 8), (4, 32, 8)])
@pytest.mark.parametrize("blocks_per_cta", [0, 1, 3])
def test_wide_multi_token(kvc, T, hq, hkv, blocks_per_cta):
    # T x group = 16, 32, 12, 16 queries per kv head, causal among the T new tokens
    from test_gpu_multi import multi_step
    kvc.set_option(kvc.OPT_BLOCKS_PER_CTA, blocks_per_cta)
    lens = [T, T + 1, 127 + T, 128, 129 + T, 600]
    case = W.multi_case(len(lens), T, hq, hkv, 128, 16, lens, "bf16", seed=130 + T)
    multi_step(kvc, case, TOL["bf16"])


def test_wide_long_context_sampled(kvc):
    # the long split-K shape: 64 q / 8 kv heads, contexts 32768 and 65536; sampled heads against the oracle
    case = W.gqa_case(2, 64, 8, 128, 16, [32768, 65536], "bf16", seed=45)
    dev = device_case(case)
    out = run_decode(kvc, dev, 1.0 / math.sqrt(128))
    pairs = [(0, 0), (0, 37), (1, 7), (1, 63)]
    ref = oracle_decode_sampled(case, 1.0 / math.sqrt(128), pairs)
    for (i, h), r in ref.items():
        assert float(np.max(np.abs(f64(out[i, h]) - r))) <= TOL["bf16"]
    assert kvc.get_error_flags() == 0


def test_config4_long_splitk_full_size_sampled(kvc):
    # the long split-K configuration at full size, in the launch configuration bench.py times: batch 4, 64 q / 8 kv
    # heads, contexts 32768 / 65536 / 131072 / 131072, block 16 (tensor-core kernel, many split-K records per unit)
    lens = [32768, 65536, 131072, 131072]
    case = W.gqa_case(4, 64, 8, 128, 16, lens, "bf16", seed=45)
    dev = device_case(case)
    out = run_decode(kvc, dev, 1.0 / math.sqrt(128))
    pairs = [(0, 0), (1, 31), (2, 8), (3, 63), (3, 1)]
    ref = oracle_decode_sampled(case, 1.0 / math.sqrt(128), pairs)
    for (i, h), r in ref.items():
        assert float(np.max(np.abs(f64(out[i, h]) - r))) <= TOL["bf16"], (i, h)
    assert kvc.get_error_flags() == 0
