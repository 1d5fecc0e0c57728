"""GPU parity of the warp-MMA decode kernel (KVC_OPT_GQA_ENGINE = 3) against the oracle.

The kernel takes bf16/f16 caches with head_dim 128 and computes each 16-row
tile's scores and output on m16n8k16 MMAs over 128B-swizzled TMA tiles. These
cases cover every head grouping it plans for (1, 2, 4, 8 and 16 query heads per
kv head, the last over two warps), every block size, ragged tails, forced
split-K partials, the window / several-token / start-row extensions, and the
exact special cases; the CUDA-core kernel (engine 1) runs beside it on the same
inputs.
"""

import math

import numpy as np
import pytest
import torch

from oracle import paged as OP
from paged_kv_cache_157_gb300 import workloads as W

from gpu_helpers import TOL, device_case, f64, max_err, oracle_decode, oracle_decode_sampled, run_decode

pytestmark = pytest.mark.gpu

OPTS = ("OPT_BLOCKS_PER_CTA", "OPT_MAX_CTAS", "OPT_CHECKED", "OPT_GQA_ENGINE", "OPT_DYNAMIC_SHARE",
        "OPT_DYNAMIC_CHUNK")


@pytest.fixture(autouse=True)
def _mma_engine(kvc):
    for o in OPTS:
        kvc.set_option(getattr(kvc, o), 0)
    kvc.set_option(kvc.OPT_GQA_ENGINE, 3)
    yield
    for o in OPTS:
        kvc.set_option(getattr(kvc, o), 0)


def _check(kvc, case, scale, tol, out_dtype=torch.float32, workspace="auto"):
    dev = device_case(case)
    out = run_decode(kvc, dev, scale, out_dtype, workspace)
    ref = oracle_decode(case, scale)
    err = max_err(out, ref)
    assert err <= tol, f"max abs error {err:.3e} > {tol}"
    assert torch.isfinite(out).all()
    assert kvc.get_error_flags() == 0
    return out, dev


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 8), (8, 1), (16, 2), (6, 2), (64, 8), (32, 2), (24, 2), (12, 4),
                                    (4, 4), (128, 8)])
def test_head_groupings_ragged(kvc, dtype, hq, hkv):
    lens = [1, 15, 16, 17, 31, 32, 33, 47, 200, 129]
    case = W.gqa_case(len(lens), hq, hkv, 128, 16, lens, dtype, seed=101)
    _check(kvc, case, 1.0 / math.sqrt(128), TOL[dtype])


@pytest.mark.parametrize("bs", [16, 32, 48, 64, 128])
@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 8), (64, 8)])
def test_block_sizes(kvc, bs, hq, hkv):
    case = W.gqa_case(5, hq, hkv, 128, bs, [1, bs - 1, bs + 1, 3 * bs, 700], "bf16", seed=102)
    _check(kvc, case, 1.0 / math.sqrt(128), TOL["bf16"])


@pytest.mark.parametrize("blocks_per_cta", [1, 2, 3, 7])
@pytest.mark.parametrize("hq,hkv", [(32, 8), (64, 8), (32, 2)])
def test_forced_split_k(kvc, blocks_per_cta, hq, hkv):
    kvc.set_option(kvc.OPT_BLOCKS_PER_CTA, blocks_per_cta)
    case = W.gqa_case(5, hq, hkv, 128, 16, [1, 17, 160, 333, 64], "bf16", seed=103)
    _check(kvc, case, 1.0 / math.sqrt(128), TOL["bf16"])


def test_few_ctas_many_segments(kvc):
    kvc.set_option(kvc.OPT_MAX_CTAS, 3)
    case = W.gqa_case(9, 8, 2, 128, 16, (1, 120), "f16", seed=104)
    _check(kvc, case, 1.0 / math.sqrt(128), TOL["f16"])


def test_without_workspace(kvc):
    case = W.gqa_case(4, 32, 8, 128, 16, [5, 700, 64, 1], "bf16", seed=105)
    _check(kvc, case, 1.0 / math.sqrt(128), TOL["bf16"], workspace=None)


def test_matches_cuda_core_kernel(kvc):
    case = W.gqa_case(6, 32, 8, 128, 16, (1, 900), "bf16", seed=106)
    dev = device_case(case)
    a = run_decode(kvc, dev, 0.088)
    kvc.set_option(kvc.OPT_GQA_ENGINE, 1)
    b = run_decode(kvc, dev, 0.088)
    assert float((a - b).abs().max()) <= 2e-3


def test_n1_returns_value_row_exactly(kvc):
    case = W.gqa_case(3, 16, 2, 128, 16, [1, 1, 1], "bf16", seed=107)
    out, _ = _check(kvc, case, 0.1, TOL["bf16"])
    for i in range(3):
        blk = int(case["block_tables"][i, 0])
        for h in range(16):
            assert torch.equal(out[i, h].cpu(), case["v_cache"][blk, h // 8, 0].float())


def test_zero_query_gives_mean(kvc):
    case = W.gqa_case(2, 8, 2, 128, 16, [40, 7], "f16", seed=108)
    case["q"].zero_()
    out, _ = _check(kvc, case, 0.3, TOL["f16"])
    for i, n in enumerate([40, 7]):
        for h in range(8):
            rows = OP.gather_logical(f64(case["v_cache"]), case["block_tables"][i].numpy(), n, h // 4)
            assert np.max(np.abs(f64(out[i, h]) - rows.mean(axis=0))) < 1e-5


def test_nan_in_tail_and_unused_blocks(kvc):
    lens = [17, 31, 40, 1, 64]
    case = W.gqa_case(5, 32, 8, 128, 32, lens, "bf16", seed=109)
    for i, n in enumerate(lens):
        blk = int(case["block_tables"][i, (n - 1) // 32])
        for c in ("k_cache", "v_cache"):
            if n % 32:
                case[c][blk, :, n % 32:, :] = float("nan")
    _check(kvc, case, 1.0 / math.sqrt(128), TOL["bf16"])


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
def test_low_precision_output(kvc, out_dtype):
    case = W.gqa_case(4, 32, 8, 128, 16, [17, 100, 3, 64], "bf16", seed=110)
    dev = device_case(case)
    out = run_decode(kvc, dev, 1.0 / math.sqrt(128), out_dtype=out_dtype)
    ref = oracle_decode(case, 1.0 / math.sqrt(128))
    rounded = torch.from_numpy(ref).to(out_dtype).to(torch.float64).numpy()
    ulp = np.abs(rounded) * (2.0 ** -7 if out_dtype == torch.bfloat16 else 2.0 ** -10)
    assert np.all(np.abs(f64(out) - rounded) <= np.maximum(ulp, 2e-3))


def test_bad_block_and_bad_length_flags(kvc):
    case = W.gqa_case(3, 8, 2, 128, 16, [40, 20, 5], "bf16", seed=111)
    case["block_tables"][0, 1] = case["num_blocks"] + 5
    dev = device_case(case)
    run_decode(kvc, dev, 0.1)
    assert kvc.get_error_flags() & kvc.FLAG_BAD_BLOCK
    case = W.gqa_case(3, 8, 2, 128, 16, [40, 20, 5], "bf16", seed=112)
    case["context_lens"][1] = 0
    dev = device_case(case)
    out = run_decode(kvc, dev, 0.1)
    assert kvc.get_error_flags() & kvc.FLAG_BAD_LEN
    assert torch.count_nonzero(out[1]) == 0


@pytest.mark.parametrize("window", [1, 15, 16, 17, 100, 1000])
def test_window(kvc, window):
    lens = [1, 15, 16, 17, 31, 200, 129, 1500]
    case = W.gqa_case(len(lens), 32, 8, 128, 16, lens, "bf16", seed=113)
    dev = device_case(case)
    B, Hq, D = case["q"].shape
    out = torch.empty((B, Hq, D), device="cuda")
    ws = kvc.new_decode_workspace(B, Hq, 8, D, 16, case["block_tables"].shape[1])
    scale = 1.0 / math.sqrt(D)
    kvc.decode_attention_window(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"],
                                scale, window, out, ws)
    torch.cuda.synchronize()
    ref = OP.paged_decode_window(f64(case["q"]), f64(case["k_cache"]), f64(case["v_cache"]),
                                 case["block_tables"].numpy(), case["context_lens"].numpy(), scale, window)
    assert max_err(out, ref) <= TOL["bf16"]
    assert kvc.get_error_flags() == 0


@pytest.mark.parametrize("T,hq,hkv", [(2, 32, 8), (4, 32, 8), (3, 8, 8), (2, 64, 8)])
def test_several_new_tokens(kvc, T, hq, hkv):
    lens = [T, T + 1, 17, 40, 300]
    case = W.multi_case(len(lens), T, hq, hkv, 128, 16, lens, "bf16", seed=114)
    dev = device_case(case)
    B = len(lens)
    out = torch.empty((B, T, hq, 128), device="cuda")
    ws = kvc.new_multi_workspace(B, T, hq, hkv, 128, 16, case["block_tables"].shape[1])
    kvc.decode_attention_multi(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"],
                               1.0 / math.sqrt(128), out, ws)
    torch.cuda.synchronize()
    ref = OP.paged_decode_multi(f64(case["q"]), f64(case["k_cache"]), f64(case["v_cache"]),
                                case["block_tables"].numpy(), case["context_lens"].numpy(), 1.0 / math.sqrt(128))
    assert max_err(out, ref) <= TOL["bf16"]
    assert kvc.get_error_flags() == 0


def test_shared_prefix_passes(kvc):
    # the two passes of the shared-prefix decode (several tokens without the
    # causal rule, then start rows) must equal the plain decode
    case = W.shared_case(2, 4, 64, 40, 8, 128, 16, "f16", seed=115)
    dev = device_case(case)
    B, H, D = case["q"].shape
    out = torch.empty((B, H, D), device="cuda")
    prefix = torch.full((2,), 64, dtype=torch.int32, device="cuda")
    ws = kvc.shared_prefix_workspace(B, 4, H, H, D, 16, case["block_tables"].shape[1])
    kvc.decode_attention_shared_prefix(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                       dev["context_lens"], 4, prefix, 1.0 / math.sqrt(D), out, ws)
    torch.cuda.synchronize()
    ref = oracle_decode(case, 1.0 / math.sqrt(D))
    assert max_err(out, ref) <= TOL["f16"]
    assert kvc.get_error_flags() == 0


@pytest.mark.parametrize("chunk,share,max_ctas", [(1, 128, 3), (2, 200, 0), (5, 64, 7), (3, 255, 0), (8, 256, 0),
                                                  (1, 255, 1)])
def test_dynamic_work_split(kvc, chunk, share, max_ctas):
    # Part of the blocks is claimed at run time in chunks; every chunk that cuts
    # a unit leaves records the last contributor merges. Two calls in a row on
    # one workspace: the claim counter must be back at zero after each.
    kvc.set_option(kvc.OPT_DYNAMIC_CHUNK, chunk)
    kvc.set_option(kvc.OPT_DYNAMIC_SHARE, share)
    kvc.set_option(kvc.OPT_MAX_CTAS, max_ctas)
    lens = [1, 17, 160, 333, 64, 2000, 45]
    case = W.gqa_case(len(lens), 32, 8, 128, 16, lens, "bf16", seed=116)
    dev = device_case(case)
    ws = kvc.new_decode_workspace(len(lens), 32, 8, 128, 16, case["block_tables"].shape[1])
    ref = oracle_decode(case, 1.0 / math.sqrt(128))
    for _ in range(2):
        out = run_decode(kvc, dev, 1.0 / math.sqrt(128), workspace=ws)
        assert max_err(out, ref) <= TOL["bf16"]
        assert kvc.get_error_flags() == 0


def test_dynamic_split_on_large_batch(kvc):
    # a quarter of every unit's blocks claimed in chunks of 8 on a large batch,
    # three calls on one workspace (the claim counter resets itself)
    kvc.set_option(kvc.OPT_DYNAMIC_SHARE, 64)
    kvc.set_option(kvc.OPT_DYNAMIC_CHUNK, 8)
    case = W.gqa_case(16, 32, 8, 128, 16, (1024, 4096), "bf16", seed=117)
    dev = device_case(case)
    ws = kvc.new_decode_workspace(16, 32, 8, 128, 16, case["block_tables"].shape[1])
    outs = [run_decode(kvc, dev, 1.0 / math.sqrt(128), workspace=ws) for _ in range(3)]
    ref = oracle_decode(case, 1.0 / math.sqrt(128))
    for o in outs:
        assert max_err(o, ref) <= TOL["bf16"]
    assert kvc.get_error_flags() == 0


def test_one_long_sequence_many_contributors(kvc):
    # one sequence of 32768 rows with 8 queries per kv head: a single unit cut
    # into every CTA's range, so its merge folds ~150 records in several rounds
    case = W.gqa_case(1, 64, 8, 128, 16, [32768], "bf16", seed=118)
    dev = device_case(case)
    scale = 1.0 / math.sqrt(128)
    out = run_decode(kvc, dev, scale)
    ref = oracle_decode_sampled(case, scale, [(0, h) for h in (0, 7, 8, 31, 56, 63)])
    for (i, h), r in ref.items():
        assert float(np.max(np.abs(f64(out[i, h]) - r))) <= TOL["bf16"]
    assert torch.isfinite(out).all()
    assert kvc.get_error_flags() == 0
