"""GPU parity: append + paged decode attention (kvc_append, kvc_decode_attention) against the oracle."""

import math

import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import paged as OP
from paged_kv_cache_157_gb300 import workloads as W

from gpu_helpers import TOL, append_new_tokens, device_case, f64, last_position_slots, max_err, oracle_decode, \
    run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_options(kvc):
    kvc.set_option(kvc.OPT_BLOCKS_PER_CTA, 0)
    kvc.set_option(kvc.OPT_MAX_CTAS, 0)
    kvc.set_option(kvc.OPT_CHECKED, 0)
    yield
    kvc.set_option(kvc.OPT_BLOCKS_PER_CTA, 0)
    kvc.set_option(kvc.OPT_MAX_CTAS, 0)
    kvc.set_option(kvc.OPT_CHECKED, 0)


def step_and_compare(kvc, case, scale, tol, out_dtype=torch.float32, workspace="auto"):
    """One decode step: append the new token of every sequence, attend, compare with the oracle."""
    dev = device_case(case)
    slots = last_position_slots(kvc, case)
    append_new_tokens(kvc, case, dev, slots)
    out = run_decode(kvc, dev, scale, out_dtype, workspace)
    kc, vc = OP.append_to_paged(f64(case["k_new"]), f64(case["v_new"]), slots.numpy(), f64(case["k_cache"]),
                                f64(case["v_cache"]))
    ref = OP.paged_decode(f64(case["q"]), kc, vc, case["block_tables"].numpy(), case["context_lens"].numpy(), scale)
    err = max_err(out, ref)
    assert err <= tol, f"max abs error {err:.3e} > {tol}"
    assert kvc.get_error_flags() == 0
    return out, ref, dev


def test_config1_tiny_mha_fp32_every_step_vs_recompute(kvc):
    # 1 sequence, 2 layers, 4 heads, d 32, fp32, block 16: prompt of 5 tokens, then 64 decode steps;
    # every step is checked against full causal recomputation (no cache).
    H, D, bs, T = 4, 32, 16, 69
    layers = W.tiny_sequence(T, 2, H, D, "f32", seed=42)
    pool = kvc.BlockPool(8, bs)
    sid = pool.add()
    caches = [(torch.zeros((8, H, bs, D), device="cuda"), torch.zeros((8, H, bs, D), device="cuda"))
              for _ in layers]
    slots = torch.tensor(pool.reserve(sid, 5), dtype=torch.int64, device="cuda")
    for l, lay in enumerate(layers):
        kvc.append(lay["k"][:5].cuda(), lay["v"][:5].cuda(), slots, *caches[l])
    scale = 1.0 / math.sqrt(D)
    ws = kvc.new_decode_workspace(1, H, H, D, bs, 5)
    worst = 0.0
    for t in range(5, T):
        slot = torch.tensor(pool.reserve(sid, 1), dtype=torch.int64, device="cuda")
        rows, lens = pool.tables([sid], 5)
        bt = torch.tensor(rows, dtype=torch.int32, device="cuda")
        cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
        for l, lay in enumerate(layers):
            kvc.append(lay["k"][t:t + 1].cuda(), lay["v"][t:t + 1].cuda(), slot, *caches[l])
            out = torch.empty((1, H, D), device="cuda")
            kvc.decode_attention(lay["q"][t:t + 1].cuda(), caches[l][0], caches[l][1], bt, cl, scale, out, ws)
            got = f64(out)[0]
            for h in range(H):
                ref = OA.decode_by_recompute(f64(lay["q"][: t + 1, h]), f64(lay["k"][: t + 1, h]),
                                             f64(lay["v"][: t + 1, h]), scale)
                worst = max(worst, float(np.max(np.abs(got[h] - ref))))
    assert worst <= TOL["f32"], worst
    assert kvc.get_error_flags() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("hq,hkv,D", [(32, 8, 128), (8, 8, 128), (8, 1, 128), (16, 2, 64), (6, 2, 64),
                                      (16, 2, 256), (8, 4, 32), (64, 8, 128), (32, 2, 128), (32, 1, 64),
                                      (24, 2, 128), (32, 2, 256)])
def test_small_batch_ragged(kvc, dtype, hq, hkv, D):
    lens = [1, 15, 16, 17, 31, 32, 33, 47, 200, 129]
    case = W.gqa_case(len(lens), hq, hkv, D, 16, lens, dtype, seed=7)
    step_and_compare(kvc, case, 1.0 / math.sqrt(D), TOL[dtype])


@pytest.mark.parametrize("bs", [32, 64])
def test_larger_blocks(kvc, bs):
    case = W.gqa_case(6, 16, 4, 128, bs, (1, 500), "bf16", seed=11)
    step_and_compare(kvc, case, 1.0 / math.sqrt(128), TOL["bf16"])


@pytest.mark.parametrize("blocks_per_cta", [1, 2, 3, 5, 16])
def test_forced_split_k(kvc, blocks_per_cta):
    kvc.set_option(kvc.OPT_BLOCKS_PER_CTA, blocks_per_cta)
    case = W.gqa_case(5, 32, 8, 128, 16, [1, 17, 160, 333, 64], "bf16", seed=13)
    step_and_compare(kvc, case, 1.0 / math.sqrt(128), TOL["bf16"])


@pytest.mark.parametrize("hq,hkv,D", [(64, 8, 128), (32, 2, 128), (32, 2, 256)])
def test_forced_split_k_wide_groups(kvc, hq, hkv, D):
    # 8 and 16 query heads per unit, split over warps that share one page stream
    kvc.set_option(kvc.OPT_BLOCKS_PER_CTA, 3)
    case = W.gqa_case(4, hq, hkv, D, 16, [1, 90, 333, 17], "bf16", seed=14)
    step_and_compare(kvc, case, 1.0 / math.sqrt(D), TOL["bf16"])


def test_without_workspace_single_cta_per_unit(kvc):
    case = W.gqa_case(4, 32, 8, 128, 16, [5, 700, 64, 1], "bf16", seed=17)
    step_and_compare(kvc, case, 1.0 / math.sqrt(128), TOL["bf16"], workspace=None)


def test_few_ctas_many_segments(kvc):
    # three CTAs for the whole batch: every CTA crosses many units
    kvc.set_option(kvc.OPT_MAX_CTAS, 3)
    case = W.gqa_case(9, 8, 2, 128, 16, (1, 120), "f16", seed=19)
    step_and_compare(kvc, case, 1.0 / math.sqrt(128), TOL["f16"])


def test_physical_placement_is_invisible_bitwise(kvc):
    # Same logical data in an ascending pool and in a permuted pool: identical bits out.
    lens = [33, 250, 16, 97]
    a = W.gqa_case(4, 32, 8, 128, 16, lens, "bf16", seed=23, permute=False)
    b = dict(a)
    nb = a["num_blocks"]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(5))
    # physical block p of pool a moves to perm[p] in pool b
    b["k_cache"] = torch.empty_like(a["k_cache"])
    b["v_cache"] = torch.empty_like(a["v_cache"])
    b["k_cache"][perm] = a["k_cache"]
    b["v_cache"][perm] = a["v_cache"]
    b["block_tables"] = perm[a["block_tables"].long()].to(torch.int32)
    outs = []
    for c in (a, b):
        dev = device_case(c)
        outs.append(run_decode(kvc, dev, 1.0 / math.sqrt(128)))
    assert torch.equal(outs[0], outs[1])


def test_nan_in_unused_tail_slots_does_not_leak(kvc):
    lens = [17, 31, 40, 1]
    case = W.gqa_case(4, 16, 4, 128, 16, lens, "bf16", seed=29)
    for i, n in enumerate(lens):
        blk = int(case["block_tables"][i, (n - 1) // 16])
        for c in ("k_cache", "v_cache"):
            case[c][blk, :, n % 16 if n % 16 else 16:, :] = float("nan")
    dev = device_case(case)
    out = run_decode(kvc, dev, 1.0 / math.sqrt(128))
    assert torch.isfinite(out).all()
    ref = oracle_decode(case, 1.0 / math.sqrt(128))
    assert max_err(out, ref) <= TOL["bf16"]


def test_special_cases_exact(kvc):
    # n = 1: the output is that value row exactly, even through the split path
    case = W.gqa_case(3, 8, 2, 128, 16, [1, 1, 1], "bf16", seed=31)
    dev = device_case(case)
    out = run_decode(kvc, dev, 0.1)
    for i in range(3):
        blk = int(case["block_tables"][i, 0])
        for h in range(8):
            assert torch.equal(out[i, h].cpu(), case["v_cache"][blk, h // 4, 0].float())
    # q = 0: the mean of the value rows
    case = W.gqa_case(2, 4, 4, 64, 16, [40, 7], "f32", seed=37)
    case["q"].zero_()
    dev = device_case(case)
    out = run_decode(kvc, dev, 0.3)
    for i, n in enumerate([40, 7]):
        for h in range(4):
            rows = OP.gather_logical(f64(case["v_cache"]), case["block_tables"][i].numpy(), n, h)
            assert np.max(np.abs(f64(out[i, h]) - rows.mean(axis=0))) < 1e-6


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
def test_low_precision_output(kvc, out_dtype):
    case = W.gqa_case(4, 32, 8, 128, 16, [17, 100, 3, 64], "bf16", seed=41)
    dev = device_case(case)
    out = run_decode(kvc, dev, 1.0 / math.sqrt(128), out_dtype=out_dtype)
    ref = oracle_decode(case, 1.0 / math.sqrt(128))
    rounded = torch.from_numpy(ref).to(out_dtype).to(torch.float64).numpy()
    ulp = np.abs(rounded) * (2.0 ** -7 if out_dtype == torch.bfloat16 else 2.0 ** -10)
    err = np.abs(f64(out) - rounded)
    assert np.all(err <= np.maximum(ulp, 2e-3))


def test_bad_block_id_sets_flag_without_fault(kvc):
    case = W.gqa_case(2, 8, 2, 128, 16, [40, 20], "bf16", seed=43)
    case["block_tables"][0, 1] = case["num_blocks"] + 5
    case["block_tables"][1, 0] = -3
    dev = device_case(case)
    run_decode(kvc, dev, 0.1)
    flags = kvc.get_error_flags()
    assert flags & kvc.FLAG_BAD_BLOCK
    assert kvc.get_error_flags() == 0  # reading clears


def test_bad_context_len_zeroes_output_and_flags(kvc):
    case = W.gqa_case(3, 8, 2, 128, 16, [40, 20, 5], "bf16", seed=47)
    case["context_lens"][1] = 0
    for ws in ("auto", None):
        dev = device_case(case)
        out = run_decode(kvc, dev, 0.1, workspace=ws)
        assert kvc.get_error_flags() & kvc.FLAG_BAD_LEN
        assert torch.count_nonzero(out[1]) == 0
        c2 = dict(case)
        c2["context_lens"] = case["context_lens"].clone()
        c2["context_lens"][1] = 1
        ref = oracle_decode(c2, 0.1)
        for i in (0, 2):
            assert np.max(np.abs(f64(out[i]) - ref[i])) <= 2e-3


def test_checked_mode_reports_out_of_range(kvc):
    case = W.gqa_case(2, 8, 2, 128, 16, [40, 20], "bf16", seed=53)
    case["block_tables"][1, 1] = 10 ** 6
    dev = device_case(case)
    kvc.set_option(kvc.OPT_CHECKED, 1)
    out = torch.empty((2, 8, 128), device="cuda")
    with pytest.raises(kvc.KvcError) as e:
        kvc.decode_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"], 0.1,
                             out, None)
    assert e.value.status == kvc.ERR_OUT_OF_RANGE


def test_config2_gqa_full_size(kvc):
    # Llama-3-8B-shaped layer: 32/8 heads, d 128, bf16, batch 32, lengths U[512, 4096], block 16, permuted pool.
    case = W.gqa_case(32, 32, 8, 128, 16, (512, 4096), "bf16", seed=43)
    step_and_compare(kvc, case, 1.0 / math.sqrt(128), TOL["bf16"])


def test_config2_target_variant_4096(kvc):
    case = W.gqa_case(32, 32, 8, 128, 16, [4096] * 32, "bf16", seed=43)
    step_and_compare(kvc, case, 1.0 / math.sqrt(128), TOL["bf16"])
