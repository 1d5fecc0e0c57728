"""GPU parity of the warp-MMA decode kernel over one-byte caches (e4m3 or int8 codes with per-channel K scales and
per-token V scales, bf16 queries) against the oracle's float64 attention over the dequantised pools.

The kernel converts each lane's codes straight into f16 MMA fragments, folds the K scales into the query (hi + lo
f16 parts, scaled by a power of two per segment) and the V scales into the softmax weights (scaled by a power of two
that drops when a later tile's scales are larger). These cases cover every head grouping, block size, ragged tails,
forced split-K partials, the unit mode without a workspace, scales far from the usual range, garbage in the rows
past each sequence's end, the int8 code -128 and the e4m3 extremes, and agreement with the CUDA-core kernel.
"""

import math

import numpy as np
import pytest
import torch

from oracle import paged as OP
from oracle import quant as Q
from paged_kv_cache_157_gb300 import workloads as W

from gpu_helpers import device_case, f64, max_err

pytestmark = pytest.mark.gpu

OPTS = ("OPT_BLOCKS_PER_CTA", "OPT_MAX_CTAS", "OPT_CHECKED", "OPT_GQA_ENGINE", "OPT_DYNAMIC_SHARE",
        "OPT_DYNAMIC_CHUNK")
KINDS = {
    "fp8": (W.fp8_case, Q.dequantized_pools, "decode_attention_fp8"),
    "int8": (W.int8_case, Q.dequantized_pools_int8, "decode_attention_int8"),
}
# S and the weights keep ~2^-22 relative accuracy (f16 hi + lo parts), the sums are fp32
TOL = 1e-4


@pytest.fixture(autouse=True)
def _mma_engine(kvc):
    for o in OPTS:
        kvc.set_option(getattr(kvc, o), 0)
    kvc.set_option(kvc.OPT_GQA_ENGINE, 3)
    yield
    for o in OPTS:
        kvc.set_option(getattr(kvc, o), 0)


def _decode(kvc, kind, dev, scale, workspace=True, out_dtype=torch.float32):
    B, Hq, D = dev["q"].shape
    _, Hkv, bs, _ = dev["k_cache"].shape
    out = torch.empty((B, Hq, D), dtype=out_dtype, device="cuda")
    ws = kvc.new_decode_workspace(B, Hq, Hkv, D, bs, dev["block_tables"].shape[1]) if workspace else None
    getattr(kvc, KINDS[kind][2])(dev["q"], dev["k_cache"], dev["v_cache"], dev["k_scale"], dev["v_scale"],
                                 dev["block_tables"], dev["context_lens"], scale, out, ws)
    torch.cuda.synchronize()
    return out


def _oracle(kind, case, scale):
    K, V = KINDS[kind][1](case["k_cache"].numpy(), case["v_cache"].numpy(), case["v_scale"].numpy(),
                          case["k_scale"].numpy())
    return OP.paged_decode(f64(case["q"]), K, V, case["block_tables"].numpy(), case["context_lens"].numpy(), scale)


def _check(kvc, kind, case, scale=None, tol=TOL, rel=False, **kw):
    scale = 1.0 / math.sqrt(case["q"].shape[2]) if scale is None else scale
    dev = device_case(case)
    out = _decode(kvc, kind, dev, scale, **kw)
    ref = _oracle(kind, case, scale)
    err = max_err(out, ref)
    bound = tol * max(1.0, float(np.max(np.abs(ref)))) if rel else tol
    assert err <= bound, f"max abs error {err:.3e} > {bound:.3e}"
    assert torch.isfinite(out).all()
    assert kvc.get_error_flags() == 0
    return out, dev


@pytest.mark.parametrize("kind", ["fp8", "int8"])
@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 8), (8, 1), (16, 2), (6, 2), (64, 8), (32, 2), (24, 2), (12, 4),
                                    (128, 8)])
def test_head_groupings_ragged(kvc, kind, hq, hkv):
    lens = [1, 15, 16, 17, 31, 32, 33, 47, 200, 129]
    case = KINDS[kind][0](len(lens), hq, hkv, 128, 16, lens, seed=301)
    _check(kvc, kind, case)


@pytest.mark.parametrize("kind", ["fp8", "int8"])
@pytest.mark.parametrize("bs", [16, 32, 48, 64, 128])
def test_block_sizes(kvc, kind, bs):
    case = KINDS[kind][0](5, 32, 8, 128, bs, [1, bs - 1, bs + 1, 3 * bs, 700], seed=302)
    _check(kvc, kind, case)


@pytest.mark.parametrize("kind", ["fp8", "int8"])
@pytest.mark.parametrize("blocks_per_cta", [1, 3, 7])
@pytest.mark.parametrize("hq,hkv", [(32, 8), (32, 2)])
def test_forced_split_k(kvc, kind, blocks_per_cta, hq, hkv):
    kvc.set_option(kvc.OPT_BLOCKS_PER_CTA, blocks_per_cta)
    case = KINDS[kind][0](5, hq, hkv, 128, 16, [1, 17, 160, 333, 64], seed=303)
    _check(kvc, kind, case)


@pytest.mark.parametrize("kind", ["fp8", "int8"])
def test_without_workspace(kvc, kind):
    case = KINDS[kind][0](4, 32, 8, 128, 16, [5, 700, 64, 1], seed=304)
    _check(kvc, kind, case, workspace=False)


@pytest.mark.parametrize("kind", ["fp8", "int8"])
def test_automatic_engine_choice_matches(kvc, kind):
    # 4 queries per kv head: the automatic choice takes this kernel
    kvc.set_option(kvc.OPT_GQA_ENGINE, 0)
    case = KINDS[kind][0](6, 32, 8, 128, 16, (1, 900), seed=305)
    _check(kvc, kind, case)


@pytest.mark.parametrize("kind", ["fp8", "int8"])
def test_matches_cuda_core_kernel(kvc, kind):
    case = KINDS[kind][0](6, 32, 8, 128, 16, (1, 900), seed=306)
    dev = device_case(case)
    a = _decode(kvc, kind, dev, 0.088)
    kvc.set_option(kvc.OPT_GQA_ENGINE, 1)
    b = _decode(kvc, kind, dev, 0.088)
    assert float((a - b).abs().max()) <= 2e-3


@pytest.mark.parametrize("kind", ["fp8", "int8"])
@pytest.mark.parametrize("k_mul,v_lo,v_hi,tol", [(1e3, 1e-4, 1e2, 1e-3), (1e-5, 1e-6, 1.0, 1e-4),
                                              (1.0, 1e-3, 30.0, 1e-4)])
def test_scales_far_from_the_usual_range(kvc, kind, k_mul, v_lo, v_hi, tol):
    # per-token V scales spread log-uniformly over several decades (later tiles
    # with larger scales lower the weights' factor), K scales far above or below
    # the usual amax / 448. With K scales x 1000 the scores reach ~10^3 (log2
    # units), where fp32 score sums alone carry ~10^-4 relative error.
    case = KINDS[kind][0](5, 32, 8, 128, 16, [3, 80, 400, 1000, 33], seed=307)
    g = torch.Generator().manual_seed(3070)
    case["k_scale"] = (case["k_scale"] * k_mul).float()
    u = torch.rand(case["v_scale"].shape, generator=g, dtype=torch.float64)
    case["v_scale"] = torch.exp(math.log(v_lo) + u * (math.log(v_hi) - math.log(v_lo))).float()
    _check(kvc, kind, case, scale=0.088, tol=tol, rel=True)


@pytest.mark.parametrize("kind", ["fp8", "int8"])
@pytest.mark.parametrize("bs", [16, 32])
def test_garbage_past_the_end_of_each_sequence(kvc, kind, bs):
    # rows past each sequence's end hold the e4m3 NaN code 0x7F (int8: -128)
    # and NaN / inf V scales: they must not reach the output (with 16-row
    # blocks the partial last block is often the second block of a stage)
    lens = [17, 31, 40, 1, 64, 47, 33]
    case = KINDS[kind][0](len(lens), 32, 8, 128, bs, lens, seed=308)
    bad = 0x7F if kind == "fp8" else -128
    for i, n in enumerate(lens):
        if n % bs == 0:
            continue
        blk = int(case["block_tables"][i, (n - 1) // bs])
        for c in ("k_cache", "v_cache"):
            case[c][blk, :, n % bs:, :] = bad
        case["v_scale"][blk, :, n % bs:] = float("nan")
        case["v_scale"][blk, :, -1] = float("inf")
    _check(kvc, kind, case)


def test_int8_extreme_codes(kvc):
    # every code from -128 to 127 appears in K and V
    case = W.int8_case(3, 16, 2, 128, 16, [256, 100, 255], seed=309)
    g = torch.Generator().manual_seed(3090)
    for c in ("k_cache", "v_cache"):
        case[c] = torch.randint(-128, 128, case[c].shape, generator=g, dtype=torch.int32).to(torch.int8)
    _check(kvc, "int8", case)


def test_fp8_extreme_codes(kvc):
    # the largest e4m3 magnitudes (+-448) and the subnormals (+-2^-9 .. +-7 x 2^-9) and zeros in K and V
    case = W.fp8_case(3, 16, 2, 128, 16, [256, 100, 255], seed=310)
    g = torch.Generator().manual_seed(3100)
    pick = torch.tensor([0x7E, 0xFE, 0x01, 0x81, 0x07, 0x87, 0x00, 0x80, 0x08, 0x88], dtype=torch.uint8)
    for c in ("k_cache", "v_cache"):
        idx = torch.randint(0, len(pick), case[c].shape, generator=g)
        case[c] = pick[idx]
    _check(kvc, "fp8", case, scale=0.01)


@pytest.mark.parametrize("kind", ["fp8", "int8"])
def test_zero_query_gives_scaled_mean(kvc, kind):
    lens = [40, 7]
    case = KINDS[kind][0](2, 8, 2, 128, 16, lens, seed=311)
    case["q"].zero_()
    out, _ = _check(kvc, kind, case, scale=0.3)
    _, V = KINDS[kind][1](case["k_cache"].numpy(), case["v_cache"].numpy(), case["v_scale"].numpy(),
                          case["k_scale"].numpy())
    for i, n in enumerate(lens):
        for h in range(8):
            rows = OP.gather_logical(V, case["block_tables"][i].numpy(), n, h // 4)
            assert np.max(np.abs(f64(out[i, h]) - rows.mean(axis=0))) < 1e-5


@pytest.mark.parametrize("kind", ["fp8", "int8"])
def test_bf16_output(kvc, kind):
    case = KINDS[kind][0](4, 32, 8, 128, 16, [17, 100, 3, 64], seed=312)
    dev = device_case(case)
    out = _decode(kvc, kind, dev, 0.088, out_dtype=torch.bfloat16)
    ref = _oracle(kind, case, 0.088)
    rounded = torch.from_numpy(ref).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.all(np.abs(f64(out) - rounded) <= np.maximum(np.abs(rounded) * 2.0 ** -7, 1e-4))


@pytest.mark.parametrize("kind", ["fp8", "int8"])
def test_bad_block_flag(kvc, kind):
    case = KINDS[kind][0](3, 8, 2, 128, 16, [40, 20, 5], seed=313)
    case["block_tables"][0, 1] = case["num_blocks"] + 5
    dev = device_case(case)
    _decode(kvc, kind, dev, 0.1)
    assert kvc.get_error_flags() & kvc.FLAG_BAD_BLOCK
