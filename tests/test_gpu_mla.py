"""GPU parity: MLA absorbed decode (kvc_append_latent + kvc_decode_attention_mla) against the oracle."""

import numpy as np
import pytest
import torch

from oracle import mla as OM
from oracle import paged as OP
from paged_kv_cache_157_gb300 import workloads as W

from gpu_helpers import f64

pytestmark = pytest.mark.gpu

D_C, D_R, H = 512, 64, 128
SCALE = 1.0 / 24.0
TOL = 2e-3


@pytest.fixture(autouse=True)
def _reset_options(kvc):
    for o in (kvc.OPT_BLOCKS_PER_CTA, kvc.OPT_MAX_CTAS, kvc.OPT_CHECKED):
        kvc.set_option(o, 0)
    yield
    for o in (kvc.OPT_BLOCKS_PER_CTA, kvc.OPT_MAX_CTAS, kvc.OPT_CHECKED):
        kvc.set_option(o, 0)


def run_mla(kvc, case, out_dtype=torch.float32, workspace="auto", append=True):
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in case.items()}
    B = case["q"].shape[0]
    bs = case["block_size"]
    lens = case["context_lens"].tolist()
    slots = kvc.slots_from_tables(case["block_tables"], bs, list(range(B)), [n - 1 for n in lens])
    if append:
        kvc.append_latent(dev["c_new"], slots.cuda(), dev["latent_cache"], D_C)
    out = torch.empty((B, H, D_C), dtype=out_dtype, device="cuda")
    ws = None
    if workspace == "auto":
        n = kvc.decode_mla_workspace_size(B, H, D_C, D_R, bs, case["block_tables"].shape[1])
        ws = torch.zeros(max(1, n), dtype=torch.uint8, device="cuda")
    kvc.decode_attention_mla(dev["q"], dev["latent_cache"], dev["block_tables"], dev["context_lens"], SCALE, D_C,
                             out, ws)
    torch.cuda.synchronize()
    return out, slots


def oracle_mla(case, slots, append=True, pairs=None):
    if pairs is not None:
        return oracle_mla_sampled(case, pairs)
    lat = f64(case["latent_cache"])
    if append:
        c = f64(case["c_new"])
        lat2, _ = OP.append_to_paged(c[:, None, :], c[:, None, :], slots.numpy(), lat[:, None], lat[:, None])
        lat = lat2[:, 0]
    q = f64(case["q"])
    out, _ = OM.mla_absorbed_decode(q, lat, case["block_tables"].numpy(), case["context_lens"].numpy(), SCALE, D_C)
    return out


def oracle_mla_sampled(case, pairs):
    """Selected (sequence, head) outputs: the sequence's own blocks are copied out in table order, the new
    row is appended at its last position through the oracle, then the oracle attends."""
    bs = case["block_size"]
    res = {}
    for (i, h) in pairs:
        n = int(case["context_lens"][i])
        nblk = -(-n // bs)
        used = case["block_tables"][i, :nblk].long()
        lat = f64(case["latent_cache"][used])
        c = f64(case["c_new"][i:i + 1])
        lat2, _ = OP.append_to_paged(c[:, None, :], c[:, None, :], np.array([n - 1]), lat[:, None], lat[:, None])
        res[(i, h)], _ = OM.mla_absorbed_one(f64(case["q"][i, h]), lat2[:, 0], np.arange(nblk), n, SCALE, D_C)
    return res


@pytest.mark.parametrize("lens", [[1], [1, 33, 100], [64, 65, 31, 32, 200, 129]])
def test_mla_small(kvc, lens):
    case = W.mla_case(len(lens), H, D_C, D_R, 64, lens, "bf16", seed=46)
    out, slots = run_mla(kvc, case)
    ref = oracle_mla(case, slots)
    err = float(np.max(np.abs(f64(out) - ref)))
    assert err <= TOL, err
    assert kvc.get_error_flags() == 0


@pytest.mark.parametrize("bs", [16, 32, 64, 256])
def test_mla_tiles_across_block_boundaries(kvc, bs):
    # 48-token tiles straddle cache blocks: lengths around tile and block edges, several block sizes
    lens = [47, 48, 49, 95, 96, 97, 63, 64, 65, 127, 128, 129, 500]
    case = W.mla_case(len(lens), H, D_C, D_R, bs, lens, "bf16", seed=51)
    out, slots = run_mla(kvc, case)
    ref = oracle_mla(case, slots)
    err = float(np.max(np.abs(f64(out) - ref)))
    assert err <= TOL, err
    assert kvc.get_error_flags() == 0


@pytest.mark.parametrize("blocks_per_cta", [1, 2, 5])
def test_mla_forced_split(kvc, blocks_per_cta):
    kvc.set_option(kvc.OPT_BLOCKS_PER_CTA, blocks_per_cta)
    lens = [700, 64, 1, 333]
    case = W.mla_case(len(lens), H, D_C, D_R, 64, lens, "bf16", seed=47)
    out, slots = run_mla(kvc, case)
    ref = oracle_mla(case, slots)
    err = float(np.max(np.abs(f64(out) - ref)))
    assert err <= TOL, err
    assert kvc.get_error_flags() == 0


def test_mla_merge_of_more_than_64_records(kvc):
    # one block per CTA pair: the 6400-row sequence is cut into ~100 parts, so the merging warpgroup lists the
    # record slots in several chunks; bf16 output takes the vector stores of the merge
    kvc.set_option(kvc.OPT_BLOCKS_PER_CTA, 1)
    lens = [6400, 300]
    case = W.mla_case(len(lens), H, D_C, D_R, 64, lens, "bf16", seed=49)
    out, slots = run_mla(kvc, case)
    ref = oracle_mla(case, slots)
    err = float(np.max(np.abs(f64(out) - ref)))
    assert err <= TOL, err
    assert kvc.get_error_flags() == 0
    out16, _ = run_mla(kvc, case, out_dtype=torch.bfloat16)  # a fresh device copy, the same append
    # bf16 rounding of the same result
    excess = np.abs(f64(out16) - ref) - (TOL + 2.0 ** -8 * np.abs(ref))
    assert float(np.max(excess)) <= 0.0
    assert kvc.get_error_flags() == 0


def test_mla_nan_in_unused_rows_of_the_last_block(kvc):
    # the rows of a sequence's last block past its length may hold anything; NaN there must not reach the output
    lens = [1, 33, 100, 64, 65]
    case = W.mla_case(len(lens), H, D_C, D_R, 64, lens, "bf16", seed=50)
    bs = case["block_size"]
    for i, n in enumerate(lens):
        blk = int(case["block_tables"][i, (n - 1) // bs])
        case["latent_cache"][blk, n % bs if n % bs else bs:, :] = float("nan")
    out, slots = run_mla(kvc, case)
    ref = oracle_mla(case, slots)
    assert torch.isfinite(out).all()
    err = float(np.max(np.abs(f64(out) - ref)))
    assert err <= TOL, err
    assert kvc.get_error_flags() == 0


def test_mla_without_workspace(kvc):
    lens = [300, 5, 129]
    case = W.mla_case(len(lens), H, D_C, D_R, 64, lens, "bf16", seed=48)
    out, slots = run_mla(kvc, case, workspace=None)
    ref = oracle_mla(case, slots)
    assert float(np.max(np.abs(f64(out) - ref))) <= TOL
    assert kvc.get_error_flags() == 0


def test_mla_bf16_out_and_block_128(kvc):
    lens = [257, 90]
    case = W.mla_case(len(lens), H, D_C, D_R, 128, lens, "bf16", seed=49)
    out, slots = run_mla(kvc, case, out_dtype=torch.bfloat16)
    ref = oracle_mla(case, slots)
    rounded = torch.from_numpy(ref).to(torch.bfloat16).to(torch.float64).numpy()
    err = np.abs(f64(out) - rounded)
    assert np.all(err <= np.maximum(np.abs(rounded) * 2.0 ** -7, TOL))


def test_mla_config5_full_size_sampled(kvc):
    # DeepSeek-V2 shape: 128 heads, d_c 512 + d_R 64, bf16, batch 64, lengths U[1024, 8192], block 64.
    case = W.mla_case(64, H, D_C, D_R, 64, (1024, 8192), "bf16", seed=46)
    out, slots = run_mla(kvc, case)
    rng = np.random.default_rng(0)
    pairs = [(int(i), int(h)) for i, h in zip(rng.integers(0, 64, 12), rng.integers(0, H, 12))]
    pairs += [(0, 0), (63, 127)]
    ref = oracle_mla(case, slots, pairs=pairs)
    got = f64(out)
    err = max(float(np.max(np.abs(got[i, h] - ref[(i, h)]))) for (i, h) in pairs)
    assert err <= TOL, err
    assert torch.isfinite(out).all()
    assert kvc.get_error_flags() == 0
