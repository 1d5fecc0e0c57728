"""GPU parity: several new query tokens per sequence (kvc_decode_attention_multi) against the oracle.

Each step appends the T new tokens' K/V rows through kvc_append and then
attends them causally: token t of a sequence with n rows sees rows
0 .. n - T + t (the prefill/decode mask rule of "单请求 KV Cache").
"""

import math

import numpy as np
import pytest
import torch

from oracle import paged as OP
from paged_kv_cache_157_gb300 import workloads as W

from gpu_helpers import TOL, device_case, f64, max_err

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_options(kvc):
    for o in (kvc.OPT_BLOCKS_PER_CTA, kvc.OPT_MAX_CTAS, kvc.OPT_CHECKED):
        kvc.set_option(o, 0)
    yield
    for o in (kvc.OPT_BLOCKS_PER_CTA, kvc.OPT_MAX_CTAS, kvc.OPT_CHECKED):
        kvc.set_option(o, 0)


def new_token_slots(kvc, case):
    """Pool slots of the T newest positions of every sequence, [B * T] in (sequence, token) order."""
    T = case["n_tok"]
    lens = case["context_lens"].tolist()
    rows = [i for i in range(len(lens)) for _ in range(T)]
    pos = [n - T + t for n in lens for t in range(T)]
    return kvc.slots_from_tables(case["block_tables"], case["block_size"], rows, pos)


def append_and_reference(kvc, case, dev):
    """Appends the new rows on the device (kvc_append) and returns the oracle's caches after the same append."""
    B, T, Hkv, D = case["k_new"].shape
    slots = new_token_slots(kvc, case)
    kvc.append(dev["k_new"].reshape(B * T, Hkv, D), dev["v_new"].reshape(B * T, Hkv, D),
               torch.as_tensor(slots, dtype=torch.int64, device="cuda"), dev["k_cache"], dev["v_cache"])
    return OP.append_to_paged(f64(case["k_new"]).reshape(B * T, Hkv, D), f64(case["v_new"]).reshape(B * T, Hkv, D),
                              np.asarray(slots), f64(case["k_cache"]), f64(case["v_cache"]))


def run_multi(kvc, dev, case, scale, workspace=True, out_dtype=torch.float32):
    B, T, Hq, D = case["q"].shape
    _, Hkv, bs, _ = case["k_cache"].shape
    out = torch.full((B, T, Hq, D), float("nan"), dtype=out_dtype, device="cuda")
    ws = kvc.new_multi_workspace(B, T, Hq, Hkv, D, bs, case["block_tables"].shape[1]) if workspace else None
    kvc.decode_attention_multi(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"],
                               scale, out, ws)
    torch.cuda.synchronize()
    return out


def multi_step(kvc, case, tol, workspace=True, out_dtype=torch.float32):
    dev = device_case(case)
    kc, vc = append_and_reference(kvc, case, dev)
    scale = 1.0 / math.sqrt(case["q"].shape[-1])
    out = run_multi(kvc, dev, case, scale, workspace, out_dtype)
    ref = OP.paged_decode_multi(f64(case["q"]), kc, vc, case["block_tables"].numpy(),
                                case["context_lens"].numpy(), scale)
    if out_dtype != torch.float32:
        # the output's own rounding (half an ulp: 2^-9 relative for bf16, 2^-12 for f16) comes on top
        rel = 2.0 ** -8 if out_dtype == torch.bfloat16 else 2.0 ** -11
        excess = np.abs(f64(out) - ref) - (tol + rel * np.abs(ref))
        assert float(np.max(excess)) <= 0.0, f"T={case['n_tok']}: error above tolerance by {np.max(excess):.3e}"
    else:
        err = max_err(out, ref)
        assert err <= tol, f"T={case['n_tok']}: max abs error {err:.3e} > {tol}"
    assert torch.isfinite(out).all()
    assert kvc.get_error_flags() == 0
    return out, dev


@pytest.mark.parametrize("T", [2, 4, 8])
def test_multi_ragged_bf16(kvc, T):
    # lengths around tile (16) and block edges, the shortest equal to T
    lens = [T, T + 1, 15 + T, 16 + T, 17, 31, 32 + T, 47, 200, 129]
    lens = [max(n, T) for n in lens]
    case = W.multi_case(len(lens), T, 32, 8, 128, 16, lens, "bf16", seed=70 + T)
    multi_step(kvc, case, TOL["bf16"])


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("hq,hkv,D,T", [(8, 8, 64, 3), (16, 2, 128, 5), (8, 4, 32, 2), (16, 2, 256, 4),
                                          (4, 1, 128, 6), (32, 8, 128, 16)])
def test_multi_dtypes_and_groups(kvc, dtype, hq, hkv, D, T):
    lens = [T, 40, 77, 130]
    case = W.multi_case(len(lens), T, hq, hkv, D, 16, lens, dtype, seed=80 + T)
    multi_step(kvc, case, TOL[dtype])


@pytest.mark.parametrize("blocks_per_cta", [1, 2, 5])
@pytest.mark.parametrize("T", [4, 17])
def test_multi_forced_split_k(kvc, blocks_per_cta, T):
    # T = 17 > 16: several boundary tiles, and split parts whose blocks some tokens may not see at all
    kvc.set_option(kvc.OPT_BLOCKS_PER_CTA, blocks_per_cta)
    case = W.multi_case(5, T, 32, 8, 128, 16, [T, T + 16, 160, 333, 64], "bf16", seed=90 + blocks_per_cta)
    multi_step(kvc, case, TOL["bf16"])


def test_multi_without_workspace_and_larger_blocks(kvc):
    case = W.multi_case(4, 7, 16, 4, 128, 64, [7, 700, 64, 130], "bf16", seed=95)
    multi_step(kvc, case, TOL["bf16"], workspace=False)


@pytest.mark.parametrize("T", [64, 256])
def test_multi_chunked_prefill_lengths(kvc, T):
    # a prompt continuation of T tokens (T = 256 is the largest accepted)
    case = W.multi_case(3, T, 8, 2, 128, 16, [T, T + 100, 3 * T], "bf16", seed=96)
    multi_step(kvc, case, TOL["bf16"], out_dtype=torch.bfloat16)


def test_earlier_tokens_never_see_later_rows(kvc):
    # Changing the newest row (position n - 1) must leave tokens 0 .. T-2 bit-identical.
    T = 5
    case = W.multi_case(4, T, 32, 8, 128, 16, [5, 33, 64, 300], "bf16", seed=97)
    out, dev = multi_step(kvc, case, TOL["bf16"])
    bs = case["block_size"]
    for i, n in enumerate(case["context_lens"].tolist()):
        blk = int(case["block_tables"][i, (n - 1) // bs])
        dev["k_cache"][blk, :, (n - 1) % bs, :] = 30.0
        dev["v_cache"][blk, :, (n - 1) % bs, :] = 1000.0
    scale = 1.0 / math.sqrt(128)
    out2 = run_multi(kvc, dev, case, scale)
    assert torch.equal(out2[:, :T - 1], out[:, :T - 1])
    assert not torch.equal(out2[:, T - 1], out[:, T - 1])


def test_one_token_is_the_single_token_decode(kvc):
    case = W.multi_case(6, 1, 32, 8, 128, 16, (1, 500), "bf16", seed=98)
    out, dev = multi_step(kvc, case, TOL["bf16"])
    ref = torch.empty((6, 32, 128), dtype=torch.float32, device="cuda")
    ws = kvc.new_decode_workspace(6, 32, 8, 128, 16, case["block_tables"].shape[1])
    kvc.decode_attention(dev["q"][:, 0].contiguous(), dev["k_cache"], dev["v_cache"], dev["block_tables"],
                         dev["context_lens"], 1.0 / math.sqrt(128), ref, ws)
    torch.cuda.synchronize()
    assert torch.equal(out[:, 0], ref)


@pytest.mark.parametrize("workspace", [True, False])
def test_context_shorter_than_the_tokens_is_invalid(kvc, workspace):
    T = 4
    case = W.multi_case(3, T, 16, 4, 64, 16, [4, 40, 9], "f32", seed=99)
    case["context_lens"] = torch.tensor([4, 3, 9], dtype=torch.int32)  # sequence 1 is too short
    dev = device_case(case)
    out = run_multi(kvc, dev, case, 0.125, workspace)
    assert kvc.get_error_flags() & kvc.FLAG_BAD_LEN
    assert torch.count_nonzero(out[1]) == 0
    assert torch.isfinite(out).all()
    kvc.get_error_flags()  # clears


def test_too_many_tokens_is_rejected(kvc):
    case = W.multi_case(1, 257, 8, 8, 64, 16, [300], "bf16", seed=100)
    dev = device_case(case)
    out = torch.empty((1, 257, 8, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(kvc.KvcError) as e:
        kvc.decode_attention_multi(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                   dev["context_lens"], 0.125, out, None)
    assert e.value.status == kvc.ERR_INVALID_ARG


def test_speculative_full_size_sampled(kvc):
    # Llama-3-8B-shaped layer verifying 4 speculated tokens: batch 32, lengths 4096 (after the append)
    case = W.multi_case(32, 4, 32, 8, 128, 16, [4096] * 32, "bf16", seed=101)
    multi_step(kvc, case, TOL["bf16"])
