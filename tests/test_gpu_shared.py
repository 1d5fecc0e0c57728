"""GPU parity: decode with shared prefixes (kvc_decode_attention_shared_prefix) against the oracle's plain
paged decode, which it must equal: forks of one prompt read the shared blocks once per group."""

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
    opts = (kvc.OPT_BLOCKS_PER_CTA, kvc.OPT_MAX_CTAS, kvc.OPT_CHECKED, kvc.OPT_GQA_ENGINE)
    for o in opts:
        kvc.set_option(o, 0)
    yield
    for o in opts:
        kvc.set_option(o, 0)


def forked_case(n_prompts, fanout, prompt_len, private_len, hq, hkv, D, bs, dtype, seed):
    """Groups of `fanout` sequences sharing a `prompt_len`-row prompt (whole blocks), then private rows."""
    g = torch.Generator()
    g.manual_seed(seed)
    table, lens, nb = W.shared_prefix_block_tables(n_prompts, fanout, prompt_len, private_len, bs, g)
    B = n_prompts * fanout
    shape = (nb, hkv, bs, D)
    return {"context_lens": lens, "block_tables": table, "num_blocks": nb, "block_size": bs,
            "k_cache": W.normal(shape, dtype, g), "v_cache": W.normal(shape, dtype, g),
            "q": W.normal((B, hq, D), dtype, g), "k_new": W.normal((B, hkv, D), dtype, g),
            "v_new": W.normal((B, hkv, D), dtype, g)}


def shared_step(kvc, case, fanout, prefix, tol, append=True, out_dtype=torch.float32):
    dev = device_case(case)
    B, Hq, D = case["q"].shape
    _, Hkv, bs, _ = case["k_cache"].shape
    kc, vc = f64(case["k_cache"]), f64(case["v_cache"])
    if append:
        lens = case["context_lens"].tolist()
        slots = kvc.slots_from_tables(case["block_tables"], bs, list(range(B)), [n - 1 for n in lens])
        kvc.append(dev["k_new"], dev["v_new"], slots.cuda(), dev["k_cache"], dev["v_cache"])
        kc, vc = OP.append_to_paged(f64(case["k_new"]), f64(case["v_new"]), slots.numpy(), kc, vc)
    prefix_lens = torch.as_tensor(prefix, dtype=torch.int32).cuda()
    ws = kvc.shared_prefix_workspace(B, fanout, Hq, Hkv, D, bs, case["block_tables"].shape[1])
    out = torch.full((B, Hq, D), float("nan"), dtype=out_dtype, device="cuda")
    scale = 1.0 / math.sqrt(D)
    kvc.decode_attention_shared_prefix(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                       dev["context_lens"], fanout, prefix_lens, scale, out, ws)
    torch.cuda.synchronize()
    ref = OP.paged_decode(f64(case["q"]), kc, vc, case["block_tables"].numpy(), case["context_lens"].numpy(), scale)
    if out_dtype == torch.float32:
        err = max_err(out, ref)
        assert err <= tol, f"max abs error {err:.3e} > {tol}"
    else:
        excess = np.abs(f64(out) - ref) - (tol + 2.0 ** -8 * np.abs(ref))
        assert float(np.max(excess)) <= 0.0
    assert torch.isfinite(out).all()
    return out, dev, ws


@pytest.mark.parametrize("hq,hkv,dtype", [(8, 8, "f16"), (16, 4, "bf16"), (32, 4, "bf16"), (16, 16, "bf16")])
@pytest.mark.parametrize("fanout", [1, 4, 8])
@pytest.mark.parametrize("engine", [0, 2])
def test_shared_prefix_equals_decode(kvc, hq, hkv, dtype, fanout, engine):
    # the prefix pass has fanout x group queries per kv head: 1 to 64; engine 2 puts the 8-32 query passes on
    # the tensor-core kernel at these small sizes
    kvc.set_option(kvc.OPT_GQA_ENGINE, engine)
    case = forked_case(3, fanout, 64, 37, hq, hkv, 128, 16, dtype, seed=140 + hq + fanout)
    shared_step(kvc, case, fanout, [64] * 3, TOL[dtype])
    assert kvc.get_error_flags() == 0


def test_prefix_shorter_than_the_shared_blocks(kvc):
    # the prefix pass may cover fewer rows than the members share; the rest go through each table
    case = forked_case(2, 4, 64, 20, 16, 4, 128, 16, "bf16", seed=150)
    shared_step(kvc, case, 4, [50, 1], TOL["bf16"])
    assert kvc.get_error_flags() == 0


def test_no_private_rows(kvc):
    # every member's rows are all shared: the second pass sees no row (its log-sum-exp is -inf)
    case = forked_case(2, 4, 64, 0, 16, 4, 128, 16, "bf16", seed=151)
    shared_step(kvc, case, 4, [64, 64], TOL["bf16"], append=False)
    assert kvc.get_error_flags() == 0


@pytest.mark.parametrize("blocks_per_cta", [1, 3])
@pytest.mark.parametrize("engine", [0, 1, 2])
def test_shared_prefix_split_k_and_engines(kvc, blocks_per_cta, engine):
    kvc.set_option(kvc.OPT_BLOCKS_PER_CTA, blocks_per_cta)
    kvc.set_option(kvc.OPT_GQA_ENGINE, engine)
    case = forked_case(2, 4, 320, 90, 32, 8, 128, 16, "bf16", seed=152)
    shared_step(kvc, case, 4, [320, 320], TOL["bf16"], out_dtype=torch.bfloat16)
    assert kvc.get_error_flags() == 0


@pytest.mark.parametrize("engine", [0, 1, 3])
def test_config3_shape_sampled_against_plain_decode(kvc, engine):
    # Llama-2-7B-shaped MHA, 8 prompts of 2048 tokens forked 8 ways + 256 private tokens: equals the plain decode.
    # Each engine's first pass leaves split-K records that must not reach the second pass's counters.
    kvc.set_option(kvc.OPT_GQA_ENGINE, engine)
    case = W.shared_case(8, 8, 2048, 256, 32, 128, 16, "f16", 44, device="cuda")
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in case.items()}
    B = 64
    scale = 1.0 / math.sqrt(128)
    plain = torch.empty((B, 32, 128), dtype=torch.float32, device="cuda")
    kvc.decode_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"], scale,
                         plain, kvc.new_decode_workspace(B, 32, 32, 128, 16, case["block_tables"].shape[1]))
    ws = kvc.shared_prefix_workspace(B, 8, 32, 32, 128, 16, case["block_tables"].shape[1])
    out = torch.empty_like(plain)
    kvc.decode_attention_shared_prefix(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                       dev["context_lens"], 8, torch.full((8,), 2048, dtype=torch.int32).cuda(),
                                       scale, out, ws)
    torch.cuda.synchronize()
    assert float((out - plain).abs().max()) <= 2e-3
    assert kvc.get_error_flags() == 0


def test_bad_arguments(kvc):
    case = forked_case(2, 4, 32, 5, 8, 8, 64, 16, "bf16", seed=153)
    dev = device_case(case)
    out = torch.empty((8, 8, 64), dtype=torch.float32, device="cuda")
    ws = kvc.shared_prefix_workspace(8, 4, 8, 8, 64, 16, case["block_tables"].shape[1])
    with pytest.raises(kvc.KvcError) as e:  # 8 sequences are not groups of 3
        _call_raw(kvc, dev, 3, out, ws)
    assert e.value.status == kvc.ERR_INVALID_ARG
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvc.KvcError) as e:
        kvc.decode_attention_shared_prefix(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                           dev["context_lens"], 4, torch.full((2,), 32, dtype=torch.int32).cuda(),
                                           0.1, out, small)
    assert e.value.status == kvc.ERR_WORKSPACE


def _call_raw(kvc, dev, group_size, out, ws):
    # a group size that does not divide the batch, past the binding's own shape check
    import ctypes
    pl = torch.full((3,), 32, dtype=torch.int32).cuda()
    st = kvc.raw().kvc_decode_attention_shared_prefix(
        ctypes.c_void_p(dev["q"].data_ptr()), ctypes.c_void_p(dev["k_cache"].data_ptr()),
        ctypes.c_void_p(dev["v_cache"].data_ptr()), ctypes.c_void_p(dev["block_tables"].data_ptr()),
        dev["block_tables"].shape[1], ctypes.c_void_p(dev["context_lens"].data_ptr()), 8, group_size,
        ctypes.c_void_p(pl.data_ptr()), 0.1, 8, 8, 64, 16, dev["k_cache"].shape[0], kvc.BF16,
        ctypes.c_void_p(out.data_ptr()), kvc.F32, ctypes.c_void_p(ws.data_ptr()), ws.numel(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if st != 0:
        raise kvc.KvcError(st, "kvc_decode_attention_shared_prefix", "")


def test_prefix_longer_than_a_member_is_flagged(kvc):
    case = forked_case(1, 4, 32, 5, 8, 8, 64, 16, "bf16", seed=154)
    dev = device_case(case)
    out = torch.empty((4, 8, 64), dtype=torch.float32, device="cuda")
    ws = kvc.shared_prefix_workspace(4, 4, 8, 8, 64, 16, case["block_tables"].shape[1])
    kvc.decode_attention_shared_prefix(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                       dev["context_lens"], 4, torch.full((1,), 100, dtype=torch.int32).cuda(),
                                       0.1, out, ws)
    assert kvc.get_error_flags() & kvc.FLAG_BAD_LEN


def test_config3_full_size_sampled_against_oracle(kvc):
    # 8 prompts x 2048 tokens forked 8 ways + 256 private tokens, 32 heads x 128, fp16: both the plain decode and
    # the shared-prefix decode against the oracle on sampled (sequence, head) pairs
    from gpu_helpers import oracle_decode_sampled
    case = W.shared_case(8, 8, 2048, 256, 32, 128, 16, "f16", 44)
    dev = device_case(case)
    B = 64
    scale = 1.0 / math.sqrt(128)
    plain = torch.empty((B, 32, 128), dtype=torch.float32, device="cuda")
    kvc.decode_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"], scale,
                         plain, kvc.new_decode_workspace(B, 32, 32, 128, 16, case["block_tables"].shape[1]))
    shared = torch.empty_like(plain)
    ws = kvc.shared_prefix_workspace(B, 8, 32, 32, 128, 16, case["block_tables"].shape[1])
    kvc.decode_attention_shared_prefix(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"],
                                       dev["context_lens"], 8, torch.full((8,), 2048, dtype=torch.int32).cuda(),
                                       scale, shared, ws)
    torch.cuda.synchronize()
    pairs = [(0, 0), (7, 31), (8, 5), (33, 17), (63, 30)]
    ref = oracle_decode_sampled(case, scale, pairs)
    for (i, h), r in ref.items():
        assert float(np.max(np.abs(f64(plain[i, h]) - r))) <= TOL["f16"], ("plain", i, h)
        assert float(np.max(np.abs(f64(shared[i, h]) - r))) <= TOL["f16"], ("shared", i, h)
    assert kvc.get_error_flags() == 0
