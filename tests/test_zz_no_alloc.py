"""GPU: kvc_decode_attention_static, the decode entry point that allocates nothing.

It exists for callers that cannot allocate device memory on the decode path
(a plugin handed only its buffers, a fixed memory budget, plain C without an
allocator). It must give the same results as kvc_decode_attention with a
caller-provided workspace, on consecutive calls (the built-in scratch keeps
the previous call's contents). This file is named to run after every other
test file.
"""

import ctypes
import math

import numpy as np
import pytest
import torch

from paged_kv_cache_157_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _c_abi_static(kvc, dev, scale, out):
    lib = kvc.raw()
    B, hq, d = dev["q"].shape
    nb, hkv, bs, _ = dev["k_cache"].shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.kvc_decode_attention_static(p(dev["q"]), p(dev["k_cache"]), p(dev["v_cache"]), p(dev["block_tables"]),
                                           dev["block_tables"].shape[1], p(dev["context_lens"]), B, scale, hq, hkv,
                                           d, bs, nb, kvc.BF16, p(out), kvc.F32, stream)


def _reference(kvc, dev, scale):
    B, hq, d = dev["q"].shape
    _, hkv, bs, _ = dev["k_cache"].shape
    ws = kvc.new_decode_workspace(B, hq, hkv, d, bs, dev["block_tables"].shape[1])
    out = torch.empty((B, hq, d), device="cuda")
    kvc.decode_attention(dev["q"], dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"], scale,
                         out, ws)
    return out


def test_static_scratch_matches_workspace_path_twice(kvc):
    for o in (kvc.OPT_BLOCKS_PER_CTA, kvc.OPT_MAX_CTAS, kvc.OPT_CHECKED, kvc.OPT_DYNAMIC_SHARE,
              kvc.OPT_DYNAMIC_CHUNK):
        kvc.set_option(o, 0)
    scale = 1.0 / math.sqrt(128)
    cases = [W.gqa_case(32, 32, 8, 128, 16, (512, 4096), "bf16", seed=43),
             W.gqa_case(5, 32, 8, 128, 16, [1, 17, 300, 2000, 64], "bf16", seed=44)]
    for case in cases:  # two calls in a row, different shapes, same scratch
        dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in case.items()}
        ref = _reference(kvc, dev, scale)
        out = torch.full_like(ref, float("nan"))
        assert _c_abi_static(kvc, dev, scale, out) == kvc.OK, kvc.raw().kvc_last_error_message()
        torch.cuda.synchronize()
        err = float((out - ref).abs().max())
        assert err <= 2e-3, err
        assert kvc.get_error_flags() == 0


def test_static_scratch_on_the_tensor_core_engine(kvc):
    # 64 query / 8 kv heads: 8 queries per kv head, which the tensor-core
    # kernel takes (forced here at any size); its counters and records sit in
    # the same built-in array in a different layout.
    for o in (kvc.OPT_BLOCKS_PER_CTA, kvc.OPT_MAX_CTAS, kvc.OPT_CHECKED, kvc.OPT_DYNAMIC_SHARE,
              kvc.OPT_DYNAMIC_CHUNK):
        kvc.set_option(o, 0)
    kvc.set_option(kvc.OPT_GQA_ENGINE, 2)
    try:
        scale = 1.0 / math.sqrt(128)
        cases = [W.gqa_case(8, 64, 8, 128, 16, [4096, 3000, 1, 17, 2500, 4096, 640, 1024], "bf16", seed=47),
                 W.gqa_case(4, 64, 8, 128, 16, (512, 4096), "bf16", seed=48)]
        for case in cases:
            dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in case.items()}
            ref = _reference(kvc, dev, scale)
            for _ in range(2):
                out = torch.full_like(ref, float("nan"))
                assert _c_abi_static(kvc, dev, scale, out) == kvc.OK, kvc.raw().kvc_last_error_message()
                torch.cuda.synchronize()
                err = float((out - ref).abs().max())
                assert err <= 2e-3, err
            assert kvc.get_error_flags() == 0
    finally:
        kvc.set_option(kvc.OPT_GQA_ENGINE, 0)


def test_static_scratch_after_a_call_with_a_bad_block_id(kvc):
    # A call that meets an out-of-pool block id flags it (and leaves its output
    # undefined); the next call with valid inputs must match the workspace path.
    for o in (kvc.OPT_BLOCKS_PER_CTA, kvc.OPT_MAX_CTAS, kvc.OPT_CHECKED, kvc.OPT_GQA_ENGINE,
              kvc.OPT_DYNAMIC_SHARE, kvc.OPT_DYNAMIC_CHUNK):
        kvc.set_option(o, 0)
    scale = 1.0 / math.sqrt(128)
    case = W.gqa_case(6, 32, 8, 128, 16, [3000, 40, 1, 4096, 777, 2048], "bf16", seed=49)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in case.items()}
    ref = _reference(kvc, dev, scale)
    torch.cuda.synchronize()
    assert kvc.get_error_flags() == 0
    bad = dict(dev)
    bad["block_tables"] = dev["block_tables"].clone()
    bad["block_tables"][3, 10] = case["num_blocks"] + 5  # outside the pool
    out = torch.empty_like(ref)
    assert _c_abi_static(kvc, bad, scale, out) == kvc.OK
    assert kvc.get_error_flags() & kvc.FLAG_BAD_BLOCK
    out = torch.full_like(ref, float("nan"))
    assert _c_abi_static(kvc, dev, scale, out) == kvc.OK
    torch.cuda.synchronize()
    assert float((out - ref).abs().max()) <= 2e-3
    assert kvc.get_error_flags() == 0


def test_static_scratch_after_a_call_that_gave_up_waiting(kvc):
    # A call whose waits give up (the KVC_OPT_WAIT_POLLS test hook) leaves the
    # counters in the built-in scratch non-zero; the next call clears them
    # itself and must match the workspace path.
    for o in (kvc.OPT_BLOCKS_PER_CTA, kvc.OPT_MAX_CTAS, kvc.OPT_CHECKED, kvc.OPT_GQA_ENGINE,
              kvc.OPT_DYNAMIC_SHARE, kvc.OPT_DYNAMIC_CHUNK, kvc.OPT_WAIT_POLLS):
        kvc.set_option(o, 0)
    scale = 1.0 / math.sqrt(128)
    case = W.gqa_case(6, 32, 8, 128, 16, [3000, 40, 1, 4096, 777, 2048], "bf16", seed=50)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in case.items()}
    ref = _reference(kvc, dev, scale)
    torch.cuda.synchronize()
    assert kvc.get_error_flags() == 0
    out = torch.empty_like(ref)
    kvc.set_option(kvc.OPT_WAIT_POLLS, 1)
    try:
        assert _c_abi_static(kvc, dev, scale, out) == kvc.OK
        assert kvc.get_error_flags() & kvc.FLAG_TIMEOUT
    finally:
        kvc.set_option(kvc.OPT_WAIT_POLLS, 0)
    out = torch.full_like(ref, float("nan"))
    assert _c_abi_static(kvc, dev, scale, out) == kvc.OK
    torch.cuda.synchronize()
    assert float((out - ref).abs().max()) <= 2e-3
    assert kvc.get_error_flags() == 0


def test_static_scratch_refuses_oversized_shapes(kvc):
    kvc.set_option(kvc.OPT_BLOCKS_PER_CTA, 1)  # one cache block per CTA: far more records than 16 MiB hold
    try:
        case = W.gqa_case(8, 32, 8, 128, 16, [4096] * 8, "bf16", seed=45)
        dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in case.items()}
        out = torch.empty((8, 32, 128), device="cuda")
        status = _c_abi_static(kvc, dev, 0.1, out)
        assert status == kvc.ERR_WORKSPACE
        assert b"built-in scratch" in kvc.raw().kvc_last_error_message()
    finally:
        kvc.set_option(kvc.OPT_BLOCKS_PER_CTA, 0)
