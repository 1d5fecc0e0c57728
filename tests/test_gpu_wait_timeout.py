"""GPU: the decode kernels' bounded waits give up cleanly (KVC_OPT_WAIT_POLLS test hook).

No fault is made on the device: the hook only makes a wait for copied data
give up after one poll, long before the data lands, so the kernel runs its
abort path (flag KVC_FLAG_TIMEOUT, every warp stops, the CTA waits with the
normal bound for its own copies still in flight). The GPU stays usable: the
next call, on a freshly zeroed workspace, must match the oracle bit for bit
in its flags and within tolerance in its output.
"""

import math

import pytest
import torch

from paged_kv_cache_157_gb300 import workloads as W

from gpu_helpers import TOL, device_case, max_err, oracle_decode, run_decode

pytestmark = pytest.mark.gpu

OPTS = ("OPT_BLOCKS_PER_CTA", "OPT_MAX_CTAS", "OPT_CHECKED", "OPT_GQA_ENGINE", "OPT_DYNAMIC_SHARE",
        "OPT_DYNAMIC_CHUNK", "OPT_WAIT_POLLS")


@pytest.fixture(autouse=True)
def _reset_options(kvc):
    for o in OPTS:
        kvc.set_option(getattr(kvc, o), 0)
    yield
    for o in OPTS:
        kvc.set_option(getattr(kvc, o), 0)


@pytest.mark.parametrize("engine,hq", [(1, 32), (3, 32), (1, 8), (3, 64)])
@pytest.mark.parametrize("workspace", ["auto", None])
def test_wait_that_gives_up_sets_timeout_then_next_call_is_right(kvc, engine, hq, workspace):
    kvc.set_option(kvc.OPT_GQA_ENGINE, engine)
    scale = 1.0 / math.sqrt(128)
    case = W.gqa_case(8, hq, 8, 128, 16, [3000, 17, 1, 640, 2048, 96, 4000, 333], "bf16", seed=131)
    dev = device_case(case)
    ref = oracle_decode(case, scale)
    assert kvc.get_error_flags() == 0
    kvc.set_option(kvc.OPT_WAIT_POLLS, 1)
    run_decode(kvc, dev, scale, workspace=workspace)
    assert kvc.get_error_flags() & kvc.FLAG_TIMEOUT
    kvc.set_option(kvc.OPT_WAIT_POLLS, 0)
    out = run_decode(kvc, dev, scale, workspace=workspace)  # a new zero-filled workspace
    assert max_err(out, ref) <= TOL["bf16"]
    assert kvc.get_error_flags() == 0
