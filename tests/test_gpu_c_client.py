"""GPU parity through the C ABI from plain C: tests/c/decode_from_c.c runs the pool, kvc_append and
kvc_decode_attention with its own cudaMalloc'd buffers and writes inputs and results; here they are checked
against the oracle (slots and tables against the pool model, the pools bit-exact, the output within 2e-3)."""

import math
import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle import paged as OP
from oracle.pool_model import PoolModel

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
# the shapes fixed in decode_from_c.c
B, HQ, HKV, D, BS, NB, MAXB = 3, 8, 2, 128, 16, 16, 4
LENS = [1, 17, 40]
T = sum(LENS)


def _bf16(raw):
    return (raw.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _load(d, name, dtype, shape):
    return np.fromfile(os.path.join(d, name), dtype=dtype).reshape(shape)


def test_whole_path_from_plain_c(kvc, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if cc is None or not os.path.exists(nvcc):
        pytest.skip("no C compiler or nvcc")
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "include")
    libdir = os.path.dirname(kvc.lib_path())
    obj, exe = str(tmp_path / "decode_from_c.o"), str(tmp_path / "decode_from_c")
    subprocess.run([cc, "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", cuda_inc, "-c", os.path.join(ROOT, "tests", "c", "decode_from_c.c"), "-o", obj],
                   check=True, capture_output=True, text=True)
    subprocess.run([nvcc, obj, "-L", libdir, "-lkvc", "-lm", "-Xlinker", "-rpath", "-Xlinker", libdir, "-o", exe],
                   check=True, capture_output=True, text=True)
    out_dir = tmp_path / "out"
    out_dir.mkdir()
    r = subprocess.run([exe, str(out_dir)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    d = str(out_dir)

    # host pool: the same slots and tables as the pool model
    model = PoolModel(NB, BS)
    want_slots = []
    for n in LENS:
        sid = model.add()
        want_slots += model.reserve(sid, n)
    slots = _load(d, "slots.bin", np.int64, (T,))
    assert slots.tolist() == want_slots
    table = _load(d, "table.bin", np.int32, (B, MAXB))
    assert table.tolist() == [model.table(i, MAXB) for i in range(B)]
    assert _load(d, "lens.bin", np.int32, (B,)).tolist() == LENS

    # append: bit-exact pools
    k_all = _bf16(_load(d, "k_all.bin", np.uint16, (T, HKV, D)))
    v_all = _bf16(_load(d, "v_all.bin", np.uint16, (T, HKV, D)))
    zeros = np.zeros((NB, HKV, BS, D))
    kc, vc = OP.append_to_paged(k_all, v_all, slots, zeros, zeros)
    assert np.array_equal(_bf16(_load(d, "k_cache.bin", np.uint16, (NB, HKV, BS, D))), kc)
    assert np.array_equal(_bf16(_load(d, "v_cache.bin", np.uint16, (NB, HKV, BS, D))), vc)

    # decode: within the bf16-input bound
    q = _bf16(_load(d, "q.bin", np.uint16, (B, HQ, D)))
    ref = OP.paged_decode(q, kc, vc, table.astype(np.int64), np.array(LENS), 1.0 / math.sqrt(D))
    out = _load(d, "out.bin", np.float32, (B, HQ, D)).astype(np.float64)
    assert np.all(np.isfinite(out))
    assert float(np.max(np.abs(out - ref))) <= 2e-3
