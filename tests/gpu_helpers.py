"""Shared helpers for the GPU parity tests: move seeded inputs to the device,
call the library through its binding, compare with the oracle."""

import math

import numpy as np
import torch

import oracle
from oracle import paged as OP

TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}


def f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def device_case(case):
    d = {}
    for k, v in case.items():
        d[k] = v.cuda() if isinstance(v, torch.Tensor) else v
    return d


def run_decode(kvc, dev, scale, out_dtype=torch.float32, workspace="auto"):
    q = dev["q"]
    B, Hq, D = q.shape
    nb, Hkv, bs, _ = dev["k_cache"].shape
    out = torch.empty((B, Hq, D), dtype=out_dtype, device="cuda")
    ws = None
    if workspace == "auto":
        ws = kvc.new_decode_workspace(B, Hq, Hkv, D, bs, dev["block_tables"].shape[1])
    elif workspace is not None:
        ws = workspace
    kvc.decode_attention(q, dev["k_cache"], dev["v_cache"], dev["block_tables"], dev["context_lens"], scale, out, ws)
    torch.cuda.synchronize()
    return out


def oracle_decode(case, scale):
    return OP.paged_decode(f64(case["q"]), f64(case["k_cache"]), f64(case["v_cache"]),
                           case["block_tables"].numpy(), case["context_lens"].numpy(), scale)


def oracle_decode_sampled(case, scale, pairs):
    """Oracle output for selected (seq, q_head) pairs, one at a time."""
    q = case["q"]
    Hq = q.shape[1]
    Hkv = case["k_cache"].shape[1]
    g = Hq // Hkv
    res = {}
    kc = case["k_cache"]
    vc = case["v_cache"]
    for (i, h) in pairs:
        n = int(case["context_lens"][i])
        kvh = h // g
        row = case["block_tables"][i].numpy()
        nblk = -(-n // kc.shape[2])
        # only the blocks this sequence uses, widened to float64 (the oracle reads them as the definition says)
        used = row[:nblk]
        sub_k = f64(kc[torch.as_tensor(used, dtype=torch.long)][:, kvh:kvh + 1])
        sub_v = f64(vc[torch.as_tensor(used, dtype=torch.long)][:, kvh:kvh + 1])
        local = np.arange(nblk)
        out, _ = OP.paged_decode_one(f64(q[i, h]), sub_k, sub_v, local, n, 0, scale)
        res[(i, h)] = out
    return res


def max_err(gpu, ref):
    return float(np.max(np.abs(f64(gpu) - ref)))


def append_new_tokens(kvc, case, dev, pool_slots):
    """Writes each sequence's new token (k_new/v_new) at its slot through kvc_append."""
    slots = torch.as_tensor(pool_slots, dtype=torch.int64, device="cuda")
    kvc.append(dev["k_new"], dev["v_new"], slots, dev["k_cache"], dev["v_cache"])


def last_position_slots(kvc, case):
    lens = case["context_lens"].tolist()
    bs = case["block_size"]
    return kvc.slots_from_tables(case["block_tables"], bs, list(range(len(lens))), [n - 1 for n in lens])


def oracle_after_append(case, slots):
    """Oracle view of the case after the append: caches with the new rows written."""
    kc, vc = OP.append_to_paged(f64(case["k_new"]), f64(case["v_new"]), slots.numpy(), f64(case["k_cache"]),
                                f64(case["v_cache"]))
    c = dict(case)
    c["k_cache_f64"], c["v_cache_f64"] = kc, vc
    return c


def default_scale(D):
    return 1.0 / math.sqrt(D)
