"""The C ABI library loads and exports every symbol include/kvc.h declares (no GPU needed)."""

import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "kvc.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc_[a-z0-9_]+)\s*\(", text)))


def test_header_declarations_match_binding(kvc):
    assert declared_functions() == kvc.symbols()


def test_library_exports_every_declared_symbol(kvc):
    out = subprocess.run(["nm", "-D", "--defined-only", kvc.lib_path()], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\b(kvc_[a-z0-9_]+)\b", out.stdout))
    missing = [s for s in declared_functions() if s not in exported]
    assert not missing, missing
    lib = kvc.raw()
    for s in declared_functions():
        assert getattr(lib, s) is not None


def test_status_strings_and_version(kvc):
    lib = kvc.raw()
    assert lib.kvc_abi_version() == 1
    assert lib.kvc_status_string(0) == b"KVC_OK"
    assert lib.kvc_status_string(3) == b"KVC_ERR_NO_BLOCKS"
    assert lib.kvc_status_string(99) == b"KVC_ERR_UNKNOWN"


def test_options_roundtrip(kvc):
    kvc.set_option(kvc.OPT_BLOCKS_PER_CTA, 7)
    assert kvc.get_option(kvc.OPT_BLOCKS_PER_CTA) == 7
    kvc.set_option(kvc.OPT_BLOCKS_PER_CTA, 0)
    with pytest.raises(kvc.KvcError):
        kvc.set_option(kvc.OPT_CHECKED, 2)
    with pytest.raises(kvc.KvcError):
        kvc.set_option(9, 1)
    lib = kvc.raw()
    assert lib.kvc_set_checked(1) == kvc.OK and kvc.get_option(kvc.OPT_CHECKED) == 1
    assert lib.kvc_set_checked(0) == kvc.OK and kvc.get_option(kvc.OPT_CHECKED) == 0
    for o, v in ((kvc.OPT_DYNAMIC_SHARE, 256), (kvc.OPT_DYNAMIC_CHUNK, 3), (kvc.OPT_WAIT_POLLS, 5)):
        kvc.set_option(o, v)
        assert kvc.get_option(o) == v
        kvc.set_option(o, 0)
    with pytest.raises(kvc.KvcError):
        kvc.set_option(kvc.OPT_DYNAMIC_SHARE, 257)
    for e in (1, 2, 3, 0):
        kvc.set_option(kvc.OPT_GQA_ENGINE, e)
        assert kvc.get_option(kvc.OPT_GQA_ENGINE) == e
    with pytest.raises(kvc.KvcError):
        kvc.set_option(kvc.OPT_GQA_ENGINE, 4)


def test_host_validation_before_any_device_work(kvc):
    import ctypes
    lib = kvc.raw()
    z = ctypes.c_void_p(0)
    # n_q_heads not a multiple of n_kv_heads
    s = lib.kvc_decode_attention(z, z, z, z, 4, z, 2, 0.1, 6, 4, 128, 16, 10, 2, z, 0, z, 0, z)
    assert s == kvc.ERR_INVALID_ARG
    assert b"multiple" in lib.kvc_last_error_message()
    # unsupported head_dim
    assert lib.kvc_decode_attention(z, z, z, z, 4, z, 2, 0.1, 8, 4, 96, 16, 10, 2, z, 0, z, 0, z) == kvc.ERR_UNSUPPORTED
    # block size not a multiple of 16
    assert lib.kvc_decode_attention(z, z, z, z, 4, z, 2, 0.1, 8, 4, 128, 8, 10, 2, z, 0, z, 0, z) == kvc.ERR_UNSUPPORTED
    # empty batch
    assert lib.kvc_decode_attention(z, z, z, z, 4, z, 0, 0.1, 8, 4, 128, 16, 10, 2, z, 0, z, 0, z) == kvc.ERR_INVALID_ARG
    # append of zero tokens is a no-op that succeeds without touching the device
    assert lib.kvc_append(z, z, z, 0, z, z, 10, 16, 8, 128, 2, z) == kvc.OK
    # bad dtype
    assert lib.kvc_append(z, z, z, 1, z, z, 10, 16, 8, 128, 7, z) == kvc.ERR_INVALID_ARG
    # workspace query validates shapes too
    n = ctypes.c_size_t()
    assert lib.kvc_decode_workspace_size(2, 6, 4, 128, 16, 4, ctypes.byref(n)) == kvc.ERR_INVALID_ARG


def test_one_byte_cache_entries_validate_on_the_host(kvc):
    import ctypes
    lib = kvc.raw()
    z = ctypes.c_void_p(0)
    p16 = ctypes.c_void_p(0x1000)  # never dereferenced: every call below fails before any device work
    for name in ("kvc_decode_attention_fp8", "kvc_decode_attention_int8"):
        fn = getattr(lib, name)
        # NULL scales
        assert fn(z, z, z, z, z, z, 4, z, 2, 0.1, 8, 4, 128, 16, 10, z, 0, z, 0, z) == kvc.ERR_INVALID_ARG
        # head_dim 32 is not instantiated for one-byte caches
        assert fn(z, z, z, p16, p16, z, 4, z, 2, 0.1, 8, 4, 32, 16, 10, z, 0, z, 0, z) == kvc.ERR_UNSUPPORTED
        # unaligned scales
        odd = ctypes.c_void_p(0x1004)
        assert fn(z, z, z, odd, p16, z, 4, z, 2, 0.1, 8, 4, 128, 16, 10, z, 0, z, 0, z) == kvc.ERR_INVALID_ARG
    for name in ("kvc_append_fp8", "kvc_append_int8"):
        fn = getattr(lib, name)
        # zero tokens: a no-op; a bad dtype or an odd head_dim: invalid
        assert fn(z, z, z, 0, z, z, z, z, 10, 16, 8, 128, 2, z) == kvc.OK
        assert fn(z, z, z, 1, z, z, z, z, 10, 16, 8, 128, 7, z) == kvc.ERR_INVALID_ARG
        assert fn(z, z, z, 1, z, z, z, z, 10, 16, 8, 127, 2, z) == kvc.ERR_INVALID_ARG
        # NULL scale pointers with tokens to write
        assert fn(p16, p16, p16, 1, p16, p16, z, z, 10, 16, 8, 128, 2, z) == kvc.ERR_INVALID_ARG
