"""The int8 -> fp32 identity the INT8 decode relies on, checked for all 256 byte values (host only): with the
sign bit flipped, a code c becomes the byte c + 128; placed in the low mantissa byte of the float 2^23 it reads
as 2^23 + c + 128, and subtracting 2^23 + 128 (exact in fp32) leaves c."""

import numpy as np


def test_every_byte_converts_exactly():
    b = np.arange(256, dtype=np.uint32)
    flipped = b ^ 0x80
    as_float = (np.uint32(0x4B000000) | flipped).view(np.float32)
    got = as_float - np.float32(8388736.0)
    want = b.astype(np.uint8).view(np.int8).astype(np.float32)
    assert np.array_equal(got, want)
    assert np.float32(8388736.0) == 2.0 ** 23 + 128  # the constant is exact in fp32
