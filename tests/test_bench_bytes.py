"""The roofline numerator: bench.py's algorithmic bytes per step, checked against sums written out by hand for
the workloads of the measurement plan (host only)."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_gqa_batch_32_by_4096():
    # Llama-3-8B layer: 32 sequences x 4096 rows x 8 kv heads x 128 dims x 2 bytes x (K and V) = 512 MiB,
    # plus q and out (32 x 32 x 128 x 2 bytes each), 256 table entries per sequence and the 32 lengths
    dec, app = bench.step_bytes([4096] * 32, 32, 8, 128, 16, 2, 2)
    assert dec == 536_870_912 + 262_144 + 262_144 + 32 * 256 * 4 + 32 * 4
    # the append reads the new K/V rows and writes them (2 x 2 x 32 x 8 x 128 x 2 bytes) and reads 32 slots
    assert app == 4 * 32 * 8 * 128 * 2 + 32 * 8


def test_only_valid_rows_count():
    # lengths 17/31/32 with 16-row blocks: 80 rows of K/V (not the 96 slots of 6 blocks), 6 table entries
    dec, _ = bench.step_bytes([17, 31, 32], 64, 8, 128, 16, 2, 2)
    assert dec == 80 * 8 * 128 * 2 * 2 + 2 * 3 * 64 * 128 * 2 + 6 * 4 + 3 * 4


def test_shared_blocks_count_once():
    # 64 forks of 2304 rows whose first 2048 are 8 shared prompts: 8 x 2048 + 64 x 256 unique rows
    lens = [2304] * 64
    dec, _ = bench.step_bytes(lens, 32, 32, 128, 16, 2, 2, unique_kv_rows=8 * 2048 + 64 * 256)
    assert dec == 32768 * 32 * 128 * 2 * 2 + 2 * 64 * 32 * 128 * 2 + 64 * 144 * 4 + 64 * 4
    assert 32768 * 32 * 128 * 2 * 2 == 536_870_912  # the unique bytes of the sharing batch
