"""The benchmark's roofline denominator: the decode's algorithmic bytes per
call, against a count made independently from the layout (packed codes +
fp16 scale/zero per group + BF16 sink/recent windows + page-table entries)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_bytes_per_history_token_and_head():
    # 64 B of K and V codes + (128 / g) groups x 2 x 4 B of (s, z)
    assert bench.algorithmic_bytes(64, 64 + 64, 1, 128) - bench.algorithmic_bytes(0, 64, 1, 128) == 64 * 72 + 4
    assert bench.algorithmic_bytes(64, 64 + 64, 1, 32) - bench.algorithmic_bytes(0, 64, 1, 32) == 64 * 96 + 4


def test_workload_bytes():
    # one layer, 100K tokens, 8 kv heads, g128: 99,680 history tokens x 8 x 72 B
    # + 320 window tokens x 8 x 512 B + 1,558 page-table entries x 4 B
    assert bench.algorithmic_bytes(100_000 - 320, 100_000, 8, 128) == 99_680 * 8 * 72 + 320 * 8 * 512 + 1_558 * 4
    assert abs(bench.algorithmic_bytes(100_000 - 320, 100_000, 8, 128) / 1e6 - 58.73) < 0.01
    # batch 8 at 131,072 tokens: 613.1 MB; the 36-layer batch-16 g32 stack at 65,536: 29.6 GB per step
    assert abs(8 * bench.algorithmic_bytes(131_072 - 320, 131_072, 8, 128) / 1e6 - 613.1) < 0.1
    assert abs(36 * 16 * bench.algorithmic_bytes(65_536 - 320, 65_536, 8, 32) / 1e9 - 29.6) < 0.01
    # the 1,024-token single-head case: 0.215 MB
    assert abs(bench.algorithmic_bytes(704, 1024, 1, 128) / 1e6 - 0.215) < 0.001
