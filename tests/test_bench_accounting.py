"""bench.py's byte accounting on the CPU, against the cache layout (the oracle's Geometry) and the
hand count for the batch-1 32K workload: 32,636 INT2 history tokens x 8 kv heads x 96 B (K and V codes
and (scale, zero) pairs), 132 BF16 window tokens x 8 kv heads x 2 x 256 B, q BF16 and o float32."""
import os
import sys

from oracle import cache

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_decode_bytes_batch1_32k_hand_count():
    d = bench.decode_bytes(32768)
    assert d["int2"] == 32636 * 8 * 96
    assert d["window"] == 132 * 8 * 2 * 128 * 2
    assert d["q"] == 32 * 128 * 2 and d["o"] == 32 * 128 * 4
    assert abs(sum(d.values()) - 25.63e6) < 0.01e6


def test_int2_bytes_per_token_match_the_page_layout():
    for dim, p in ((128, 64), (64, 16)):
        g = cache.Geometry(1, 8, dim, p, 32, 4, 128, 1, 1)
        per_token_head = g.block_bytes // p          # K and V codes + (scale, zero) pairs of one slot
        assert bench.decode_bytes(10_000, d=dim)["int2"] == (10_000 - 132) * 8 * per_token_head


def test_window_only_context_has_no_int2_bytes():
    d = bench.decode_bytes(100)
    assert d["int2"] == 0 and d["window"] == 100 * 8 * 2 * 128 * 2


def test_extend_config_parser():
    assert bench.parse_extend_configs("4,32768,2048;8,0,4096") == ((4, 32768, 2048), (8, 0, 4096))
    assert bench.parse_extend_configs("1,8192,512") == ((1, 8192, 512),)
