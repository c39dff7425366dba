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


def _fake_smi(tmp_path, mhz, reason_col=""):
    """An nvidia-smi stand-in that prints one timestamped sample line every 20 ms until killed."""
    script = tmp_path / "nvidia-smi"
    script.write_text(
        "#!/usr/bin/env python3\n"
        "import sys, time\n"
        "while True:\n"
        "    t = time.time()\n"
        "    stamp = time.strftime('%Y/%m/%d %H:%M:%S', time.localtime(t)) + '.%03d' % int((t % 1) * 1000)\n"
        f"    print(stamp + ', 0, {mhz}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, {reason_col or 'Not Active'}',"
        " flush=True)\n"
        "    time.sleep(0.02)\n")
    script.chmod(0o755)
    return str(tmp_path)


def test_clock_sampler_counts_samples_inside_the_timed_window(tmp_path, monkeypatch):
    import time
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, 1980, "Active") + os.pathsep + os.environ["PATH"])
    c = bench.ClockSampler(0)
    c.start()
    time.sleep(0.2)
    c.mark_start()
    time.sleep(0.6)
    c.mark_end()
    time.sleep(0.2)
    rec = c.stop()
    # the stand-in prints every 20 ms; the sampler's own period does not apply to it
    assert rec["samples"] >= 10 and rec["sm_mhz"] == 1980 and rec["sm_max_mhz"] == 2070
    assert rec["reasons"] == ["sw_power_cap"]
    assert 0.55 < rec["window_s"] < 0.9
    assert "phase" not in rec


def test_clock_sampler_short_window_reports_the_phase(tmp_path, monkeypatch):
    import time
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, 2070) + os.pathsep + os.environ["PATH"])
    c = bench.ClockSampler(0)
    c.start()
    time.sleep(0.3)
    c.mark_start()
    c.mark_end()          # a window with no sample in it
    time.sleep(0.3)
    rec = c.stop()
    assert rec["samples"] == 0
    assert rec["phase"]["samples"] >= 10 and rec["sm_mhz"] == 2070 and rec["reasons"] == []


def test_clock_sampler_without_nvidia_smi(monkeypatch, tmp_path):
    monkeypatch.setenv("PATH", str(tmp_path))
    c = bench.ClockSampler(0)
    c.start()
    c.mark_start()
    c.mark_end()
    rec = c.stop()
    assert rec["samples"] == 0 and rec["reasons"] == ["nvidia-smi unavailable"]
