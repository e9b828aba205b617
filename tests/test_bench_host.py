"""Host-side arithmetic of bench.py: the byte and flop counts its roofline figures divide by."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _mm(m, n, k):
    return 2 * m * n * k


def test_prefill_mma_flops_counts_blocks_and_products():
    # chunks of 300, 256 and 1 tokens: 3 + 2 + 1 blocks of at most 128 tokens
    cu = np.array([0, 300, 556, 557], np.int32)
    H, P, N = 3, 64, 128
    # per block and head: S = C B^T, Y1 = P X, Y2 = C Hprev^T, dS = B^T (w x), as (m, n, k)
    per = _mm(128, 128, N) + _mm(128, P, 128) + _mm(128, P, N) + _mm(N, P, 128)
    assert bench.prefill_mma_flops(cu, H, P, N) == 6 * H * per
    assert per == 10_485_760


def test_prefill_mma_flops_long_batch():
    # 8 sequences of 65536 tokens in 256-token chunks: 4096 blocks of 128 tokens per head
    cu = np.arange(0, 8 * 65536 + 1, 256, dtype=np.int32)
    assert bench.prefill_mma_flops(cu, 128, 64, 128) == 4096 * 128 * 10_485_760


def test_prefill_and_decode_bytes_by_hand():
    # one token, one chunk, every size 1, 2-byte elements: x, y (2 + 2), dt (2), B, C (2 + 2),
    # one fp32 state store (4)
    assert bench.prefill_bytes(1, 1, 1, 1, 1, 1, 2) == 14
    # plus one initial-state load
    assert bench.prefill_bytes(1, 1, 1, 1, 1, 1, 2, init_reads=1) == 18
    # one live request, one token, one column written: a state load and a store (8) and the
    # token's tensors (10)
    assert bench.decode_bytes(1, 1, 1, 1, 1, 1, 1, 2) == 18
    # the fused kernel's share: all but dt (2), which the prep kernel reads
    assert bench.fused_bytes(1, 1, 1, 1, 1, 1, 2) == 12
    # the long batch: 524,288 tokens, 2048 chunks, H=128: 28.05 GB for the call, 0.13 GB of it dt
    call = bench.prefill_bytes(524288, 2048, 128, 64, 128, 8, 2)
    assert call == 28051505152 and call - bench.fused_bytes(524288, 2048, 128, 64, 128, 8, 2) == 524288 * 128 * 2


def test_peaks_come_from_the_measured_file_when_present():
    path = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    hbm, kind = bench._peaks()
    bf16, bkind = bench._bf16_peak()
    if os.path.exists(path):
        import json
        m = json.load(open(path))
        assert (hbm, kind) == (float(m["hbm_gbs"]), "measured")
        assert bf16 == float(m["bf16_tflops"]) and bkind.startswith("measured")
        assert bench._sm_max_mhz() == float(m["sm_max_mhz"])
    else:
        assert kind == "fallback" and bkind == "fallback"


def test_reference_arm_prints_one_json_line():
    """`bench.py --impl reference` (the oracle on the host cores) needs no GPU: one JSON line with
    the native arm's metric and unit, impl "reference", its cpu_baseline and a host-only e2e."""
    import json
    import subprocess
    root = bench.ROOT
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["steps"] == 1 and d["higher_is_better"] is True
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"]
