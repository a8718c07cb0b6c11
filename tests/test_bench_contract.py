"""The oracle arm of bench.py stays apart from the product: an oracle worker
(the process the reference arm and the CPU baseline time) quantizes and
attends with `oracle/` only, and never maps the CUDA library."""

import os

import pytest

import bench


@pytest.mark.skipif(not os.path.exists("/proc/self/maps"), reason="needs /proc")
def test_oracle_worker_maps_no_product_library():
    pool = bench.OraclePool(1)
    try:
        pool.prep([{"workload": "q4_0_mha_1k", "heads": 1, "T": 64, "seed": 0}])
        out = pool._ask([{"cmd": "run"}])
        assert out[0]["bytes"] > 0 and out[0]["dt"] >= 0
        with open(f"/proc/{pool.procs[0].pid}/maps") as fh:
            maps = fh.read()
        assert "libkvq" not in maps
    finally:
        for p in pool.procs:
            try:
                p.stdin.write('{"cmd": "quit"}\n')
                p.stdin.flush()
            except (BrokenPipeError, ValueError):
                pass
            p.wait(timeout=60)


@pytest.mark.skipif(not os.path.exists("/proc/self/maps"), reason="needs /proc")
def test_the_map_check_sees_the_library_when_it_is_loaded():
    import subprocess
    import sys

    lib = os.path.join(bench.ROOT, "bit_kv_cache_04_gb300", "libkvq.so")
    if not os.path.exists(lib):
        pytest.skip("libkvq.so not built")
    code = "from bit_kv_cache_04_gb300 import kvq; print(open('/proc/self/maps').read().count('libkvq'))"
    out = subprocess.run([sys.executable, "-c", code], cwd=bench.ROOT, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert int(out.stdout.strip().splitlines()[-1]) > 0
