"""Host-side pieces of bench.py that need no GPU: the gate that holds the CPU
oracle's worker processes until the GPU timing is done."""
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_gated_oracle_workers_wait_until_the_gate_opens():
    sys.path.insert(0, ROOT)
    import bench
    pool, gate = bench.oracle_pool(1, gated=True)
    try:
        res = pool.apply_async(bench._gate_wait)
        time.sleep(1.0)
        assert not res.ready()  # held while the GPU would be timed
        gate.set()
        res.get(timeout=60)
    finally:
        pool.terminate()
    pool, gate = bench.oracle_pool(1, gated=False)  # the reference arm: open from the start
    try:
        assert gate.is_set()
        pool.apply_async(bench._gate_wait).get(timeout=60)
    finally:
        pool.terminate()
