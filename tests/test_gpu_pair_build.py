"""The prefill on CTA pairs (libkvq_pair.so, built with KVQ_PREFILL_PAIR=1).

A build option: quantised caches at head_dim 128 and 256 run the prefill's
MMAs on pairs of CTAs of a cluster (cta_group::2, M = 256: two consecutive
128-row tiles of one kv head share each converted KV tile, each CTA
converting half of it).  It is measured slower than single CTAs on the
prefill workloads, so the default build does not use it; this test keeps it
correct.  The pair library runs, in a child process (KVQ_LIBRARY selects
it), the plan checks (pair tiles at list entries 2i, 2i + 1) and the whole
prefill parity suite against the oracle.
"""
import os
import subprocess
import sys

import pytest

from int8_kv_cache_reshape_gb300 import build as kvq_build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

CHILD = r"""
import sys
import numpy as np
from int8_kv_cache_reshape_gb300 import kvq
assert kvq.LIB_PATH.endswith("libkvq_pair.so"), kvq.LIB_PATH
qsl = np.array([0, 300, 301], np.int32)
s = kvq.get_scheduler_metadata(2, 16, 4, 256, np.array([300, 900], np.int32), qsl, True, 0, "fp8_e4m3")
assert s.info()["prefill_cta_group"] == 2
s.close()
s = kvq.get_scheduler_metadata(2, 16, 4, 128, np.array([300, 900], np.int32), qsl, True, 0, "auto")
assert s.info()["prefill_cta_group"] == 1
s.close()
print("pair build ok")
"""


def test_pair_build_plan_and_prefill_parity(cuda_device):
    lib = kvq_build.build(pair=True)
    env = dict(os.environ, KVQ_LIBRARY=lib, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    res = subprocess.run([sys.executable, "-c", CHILD], env=env, capture_output=True, text=True,
                         timeout=300, cwd=ROOT)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          os.path.join(HERE, "test_plan.py"), os.path.join(HERE, "test_gpu_prefill.py")],
                         env=env, capture_output=True, text=True, timeout=1500, cwd=ROOT)
    assert res.returncode == 0, res.stdout[-4000:] + res.stderr[-2000:]
