"""The bounds-checked build: libkvq_checked.so, the same sources compiled
with KVQ_CHECKED=1.  Its kernels also check the indices they derive from
device arrays the host did not plan from -- each decode piece's (and each
merged tile's) rows against q and out through the device query_start_loc,
the decode's block-table positions against the table width -- and an index
outside its array sets the schedule's error word to 2
(kvq_sched_check_device: KVQ_E_INVALID_ARG) while the access is skipped.
Nothing traps.

The checked library runs in a child process (KVQ_LIBRARY selects it):
  * on valid inputs its output is bit-identical to the regular build's;
  * with the decode requests' device row offsets moved far past q and out
    (the host plan still holds the true ones) it reports KVQ_E_INVALID_ARG,
    leaves those requests' output rows untouched (the canary bands around
    every buffer intact) and still computes the prefill request, which is
    planned from the host's offsets.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from int8_kv_cache_reshape_gb300 import build as kvq_build
from int8_kv_cache_reshape_gb300 import workloads as W

from _harness import GpuRun

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

# one prefill request (40 tokens) and two long decodes (tiles cut among warps)
SHAPE = dict(query_lens=[40, 1, 1], seq_lens=[40, 3000, 2000], heads_q=16, heads_kv=4,
             head_dim=128, block_size=16, kv_cache_dtype="fp8_e4m3", seed=431)

CHILD = r"""
import json, os, sys
import numpy as np, torch
sys.path.insert(0, os.environ["KVQ_TEST_DIR"])
sys.path.insert(0, os.environ["KVQ_ROOT"])
from int8_kv_cache_reshape_gb300 import workloads as W
from int8_kv_cache_reshape_gb300 import kvq
from _harness import GpuRun, Guarded
shape = json.loads(os.environ["KVQ_SHAPE"])
out_dir = os.environ["KVQ_OUT"]
wl = W.custom("checked", shape["query_lens"], shape["seq_lens"], shape["heads_q"], shape["heads_kv"],
              shape["head_dim"], shape["block_size"], shape["kv_cache_dtype"], shape["seed"])
assert kvq.LIB_PATH.endswith("libkvq_checked.so"), kvq.LIB_PATH

# valid inputs
g = GpuRun(wl).write_cache().attention()
np.save(os.path.join(out_dir, "valid.npy"), g.out.view(torch.int16).cpu().numpy())

# the decode requests' device row offsets far past q and out
g2 = GpuRun(wl).write_cache()
bad = wl.query_start_loc.clone()
bad[1] += 10_000_000
bad[2] += 10_000_000
g2.qsl = bad.to(g2.dev)
sched = kvq.get_scheduler_metadata(wl.num_req, wl.heads_q, wl.heads_kv, wl.head_dim,
                                   wl.seq_lens_t.numpy(), wl.query_start_loc.numpy(),
                                   wl.causal, wl.window, wl.kv_cache_dtype)
ws = Guarded((max(sched.workspace_bytes, 1),), torch.uint8, 0, g2.dev)
kvq.attention_with_kv_cache(sched, g2.q, g2.kc, g2.vc, g2.qsl, g2.sl, g2.bt, wl.sm_scale,
                            wl.causal, wl.window, wl.soft_cap, wl.k_scale, wl.v_scale, g2.out,
                            ws.t, wl.kv_cache_dtype, wl.heads_kv)
torch.cuda.synchronize()
status = 0
try:
    sched.check_device()
except kvq.KvqError as e:
    status = e.status
ws.check("workspace")
g2._out.check("output")
g2._kc.check("key cache")
g2._vc.check("value cache")
info = sched.info()
sched.close()
np.save(os.path.join(out_dir, "invalid.npy"), g2.out.view(torch.int16).cpu().numpy())
json.dump({"status": status, "merges": info["num_merge_items"]}, open(os.path.join(out_dir, "res.json"), "w"))
"""


def test_checked_build_matches_and_catches_bad_row_offsets(cuda_device, tmp_path):
    lib = kvq_build.build(checked=True)
    wl = W.custom("checked", SHAPE["query_lens"], SHAPE["seq_lens"], SHAPE["heads_q"],
                  SHAPE["heads_kv"], SHAPE["head_dim"], SHAPE["block_size"],
                  SHAPE["kv_cache_dtype"], SHAPE["seed"])
    ref = GpuRun(wl).write_cache().attention().out.view(torch.int16).cpu().numpy()
    env = dict(os.environ, KVQ_LIBRARY=lib, KVQ_TEST_DIR=HERE, KVQ_ROOT=ROOT,
               KVQ_SHAPE=json.dumps(SHAPE), KVQ_OUT=str(tmp_path))
    res = subprocess.run([sys.executable, "-c", CHILD], env=env, capture_output=True, text=True,
                         timeout=600)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    valid = np.load(tmp_path / "valid.npy")
    invalid = np.load(tmp_path / "invalid.npy")
    r = json.load(open(tmp_path / "res.json"))
    assert r["merges"] > 0                       # the decode tiles were cut and merged
    assert np.array_equal(valid, ref)             # the checks change no result
    from int8_kv_cache_reshape_gb300 import kvq
    assert r["status"] == kvq.E_INVALID_ARG
    n_pre = SHAPE["query_lens"][0]
    assert np.array_equal(invalid[:n_pre], ref[:n_pre])        # the prefill request, from the host plan
    nan_bits = torch.tensor(float("nan"), dtype=torch.bfloat16).view(torch.int16).item()
    assert np.all(invalid[n_pre:] == nan_bits)                 # decode rows untouched (NaN fill)
