"""Full-size parity of the five workloads against the oracle, in the launch
configuration the benchmark times (the whole batch runs on the GPU at full
size; the oracle writes the keys the compared requests can see).

  * decode workloads (tiny, decode batch, long context): every query row of
    every request, all heads;
  * large prefill: every row of a whole request (all heads);
  * mixed batch (each per-token-head dtype): every row of its longest
    prefill and of every decode request (the longest context is a decode).

The tiny, decode-batch and long-context workloads draw N(0, 1) values and
must meet the stated bounds (max-abs 1e-2, mean-abs 1e-3) plainly.  The
large prefill (x20 outliers) and the mixed batch (x10 token scales) have
outputs far above 4 in magnitude, where the bf16 result itself is coarser
than 1e-2: they are held to the bound of tests/_harness.py, and the test
checks that the oracle's own result rounded to bf16 misses the stated
max-abs bound there (the stated bound is infeasible, not merely missed).
vllm PR 50194 page, Key source snippet (the large fp8 prefill);
vllm PR 38378 page, Review (the reference quantiser matches the kernel's).
"""
import numpy as np
import pytest

from int8_kv_cache_reshape_gb300 import workloads as W

from _harness import (GpuRun, assert_attention_close, describe, oracle_cache, oracle_reference,
                      visible_window_mask)

pytestmark = pytest.mark.gpu


def _compare(wl, reqs, stated):
    g = GpuRun(wl).write_cache().attention()
    qsl = wl.query_start_loc.numpy()
    toks = np.concatenate([np.arange(qsl[r], qsl[r + 1]) for r in reqs])
    mask = visible_window_mask(wl, reqs)
    kc, vc = oracle_cache(wl, write_mask=mask)
    ref, bnd = oracle_reference(wl, kc, vc, tokens=toks)
    e = assert_attention_close(g.out_f32(toks), ref, f"full: {wl.name}", bnd, stated=stated)
    print(f"{wl.name}: {len(reqs)} requests, {toks.size} query tokens: {describe(e)}")
    return e


@pytest.mark.parametrize("index", [1, 2, 5])
def test_decode_workloads_every_row(cuda_device, index):
    wl = W.config(index)
    _compare(wl, list(range(wl.num_req)), stated=True)


def test_large_prefill_whole_request(cuda_device):
    wl = W.config(3)
    r = int(np.argmax(wl.seq_lens))
    e = _compare(wl, [r], stated=False)
    if not e["stated_max_ok"]:
        assert e["floor_max"] > 1e-2, "beyond 1e-2 although bf16(oracle) is within it"


@pytest.mark.parametrize("dtype", ["int8_per_token_head", "fp8_per_token_head",
                                   "fp8_e5m2_per_token_head"])
def test_mixed_longest_prefill_and_every_decode(cuda_device, dtype):
    wl = W.config(4, dtype)
    ql, sl = np.array(wl.query_lens), np.array(wl.seq_lens)
    prefills = [r for r in range(wl.num_req) if ql[r] > 1]
    decodes = [r for r in range(wl.num_req) if ql[r] == 1]
    longest_prefill = max(prefills, key=lambda r: sl[r])
    assert int(np.argmax(sl)) in decodes
    e = _compare(wl, sorted([longest_prefill] + decodes), stated=False)
    if not e["stated_max_ok"]:
        assert e["floor_max"] > 1e-2, "beyond 1e-2 although bf16(oracle) is within it"
