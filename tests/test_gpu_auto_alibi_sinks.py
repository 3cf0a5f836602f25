"""GPU parity of the bf16 ("auto") cache and of the ALiBi / sink options.

kv_cache_dtype "auto" is the default of the vllm PR 50194 page (Breakdown
item 2) and the non-quantised path the pages compare against (vllm PR 39445
page, Risks: an fp8 cache halves the bytes of a bf16 one; vllm PR 38378
page, Risks: the non-quantised path's throughput).  The cache writer copies
the bf16 rows; both attention kernels read them with bf16 MMAs and carry P
as the sum of two bf16 numbers, so the parity bound is the one of every
other dtype (tests/_harness.py).

use_alibi and use_sink are options of the attention the vllm PR 50194 page
tests (Key source snippet): ALiBi adds slope_h * (j - p) after the soft cap,
a sink is one extra per-head logit in the softmax normaliser.  Covered on
decode rows (whole and split tiles, whose merge adds the sink once) and on
prefill rows, for several dtypes.
"""
import numpy as np
import pytest

from int8_kv_cache_reshape_gb300 import workloads as W

from _harness import GpuRun, assert_attention_close, oracle_cache, oracle_reference

pytestmark = pytest.mark.gpu


def _check(wl, alibi=None, sinks=None, stated=False):
    g = GpuRun(wl, alibi_slopes=alibi, sinks=sinks).write_cache().attention()
    kc, vc = oracle_cache(wl)
    assert np.array_equal(g.kc.cpu().numpy(), kc) and np.array_equal(g.vc.cpu().numpy(), vc)
    ref, bnd = oracle_reference(wl, kc, vc, alibi_slopes=alibi, sinks=sinks)
    return assert_attention_close(g.out_f32(), ref, wl.name, bnd, stated=stated), g


@pytest.mark.parametrize("D,hq,hkv", [(64, 8, 2), (128, 32, 8), (256, 16, 2), (128, 12, 3)])
def test_auto_decode_and_prefill(cuda_device, D, hq, hkv):
    wl = W.custom(f"auto-{D}-{hq}/{hkv}", [1, 70, 1, 3, 150], [900, 70, 33, 300, 400], hq, hkv, D,
                  16, "auto", 500 + D + hq)
    e, g = _check(wl)
    assert g.sched_info["num_prefill_tiles"] > 0 and g.sched_info["num_tiles"] > 0
    assert g.sched_info["kv_elem_bytes"] == 2 and g.sched_info["row_bytes"] == 2 * D


@pytest.mark.parametrize("window,soft_cap", [(0, 0.0), (37, 0.0), (200, 30.0), (0, 5.0)])
def test_auto_window_soft_cap(cuda_device, window, soft_cap):
    wl = W.custom("auto-win", [1, 150, 2], [1200, 300, 90], 16, 4, 128, 16, "auto", 510,
                  window=window, soft_cap=soft_cap, outlier_p=0.01)
    _check(wl)


def test_auto_large_blocks_and_holes(cuda_device):
    """block_size 2176 and a request whose 16-key chunks straddle block ends."""
    wl = W.custom("auto-B2176", [300, 1], [2400, 2300], 16, 2, 256, 2176, "auto", 511,
                  window=700)
    _check(wl)


def test_auto_forced_splits(cuda_device, monkeypatch):
    monkeypatch.setenv("KVQ_DECODE_WARPS", "100000")
    wl = W.custom("auto-splits", [1, 1, 4], [2000, 129, 700], 32, 8, 128, 16, "auto", 512)
    e, g = _check(wl)
    assert g.sched_info["num_merge_items"] > 0


DT_CASES = [("fp8_e4m3", None), ("int8_per_token_head", (0.1, 10.0)), ("auto", None),
            ("fp8_e5m2_per_token_head", (0.1, 10.0))]


@pytest.mark.parametrize("dtype,tsr", DT_CASES)
@pytest.mark.parametrize("use_alibi,use_sink", [(True, False), (False, True), (True, True)])
def test_alibi_and_sinks(cuda_device, dtype, tsr, use_alibi, use_sink):
    hq = 16
    wl = W.custom(f"ext-{dtype}-{use_alibi}-{use_sink}", [1, 90, 2, 1], [1500, 200, 40, 16], hq,
                  4, 128, 16, dtype, 520, token_scale_range=tsr, soft_cap=30.0 if use_alibi else 0.0)
    alibi = W.alibi_slopes(hq) if use_alibi else None
    sinks = W.sink_logits(hq, 521) if use_sink else None
    e, g = _check(wl, alibi, sinks)
    assert g.sched_info["num_prefill_tiles"] > 0 and g.sched_info["num_tiles"] > 0


@pytest.mark.parametrize("warps", [8, 100000])
def test_sinks_on_split_tiles(cuda_device, monkeypatch, warps):
    """A tile cut among warps gets its sink once, in the merge."""
    monkeypatch.setenv("KVQ_DECODE_WARPS", str(warps))
    hq = 32
    wl = W.custom("sink-splits", [1, 1, 3, 1], [3000, 129, 700, 16], hq, 8, 128, 16, "fp8_e4m3",
                  530, window=1000)
    e, g = _check(wl, W.alibi_slopes(hq), W.sink_logits(hq, 531))
    if warps > 8:
        assert g.sched_info["num_merge_items"] > 0


@pytest.mark.parametrize("D", [64, 256])
def test_alibi_sinks_head_dims(cuda_device, D):
    hq = 8
    wl = W.custom(f"ext-D{D}", [1, 40, 1], [600, 40, 2177], hq, 2, D, 16, "fp8_e5m2", 540 + D,
                  window=300)
    _check(wl, W.alibi_slopes(hq), W.sink_logits(hq, 541))
