"""GPU parity of the tensor-core prefill path against the oracle.

Requests with more than 16 (query, head) rows per kv head run on the
128-row tcgen05 prefill kernel: vllm PR 39445 page, Breakdown items 2-3
(tile GEMMs with the fp8 cache dequantised into a bf16 tile, scales folded);
vllm PR 38378 page, Breakdown item 3 (per-token-head scales in the tile);
vllm PR 50194 page, Key source snippet (causal, window_size, soft_cap,
paged blocks, block_size 2176).  These cases span several 128-row tiles and
64-key tiles with ragged tails, every cache dtype and head size, windows
that start inside a key tile, soft caps, mixed prefill + decode batches and
rows that see no written key.  Tolerances: see tests/_harness.py.
"""
import pytest
import torch

import oracle
from int8_kv_cache_reshape_gb300 import workloads as W

from _harness import (GpuRun, _oracle_args, assert_attention_close, oracle_cache,
                      oracle_reference)

pytestmark = pytest.mark.gpu

DTYPES = ["fp8_e4m3", "fp8_e5m2", "int8_per_token_head", "fp8_per_token_head",
          "fp8_e5m2_per_token_head"]


def _check(wl):
    g = GpuRun(wl).write_cache().attention()
    kc, vc = oracle_cache(wl)
    ref, bnd = oracle_reference(wl, kc, vc)
    e = assert_attention_close(g.out_f32(), ref, wl.name, bnd)
    return e, g


def _pth(dtype):
    return (0.1, 10.0) if "per_token" in dtype else None


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D,hq,hkv", [(64, 8, 8), (128, 32, 8), (128, 8, 1), (256, 16, 4)])
def test_prefill_dtypes_and_heads(cuda_device, dtype, D, hq, hkv):
    # query rows per kv head: 77*G (several 128-row tiles, ragged tail), 130*G, 17*G
    wl = W.custom(f"pf-{dtype}-{D}-{hq}/{hkv}", [77, 130, 17], [77, 300, 1000], hq, hkv, D, 16,
                  dtype, 400 + D + hq, outlier_p=0.01, token_scale_range=_pth(dtype))
    e, g = _check(wl)
    assert g.sched_info["num_prefill_tiles"] > 0 and g.sched_info["num_tiles"] == 0


@pytest.mark.parametrize("window,soft_cap", [(1, 0.0), (50, 0.0), (100, 20.0), (0, 5.0),
                                             (4000, 0.0)])
def test_prefill_window_and_soft_cap(cuda_device, window, soft_cap):
    wl = W.custom("pf-win", [150, 70], [900, 70], 16, 4, 128, 16, "fp8_e4m3", 410,
                  window=window, soft_cap=soft_cap)
    _check(wl)


def test_prefill_non_causal(cuda_device):
    wl = W.custom("pf-noncausal", [40, 100], [200, 100], 16, 4, 128, 16,
                  "int8_per_token_head", 411, causal=False, token_scale_range=(0.1, 10.0))
    _check(wl)


def test_mixed_prefill_and_decode(cuda_device):
    wl = W.custom("pf-mixed", [1, 300, 1, 1, 64, 3], [2000, 300, 45, 700, 1100, 3], 32, 8, 128,
                  16, "fp8_per_token_head", 412, token_scale_range=(0.1, 10.0))
    e, g = _check(wl)
    assert g.sched_info["num_prefill_tiles"] > 0 and g.sched_info["num_tiles"] > 0


def test_prefill_large_block_size(cuda_device):
    wl = W.custom("pf-B2176", [500, 64], [2500, 2176], 8, 1, 256, 2176, "fp8_e4m3", 413)
    _check(wl)


def test_prefill_scaled_outliers(cuda_device):
    """Heavy outliers (x64 on 2% of values): per-token-head scales differ by
    orders of magnitude between neighbouring keys inside one 64-key tile."""
    wl = W.custom("pf-outliers", [200], [450], 16, 2, 128, 16, "int8_per_token_head", 414,
                  outlier_p=0.02, outlier_mul=64.0, token_scale_range=(0.01, 100.0))
    _check(wl)


def test_prefill_rows_without_blocks(cuda_device):
    """Table entries outside [0, num_blocks) read as masked keys: a prefill
    whose table holds only -1 gets zero output, and the other request of the
    batch matches the oracle (computed for its tokens only)."""
    wl = W.custom("pf-holes", [64, 40], [64, 200], 8, 2, 64, 16, "fp8_e5m2", 415)
    g0 = GpuRun(wl).write_cache()
    g0.bt[0, :] = -1
    g = g0.attention()
    kc, vc = oracle_cache(wl)
    ref, bnd = oracle_reference(wl, kc, vc, tokens=range(64, 104))
    assert_attention_close(g.out_f32(range(64, 104)), ref, "holes", bnd)
    assert float(abs(g.out_f32(range(64))).max()) == 0.0


@pytest.mark.parametrize("dtype", ["int8_per_token_head", "fp8_per_token_head",
                                   "fp8_e5m2_per_token_head"])
def test_prefill_large_blocks_window_per_token_head(cuda_device, dtype):
    """block_size 2176 (vllm PR 50194 page, Key source snippet) with a
    sliding window and per-token-head scales at D = 256: the 16-key copies
    of codes and of their scale tails cross a block boundary mid-tile."""
    wl = W.custom(f"pf-B2176-win-{dtype}", [300, 90, 1], [2400, 2176, 4500], 16, 4, 256, 2176,
                  dtype, 416, window=700, token_scale_range=(0.1, 10.0), outlier_p=0.01)
    e, g = _check(wl)
    assert g.sched_info["num_prefill_tiles"] > 0 and g.sched_info["num_tiles"] > 0


def _without_block(bt, sl, block_size, req, blk):
    """Block table and sequence lengths with block `blk` of request `req`
    taken out of its table and its sequence one block shorter.  When every
    query of the request sees that block whole (no window, the block ends at
    or before L - Q), the keys that remain keep their causal relation to
    every query, so on the same caches this is what a table hole at `blk`
    must give."""
    bt, sl = bt.clone(), sl.clone()
    row = bt[req].tolist()
    bt[req] = torch.tensor(row[:blk] + row[blk + 1:] + [row[0]], dtype=bt.dtype)
    sl[req] -= block_size
    return bt, sl


@pytest.mark.parametrize("dtype,D", [("fp8_e4m3", 128), ("int8_per_token_head", 256),
                                     ("fp8_e5m2", 64)])
def test_table_hole_mid_sequence(cuda_device, dtype, D):
    """A -1 in the middle of a block table masks that block's keys, for a
    prefill request (the hole inside one key tile) and a decode request of
    the same batch; the rest of each row matches the oracle without them."""
    wl = W.custom(f"hole-{dtype}-{D}", [120, 1], [700, 900], 16, 4, D, 16, dtype, 417,
                  token_scale_range=_pth(dtype))
    g0 = GpuRun(wl).write_cache()
    holes = {0: 9, 1: 30}                       # keys 144..159 and 480..495
    for r, blk in holes.items():
        assert (blk + 1) * wl.block_size <= wl.seq_lens[r] - wl.query_lens[r]
        g0.bt[r, blk] = -1
    g = g0.attention()
    assert g.sched_info["num_prefill_tiles"] > 0 and g.sched_info["num_tiles"] > 0
    kc, vc = oracle_cache(wl)
    bt, sl = wl.block_table, wl.seq_lens_t
    for r, blk in holes.items():
        bt, sl = _without_block(bt, sl, wl.block_size, r, blk)
    args = list(_oracle_args(wl, kc, vc))
    args[4], args[5] = sl, bt
    ref = oracle.attention(*args)
    bnd = oracle.attention_fp32_bound(*args)
    assert_attention_close(g.out_f32(), ref, "table hole", bnd)


def test_reruns_are_bit_identical(cuda_device, monkeypatch):
    """Two calls on the same inputs give the same bits: the split-KV merge
    order is fixed by the schedule, not by which piece arrives last."""
    monkeypatch.setenv("KVQ_DECODE_WARPS", "96")
    wl = W.custom("rerun", [1, 200, 1, 33], [3000, 500, 1200, 40], 32, 8, 128, 16,
                  "fp8_per_token_head", 418, token_scale_range=(0.1, 10.0))
    g = GpuRun(wl).write_cache()
    a = g.attention().out.clone()
    g.out.fill_(float("nan"))
    b = g.attention().out.clone()
    assert g.sched_info["num_merge_items"] > 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("dtype,D,ctas", [("fp8_e4m3", 256, 1), ("int8_per_token_head", 128, 3),
                                          ("fp8_e5m2_per_token_head", 64, 2), ("auto", 128, 5),
                                          ("fp8_per_token_head", 128, 7)])
def test_persistent_ctas_walk_many_tiles(cuda_device, monkeypatch, dtype, D, ctas):
    """The prefill runs one persistent CTA per SM over the dealt tile list;
    with KVQ_PREFILL_CTAS forcing a few CTAs, each walks many tiles of
    different requests, kv heads and key ranges back to back (the rings,
    Q and O carried over tile boundaries).  The output is bit-identical to
    the one-tile-per-CTA run and matches the oracle."""
    wl = W.custom(f"pf-persist-{dtype}-{D}", [150, 40, 1, 300, 17], [400, 40, 900, 1300, 17], 16, 4, D,
                  16, dtype, 420 + D, window=0, token_scale_range=_pth(dtype), outlier_p=0.01)
    monkeypatch.delenv("KVQ_PREFILL_CTAS", raising=False)
    g = GpuRun(wl).write_cache().attention()
    a = g.out.clone()
    tiles = g.sched_info["num_prefill_tiles"]
    assert tiles > 4 * ctas
    monkeypatch.setenv("KVQ_PREFILL_CTAS", str(ctas))
    g.out.fill_(float("nan"))
    b = g.attention().out.clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    kc, vc = oracle_cache(wl)
    ref, bnd = oracle_reference(wl, kc, vc)
    assert_attention_close(g.out_f32(), ref, wl.name, bnd)
