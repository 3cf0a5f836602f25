"""GPU parity of attention_with_kv_cache against the oracle.

vllm PR 39445 page, Breakdown items 2-3 (attention over the fp8 cache with
fused dequantisation and scale folding); vllm PR 50194 page, Key source
snippet (causal, window_size, soft_cap, paged blocks, KV split); vllm PR
38378 page, Breakdown item 3 (per-token-head dequantisation in the tile).
Tolerances: see tests/_harness.py.
"""
import numpy as np
import pytest
import torch

from int8_kv_cache_reshape_gb300 import workloads as W

from _harness import (GpuRun, assert_attention_close, oracle_cache, oracle_reference,
                      visible_window_mask)

pytestmark = pytest.mark.gpu


def _check(wl, warps=None, monkeypatch=None, tokens=None):
    if monkeypatch is not None:
        if warps is None:
            monkeypatch.delenv("KVQ_DECODE_WARPS", raising=False)
        else:
            monkeypatch.setenv("KVQ_DECODE_WARPS", str(warps))
    g = GpuRun(wl).write_cache().attention()
    kc, vc = oracle_cache(wl)
    ref, bnd = oracle_reference(wl, kc, vc, tokens=tokens)
    return assert_attention_close(g.out_f32(tokens), ref, wl.name, bnd), g


def test_config1_tiny(cuda_device):
    e, g = _check(W.config(1))
    assert e["max_abs"] <= 1e-2


@pytest.mark.parametrize("index,dtype", [(2, None), (3, None), (4, "int8_per_token_head"),
                                         (4, "fp8_per_token_head"),
                                         (4, "fp8_e5m2_per_token_head"), (5, None)])
def test_scaled_configs(cuda_device, index, dtype):
    _check(W.scaled(index, kv_cache_dtype=dtype))


DTYPES = ["fp8_e4m3", "fp8_e5m2", "int8_per_token_head", "fp8_per_token_head",
          "fp8_e5m2_per_token_head"]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D,hq,hkv", [(64, 8, 8), (64, 8, 1), (128, 16, 8), (128, 12, 3),
                                      (256, 16, 2), (128, 16, 1)])
def test_shapes_and_dtypes(cuda_device, dtype, D, hq, hkv):
    wl = W.custom(f"{dtype}-{D}-{hq}/{hkv}", [1, 2, 1, 5, 1], [1, 17, 100, 5, 333], hq, hkv, D,
                  16, dtype, 200 + D + hq, outlier_p=0.01,
                  token_scale_range=(0.1, 10.0) if "per_token" in dtype else None)
    _check(wl)


@pytest.mark.parametrize("window,soft_cap", [(0, 0.0), (1, 0.0), (16, 0.0), (37, 30.0),
                                             (0, 5.0), (1000, 0.0)])
def test_window_and_soft_cap(cuda_device, window, soft_cap):
    wl = W.custom("win", [1, 3, 1, 2], [700, 90, 16, 256], 32, 8, 128, 16, "fp8_e4m3", 300,
                  window=window, soft_cap=soft_cap)
    _check(wl)


def test_non_causal(cuda_device):
    wl = W.custom("noncausal", [4, 1, 7], [60, 30, 7], 16, 4, 128, 16, "fp8_e5m2", 301,
                  causal=False)
    _check(wl)


@pytest.mark.parametrize("warps", [4, 12, 40, 400, 100000])
def test_forced_warp_counts(cuda_device, monkeypatch, warps):
    """Few warps: each streams many pieces of many tiles; many warps: tiles
    are cut into many pieces and merged (one chunk per warp at the end)."""
    wl = W.custom("splits", [1, 1, 2, 1], [1000, 129, 300, 16], 32, 8, 128, 16,
                  "int8_per_token_head", 302, token_scale_range=(0.1, 10.0),
                  window=200 if warps == 40 else 0)
    e, g = _check(wl, warps=warps, monkeypatch=monkeypatch)
    assert g.sched_info["num_decode_warps"] <= max(warps, 4)


@pytest.mark.parametrize("warps", [4, 100000])
def test_forced_warp_counts_prefill_rows(cuda_device, monkeypatch, warps):
    wl = W.custom("rows-split", [37, 1, 9], [300, 600, 9], 16, 2, 128, 16, "fp8_e4m3", 309,
                  window=100)
    _check(wl, warps=warps, monkeypatch=monkeypatch)


def test_block_permutation_is_bit_identical(cuda_device):
    wl = W.custom("perm", [1, 2], [500, 77], 32, 8, 128, 16, "fp8_e4m3", 303, extra_blocks=9)
    a = GpuRun(wl).write_cache().attention().out.cpu()
    perm = torch.randperm(wl.num_blocks, generator=torch.Generator().manual_seed(1))
    wl2 = W.custom("perm", [1, 2], [500, 77], 32, 8, 128, 16, "fp8_e4m3", 303, extra_blocks=9)
    wl2.block_table = perm[wl.block_table.long()].to(torch.int32)
    blk = perm[wl.slot_mapping // 16]
    wl2.slot_mapping = blk * 16 + wl.slot_mapping % 16
    b = GpuRun(wl2).write_cache().attention().out.cpu()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_large_block_size(cuda_device):
    wl = W.custom("B2176", [40, 1, 3], [1000, 2176, 3000], 16, 2, 256, 2176, "fp8_e4m3", 304)
    _check(wl)


def test_empty_and_zero_query_requests(cuda_device):
    wl = W.custom("zeroq", [0, 1, 0, 2], [10, 40, 0, 20], 8, 2, 64, 16, "fp8_e4m3", 305)
    _check(wl)
    wl = W.custom("empty", [], [], 8, 2, 64, 16, "fp8_e4m3", 306)
    g = GpuRun(wl).write_cache().attention()
    assert g.out.numel() == 0


def test_queries_spanning_many_rows(cuda_device):
    """Requests whose query rows span several 16-row tiles and more than one
    KV chunk: causal masks inside a tile differ per row."""
    wl = W.custom("rows", [33, 9, 16], [50, 9, 300], 8, 2, 128, 16, "fp8_per_token_head", 307,
                  window=20, token_scale_range=(0.1, 10.0))
    _check(wl)


def test_unwritten_pages_outside_window_are_ignored(cuda_device):
    """Keys that no query can see are never read: leave their rows unwritten
    (0xCD bytes = NaN-free but arbitrary) and the output is unchanged."""
    wl = W.custom("win", [1, 1], [3000, 500], 32, 8, 128, 16, "fp8_e5m2", 308, window=128,
                  soft_cap=50.0)
    mask = visible_window_mask(wl, range(wl.num_req))
    g = GpuRun(wl, write_mask=mask).write_cache().attention()
    kc, vc = oracle_cache(wl, write_mask=mask)
    ref, bnd = oracle_reference(wl, kc, vc)
    assert_attention_close(g.out_f32(), ref, "unwritten", bnd)
