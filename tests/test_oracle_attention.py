"""Pins for the oracle's paged attention.

The attention is the plain definition (vllm PR 39445 page, Breakdown items
2-3; vllm PR 50194 page, Key source snippet: causal, window_size, soft_cap
over paged blocks; vllm PR 38378 page, Breakdown item 3: per-token-head
dequantisation).  Pins: torch's scaled_dot_product_attention in float64 on
dequantised K/V gathered with numpy indexing and torch's fp8 casts,
invariants (block permutation, paging, masking), closed forms (L = 1, equal
keys) and the soft-cap bound.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from int8_kv_cache_reshape_gb300 import workloads as W

DT = {"auto": oracle.AUTO, "fp8_e4m3": oracle.FP8_E4M3,
      "fp8_e5m2": oracle.FP8_E5M2, "int8_per_token_head": oracle.INT8_PER_TOKEN_HEAD,
      "fp8_per_token_head": oracle.FP8_PER_TOKEN_HEAD,
      "fp8_e5m2_per_token_head": oracle.FP8_E5M2_PER_TOKEN_HEAD}


def _cache(wl):
    dt = DT[wl.kv_cache_dtype]
    row = oracle.row_bytes(dt, wl.head_dim)
    kc = np.zeros((wl.num_blocks, wl.block_size, wl.heads_kv, row), np.uint8)
    vc = np.zeros_like(kc)
    oracle.reshape_and_cache(W.bf16_bits(wl.key), W.bf16_bits(wl.value), kc, vc,
                             wl.slot_mapping.numpy(), dt, wl.k_scale, wl.v_scale,
                             wl.block_size)
    return kc, vc


def _attn(wl, kc, vc, **over):
    a = dict(heads_kv=wl.heads_kv, block_size=wl.block_size,
             dtype=DT[wl.kv_cache_dtype], sm_scale=wl.sm_scale,
             causal=wl.causal, window=wl.window, soft_cap=wl.soft_cap,
             k_scale=wl.k_scale, v_scale=wl.v_scale)
    a.update(over)
    bt = over.pop("block_table", wl.block_table)
    a.pop("block_table", None)
    return oracle.attention(W.bf16_bits(wl.q), kc, vc, wl.query_start_loc,
                            wl.seq_lens_t, bt, **a)


def _dequant_library(wl, cache, scale):
    """[T, Hkv, D] float64 dequantised rows via torch casts (not the oracle)."""
    D = wl.head_dim
    flat = torch.from_numpy(cache.reshape(-1, wl.heads_kv, cache.shape[-1]).copy())
    rows = flat[wl.slot_mapping]
    dt = wl.kv_cache_dtype
    if dt == "auto":
        return rows.view(torch.bfloat16).to(torch.float64)
    codes = rows[..., :D].contiguous()
    if dt in ("fp8_e4m3", "fp8_per_token_head"):
        val = codes.view(torch.float8_e4m3fn).to(torch.float64)
    elif dt in ("fp8_e5m2", "fp8_e5m2_per_token_head"):
        val = codes.view(torch.float8_e5m2).to(torch.float64)
    else:
        val = codes.view(torch.int8).to(torch.float64)
    if dt in ("fp8_e4m3", "fp8_e5m2"):
        return val * float(scale)
    s = rows[..., D:D + 4].contiguous().view(torch.float32).to(torch.float64)
    return val * s


def _sdpa_reference(wl, kc, vc, soft_cap_ok=False):
    """float64 torch SDPA on dequantised K/V with an explicit boolean mask."""
    K = _dequant_library(wl, kc, wl.k_scale)
    V = _dequant_library(wl, vc, wl.v_scale)
    q = wl.q.to(torch.float64)
    G = wl.heads_q // wl.heads_kv
    out = torch.zeros(q.shape, dtype=torch.float64)
    qsl = wl.query_start_loc.tolist()
    for r, (Q, L) in enumerate(zip(wl.query_lens, wl.seq_lens)):
        sel = (wl.token_req == r)
        pos = wl.token_pos[sel].long()
        Kr = torch.zeros((L, wl.heads_kv, wl.head_dim), dtype=torch.float64)
        Vr = torch.zeros_like(Kr)
        Kr[pos], Vr[pos] = K[sel], V[sel]
        p = torch.arange(L - Q, L).view(Q, 1)
        j = torch.arange(L).view(1, L)
        mask = torch.ones((Q, L), dtype=torch.bool)
        if wl.causal:
            mask &= j <= p
        if wl.window > 0:
            mask &= (p - j) < wl.window
        qr = q[qsl[r]:qsl[r + 1]].transpose(0, 1)                  # [Hq, Q, D]
        Kh = Kr.transpose(0, 1).repeat_interleave(G, dim=0)        # [Hq, L, D]
        Vh = Vr.transpose(0, 1).repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(
            qr, Kh, Vh, attn_mask=mask, scale=wl.sm_scale)
        out[qsl[r]:qsl[r + 1]] = o.transpose(0, 1)
    return out.numpy()


CASES = [
    ("fp8_e4m3", dict(query_lens=[1, 8], seq_lens=[37, 8], hq=4, hkv=2, D=64)),
    ("fp8_e5m2", dict(query_lens=[3, 1, 6], seq_lens=[50, 70, 6], hq=8, hkv=2, D=64)),
    ("int8_per_token_head", dict(query_lens=[5, 1], seq_lens=[40, 33], hq=4, hkv=4, D=128)),
    ("fp8_per_token_head", dict(query_lens=[2, 4], seq_lens=[19, 64], hq=6, hkv=2, D=64)),
    ("fp8_e5m2_per_token_head", dict(query_lens=[3, 1], seq_lens=[30, 45], hq=4, hkv=2, D=64)),
    ("auto", dict(query_lens=[4], seq_lens=[21], hq=2, hkv=1, D=64)),
]


@pytest.mark.parametrize("dtype,c", CASES)
@pytest.mark.parametrize("window", [0, 7])
def test_matches_torch_sdpa(dtype, c, window):
    wl = W.custom("t", c["query_lens"], c["seq_lens"], c["hq"], c["hkv"], c["D"],
                  16, dtype, 21, window=window, outlier_p=0.02,
                  token_scale_range=(0.1, 10) if "per_token" in dtype else None)
    kc, vc = _cache(wl)
    got = _attn(wl, kc, vc)
    ref = _sdpa_reference(wl, kc, vc)
    assert np.max(np.abs(got - ref)) < 2e-6 * max(1.0, np.max(np.abs(ref)))


def test_non_causal_matches_sdpa():
    wl = W.custom("t", [3, 2], [9, 30], 4, 2, 64, 16, "fp8_e4m3", 22, causal=False)
    kc, vc = _cache(wl)
    assert np.max(np.abs(_attn(wl, kc, vc) - _sdpa_reference(wl, kc, vc))) < 2e-6


def test_block_permutation_invariance():
    wl = W.custom("t", [2, 1], [45, 31], 4, 2, 64, 16, "fp8_e4m3", 23,
                  extra_blocks=5)
    kc, vc = _cache(wl)
    base = _attn(wl, kc, vc)
    perm = np.random.default_rng(1).permutation(wl.num_blocks)
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    bt2 = perm[wl.block_table.numpy()].astype(np.int32)
    assert np.array_equal(_attn(wl, kc2, vc2, block_table=bt2), base)


def test_paged_equals_contiguous():
    args = ([3, 1], [40, 29], 4, 2, 64)
    paged = W.custom("t", *args, 16, "fp8_e5m2", 24, k_scale=0.02, v_scale=0.03)
    contig = W.custom("t", *args, 64, "fp8_e5m2", 24, k_scale=0.02, v_scale=0.03)
    assert torch.equal(paged.key, contig.key) and torch.equal(paged.q, contig.q)
    a = _attn(paged, *_cache(paged))
    b = _attn(contig, *_cache(contig))
    assert np.array_equal(a, b)


def test_softmax_rows_sum_to_one_and_masks():
    wl = W.custom("t", [6], [50], 4, 2, 64, 16, "int8_per_token_head", 25,
                  window=9, token_scale_range=(0.1, 10))
    kc, _ = _cache(wl)
    for t in range(6):
        p_pos = 50 - 6 + t
        for h in range(4):
            P = oracle.attention_probs(W.bf16_bits(wl.q), kc, wl.query_start_loc,
                                       wl.seq_lens_t, wl.block_table, 2, 16,
                                       oracle.INT8_PER_TOKEN_HEAD, wl.sm_scale,
                                       True, 9, 0.0, 1.0, t, h)
            assert abs(P.sum() - 1.0) < 1e-12
            j = np.arange(50)
            visible = (j <= p_pos) & (p_pos - j < 9)
            assert np.all(P[~visible] == 0) and np.all(P[visible] > 0)


def test_single_key_returns_its_value():
    wl = W.custom("t", [1], [1], 4, 2, 64, 16, "fp8_e4m3", 26)
    kc, vc = _cache(wl)
    out = _attn(wl, kc, vc)
    V = _dequant_library(wl, vc, wl.v_scale).numpy()       # [1, Hkv, D]
    for h in range(4):
        assert np.array_equal(out[0, h], V[0, h // 2].astype(np.float32))


def test_equal_keys_give_mean_of_values():
    wl = W.custom("t", [3], [20], 2, 1, 64, 16, "fp8_e4m3", 27)
    wl.key[:] = wl.key[0]                 # every key identical
    kc, vc = _cache(wl)
    out = _attn(wl, kc, vc)
    V = _dequant_library(wl, vc, wl.v_scale).numpy()[:, 0]  # [20, D]
    for t in range(3):
        p = 20 - 3 + t
        assert np.allclose(out[t, 0], V[:p + 1].mean(0), atol=1e-6, rtol=0)


def test_window_at_least_L_is_no_window_and_huge_cap_is_off():
    wl = W.custom("t", [2, 1], [25, 40], 4, 2, 64, 16, "fp8_e4m3", 28)
    kc, vc = _cache(wl)
    base = _attn(wl, kc, vc)
    assert np.array_equal(_attn(wl, kc, vc, window=40), base)
    assert np.array_equal(_attn(wl, kc, vc, window=1000), base)
    assert np.max(np.abs(_attn(wl, kc, vc, soft_cap=1e12) - base)) < 1e-6


def test_soft_cap_bounds_log_odds():
    """With cap c every score lies in (-c, c): log(P_i / P_j) <= 2c."""
    wl = W.custom("t", [1], [64], 2, 1, 64, 16, "fp8_e4m3", 29, sm_scale=3.0)
    kc, _ = _cache(wl)
    for cap in (0.25, 2.0):
        P = oracle.attention_probs(W.bf16_bits(wl.q), kc, wl.query_start_loc,
                                   wl.seq_lens_t, wl.block_table, 1, 16,
                                   oracle.FP8_E4M3, wl.sm_scale, True, 0, cap,
                                   wl.k_scale, 0, 0)
        assert math.log(P.max() / P.min()) <= 2 * cap + 1e-12
    P = oracle.attention_probs(W.bf16_bits(wl.q), kc, wl.query_start_loc,
                               wl.seq_lens_t, wl.block_table, 1, 16,
                               oracle.FP8_E4M3, wl.sm_scale, True, 0, 0.0,
                               wl.k_scale, 0, 0)
    assert math.log(P.max() / P.min()) > 4.0   # the uncapped case is sharper


def test_masked_keys_do_not_matter():
    wl = W.custom("t", [2], [48], 4, 2, 64, 16, "fp8_e4m3", 30, window=10)
    kc, vc = _cache(wl)
    base = _attn(wl, kc, vc)
    kc2, vc2 = kc.copy(), vc.copy()
    flat_k, flat_v = kc2.reshape(-1, 2, 64), vc2.reshape(-1, 2, 64)
    slots = wl.slot_mapping.numpy()
    for j in range(0, 48 - 2 - 9):        # before every query's window
        flat_k[slots[j]] = np.uint8(0x55)
        flat_v[slots[j]] = np.uint8(0x66)
    assert np.array_equal(_attn(wl, kc2, vc2), base)


def test_token_subset_matches_full():
    wl = W.custom("t", [4, 1, 3], [30, 17, 3], 4, 2, 64, 16, "fp8_e4m3", 31)
    kc, vc = _cache(wl)
    full = _attn(wl, kc, vc)
    toks = np.array([6, 0, 4, 7])
    sub = oracle.attention(W.bf16_bits(wl.q), kc, vc, wl.query_start_loc,
                           wl.seq_lens_t, wl.block_table, wl.heads_kv, 16,
                           oracle.FP8_E4M3, wl.sm_scale, True, 0, 0.0,
                           wl.k_scale, wl.v_scale, tokens=toks)
    assert np.array_equal(sub, full[toks])
