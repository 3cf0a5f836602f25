"""Pins for the oracle's ALiBi bias and attention sinks.

The vllm PR 50194 page (Key source snippet) passes use_alibi and use_sink to
its attention test helper; the pages name the options only.  Readings, the
plainest ones the rest supports (as in vLLM's own attention kernels):
  * ALiBi: score z_j <- z_j + slope_h * (j - p) for query position p, after
    sm_scale and the soft cap;
  * sink: one extra logit s_h per q head in the softmax normaliser, with no
    value: o = sum_j e^{z_j} v_j / (e^{s_h} + sum_j e^{z_j}).
Pins: torch's float64 scaled_dot_product_attention with the bias as a float
mask and the sink as an extra zero key whose bias is s_h and whose value is
zero; "off" special cases (slope 0, sink -inf) bit for bit; closed forms.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from int8_kv_cache_reshape_gb300 import workloads as W

from test_oracle_attention import DT, _cache, _dequant_library


def _attn(wl, kc, vc, **kw):
    return oracle.attention(W.bf16_bits(wl.q), kc, vc, wl.query_start_loc, wl.seq_lens_t,
                            wl.block_table, wl.heads_kv, wl.block_size,
                            DT[wl.kv_cache_dtype], wl.sm_scale, wl.causal, wl.window,
                            wl.soft_cap, wl.k_scale, wl.v_scale, **kw)


def _sdpa_ext(wl, kc, vc, alibi, sinks):
    """float64 SDPA on dequantised K/V: ALiBi as a float bias, the sink as an
    extra all-zero key with bias s_h and an all-zero value."""
    K = _dequant_library(wl, kc, wl.k_scale)
    V = _dequant_library(wl, vc, wl.v_scale)
    q = wl.q.to(torch.float64)
    G = wl.heads_q // wl.heads_kv
    Hq, D = wl.heads_q, wl.head_dim
    out = torch.zeros(q.shape, dtype=torch.float64)
    qsl = wl.query_start_loc.tolist()
    for r, (Q, L) in enumerate(zip(wl.query_lens, wl.seq_lens)):
        sel = wl.token_req == r
        pos = wl.token_pos[sel].long()
        Kr = torch.zeros((L + 1, wl.heads_kv, D), dtype=torch.float64)
        Vr = torch.zeros_like(Kr)
        Kr[pos], Vr[pos] = K[sel], V[sel]           # row L stays zero: the sink's key
        p = torch.arange(L - Q, L, dtype=torch.float64).view(1, Q, 1)
        j = torch.arange(L + 1, dtype=torch.float64).view(1, 1, L + 1)
        vis = torch.ones((1, Q, L + 1), dtype=torch.bool)
        if wl.causal:
            vis &= j <= p
        if wl.window > 0:
            vis &= (p - j) < wl.window
        bias = torch.zeros((Hq, Q, L + 1), dtype=torch.float64)
        if alibi is not None:
            bias += torch.tensor(alibi, dtype=torch.float64).view(Hq, 1, 1) * (j - p)
        vis = vis.expand(Hq, Q, L + 1).clone()
        vis[:, :, L] = sinks is not None
        if sinks is not None:
            bias[:, :, L] = torch.tensor(sinks, dtype=torch.float64).view(Hq, 1)
        mask = torch.where(vis, bias, torch.tensor(-math.inf, dtype=torch.float64))
        qr = q[qsl[r]:qsl[r + 1]].transpose(0, 1)
        Kh = Kr.transpose(0, 1).repeat_interleave(G, dim=0)
        Vh = Vr.transpose(0, 1).repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(qr, Kh, Vh, attn_mask=mask,
                                                             scale=wl.sm_scale)
        out[qsl[r]:qsl[r + 1]] = o.transpose(0, 1)
    return out.numpy()


CASES = [("fp8_e4m3", 64, 8, 2), ("int8_per_token_head", 128, 4, 4),
         ("fp8_e5m2", 64, 6, 3), ("auto", 64, 4, 2)]


@pytest.mark.parametrize("dtype,D,hq,hkv", CASES)
@pytest.mark.parametrize("use_alibi,use_sink", [(True, False), (False, True), (True, True)])
@pytest.mark.parametrize("window", [0, 9])
def test_matches_torch_sdpa(dtype, D, hq, hkv, use_alibi, use_sink, window):
    wl = W.custom("ext", [3, 1, 7], [40, 25, 7], hq, hkv, D, 16, dtype, 31, window=window,
                  outlier_p=0.02,
                  token_scale_range=(0.1, 10) if "per_token" in dtype else None)
    alibi = W.alibi_slopes(hq) if use_alibi else None
    sinks = W.sink_logits(hq, 77) if use_sink else None
    kc, vc = _cache(wl)
    got = _attn(wl, kc, vc, alibi_slopes=alibi, sinks=sinks)
    ref = _sdpa_ext(wl, kc, vc, alibi, sinks)
    assert np.max(np.abs(got - ref)) < 2e-6 * max(1.0, np.max(np.abs(ref)))


def test_off_values_are_bit_identical():
    """Slope 0 is no ALiBi and a sink of -inf is no sink, bit for bit."""
    wl = W.custom("off", [2, 5], [30, 61], 8, 2, 64, 16, "fp8_e4m3", 32, soft_cap=20.0)
    kc, vc = _cache(wl)
    base = _attn(wl, kc, vc)
    zero = _attn(wl, kc, vc, alibi_slopes=np.zeros(8, np.float32))
    ninf = _attn(wl, kc, vc, sinks=np.full(8, -np.inf, np.float32))
    assert np.array_equal(base.view(np.uint32), zero.view(np.uint32))
    assert np.array_equal(base.view(np.uint32), ninf.view(np.uint32))


@pytest.mark.parametrize("s", [0.0, math.log(3.0), -2.5])
def test_single_zero_key_with_sink(s):
    """One visible key whose K row is zero (score 0) and a sink s: the weight
    of the key is 1 / (1 + e^s), so o = v / (1 + e^s)."""
    wl = W.custom("sink1", [1], [1], 2, 1, 64, 16, "fp8_e4m3", 33)
    wl.key.zero_()
    kc, vc = _cache(wl)
    v = _dequant_library(wl, vc, wl.v_scale)[0, 0].numpy()
    got = _attn(wl, kc, vc, sinks=np.full(2, s, np.float32))
    for h in range(2):
        np.testing.assert_allclose(got[0, h], v / (1.0 + math.exp(np.float32(s))), rtol=1e-6,
                                   atol=1e-7)


@pytest.mark.parametrize("slope", [0.5, 0.0625, 2.0])
def test_alibi_equal_keys_give_geometric_weights(slope):
    """All keys equal: the raw scores are equal, so the weights follow the
    bias alone, w_j proportional to e^{slope j} -- nearer keys weigh more."""
    L = 20
    wl = W.custom("geo", [1], [L], 1, 1, 64, 16, "fp8_e4m3", 34, soft_cap=7.0)
    wl.key[:] = wl.key[0:1].clone()
    kc, vc = _cache(wl)
    probs = oracle.attention_probs(W.bf16_bits(wl.q), kc, wl.query_start_loc, wl.seq_lens_t,
                                   wl.block_table, 1, 16, DT["fp8_e4m3"], wl.sm_scale, True, 0,
                                   wl.soft_cap, wl.k_scale, 0, 0,
                                   alibi_slopes=np.array([slope], np.float32))
    sl = float(np.float32(slope))
    want = np.exp(sl * (np.arange(L) - (L - 1)))
    np.testing.assert_allclose(probs, want / want.sum(), rtol=1e-12)


def test_alibi_follows_the_soft_cap():
    """Two keys with different raw scores z0, z1 under a soft cap: the bias
    is added to the capped scores, so w1 / w0 = e^{c(z1) - c(z0) + slope},
    c(z) = cap tanh(z / cap)."""
    wl = W.custom("order", [1], [2], 1, 1, 64, 16, "auto", 35, soft_cap=3.0,
                  sm_scale=1.0)
    kc, vc = _cache(wl)
    K = _dequant_library(wl, kc, 1.0)[:, 0].numpy()
    q = wl.q.to(torch.float64)[0, 0].numpy()
    z = K @ q
    c = 3.0 * np.tanh(z / 3.0)
    slope = 0.75
    probs = oracle.attention_probs(W.bf16_bits(wl.q), kc, wl.query_start_loc, wl.seq_lens_t,
                                   wl.block_table, 1, 16, DT["auto"], 1.0, True, 0, 3.0, 1.0, 0,
                                   0, alibi_slopes=np.array([slope], np.float32))
    np.testing.assert_allclose(probs[1] / probs[0], math.exp(c[1] - c[0] + slope), rtol=1e-12)


def test_sink_weight_completes_the_distribution():
    """With a sink the key weights and the sink's weight sum to 1."""
    wl = W.custom("sum", [1], [33], 4, 2, 64, 16, "fp8_e5m2", 36, window=10)
    kc, vc = _cache(wl)
    for h in range(4):
        probs, sw = oracle.attention_probs(W.bf16_bits(wl.q), kc, wl.query_start_loc,
                                           wl.seq_lens_t, wl.block_table, 2, 16,
                                           DT["fp8_e5m2"], wl.sm_scale, True, 10, 0.0,
                                           wl.k_scale, 0, h, sinks=W.sink_logits(4, 5),
                                           with_sink=True)
        assert 0.0 < sw < 1.0
        assert abs(probs.sum() + sw - 1.0) < 1e-12
        assert np.count_nonzero(probs) == 10
