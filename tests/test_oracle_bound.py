"""Pins for oracle.attention_fp32_bound, the binary32 evaluation bound the
parity tests add to the stated attention tolerance.

It is a first-order forward error bound (scores accumulated in binary32,
softmax weights rounded to 11 significant bits, binary32 sums), so it is
pinned by its closed forms (one visible key; equal values, where score
errors cannot move the output), the growth of its score term with the
scores (equal keys: affine in sm_scale, slope doubling with q), its exact
scaling with the values, its invariance under block permutation, and by
being a bound: a binary32 numpy evaluation of the same attention on inputs
with large outliers stays within it, element by element, and comes within
a twentieth of it somewhere.
"""
import numpy as np
import pytest

import oracle
from int8_kv_cache_reshape_gb300 import workloads as W

from test_oracle_attention import DT, _cache, _dequant_library

U = 2.0 ** -23


def _gamma(n):
    return n * U / (1 - n * U)


def _bound(wl, kc, vc, **over):
    a = dict(heads_kv=wl.heads_kv, block_size=wl.block_size, dtype=DT[wl.kv_cache_dtype],
             sm_scale=wl.sm_scale, causal=wl.causal, window=wl.window, soft_cap=wl.soft_cap,
             k_scale=wl.k_scale, v_scale=wl.v_scale)
    a.update(over)
    return oracle.attention_fp32_bound(W.bf16_bits(wl.q), kc, vc, wl.query_start_loc,
                                       wl.seq_lens_t, wl.block_table, **a)


def test_single_key_closed_form():
    """One visible key: the output is that key's value, score errors move
    nothing; only the weight rounding remains, (2^-11 + gamma_10) |v|."""
    wl = W.custom("b", [1], [1], 4, 2, 64, 16, "fp8_e4m3", 40)
    kc, vc = _cache(wl)
    V = _dequant_library(wl, vc, wl.v_scale).numpy()[0]      # [Hkv, D]
    b = _bound(wl, kc, vc)
    for h in range(4):
        want = (2.0 ** -11 + _gamma(10) + 2.0 ** -25) * np.abs(V[h // 2])
        assert np.allclose(b[0, h], want, rtol=1e-6, atol=0)


def test_equal_values_have_no_score_term():
    """All values equal: every weighting gives the same output, so the
    score term vanishes and the bound is (2^-11 + gamma_{2n+8}) |v| plus
    the subnormal term 2^-25 n |v| / l, l = sum of the weights over the
    largest one (equal keys: l = n)."""
    wl = W.custom("b", [3], [40], 2, 1, 64, 16, "fp8_e4m3", 41, sm_scale=2.0)
    wl.value[:] = wl.value[0]
    wl.key[:] = wl.key[0]
    kc, vc = _cache(wl)
    V = _dequant_library(wl, vc, wl.v_scale).numpy()[0, 0]   # [D]
    b = _bound(wl, kc, vc)
    for t in range(3):
        n = 40 - 3 + t + 1
        assert np.allclose(b[t, 0], (2.0 ** -11 + _gamma(2 * n + 8) + 2.0 ** -25) * np.abs(V),
                           rtol=1e-6, atol=0)


def test_score_term_grows_with_the_scores():
    """Equal keys keep every weight at 1/n whatever the score scale, so only
    the score term depends on sm_scale: the bound is affine in sm_scale,
    with a slope that doubles when q doubles and vanishes when q = 0."""
    wl = W.custom("b", [2], [24], 2, 1, 64, 16, "fp8_e4m3", 47)
    wl.key[:] = wl.key[0]
    kc, vc = _cache(wl)
    s = wl.sm_scale
    b1, b2, b4 = (_bound(wl, kc, vc, sm_scale=k * s).astype(np.float64) for k in (1, 2, 4))
    slope = b2 - b1
    assert np.all(slope > 0)
    assert np.allclose(b4 - b2, 2 * slope, rtol=1e-3, atol=0)
    q0 = wl.q.clone()
    wl.q.mul_(2)                                           # exact in bf16
    d1, d2 = (_bound(wl, kc, vc, sm_scale=k * s).astype(np.float64) for k in (1, 2))
    assert np.allclose(d2 - d1, 2 * slope, rtol=1e-3, atol=0)
    wl.q.zero_()
    z1, z2 = (_bound(wl, kc, vc, sm_scale=k * s) for k in (1, 2))
    assert np.array_equal(z1, z2)
    wl.q.copy_(q0)


def test_scales_with_the_values():
    wl = W.custom("b", [2, 1], [30, 50], 4, 2, 64, 16, "fp8_e4m3", 42)
    kc, vc = _cache(wl)
    b1 = _bound(wl, kc, vc)
    b4 = _bound(wl, kc, vc, v_scale=4 * wl.v_scale)
    assert np.allclose(b4, 4 * b1, rtol=1e-6, atol=0)


def test_block_permutation_invariance():
    wl = W.custom("b", [2, 1], [70, 33], 4, 2, 64, 16, "int8_per_token_head", 43,
                  extra_blocks=5, token_scale_range=(0.1, 10.0))
    kc, vc = _cache(wl)
    base = _bound(wl, kc, vc)
    perm = np.random.default_rng(0).permutation(wl.num_blocks)
    inv = np.argsort(perm)
    kc2, vc2 = kc[inv], vc[inv]         # physical block b moves to perm[b]
    wl.block_table = wl.block_table.clone()
    wl.block_table[:] = wl.block_table.new_tensor(perm[wl.block_table.numpy()])
    assert np.array_equal(_bound(wl, kc2, vc2), base)


def _binary32_attention(wl, kc, vc):
    """The attention evaluated as a GPU kernel does: binary32 scores in
    16-wide partial sums, binary16 weights, binary32 sums."""
    D, G = wl.head_dim, wl.heads_q // wl.heads_kv
    K = _dequant_library(wl, kc, wl.k_scale).numpy()          # [T, Hkv, D] in slot order
    V = _dequant_library(wl, vc, wl.v_scale).numpy()
    q = W.bf16_bits(wl.q).astype(np.uint32) << 16
    q = q.view(np.float32)
    qsl = wl.query_start_loc.numpy()
    L = wl.seq_lens_t.numpy()
    tok0 = np.concatenate([[0], np.cumsum(L)])                # keys of request r in slot order
    out = np.zeros(q.shape, np.float32)
    for r in range(len(L)):
        for i in range(qsl[r + 1] - qsl[r]):
            pos = L[r] - (qsl[r + 1] - qsl[r]) + i
            lo = 0 if wl.window <= 0 else max(0, pos - wl.window + 1)
            for h in range(wl.heads_q):
                Kr = K[tok0[r] + lo:tok0[r] + pos + 1, h // G].astype(np.float32)
                Vr = V[tok0[r] + lo:tok0[r] + pos + 1, h // G].astype(np.float32)
                qv = q[qsl[r] + i, h]
                s = np.zeros(len(Kr), np.float32)
                for d0 in range(0, D, 16):
                    s = s + Kr[:, d0:d0 + 16] @ qv[d0:d0 + 16]
                z = s * np.float32(wl.sm_scale)
                p = np.exp(z - z.max()).astype(np.float32)
                w16 = p.astype(np.float16).astype(np.float32)
                out[qsl[r] + i, h] = (w16 @ Vr) / p.sum(dtype=np.float32)
    return out


@pytest.mark.parametrize("dtype,seed", [("fp8_e4m3", 44), ("int8_per_token_head", 45),
                                        ("fp8_per_token_head", 46)])
def test_bounds_a_binary32_evaluation(dtype, seed):
    """x20 outliers on 2% of the elements and x10 token scales make scores
    of several hundred, where binary32 score errors dominate."""
    wl = W.custom("b", [3, 1, 2], [200, 300, 120], 8, 2, 64, 16, dtype, seed,
                  outlier_p=0.02, outlier_mul=20.0,
                  token_scale_range=(0.1, 10.0) if "per_token" in dtype else None)
    kc, vc = _cache(wl)
    ref = oracle.attention(W.bf16_bits(wl.q), kc, vc, wl.query_start_loc, wl.seq_lens_t,
                           wl.block_table, wl.heads_kv, wl.block_size, DT[dtype], wl.sm_scale,
                           True, 0, 0.0, wl.k_scale, wl.v_scale)
    b = _bound(wl, kc, vc)
    err = np.abs(_binary32_attention(wl, kc, vc).astype(np.float64) - ref)
    assert np.all(err <= b)
    assert (err / b).max() > 0.05    # and not a vacuous one: the evaluation gets close
