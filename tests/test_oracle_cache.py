"""Pins for the oracle's cache writer (reshape_and_cache).

Per-tensor fp8 (vllm PR 39445 page, Breakdown item 1; vllm PR 50194 page,
Key source snippet for fp8_e4m3 / fp8_e5m2) and per-token-head int8 / fp8
with inline absmax scales (vllm PR 38378 page, Breakdown item 3, Risks).
The expected bytes come from torch's own division, rounding and fp8 casts,
not from the oracle's code.
"""
import sys

import numpy as np
import pytest
import torch

import oracle
from int8_kv_cache_reshape_gb300 import workloads as W

FILL = 0xCD


def _caches(nb, B, H, row):
    kc = np.full((nb, B, H, row), FILL, dtype=np.uint8)
    return kc, kc.copy()


def _torch_fp8_codes(x: torch.Tensor, scale, fmt: str) -> np.ndarray:
    """Codes via torch: fp32 division, clamp to the largest finite value,
    round-to-nearest-even cast."""
    tdt, vmax = ((torch.float8_e4m3fn, 448.0) if fmt == "e4m3"
                 else (torch.float8_e5m2, 57344.0))
    y = x.float() / scale
    return y.clamp(-vmax, vmax).to(tdt).view(torch.uint8).numpy()


def _write(wl, dtype):
    H, D = wl.heads_kv, wl.head_dim
    row = oracle.row_bytes(dtype, D)
    kc, vc = _caches(wl.num_blocks, wl.block_size, H, row)
    oracle.reshape_and_cache(W.bf16_bits(wl.key), W.bf16_bits(wl.value), kc, vc,
                             wl.slot_mapping.numpy(), dtype, wl.k_scale,
                             wl.v_scale, wl.block_size)
    return kc, vc


def _rows_at_slots(cache, slots, B):
    flat = cache.reshape(-1, *cache.shape[2:])
    return flat[slots]


@pytest.mark.parametrize("fmt,dtype", [("e4m3", oracle.FP8_E4M3),
                                       ("e5m2", oracle.FP8_E5M2)])
def test_per_tensor_matches_torch(fmt, dtype):
    wl = W.custom("t", [3, 1], [40, 23], 4, 2, 64, 16,
                  "fp8_e4m3" if fmt == "e4m3" else "fp8_e5m2", 11,
                  outlier_p=0.05, outlier_mul=50.0,
                  k_scale=0.01 if fmt == "e4m3" else 1e-4,
                  v_scale=0.02 if fmt == "e4m3" else 2e-4)
    kc, vc = _write(wl, dtype)
    slots = wl.slot_mapping.numpy()
    assert np.array_equal(_rows_at_slots(kc, slots, 16),
                          _torch_fp8_codes(wl.key, wl.k_scale, fmt))
    assert np.array_equal(_rows_at_slots(vc, slots, 16),
                          _torch_fp8_codes(wl.value, wl.v_scale, fmt))
    # saturation is exercised: some codes sit at the largest magnitude
    assert np.any((_rows_at_slots(kc, slots, 16) & 0x7F) == (0x7E if fmt == "e4m3" else 0x7B))


@pytest.mark.parametrize("dtype", [oracle.INT8_PER_TOKEN_HEAD,
                                   oracle.FP8_PER_TOKEN_HEAD,
                                   oracle.FP8_E5M2_PER_TOKEN_HEAD])
def test_per_token_head_matches_torch(dtype):
    wl = W.custom("t", [2, 5], [33, 17], 4, 2, 128, 16, "int8_per_token_head",
                  12, token_scale_range=(0.1, 10.0))
    kc, vc = _write(wl, dtype)
    slots = wl.slot_mapping.numpy()
    D = wl.head_dim
    assert sys.byteorder == "little"
    for x, cache in ((wl.key, kc), (wl.value, vc)):
        xf = x.float()
        amax = xf.abs().amax(dim=-1)                      # exact in fp32
        qmax = {oracle.INT8_PER_TOKEN_HEAD: 127.0, oracle.FP8_PER_TOKEN_HEAD: 448.0,
                oracle.FP8_E5M2_PER_TOKEN_HEAD: 57344.0}[dtype]
        s = amax / torch.tensor(qmax, dtype=torch.float32)  # fp32 division
        y = xf / s.unsqueeze(-1)
        if dtype == oracle.INT8_PER_TOKEN_HEAD:
            codes = torch.round(y).clamp(-128, 127).to(torch.int8).view(torch.uint8)
        elif dtype == oracle.FP8_PER_TOKEN_HEAD:
            codes = y.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        else:
            codes = y.clamp(-57344, 57344).to(torch.float8_e5m2).view(torch.uint8)
        rows = _rows_at_slots(cache, slots, wl.block_size)
        assert np.array_equal(rows[..., :D], codes.numpy())
        assert np.array_equal(rows[..., D:D + 4].copy().view(np.float32)[..., 0],
                              s.numpy())
        assert np.all(rows[..., D + 4:] == 0)
        # the row's absmax element lands on +-qmax
        arg = xf.abs().argmax(dim=-1, keepdim=True)
        top = torch.gather(torch.from_numpy(rows[..., :D].copy()), -1, arg)
        want = {oracle.INT8_PER_TOKEN_HEAD: 127, oracle.FP8_PER_TOKEN_HEAD: 0x7E,
                oracle.FP8_E5M2_PER_TOKEN_HEAD: 0x7B}[dtype]
        assert np.all((top.numpy() & 0x7F) == want if dtype != oracle.INT8_PER_TOKEN_HEAD
                      else np.abs(top.numpy().view(np.int8)) == want)


@pytest.mark.parametrize("dtype", [oracle.INT8_PER_TOKEN_HEAD,
                                   oracle.FP8_PER_TOKEN_HEAD,
                                   oracle.FP8_E5M2_PER_TOKEN_HEAD])
def test_per_token_head_zero_row(dtype):
    D, H = 64, 1
    key = np.zeros((1, H, D), np.uint16)
    key[0, 0, 5] = 0x8000                           # -0.0 keeps the row zero
    kc, vc = _caches(1, 16, H, D + 16)
    oracle.reshape_and_cache(key, key, kc, vc, np.array([3]), dtype, 1.0, 1.0, 16)
    assert np.all(kc[0, 3, 0] == 0) and np.all(vc[0, 3, 0] == 0)


def test_skipped_slots_keep_bytes():
    wl = W.custom("t", [1], [20], 2, 1, 64, 16, "fp8_e4m3", 13)
    slots = wl.slot_mapping.numpy().copy()
    slots[[0, 7, 19]] = -1
    slots[3] = wl.num_blocks * wl.block_size   # beyond the pool
    kc, vc = _caches(wl.num_blocks, 16, 1, 64)
    oracle.reshape_and_cache(W.bf16_bits(wl.key), W.bf16_bits(wl.value), kc,
                             vc, slots, oracle.FP8_E4M3, wl.k_scale,
                             wl.v_scale, 16)
    written = set(int(s) for s in slots if 0 <= s < wl.num_blocks * 16)
    flat = kc.reshape(-1, 64)
    for s in range(flat.shape[0]):
        if s not in written:
            assert np.all(flat[s] == FILL)
    assert len(written) == 16


def test_slot_permutation_permutes_rows():
    wl = W.custom("t", [1, 1], [30, 18], 4, 2, 64, 16, "fp8_e5m2", 14)
    kc1, vc1 = _write(wl, oracle.FP8_E5M2)
    perm = np.random.default_rng(0).permutation(wl.num_blocks * 16)
    slots2 = perm[wl.slot_mapping.numpy()]
    kc2, vc2 = _caches(wl.num_blocks, 16, 2, 64)
    oracle.reshape_and_cache(W.bf16_bits(wl.key), W.bf16_bits(wl.value), kc2,
                             vc2, slots2, oracle.FP8_E5M2, wl.k_scale,
                             wl.v_scale, 16)
    f1, f2 = kc1.reshape(-1, 2, 64), kc2.reshape(-1, 2, 64)
    for s in wl.slot_mapping.numpy():
        assert np.array_equal(f1[s], f2[perm[s]])


def test_auto_is_a_copy():
    wl = W.custom("t", [1], [9], 2, 1, 64, 16, "auto", 15)
    kc, vc = _write(wl, oracle.AUTO)
    rows = _rows_at_slots(kc, wl.slot_mapping.numpy(), 16)
    assert np.array_equal(rows.view(np.uint16), W.bf16_bits(wl.key))
