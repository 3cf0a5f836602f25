"""GPU parity of reshape_and_cache: cache bytes bit-exact against the oracle.

vllm PR 39445 page, Breakdown item 1 (fp8 cache writer) and vllm PR 38378
page, Breakdown item 3 (per-token-head int8 / fp8 with inline scales).
"""
import numpy as np
import pytest
import torch

from int8_kv_cache_reshape_gb300 import workloads as W

from _harness import FILL, GpuRun, oracle_cache

pytestmark = pytest.mark.gpu

DTYPES = ["auto", "fp8_e4m3", "fp8_e5m2", "int8_per_token_head", "fp8_per_token_head",
          "fp8_e5m2_per_token_head"]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D", [64, 128, 256])
def test_cache_bytes_match_oracle(cuda_device, dtype, D):
    wl = W.custom("cache", [1, 3, 1], [37, 50, 16], 8, 2 if D == 256 else 4, D, 16, dtype,
                  100 + D, extra_blocks=3, outlier_p=0.02, outlier_mul=40.0,
                  token_scale_range=(0.01, 100.0) if "per_token" in dtype else None)
    # some tokens are not written (negative slots, a slot past the pool)
    wl.slot_mapping[[0, 5, 40]] = -1
    wl.slot_mapping[7] = wl.num_blocks * wl.block_size + 3
    g = GpuRun(wl).write_cache()
    torch.cuda.synchronize()
    kc, vc = oracle_cache(wl)
    assert np.array_equal(g.kc.cpu().numpy(), kc)
    assert np.array_equal(g.vc.cpu().numpy(), vc)
    assert np.any(kc == FILL)  # untouched rows stay untouched


def _finite_bf16_patterns():
    bits = np.arange(65536, dtype=np.uint32)
    exp = (bits >> 7) & 0xFF
    return bits[exp != 0xFF].astype(np.uint16)            # no inf / nan


@pytest.mark.parametrize("dtype", ["fp8_e4m3", "fp8_e5m2"])
@pytest.mark.parametrize("scale", [1.0, 0.05, 3.0e-3, 7.0e2, 2.0 ** -20])
def test_every_finite_bf16_value(cuda_device, dtype, scale):
    """Every finite bf16 value through the per-tensor quantiser (exact ties,
    subnormals, saturation, signed zeros), for several scales."""
    pats = _finite_bf16_patterns()
    D, H = 128, 2
    T = -(-pats.size // (H * D))
    x = np.zeros(T * H * D, np.uint16)
    x[: pats.size] = pats
    key = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).view(T, H, D)
    value = key.flip(0).contiguous()
    wl = W.custom("sweep", [1], [T], 2, H, D, 16, dtype, 7, k_scale=scale, v_scale=scale)
    wl.key, wl.value = key, value
    g = GpuRun(wl).write_cache()
    torch.cuda.synchronize()
    kc, vc = oracle_cache(wl)
    assert np.array_equal(g.kc.cpu().numpy(), kc)
    assert np.array_equal(g.vc.cpu().numpy(), vc)


@pytest.mark.parametrize("dtype", ["int8_per_token_head", "fp8_per_token_head",
                                   "fp8_e5m2_per_token_head"])
def test_per_token_head_special_rows(cuda_device, dtype):
    """Zero rows, rows of signed zeros, subnormal-only rows, huge rows and
    exact ties after the division."""
    D, H, T = 128, 2, 8
    rng = np.random.default_rng(5)
    x = rng.standard_normal((T, H, D)).astype(np.float32)
    x[0] = 0.0
    x[1, 0] = -0.0
    x[1, 1] = 1e-39                                         # fp32/bf16 subnormals
    x[2] *= 1e30
    x[3, 0] = np.arange(D) - 63.5                           # absmax 64.5
    x[4, 1] = 2.0 ** -133                                   # smallest bf16 subnormal
    key = torch.from_numpy(x).to(torch.bfloat16)
    wl = W.custom("special", [1], [T], 2, H, D, 16, dtype, 8)
    wl.key, wl.value = key, (-key).contiguous()
    g = GpuRun(wl).write_cache()
    torch.cuda.synchronize()
    kc, vc = oracle_cache(wl)
    assert np.array_equal(g.kc.cpu().numpy(), kc)
    assert np.array_equal(g.vc.cpu().numpy(), vc)


def test_strided_key_value(cuda_device):
    """Keys and values taken as views of a fused qkv tensor (token stride >
    heads * head_dim)."""
    T, Hq, H, D = 33, 8, 2, 128
    qkv = torch.randn((T, Hq + 2 * H, D), generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    wl = W.custom("strided", [1], [T], Hq, H, D, 16, "fp8_e4m3", 9, k_scale=0.02, v_scale=0.03)
    dev = torch.device("cuda:0")
    qkv_d = qkv.to(dev)
    g = GpuRun(wl)
    g.key, g.value = qkv_d[:, Hq:Hq + H], qkv_d[:, Hq + H:]
    g.write_cache()
    torch.cuda.synchronize()
    wl.key, wl.value = qkv[:, Hq:Hq + H].contiguous(), qkv[:, Hq + H:].contiguous()
    kc, vc = oracle_cache(wl)
    assert np.array_equal(g.kc.cpu().numpy(), kc)
    assert np.array_equal(g.vc.cpu().numpy(), vc)


@pytest.mark.parametrize("index,dtype", [(1, None), (2, None), (3, None),
                                         (4, "int8_per_token_head"),
                                         (4, "fp8_per_token_head"),
                                         (4, "fp8_e5m2_per_token_head"), (5, None)])
def test_full_size_cache_write_sampled(cuda_device, index, dtype):
    """The bulk cache write of each full-size workload; sampled tokens are
    compared with the oracle (written into a compact cache, block size 1)."""
    wl = W.config(index, dtype)
    g = GpuRun(wl).write_cache()
    torch.cuda.synchronize()
    rng = np.random.default_rng(index)
    n = min(wl.num_tokens, 512)
    toks = np.unique(np.concatenate([rng.choice(wl.num_tokens, n, replace=False),
                                     [0, wl.num_tokens - 1]]))
    sub = W.custom("sub", [1], [len(toks)], wl.heads_q, wl.heads_kv, wl.head_dim, 1,
                   wl.kv_cache_dtype, 0, k_scale=wl.k_scale, v_scale=wl.v_scale)
    sub.key = wl.key[toks].contiguous()
    sub.value = wl.value[toks].contiguous()
    sub.slot_mapping = torch.arange(len(toks), dtype=torch.int64)
    sub.num_blocks = len(toks)
    kc, vc = oracle_cache(sub)
    slots = wl.slot_mapping[toks].to(torch.long)
    gk = g.kc.view(-1, *g.kc.shape[2:])[slots.to(g.kc.device)].cpu().numpy()
    gv = g.vc.view(-1, *g.vc.shape[2:])[slots.to(g.vc.device)].cpu().numpy()
    assert np.array_equal(gk, kc.reshape(gk.shape))
    assert np.array_equal(gv, vc.reshape(gv.shape))
