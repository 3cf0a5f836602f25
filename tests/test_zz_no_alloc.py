"""The no-allocation attention entry point (GPU).

kvq_attention_with_kv_cache_static_scratch serves callers that cannot call
cudaMalloc where they run attention (a serving loop whose device heap is
owned by a pool or allocator hook): it takes no workspace and keeps the
split-KV partials in a fixed device array the library reserves.  These tests
call it through the C ABI and check its output against the workspace-taking
entry point, within the parity tolerance of tests/_harness.py, on two calls
in a row (the array keeps the previous call's contents), and check that a
schedule needing more scratch than the array holds is refused.

This file is collected last so that a failure here cannot stop a -x run
before the other tests have run.
"""
import numpy as np
import pytest
import torch

from int8_kv_cache_reshape_gb300 import workloads as W

from _harness import GpuRun, assert_attention_close, kvq

pytestmark = pytest.mark.gpu


def _run_static(g, sched):
    wl = g.wl
    out = torch.full(wl.q.shape, float("nan"), dtype=torch.bfloat16, device=g.q.device)
    kvq().attention_with_kv_cache_static_scratch(
        sched, g.q, g.kc, g.vc, g.qsl, g.sl, g.bt, wl.sm_scale, wl.causal, wl.window,
        wl.soft_cap, wl.k_scale, wl.v_scale, out, wl.kv_cache_dtype, wl.heads_kv)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("dtype", ["fp8_e4m3", "int8_per_token_head"])
def test_static_scratch_matches_workspace_entry_point(cuda_device, monkeypatch, dtype):
    monkeypatch.setenv("KVQ_DECODE_WARPS", "64")  # tiles cut among warps: scratch is used
    wl = W.custom("noalloc", [1, 1, 2, 1], [900, 333, 640, 1500], 32, 8, 128, 16, dtype, 77,
                  token_scale_range=(0.1, 10.0) if "per_token" in dtype else None)
    g = GpuRun(wl).write_cache().attention()         # workspace entry point
    ref = g.out_f32()
    k = kvq()
    sched = k.get_scheduler_metadata(wl.num_req, wl.heads_q, wl.heads_kv, wl.head_dim,
                                     wl.seq_lens_t.numpy(), wl.query_start_loc.numpy(),
                                     wl.causal, wl.window, wl.kv_cache_dtype)
    assert 0 < sched.workspace_bytes <= k.STATIC_SCRATCH_BYTES
    first = _run_static(g, sched)
    second = _run_static(g, sched)
    sched.close()
    for out in (first, second):
        got = out.float().cpu().numpy()
        assert np.all(np.isfinite(got))
        assert_attention_close(got, ref, "static scratch vs workspace")
    assert torch.equal(first.view(torch.int16), second.view(torch.int16))


def test_static_scratch_refuses_oversized_schedule(cuda_device, monkeypatch):
    monkeypatch.setenv("KVQ_DECODE_WARPS", "100000")   # one chunk per warp: huge scratch
    k = kvq()
    L = np.full(64, 2048, np.int32)
    qsl = np.arange(65, dtype=np.int32)
    sched = k.get_scheduler_metadata(64, 32, 8, 128, L, qsl, True, 0, "fp8_e4m3")
    assert sched.workspace_bytes > k.STATIC_SCRATCH_BYTES
    dev = torch.device("cuda:0")
    q = torch.zeros((64, 32, 128), dtype=torch.bfloat16, device=dev)
    cache = torch.zeros((64 * 128, 16, 8, 128), dtype=torch.uint8, device=dev)
    lens = torch.from_numpy(L).to(dev)
    qsl_d = torch.from_numpy(qsl).to(dev)
    bt = torch.arange(64 * 128, dtype=torch.int32, device=dev).view(64, 128)
    out = torch.zeros_like(q)
    with pytest.raises(k.KvqError) as e:
        k.attention_with_kv_cache_static_scratch(sched, q, cache, cache, qsl_d, lens, bt,
                                                 0.088, True, 0, 0.0, 1.0, 1.0, out,
                                                 "fp8_e4m3", 8)
    assert e.value.status == k.E_WORKSPACE_TOO_SMALL
    sched.close()


def test_static_scratch_with_prefill_rows(cuda_device, monkeypatch):
    """A batch with prefill tiles and cut decode tiles: both kernels run
    from the static-scratch entry point and match the workspace one."""
    monkeypatch.setenv("KVQ_DECODE_WARPS", "48")
    wl = W.custom("noalloc-mixed", [1, 150, 1, 40], [1800, 400, 700, 40], 32, 8, 128, 16,
                  "int8_per_token_head", 78, token_scale_range=(0.1, 10.0))
    g = GpuRun(wl).write_cache().attention()
    assert g.sched_info["num_prefill_tiles"] > 0 and g.sched_info["num_merge_items"] > 0
    ref = g.out_f32()
    k = kvq()
    sched = k.get_scheduler_metadata(wl.num_req, wl.heads_q, wl.heads_kv, wl.head_dim,
                                     wl.seq_lens_t.numpy(), wl.query_start_loc.numpy(),
                                     wl.causal, wl.window, wl.kv_cache_dtype)
    out = _run_static(g, sched)
    sched.check_device()
    sched.close()
    got = out.float().cpu().numpy()
    assert_attention_close(got, ref, "static scratch, mixed batch")
    assert np.array_equal(got, ref)      # same kernels, same schedule: same bits
