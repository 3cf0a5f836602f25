"""A serving step captured in a CUDA graph.

reshape_and_cache of the step's tokens plus attention_with_kv_cache over a
batch with cut decode tiles and prefill tiles, captured once and replayed:
the replays give the same bits as the direct calls, and match the oracle
within the parity tolerance of tests/_harness.py.  Neither call
synchronises with the host, allocates, or keeps state between calls that a
replay would repeat wrongly (cut decode tiles are merged by a kernel of
their own; the prefill's tensor maps are kernel arguments).
"""
import pytest
import torch

from int8_kv_cache_reshape_gb300 import workloads as W

from _harness import GpuRun, assert_attention_close, kvq, oracle_cache, oracle_reference

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["fp8_e4m3", "int8_per_token_head"])
def test_step_replayed_from_a_cuda_graph(cuda_device, monkeypatch, dtype):
    monkeypatch.setenv("KVQ_DECODE_WARPS", "48")     # cut tiles: the merge path runs
    wl = W.custom("graph", [1, 150, 1, 40], [1800, 400, 700, 40], 32, 8, 128, 16, dtype, 81,
                  token_scale_range=(0.1, 10.0) if "per_token" in dtype else None)
    g = GpuRun(wl)
    k = kvq()
    sched = k.get_scheduler_metadata(wl.num_req, wl.heads_q, wl.heads_kv, wl.head_dim,
                                     wl.seq_lens_t.numpy(), wl.query_start_loc.numpy(),
                                     wl.causal, wl.window, wl.kv_cache_dtype)
    info = sched.info()
    assert info["num_prefill_tiles"] > 0 and info["num_merge_items"] > 0
    ws = torch.empty(max(1, sched.workspace_bytes), dtype=torch.uint8, device=g.q.device)

    def step(out):
        k.reshape_and_cache(g.key, g.value, g.kc, g.vc, g.slots, dtype, wl.k_scale, wl.v_scale)
        k.attention_with_kv_cache(sched, g.q, g.kc, g.vc, g.qsl, g.sl, g.bt, wl.sm_scale,
                                  wl.causal, wl.window, wl.soft_cap, wl.k_scale, wl.v_scale,
                                  out, ws, dtype, wl.heads_kv)

    direct = torch.full_like(g.out, float("nan"))
    step(direct)
    torch.cuda.synchronize()
    graphed = torch.full_like(g.out, float("nan"))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(graphed)                                   # warm-up off the default stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graphed.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(graphed)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    sched.check_device()
    sched.close()
    assert torch.equal(direct.view(torch.int16), graphed.view(torch.int16))
    kc, vc = oracle_cache(wl)
    ref, bnd = oracle_reference(wl, kc, vc)
    assert_attention_close(graphed.float().cpu().numpy(), ref, "graph replay", bnd)
