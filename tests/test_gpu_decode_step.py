"""GPU parity of the fused decode step (kvq_decode_step): the step's new K/V
rows written into the caches, the plan built on the device from the
device's lengths, and split-KV attention -- one cooperative launch --, then
the merge of the cut tiles (a kernel of its own, a programmatic dependent).

vllm PR 50194 page, Key source snippet (get_scheduler_metadata feeding the
attention) and Breakdown item 1; vllm PR 39445 page, Breakdown items 1-3.
The caches it leaves must equal the oracle's writer bit for bit; the
output must match the oracle within the parity bound of tests/_harness.py.
A step captured once in a CUDA graph is replayed with other lengths, new
tokens and tables (the plan lives on the device), and must match the oracle
for those.
"""
import numpy as np
import pytest
import torch

from int8_kv_cache_reshape_gb300 import workloads as W

from _harness import (Guarded, GpuRun, assert_attention_close, kvq, oracle_cache,
                      oracle_reference)

pytestmark = pytest.mark.gpu


class Step:
    """A decode batch split into its cached context and the step's new rows
    (the last Q tokens of every request), on the device."""

    def __init__(self, wl, alibi=None, sinks=None, max_query_len=None):
        self.wl = wl
        self.g = GpuRun(wl, alibi_slopes=alibi, sinks=sinks)
        new = wl.new_token_mask()
        old_slots = wl.slot_mapping.clone()
        old_slots[new] = -1
        k = kvq()
        # the context written beforehand; the step writes the new rows
        k.reshape_and_cache(self.g.key, self.g.value, self.g.kc, self.g.vc, old_slots.to(self.g.dev),
                            wl.kv_cache_dtype, wl.k_scale, wl.v_scale)
        idx = torch.nonzero(new).flatten()
        dev = self.g.dev
        self.nkey = wl.key[idx].contiguous().to(dev)
        self.nval = wl.value[idx].contiguous().to(dev)
        self.nslot = wl.slot_mapping[idx].contiguous().to(dev)
        self.mql = max(wl.query_lens) if max_query_len is None else max_query_len
        nbytes = k.decode_step_workspace_size(wl.num_req, wl.heads_q, wl.heads_kv, wl.head_dim,
                                              wl.kv_cache_dtype, self.mql, alibi is not None)
        self.ws = Guarded((nbytes,), torch.uint8, 0, dev)

    def run(self):
        wl, g = self.wl, self.g
        kvq().decode_step(self.nkey, self.nval, self.nslot, g.kc, g.vc, g.q, g.qsl, g.sl, g.bt,
                          self.mql, wl.sm_scale, wl.window, wl.soft_cap, wl.k_scale, wl.v_scale,
                          g.out, self.ws.t, wl.kv_cache_dtype, wl.heads_kv,
                          alibi_slopes=g.alibi, sinks=g.sinks)
        return self

    def check(self, what):
        torch.cuda.synchronize()
        kvq().decode_step_check(self.ws.t)
        self.ws.check("decode-step workspace")
        self.g._kc.check("key cache")
        self.g._vc.check("value cache")
        self.g._out.check("output")
        wl = self.wl
        kc, vc = oracle_cache(wl)
        assert np.array_equal(self.g.kc.cpu().numpy(), kc), f"{what}: key cache"
        assert np.array_equal(self.g.vc.cpu().numpy(), vc), f"{what}: value cache"
        ref, bnd = oracle_reference(wl, kc, vc, alibi_slopes=self.g.alibi_np,
                                    sinks=self.g.sinks_np)
        return assert_attention_close(self.g.out_f32(), ref, what, bnd)


CASES = [("fp8_e4m3", 128, 32, 8, [1] * 12, 0, 0.0),
         ("fp8_e5m2", 128, 64, 8, [1] * 5, 300, 50.0),
         ("int8_per_token_head", 128, 32, 8, [1, 2, 4, 1, 3], 0, 0.0),
         ("fp8_per_token_head", 64, 8, 2, [2, 1, 4, 1], 100, 0.0),
         ("auto", 128, 16, 4, [1, 3, 1], 0, 20.0),
         ("fp8_e5m2_per_token_head", 256, 16, 2, [1, 2, 1], 0, 0.0)]


@pytest.mark.parametrize("dtype,D,hq,hkv,ql,window,cap", CASES)
def test_fused_step_matches_oracle(cuda_device, dtype, D, hq, hkv, ql, window, cap):
    rng = np.random.default_rng(len(ql) + D)
    sl = [int(x) for x in rng.integers(max(ql), 3000, len(ql))]
    sl[0] = ql[0]                          # a request that is all new tokens
    wl = W.custom(f"step-{dtype}-{D}", ql, sl, hq, hkv, D, 16, dtype, 600 + D + hq,
                  window=window, soft_cap=cap,
                  token_scale_range=(0.1, 10.0) if "per_token" in dtype else None)
    Step(wl).run().check(wl.name)


def test_fused_step_alibi_sinks(cuda_device):
    hq = 32
    wl = W.custom("step-ext", [1, 2, 1, 4], [2500, 700, 33, 1200], hq, 8, 128, 16, "fp8_e4m3", 610,
                  window=600)
    Step(wl, W.alibi_slopes(hq), W.sink_logits(hq, 611)).run().check("step alibi + sinks")


def test_fused_step_tiny_batch_and_big_batch(cuda_device):
    """Fewer chunks than warps (every segment at most one chunk) and many
    more (the decode batch's shape)."""
    wl = W.custom("step-tiny", [1, 1], [20, 47], 8, 2, 64, 16, "fp8_e4m3", 612)
    Step(wl).run().check("step tiny")
    wl = W.config(2)
    Step(wl).run().check("step decode batch")


def test_fused_step_graph_replay_with_new_lengths(cuda_device):
    """Capture one step, then change the device lengths, tables, slots, new
    rows and q in place (same capacities) and replay: the output follows."""
    hq, hkv, D = 32, 8, 128
    a = W.custom("replay-a", [1] * 6, [900, 40, 3200, 300, 1, 1500], hq, hkv, D, 16,
                 "int8_per_token_head", 620, token_scale_range=(0.1, 10.0), extra_blocks=200)
    st = Step(a)
    st.run()
    st.check("replay: direct")
    # a second batch of the same shape with other lengths, in the same pool
    b = W.custom("replay-b", [1] * 6, [1700, 2, 600, 3100, 45, 900], hq, hkv, D, 16,
                 "int8_per_token_head", 621, token_scale_range=(0.1, 10.0),
                 num_blocks=a.num_blocks)
    assert b.block_table.shape[1] <= a.block_table.shape[1]
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        st.run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        st.run()
    # swap in batch b: caches rewritten from scratch with b's context
    g = st.g
    sb = Step.__new__(Step)
    sb.wl = b
    sb.g = GpuRun(b)
    new = b.new_token_mask()
    old_slots = b.slot_mapping.clone()
    old_slots[new] = -1
    g.kc.fill_(0xCD)
    g.vc.fill_(0xCD)
    kvq().reshape_and_cache(sb.g.key, sb.g.value, g.kc, g.vc, old_slots.to(g.dev),
                            b.kv_cache_dtype, b.k_scale, b.v_scale)
    idx = torch.nonzero(new).flatten()
    st.nkey.copy_(b.key[idx])
    st.nval.copy_(b.value[idx])
    st.nslot.copy_(b.slot_mapping[idx])
    g.q.copy_(b.q)
    g.qsl.copy_(b.query_start_loc)
    g.sl.copy_(b.seq_lens_t)
    g.bt.fill_(-1)
    g.bt[:, :b.block_table.shape[1]].copy_(b.block_table)
    g.out.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    kvq().decode_step_check(st.ws.t)
    kc, vc = oracle_cache(b)
    assert np.array_equal(g.kc.cpu().numpy(), kc) and np.array_equal(g.vc.cpu().numpy(), vc)
    ref, bnd = oracle_reference(b, kc, vc)
    assert_attention_close(g.out.float().cpu().numpy(), ref, "replay with new lengths", bnd)


def test_fused_step_refuses_wide_tiles(cuda_device):
    with pytest.raises(kvq().KvqError) as e:
        kvq().decode_step_workspace_size(4, 32, 8, 128, "fp8_e4m3", 5)   # 5 * 4 rows > 16
    assert e.value.status == kvq().E_UNSUPPORTED


def test_fused_step_flags_device_lengths_beyond_the_bound(cuda_device):
    """A device query length above max_query_len: the request is skipped and
    the error word says so; the other requests still match the oracle."""
    wl = W.custom("step-bad", [1, 3, 1], [500, 90, 40], 16, 4, 128, 16, "fp8_e4m3", 630)
    st = Step(wl, max_query_len=2)
    st.run()
    torch.cuda.synchronize()
    with pytest.raises(kvq().KvqError) as e:
        kvq().decode_step_check(st.ws.t)
    assert e.value.status == kvq().E_INVALID_ARG
    kc, vc = oracle_cache(wl)
    toks = [0, 4]                                      # requests 0 and 2
    ref, bnd = oracle_reference(wl, kc, vc, tokens=toks)
    assert_attention_close(st.g.out_f32(toks), ref, "step: good requests", bnd)


def test_fused_step_from_host_buffers(cuda_device):
    """kvq_decode_step_host_io: the step's inputs packed in one pinned host
    buffer, copied to the device, the fused step run on views of the device
    copy, the output copied back to pinned host memory -- one C-ABI call.
    The caches and the host output equal the device-input step's, bit for
    bit, and match the oracle."""
    wl = W.custom("step-host-io", [1, 2, 1, 4, 1], [700, 333, 1, 2048, 96], 32, 8, 128, 16,
                  "fp8_e4m3", 907)
    ref_step = Step(wl).run()
    ref_step.check("device inputs")
    want_out = ref_step.g.out.view(torch.int16).cpu()
    want_kc, want_vc = ref_step.g.kc.cpu(), ref_step.g.vc.cpu()

    st = Step(wl)
    g = st.g
    parts = [g.q, st.nkey, st.nval, st.nslot, g.qsl, g.sl, g.bt]
    sizes = [t.numel() * t.element_size() for t in parts]
    offs, o = [], 0
    for n in sizes:
        offs.append(o)
        o += (n + 255) // 256 * 256
    h_in = torch.zeros(o, dtype=torch.uint8).pin_memory()
    for t, off, n in zip(parts, offs, sizes):
        h_in[off:off + n].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
    d_in = torch.full((o,), 0xA5, dtype=torch.uint8, device=g.dev)   # garbage until the copy
    views = [d_in[off:off + n].view(t.dtype).view(t.shape) for t, off, n in zip(parts, offs, sizes)]
    q, nkey, nval, nslot, qsl, sl, bt = views
    h_out = torch.zeros(g.out.shape, dtype=torch.bfloat16).pin_memory()
    out_bytes = g.out.numel() * g.out.element_size()
    call = kvq().prepare_decode_step_host_io(
        h_in, d_in, h_out, out_bytes, nkey, nval, nslot, g.kc, g.vc, q, qsl, sl, bt, st.mql,
        wl.sm_scale, wl.window, wl.soft_cap, wl.k_scale, wl.v_scale, g.out, st.ws.t,
        wl.kv_cache_dtype, wl.heads_kv)
    call()                                     # returns with the output on the host
    assert torch.equal(h_out.view(torch.int16), want_out)
    assert torch.equal(g.kc.cpu(), want_kc) and torch.equal(g.vc.cpu(), want_vc)
    st.check("host inputs")
    # a second call from the same buffers gives the same output (the
    # workspace is left ready; the cache rows are rewritten with equal bytes)
    h_out.zero_()
    call()
    assert torch.equal(h_out.view(torch.int16), want_out)


def test_fused_step_output_straight_to_host(cuda_device):
    """kvq_decode_step_host_io with out NULL: the kernels store the output
    rows into the pinned host buffer through its device mapping (no copy
    after the step); the rows equal the device-output step's."""
    wl = W.custom("step-host-out", [1, 3, 1, 2], [1500, 900, 33, 4000], 32, 8, 128, 16,
                  "int8_per_token_head", 911, token_scale_range=(0.1, 10.0))
    ref_step = Step(wl).run()
    ref_step.check("device output")
    want_out = ref_step.g.out.view(torch.int16).cpu()
    st = Step(wl)
    g = st.g
    h_in = torch.zeros(256, dtype=torch.uint8).pin_memory()
    d_in = torch.zeros(256, dtype=torch.uint8, device=g.dev)
    h_out = torch.full(g.out.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    call = kvq().prepare_decode_step_host_io(
        h_in, d_in, h_out, 0, st.nkey, st.nval, st.nslot, g.kc, g.vc, g.q, g.qsl, g.sl, g.bt, st.mql,
        wl.sm_scale, wl.window, wl.soft_cap, wl.k_scale, wl.v_scale, None, st.ws.t,
        wl.kv_cache_dtype, wl.heads_kv)
    call()
    assert torch.equal(h_out.view(torch.int16), want_out)
    assert torch.equal(g.kc.cpu(), ref_step.g.kc.cpu()) and torch.equal(g.vc.cpu(), ref_step.g.vc.cpu())
    kvq().decode_step_check(st.ws.t)


def _packed_inputs(st, extra_tail, host):
    """The step's inputs packed 256-byte aligned into one host buffer (plus
    `extra_tail` bytes of noise at the end), and a garbage-filled device
    buffer with views at the same offsets.  host: "pinned", "pinned+8" (a
    pinned buffer starting 8 bytes past a 16-byte boundary) or "pageable"."""
    g = st.g
    parts = [g.q, st.nkey, st.nval, st.nslot, g.qsl, g.sl, g.bt]
    sizes = [t.numel() * t.element_size() for t in parts]
    offs, o = [], 0
    for n in sizes:
        offs.append(o)
        o += (n + 255) // 256 * 256
    gen = torch.Generator().manual_seed(17)
    h_in = torch.randint(0, 256, (o + extra_tail + 8,), dtype=torch.uint8, generator=gen)
    if host != "pageable":
        h_in = h_in.pin_memory()
    h_in = h_in[8:] if host == "pinned+8" else h_in[:o + extra_tail]
    for t, off, n in zip(parts, offs, sizes):
        h_in[off:off + n].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
    d_in = torch.full((o + extra_tail,), 0xA5, dtype=torch.uint8, device=g.dev)
    views = [d_in[off:off + n].view(t.dtype).view(t.shape) for t, off, n in zip(parts, offs, sizes)]
    return h_in, d_in, views


@pytest.mark.parametrize("host", ["pinned", "pinned+8", "pageable"])
def test_fused_step_host_inputs_reach_the_device(cuda_device, host):
    """kvq_decode_step_host_io's two ways in: pinned host_in on a 16-byte
    boundary is read by the fused kernel through its device mapping and
    copied to dev_in by the kernel's CTAs (a size with a 13-byte tail beyond
    the last 16-byte word); host_in 8 bytes off that boundary goes through
    one copy first; pageable host_in takes either way, depending on whether
    the device addresses pageable memory.  Each time dev_in ends up equal to
    host_in byte for byte, and the caches and the host output equal the
    device-input step's."""
    wl = W.custom("step-host-stage", [1, 1, 2, 1, 3, 1], [64, 1200, 480, 17, 3000, 256], 32, 8, 128,
                  16, "fp8_e5m2", 913)
    ref_step = Step(wl).run()
    ref_step.check("device inputs")
    want_out = ref_step.g.out.view(torch.int16).cpu()
    want_kc, want_vc = ref_step.g.kc.cpu(), ref_step.g.vc.cpu()
    st = Step(wl)
    g = st.g
    h_in, d_in, views = _packed_inputs(st, 13, host)
    q, nkey, nval, nslot, qsl, sl, bt = views
    h_out = torch.zeros(g.out.shape, dtype=torch.bfloat16).pin_memory()
    call = kvq().prepare_decode_step_host_io(
        h_in, d_in, h_out, 0, nkey, nval, nslot, g.kc, g.vc, q, qsl, sl, bt, st.mql,
        wl.sm_scale, wl.window, wl.soft_cap, wl.k_scale, wl.v_scale, None, st.ws.t,
        wl.kv_cache_dtype, wl.heads_kv)
    call()
    assert torch.equal(d_in.cpu(), h_in)
    assert torch.equal(h_out.view(torch.int16), want_out)
    assert torch.equal(g.kc.cpu(), want_kc) and torch.equal(g.vc.cpu(), want_vc)
    kvq().decode_step_check(st.ws.t)


def _pack_into(h_in, offs, tensors):
    for t, off in zip(tensors, offs):
        n = t.numel() * t.element_size()
        h_in[off:off + n].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))


def test_fused_step_graph_from_host_buffers(cuda_device):
    """kvq_decode_step_graph_create / _launch: the host-buffer step captured
    once (inputs staged by the fused kernel from pinned host memory, output
    stored straight into pinned host memory).  A launch equals the one-call
    step bit for bit; after a second batch's rows, lengths, slots and table
    are written into the same pinned buffer (same capacities) and the caches
    are refilled with its context, a launch of the same graph matches the
    oracle for that batch."""
    hq, hkv, D = 32, 8, 128
    # dynamic per-token-head scales: the captured step's per-tensor scales
    # would be a's, not b's
    a = W.custom("graph-io-a", [1, 2, 1, 1, 3, 1], [900, 40, 3200, 300, 7, 1500], hq, hkv, D, 16,
                 "int8_per_token_head", 630, token_scale_range=(0.1, 10.0), extra_blocks=200)
    ref_step = Step(a).run()
    ref_step.check("graph io: device inputs")
    want_out = ref_step.g.out.view(torch.int16).cpu()
    st = Step(a)
    g = st.g
    parts = [g.q, st.nkey, st.nval, st.nslot, g.qsl, g.sl, g.bt]
    sizes = [t.numel() * t.element_size() for t in parts]
    offs, o = [], 0
    for n in sizes:
        offs.append(o)
        o += (n + 255) // 256 * 256
    h_in = torch.zeros(o, dtype=torch.uint8).pin_memory()
    _pack_into(h_in, offs, parts)
    d_in = torch.full((o,), 0xA5, dtype=torch.uint8, device=g.dev)
    q, nkey, nval, nslot, qsl, sl, bt = [d_in[off:off + n].view(t.dtype).view(t.shape)
                                         for t, off, n in zip(parts, offs, sizes)]
    h_out = torch.full(g.out.shape, float("nan"), dtype=torch.bfloat16).pin_memory()
    step = kvq().decode_step_graph(h_in, d_in, h_out, 0, nkey, nval, nslot, g.kc, g.vc, q, qsl,
                                   sl, bt, st.mql, a.sm_scale, a.window, a.soft_cap, a.k_scale,
                                   a.v_scale, None, st.ws.t, a.kv_cache_dtype, a.heads_kv)
    try:
        step()
        assert torch.equal(h_out.view(torch.int16), want_out)
        assert torch.equal(d_in.cpu(), h_in)
        assert torch.equal(g.kc.cpu(), ref_step.g.kc.cpu())
        assert torch.equal(g.vc.cpu(), ref_step.g.vc.cpu())
        kvq().decode_step_check(st.ws.t)

        # batch b: same request count and query lengths, other context lengths
        b = W.custom("graph-io-b", [1, 2, 1, 1, 3, 1], [1700, 2, 600, 3100, 45, 900], hq, hkv, D,
                     16, "int8_per_token_head", 631, token_scale_range=(0.1, 10.0),
                     num_blocks=a.num_blocks)
        assert b.block_table.shape[1] <= a.block_table.shape[1]
        gb = GpuRun(b)
        new = b.new_token_mask()
        old_slots = b.slot_mapping.clone()
        old_slots[new] = -1
        g.kc.fill_(0xCD)
        g.vc.fill_(0xCD)
        kvq().reshape_and_cache(gb.key, gb.value, g.kc, g.vc, old_slots.to(g.dev),
                                b.kv_cache_dtype, b.k_scale, b.v_scale)
        torch.cuda.synchronize()
        idx = torch.nonzero(new).flatten()
        bt_b = torch.full(tuple(g.bt.shape), -1, dtype=torch.int32)
        bt_b[:, :b.block_table.shape[1]] = b.block_table
        _pack_into(h_in, offs, [b.q, b.key[idx], b.value[idx], b.slot_mapping[idx],
                                b.query_start_loc, b.seq_lens_t, bt_b])
        h_out.fill_(float("nan"))
        step()
        kvq().decode_step_check(st.ws.t)
        kc, vc = oracle_cache(b)
        assert np.array_equal(g.kc.cpu().numpy(), kc) and np.array_equal(g.vc.cpu().numpy(), vc)
        ref, bnd = oracle_reference(b, kc, vc)
        assert_attention_close(h_out.float().numpy(), ref, "graph replay with new host inputs", bnd)
    finally:
        step.close()


def test_fused_step_graph_refuses_inputs_it_cannot_stage(cuda_device):
    """A host_in the fused kernel cannot stage (here: 8 bytes off a 16-byte
    boundary) would need a copy inside the graph: KVQ_E_UNSUPPORTED, and
    nothing is created."""
    wl = W.custom("graph-io-unaligned", [1, 1], [64, 200], 8, 2, 64, 16, "fp8_e4m3", 632)
    st = Step(wl)
    g = st.g
    h_in = torch.zeros(4096 + 8, dtype=torch.uint8).pin_memory()[8:]
    d_in = torch.zeros(4096, dtype=torch.uint8, device=g.dev)
    h_out = torch.zeros(g.out.shape, dtype=torch.bfloat16).pin_memory()
    with pytest.raises(kvq().KvqError) as e:
        kvq().decode_step_graph(h_in, d_in, h_out, 0, st.nkey, st.nval, st.nslot, g.kc, g.vc, g.q,
                                g.qsl, g.sl, g.bt, st.mql, wl.sm_scale, wl.window, wl.soft_cap,
                                wl.k_scale, wl.v_scale, None, st.ws.t, wl.kv_cache_dtype,
                                wl.heads_kv)
    assert e.value.status == kvq().E_UNSUPPORTED
