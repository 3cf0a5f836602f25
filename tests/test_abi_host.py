"""Host-side tests of the C ABI (no GPU): the library loads and exports
every function include/kvq.h declares; dtype parsing, row sizes, argument
checks and the scheduler's plan (built host-only when no device is present).

The scheduler and its checks restate the vllm PR 50194 page (Breakdown
item 1, Key source snippet): the plan is sized from the KV cache dtype, and
a runtime that disagrees with the plan is refused.
"""
import ctypes
import subprocess

import numpy as np
import pytest

from int8_kv_cache_reshape_gb300 import build as kbuild

kbuild.build()
from int8_kv_cache_reshape_gb300 import kvq  # noqa: E402


def test_every_declared_function_is_exported():
    names = kvq.declared_functions()
    assert {"kvq_reshape_and_cache", "kvq_get_scheduler_metadata",
            "kvq_attention_with_kv_cache", "kvq_sched_destroy"} <= set(names)
    for n in names:
        assert hasattr(kvq.lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", kvq.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(names) <= exported
    # nothing but the ABI is exported
    assert {n for n in exported if n.startswith("kvq")} == set(names)


@pytest.mark.parametrize("s,want", [("auto", 0), (None, 0), ("", 0), ("fp8", 1),
                                    ("fp8_e4m3", 1), ("fp8_e5m2", 2),
                                    ("int8_per_token_head", 3), ("fp8_per_token_head", 4),
                                    ("fp8_e5m2_per_token_head", 5)])
def test_parse_dtype(s, want):
    assert kvq.parse_kv_cache_dtype(s) == want


def test_parse_dtype_rejects_unknown():
    with pytest.raises(kvq.KvqError) as e:
        kvq.parse_kv_cache_dtype("fp8_e3m4")
    assert e.value.status == kvq.E_INVALID_ARG


def test_row_bytes():
    assert kvq.cache_row_bytes("auto", 128) == 256
    assert kvq.cache_row_bytes("fp8_e4m3", 128) == 128
    assert kvq.cache_row_bytes("fp8_e5m2", 256) == 256
    assert kvq.cache_row_bytes("int8_per_token_head", 128) == 144
    assert kvq.cache_row_bytes("fp8_per_token_head", 64) == 80
    assert kvq.cache_row_bytes("fp8_e5m2_per_token_head", 128) == 144
    with pytest.raises(kvq.KvqError):
        kvq.cache_row_bytes("fp8_e4m3", 100)


def test_status_strings():
    for s in (0, -1, -2, -3, -4, -5, -6, -7):
        assert kvq.status_string(s) and kvq.status_string(s) != "unknown status"
    assert kvq.status_string(-99) == "unknown status"


def _rac(**kw):
    """Call kvq_reshape_and_cache with fake (never dereferenced) pointers;
    only argument checks that fail before any launch are exercised."""
    a = dict(key=256, value=512, T=4, ks=256, vs=256, H=2, D=128, kc=1024,
             vc=2048, nb=4, bs=16, slots=4096, dt=1, k=1.0, v=1.0)
    a.update(kw)
    return kvq.lib.kvq_reshape_and_cache(
        ctypes.c_void_p(a["key"]), ctypes.c_void_p(a["value"]), a["T"], a["ks"], a["vs"],
        a["H"], a["D"], ctypes.c_void_p(a["kc"]), ctypes.c_void_p(a["vc"]), a["nb"], a["bs"],
        ctypes.c_void_p(a["slots"]), a["dt"], a["k"], a["v"], None)


@pytest.mark.parametrize("kw,want", [
    (dict(D=96), kvq.E_UNSUPPORTED), (dict(dt=9), kvq.E_INVALID_ARG),
    (dict(T=-1), kvq.E_INVALID_ARG), (dict(key=0), kvq.E_INVALID_ARG),
    (dict(ks=255), kvq.E_INVALID_ARG), (dict(ks=100), kvq.E_INVALID_ARG),
    (dict(key=264), kvq.E_INVALID_ARG), (dict(kc=1032), kvq.E_INVALID_ARG),
    (dict(k=0.0), kvq.E_INVALID_ARG), (dict(v=float("nan")), kvq.E_INVALID_ARG),
    (dict(k=float("inf")), kvq.E_INVALID_ARG), (dict(H=0), kvq.E_INVALID_ARG),
    (dict(T=0), kvq.OK),
])
def test_reshape_and_cache_argument_checks(kw, want):
    assert _rac(**kw) == want


def _sched(seq_lens, query_lens, hq=32, hkv=8, D=128, dtype="fp8_e4m3", causal=True,
           window=0):
    qsl = np.concatenate([[0], np.cumsum(query_lens)]).astype(np.int32)
    return kvq.get_scheduler_metadata(len(seq_lens), hq, hkv, D, np.array(seq_lens, np.int32),
                                      qsl, causal, window, dtype)


def test_scheduler_decode_plan_covers_every_chunk(monkeypatch):
    """Stream decomposition: every (request, kv head) tile's 16-token chunks
    are streamed exactly once, cut among the warps; each warp boundary cuts
    at most one tile."""
    monkeypatch.delenv("KVQ_DECODE_WARPS", raising=False)
    rng = np.random.default_rng(0)
    L = rng.integers(1024, 4097, 64)
    s = _sched(L, [1] * 64)
    info = s.info()
    assert info["kv_elem_bytes"] == 1 and info["row_bytes"] == 128
    assert info["total_query_tokens"] == 64
    assert info["num_tiles"] == 64 * 8
    assert info["num_chunks"] == int(np.sum(-(-L // 16))) * 8
    assert info["num_decode_warps"] == 152 * 4 * 4        # all SMs, 4 CTAs of 4 warps
    assert info["num_pieces"] <= info["num_tiles"] + info["num_decode_warps"] - 1
    assert info["num_merge_items"] <= info["num_tiles"]
    # the decode kernel, then the merge of the cut tiles
    assert info["num_kernel_launches"] == 1 + (info["num_merge_items"] > 0)
    # every cut tile keeps one partial row per (piece, row): 4 rows (G = 4)
    split_pieces = info["num_pieces"] - (info["num_tiles"] - info["num_merge_items"])
    assert info["workspace_bytes"] >= split_pieces * 4 * (128 + 1) * 4
    s.close()


def test_scheduler_sizes_follow_kv_element_size():
    """The vllm PR 50194 page's bug: scratch sized from the query's element
    size instead of the cache's.  The plan's row size and shared memory
    follow the cache dtype."""
    a = _sched([300], [1], dtype="fp8_e4m3").info()
    b = _sched([300], [1], dtype="int8_per_token_head").info()
    assert a["row_bytes"] == 128 and b["row_bytes"] == 144
    assert a["kv_elem_bytes"] == b["kv_elem_bytes"] == 1
    # bytes streamed per 16-token chunk: 2 * 16 * (D codes) [+ scale tails]
    assert a["decode_chunk_bytes"] == 2 * 16 * 128
    assert b["decode_chunk_bytes"] == 2 * 16 * 128 + 32 * 16
    for dt in ("fp8_e4m3", "int8_per_token_head"):
        for D in (64, 128, 256):
            assert _sched([300], [1], dtype=dt, D=D).info()["decode_smem_bytes"] <= 227 * 1024


def test_forced_warp_counts(monkeypatch):
    T = 8 * (63 + 3)                      # chunks of L = 1000 and L = 37, 8 kv heads
    monkeypatch.setenv("KVQ_DECODE_WARPS", "4")
    info = _sched([1000, 37], [1, 1]).info()
    assert info["num_decode_warps"] == 4 and info["num_chunks"] == T
    assert info["max_splits"] <= 2
    monkeypatch.setenv("KVQ_DECODE_WARPS", "100000")   # one chunk per warp
    info = _sched([1000, 37], [1, 1]).info()
    assert info["num_decode_warps"] == T
    assert info["max_splits"] == 63 and info["num_merge_items"] == 16
    assert info["num_pieces"] == T


def test_prefill_rows_make_tensor_core_tiles():
    info = _sched([100, 50], [40, 1], hq=32, hkv=8).info()   # 160 rows + 4 rows per kv head
    assert info["num_prefill_tiles"] == 8 * 2                 # 128 + 32 rows per kv head
    assert info["num_tiles"] == 8                             # the decode's 4-row tiles
    # prefill + one decode class (+ the merge of its cut tiles)
    assert info["num_kernel_launches"] == 2 + (info["num_merge_items"] > 0)
    assert info["prefill_smem_bytes"] > 0


def test_prefill_tiles_and_decode_boundary():
    # 16 rows per kv head stays a decode tile; 17 rows become a prefill tile
    # (a build with CTA pairs gives each single tile an empty partner; bf16
    # rows always run on single CTAs).
    info = _sched([64, 64], [8, 9], hq=16, hkv=8).info()      # G=2: 16 and 18 rows
    cg = info["prefill_cta_group"]
    assert cg in (1, 2)
    assert info["num_prefill_tiles"] == cg * 8
    assert info["num_tiles"] == 8
    assert info["num_kernel_launches"] == 2 + (info["num_merge_items"] > 0)
    info = _sched([64, 64], [8, 9], hq=16, hkv=8, dtype="auto").info()
    assert info["num_prefill_tiles"] == 8 and info["prefill_cta_group"] == 1
    info = _sched([64], [64], hq=8, hkv=8).info()             # only prefill
    assert info["num_prefill_tiles"] == cg * 8 and info["num_tiles"] == 0
    assert info["num_kernel_launches"] == 1 and info["workspace_bytes"] == 0


@pytest.mark.parametrize("kw,want", [
    (dict(hq=30, hkv=8), kvq.E_UNSUPPORTED), (dict(D=96), kvq.E_UNSUPPORTED),
    (dict(causal=False, window=8), kvq.E_INVALID_ARG),
])
def test_scheduler_rejects(kw, want):
    with pytest.raises(kvq.KvqError) as e:
        _sched([10, 20], [1, 2], **kw)
    assert e.value.status == want


def test_scheduler_rejects_more_queries_than_keys():
    with pytest.raises(kvq.KvqError) as e:
        _sched([3], [4])
    assert e.value.status == kvq.E_INVALID_ARG


def test_empty_batch_and_zero_query_requests():
    s = _sched([], [])
    assert s.info()["num_tiles"] == 0 and s.workspace_bytes == 0
    s = _sched([40, 0], [0, 0])
    assert s.info()["num_tiles"] == 0 and s.info()["num_kernel_launches"] == 0


def test_attention_refuses_mismatched_schedule():
    s = _sched([64], [1], dtype="fp8_e4m3")
    f = kvq.lib.kvq_attention_with_kv_cache
    args = lambda hq, hkv, D, dt, causal=1, window=0: (
        s.handle, hq, hkv, D, dt, *([ctypes.c_void_p(256)] * 6), 4, 16, 8, 0.1, causal,
        window, 0.0, None, None, 1.0, 1.0, ctypes.c_void_p(256), None, 0, None)
    assert f(*args(32, 8, 128, 3)) == kvq.E_SCHED_MISMATCH     # other dtype
    assert f(*args(32, 8, 64, 1)) == kvq.E_SCHED_MISMATCH      # other head_dim
    assert f(*args(16, 8, 128, 1)) == kvq.E_SCHED_MISMATCH     # other heads
    assert f(*args(32, 8, 128, 1, causal=0)) == kvq.E_SCHED_MISMATCH
    assert f(*args(32, 8, 128, 1, window=5)) == kvq.E_SCHED_MISMATCH


def test_decode_step_shape_checks_come_first():
    """kvq_decode_step_workspace_size refuses bad shapes on the host before
    it asks the device anything (no GPU needed for these)."""
    f = kvq.lib.kvq_decode_step_workspace_size
    out = ctypes.c_size_t()
    assert f(4, 32, 8, 128, 1, 5, 0, ctypes.byref(out)) == kvq.E_UNSUPPORTED   # 20 rows
    assert f(4, 30, 8, 128, 1, 1, 0, ctypes.byref(out)) == kvq.E_UNSUPPORTED   # GQA ratio
    assert f(4, 32, 8, 96, 1, 1, 0, ctypes.byref(out)) == kvq.E_UNSUPPORTED    # head_dim
    assert f(-1, 32, 8, 128, 1, 1, 0, ctypes.byref(out)) == kvq.E_INVALID_ARG
    assert f(4, 32, 8, 128, 1, 0, 0, ctypes.byref(out)) == kvq.E_INVALID_ARG   # max_query_len
    assert f(4, 32, 8, 128, 9, 1, 0, ctypes.byref(out)) == kvq.E_INVALID_ARG   # dtype
    assert f(4, 32, 8, 128, 1, 1, 0, None) == kvq.E_INVALID_ARG
    assert kvq.lib.kvq_decode_step_check(None) == kvq.E_INVALID_ARG


def _step_args():
    """kvq_decode_step's arguments after the host-buffer ones, with NULL
    pointers (never dereferenced: the calls below are refused first)."""
    return [4, 32, 8, 128, 1, None, None, 0, 1024, 1024, None, None, None, 16, 16, None, None,
            None, None, 1, 1, 0.088, 0, 0.0, None, None, 1.0, 1.0, None, None, 0]


def test_host_io_checks_its_buffers_before_any_device_call():
    """kvq_decode_step_host_io: a NULL buffer with a nonzero size is refused
    on the host (no GPU needed)."""
    f = kvq.lib.kvq_decode_step_host_io
    h = ctypes.create_string_buffer(64)
    assert f(None, ctypes.c_void_p(256), 64, None, 0, *_step_args(), None) == kvq.E_INVALID_ARG
    assert f(h, None, 64, None, 0, *_step_args(), None) == kvq.E_INVALID_ARG
    # out given, out_bytes > 0, host_out NULL
    args = _step_args()
    args[-3] = ctypes.c_void_p(256)
    assert f(None, None, 0, None, 16, *args, None) == kvq.E_INVALID_ARG


def test_step_graph_entry_points_refuse_null_handles():
    """kvq_decode_step_graph_create needs somewhere to put the graph, and
    refuses NULL buffers with sizes as host_io does; launch refuses a NULL
    graph; destroy accepts NULL."""
    create = kvq.lib.kvq_decode_step_graph_create
    h = ctypes.c_void_p()
    assert create(None, None, 0, None, 0, *_step_args(), None) == kvq.E_INVALID_ARG
    assert create(None, ctypes.c_void_p(256), 64, None, 0, *_step_args(),
                  ctypes.byref(h)) == kvq.E_INVALID_ARG
    assert h.value is None
    assert kvq.lib.kvq_decode_step_graph_launch(None, None) == kvq.E_INVALID_ARG
    kvq.lib.kvq_decode_step_graph_destroy(None)
