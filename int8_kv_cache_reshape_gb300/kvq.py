"""ctypes binding of libkvq.so (include/kvq.h) -- argument marshalling only.

Every function here turns tensors into pointers and sizes and calls the C
ABI of the same name; all computation runs in the library's CUDA kernels.
Importing this module loads the library and raises if it was not built
(``python -m int8_kv_cache_reshape_gb300.build`` or ``__graft_entry__.build()``):
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# KVQ_LIBRARY selects another build of the library (the bounds-checked
# libkvq_checked.so); default libkvq.so next to this file.
LIB_PATH = os.environ.get("KVQ_LIBRARY") or os.path.join(_HERE, "libkvq.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "kvq.h")

OK = 0
E_INVALID_ARG, E_UNSUPPORTED, E_SCHED_MISMATCH = -1, -2, -3
E_WORKSPACE_TOO_SMALL, E_CUDA, E_NO_MEMORY, E_TIMEOUT = -4, -5, -6, -7

DTYPES = {"auto": 0, "fp8_e4m3": 1, "fp8_e5m2": 2, "int8_per_token_head": 3,
          "fp8_per_token_head": 4, "fp8_e5m2_per_token_head": 5}


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{os.path.basename(LIB_PATH)} is not built ({LIB_PATH}); run "
                      "int8_kv_cache_reshape_gb300.build.build() first")

lib = ctypes.CDLL(LIB_PATH)


class SchedInfo(ctypes.Structure):
    _fields_ = [("num_req", ctypes.c_int), ("heads_q", ctypes.c_int),
                ("heads_kv", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("dtype", ctypes.c_int), ("kv_elem_bytes", ctypes.c_int),
                ("row_bytes", ctypes.c_int), ("causal", ctypes.c_int),
                ("window", ctypes.c_int),
                ("num_tiles", ctypes.c_int64),
                ("num_pieces", ctypes.c_int64),
                ("num_merge_items", ctypes.c_int64),
                ("num_chunks", ctypes.c_int64),
                ("num_decode_warps", ctypes.c_int64),
                ("max_splits", ctypes.c_int64),
                ("total_query_tokens", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_size_t),
                ("decode_smem_bytes", ctypes.c_size_t),
                ("decode_chunk_bytes", ctypes.c_size_t),
                ("num_prefill_tiles", ctypes.c_int64),
                ("prefill_smem_bytes", ctypes.c_size_t),
                ("num_kernel_launches", ctypes.c_int64),
                ("prefill_cta_group", ctypes.c_int64)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


_c = ctypes
_p = ctypes.c_void_p
lib.kvq_status_string.restype = _c.c_char_p
lib.kvq_status_string.argtypes = [_c.c_int]
lib.kvq_parse_kv_cache_dtype.restype = _c.c_int
lib.kvq_parse_kv_cache_dtype.argtypes = [_c.c_char_p, _c.POINTER(_c.c_int)]
lib.kvq_cache_row_bytes.restype = _c.c_int
lib.kvq_cache_row_bytes.argtypes = [_c.c_int, _c.c_int, _c.POINTER(_c.c_size_t)]
lib.kvq_reshape_and_cache.restype = _c.c_int
lib.kvq_reshape_and_cache.argtypes = [
    _p, _p, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int, _c.c_int, _p, _p,
    _c.c_int64, _c.c_int, _p, _c.c_int, _c.c_float, _c.c_float, _p]
lib.kvq_get_scheduler_metadata.restype = _c.c_int
lib.kvq_get_scheduler_metadata.argtypes = [
    _c.c_int, _c.c_int, _c.c_int, _c.c_int, _p, _p, _c.c_int, _c.c_int,
    _c.c_int, _c.POINTER(_p), _c.POINTER(_c.c_size_t)]
lib.kvq_attention_with_kv_cache.restype = _c.c_int
lib.kvq_attention_with_kv_cache.argtypes = [
    _p, _c.c_int, _c.c_int, _c.c_int, _c.c_int, _p, _p, _p, _p, _p, _p,
    _c.c_int, _c.c_int, _c.c_int64, _c.c_float, _c.c_int, _c.c_int,
    _c.c_float, _p, _p, _c.c_float, _c.c_float, _p, _p, _c.c_size_t, _p]
lib.kvq_attention_with_kv_cache_static_scratch.restype = _c.c_int
lib.kvq_attention_with_kv_cache_static_scratch.argtypes = [
    _p, _c.c_int, _c.c_int, _c.c_int, _c.c_int, _p, _p, _p, _p, _p, _p,
    _c.c_int, _c.c_int, _c.c_int64, _c.c_float, _c.c_int, _c.c_int,
    _c.c_float, _p, _p, _c.c_float, _c.c_float, _p, _p]
STATIC_SCRATCH_BYTES = 16 << 20
lib.kvq_decode_step.restype = _c.c_int
lib.kvq_decode_step.argtypes = [
    _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int, _p, _p, _c.c_int64, _c.c_int64,
    _c.c_int64, _p, _p, _p, _c.c_int64, _c.c_int, _p, _p, _p, _p, _c.c_int, _c.c_int,
    _c.c_float, _c.c_int, _c.c_float, _p, _p, _c.c_float, _c.c_float, _p, _p, _c.c_size_t, _p]
lib.kvq_decode_step_host_io.restype = _c.c_int
lib.kvq_decode_step_host_io.argtypes = [_p, _p, _c.c_size_t, _p, _c.c_size_t] + lib.kvq_decode_step.argtypes
lib.kvq_decode_step_graph_create.restype = _c.c_int
lib.kvq_decode_step_graph_create.argtypes = ([_p, _p, _c.c_size_t, _p, _c.c_size_t]
                                             + lib.kvq_decode_step.argtypes[:-1]
                                             + [_c.POINTER(_p)])
lib.kvq_decode_step_graph_launch.restype = _c.c_int
lib.kvq_decode_step_graph_launch.argtypes = [_p, _p]
lib.kvq_decode_step_graph_destroy.restype = None
lib.kvq_decode_step_graph_destroy.argtypes = [_p]
lib.kvq_decode_step_workspace_size.restype = _c.c_int
lib.kvq_decode_step_workspace_size.argtypes = [
    _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.c_int, _c.POINTER(_c.c_size_t)]
lib.kvq_decode_step_check.restype = _c.c_int
lib.kvq_decode_step_check.argtypes = [_p]
lib.kvq_sched_destroy.restype = None
lib.kvq_sched_destroy.argtypes = [_p]
lib.kvq_sched_check_device.restype = _c.c_int
lib.kvq_sched_check_device.argtypes = [_p]
lib.kvq_sched_get_info.restype = _c.c_int
lib.kvq_sched_get_info.argtypes = [_p, _c.POINTER(SchedInfo)]


class PlanSizes(ctypes.Structure):
    _fields_ = [("num_pieces", ctypes.c_int64), ("num_merges", ctypes.c_int64),
                ("num_prefill_tiles", ctypes.c_int64), ("num_chunks", ctypes.c_int64 * 2),
                ("num_warps", ctypes.c_int32 * 2), ("lockstep", ctypes.c_int32 * 2)]


# numpy layouts of kvq_plan_piece_t, kvq_plan_merge_t, kvq_plan_prefill_tile_t
PLAN_PIECE = np.dtype([(n, np.int32) for n in (
    "launch", "req", "kv_head", "row0", "nrows", "part", "merge", "key_lo", "key_hi", "flat0",
    "chunk0", "nchunks")])
PLAN_MERGE = np.dtype([(n, np.int32) for n in ("req", "kv_head", "row0", "nrows", "part",
                                                "nsplits")])
PLAN_PREFILL = np.dtype([(n, np.int32) for n in ("req", "kv_head", "row0", "nrows", "key_lo",
                                                  "key_hi")])
lib.kvq_sched_get_plan_sizes.restype = _c.c_int
lib.kvq_sched_get_plan_sizes.argtypes = [_p, _c.POINTER(PlanSizes)]
lib.kvq_sched_export_plan.restype = _c.c_int
lib.kvq_sched_export_plan.argtypes = [_p, _p, _c.c_int64, _p, _c.c_int64, _p, _c.c_int64, _p,
                                      _c.c_int64]


def declared_functions() -> list:
    """Names of the functions include/kvq.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_\w+)\s*\(", text)))


def status_string(status: int) -> str:
    return lib.kvq_status_string(int(status)).decode()


def _check(rc: int, what: str) -> None:
    if rc != OK:
        raise KvqError(rc, what)


def _ptr(t):
    return None if t is None else _p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return _p(getattr(stream, "cuda_stream", stream))


def parse_kv_cache_dtype(s) -> int:
    out = _c.c_int()
    _check(lib.kvq_parse_kv_cache_dtype(None if s is None else s.encode(), _c.byref(out)),
           "kvq_parse_kv_cache_dtype")
    return out.value


def cache_row_bytes(kv_cache_dtype, head_dim: int) -> int:
    dt = parse_kv_cache_dtype(kv_cache_dtype) if isinstance(kv_cache_dtype, str) else kv_cache_dtype
    out = _c.c_size_t()
    _check(lib.kvq_cache_row_bytes(dt, head_dim, _c.byref(out)), "kvq_cache_row_bytes")
    return out.value


def reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, kv_cache_dtype,
                      k_scale: float = 1.0, v_scale: float = 1.0, stream=None) -> None:
    """key/value: bf16 [T, Hkv, D] (token stride may exceed Hkv*D);
    caches: uint8 [NB, B, Hkv, row]; slot_mapping: int64 [T]."""
    dt = parse_kv_cache_dtype(kv_cache_dtype) if isinstance(kv_cache_dtype, str) else kv_cache_dtype
    T, H, D = key.shape
    nb, bs = key_cache.shape[0], key_cache.shape[1]
    _check(lib.kvq_reshape_and_cache(
        _ptr(key), _ptr(value), T, key.stride(0), value.stride(0), H, D,
        _ptr(key_cache), _ptr(value_cache), nb, bs, _ptr(slot_mapping), dt,
        float(k_scale), float(v_scale), _stream(stream)), "kvq_reshape_and_cache")


class Sched:
    """Owns one kvq_sched_t (freed on close / garbage collection)."""

    def __init__(self, handle, workspace_bytes: int):
        self.handle = handle
        self.workspace_bytes = workspace_bytes

    def info(self) -> dict:
        inf = SchedInfo()
        _check(lib.kvq_sched_get_info(self.handle, _c.byref(inf)), "kvq_sched_get_info")
        return inf.as_dict()

    def plan(self) -> dict:
        """The schedule's plan as numpy arrays (kvq_sched_export_plan)."""
        sz = PlanSizes()
        _check(lib.kvq_sched_get_plan_sizes(self.handle, _c.byref(sz)), "kvq_sched_get_plan_sizes")
        pieces = np.zeros(sz.num_pieces, PLAN_PIECE)
        warps = np.zeros(sz.num_warps[0] + sz.num_warps[1], np.int32)
        merges = np.zeros(sz.num_merges, PLAN_MERGE)
        tiles = np.zeros(sz.num_prefill_tiles, PLAN_PREFILL)
        _check(lib.kvq_sched_export_plan(
            self.handle, pieces.ctypes.data, pieces.size, warps.ctypes.data, warps.size,
            merges.ctypes.data, merges.size, tiles.ctypes.data, tiles.size),
            "kvq_sched_export_plan")
        return {"pieces": pieces, "warp_first_piece": warps, "merges": merges,
                "prefill_tiles": tiles, "num_chunks": list(sz.num_chunks),
                "num_warps": list(sz.num_warps), "lockstep": list(sz.lockstep)}

    def check_device(self) -> None:
        """Raise KvqError(E_TIMEOUT) if a kernel run with this schedule gave
        up a bounded wait; synchronizes the device."""
        _check(lib.kvq_sched_check_device(self.handle), "kvq_sched_check_device")

    def close(self):
        if self.handle is not None:
            lib.kvq_sched_destroy(self.handle)
            self.handle = None

    def __del__(self):
        self.close()


def get_scheduler_metadata(num_req: int, heads_q: int, heads_kv: int, head_dim: int,
                           seq_lens, query_start_loc, causal: bool, window: int,
                           kv_cache_dtype) -> Sched:
    """seq_lens / query_start_loc: host int32 tensors or arrays."""
    import numpy as np
    dt = parse_kv_cache_dtype(kv_cache_dtype) if isinstance(kv_cache_dtype, str) else kv_cache_dtype
    sl = np.ascontiguousarray(np.asarray(seq_lens), dtype=np.int32)
    qsl = np.ascontiguousarray(np.asarray(query_start_loc), dtype=np.int32)
    h = _p()
    ws = _c.c_size_t()
    _check(lib.kvq_get_scheduler_metadata(
        num_req, heads_q, heads_kv, head_dim, _p(sl.ctypes.data), _p(qsl.ctypes.data),
        int(bool(causal)), int(window), dt, _c.byref(h), _c.byref(ws)),
        "kvq_get_scheduler_metadata")
    return Sched(h, ws.value)


def attention_with_kv_cache(sched: Sched, q, key_cache, value_cache, query_start_loc,
                            seq_lens, block_table, sm_scale: float, causal: bool,
                            window: int, soft_cap: float, k_scale: float, v_scale: float,
                            out, workspace, kv_cache_dtype, heads_kv: int, stream=None,
                            num_blocks=None, alibi_slopes=None, sinks=None) -> None:
    """q / out: bf16 [sum Q, Hq, D]; caches uint8 [NB, B, Hkv, row];
    block_table int32 [R, max_blocks]; query_start_loc / seq_lens device
    int32; workspace: a uint8 device tensor of >= sched.workspace_bytes;
    alibi_slopes / sinks: device float32 [Hq] or None."""
    dt = parse_kv_cache_dtype(kv_cache_dtype) if isinstance(kv_cache_dtype, str) else kv_cache_dtype
    _, Hq, D = q.shape
    nb = key_cache.shape[0] if num_blocks is None else num_blocks
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.kvq_attention_with_kv_cache(
        sched.handle, Hq, heads_kv, D, dt, _ptr(q), _ptr(key_cache), _ptr(value_cache),
        _ptr(query_start_loc), _ptr(seq_lens), _ptr(block_table), block_table.stride(0),
        key_cache.shape[1], nb, float(sm_scale), int(bool(causal)), int(window),
        float(soft_cap), _ptr(alibi_slopes), _ptr(sinks), float(k_scale), float(v_scale),
        _ptr(out), _ptr(workspace), ws_bytes, _stream(stream)), "kvq_attention_with_kv_cache")


def attention_with_kv_cache_static_scratch(sched: Sched, q, key_cache, value_cache,
                                           query_start_loc, seq_lens, block_table,
                                           sm_scale: float, causal: bool, window: int,
                                           soft_cap: float, k_scale: float, v_scale: float,
                                           out, kv_cache_dtype, heads_kv: int, stream=None,
                                           num_blocks=None, alibi_slopes=None,
                                           sinks=None) -> None:
    """attention_with_kv_cache without a workspace argument: the library's
    fixed device scratch (STATIC_SCRATCH_BYTES) holds the split partials.
    For callers that cannot allocate device memory; calls must not overlap
    on the GPU."""
    dt = parse_kv_cache_dtype(kv_cache_dtype) if isinstance(kv_cache_dtype, str) else kv_cache_dtype
    _, Hq, D = q.shape
    nb = key_cache.shape[0] if num_blocks is None else num_blocks
    _check(lib.kvq_attention_with_kv_cache_static_scratch(
        sched.handle, Hq, heads_kv, D, dt, _ptr(q), _ptr(key_cache), _ptr(value_cache),
        _ptr(query_start_loc), _ptr(seq_lens), _ptr(block_table), block_table.stride(0),
        key_cache.shape[1], nb, float(sm_scale), int(bool(causal)), int(window),
        float(soft_cap), _ptr(alibi_slopes), _ptr(sinks), float(k_scale), float(v_scale),
        _ptr(out), _stream(stream)), "kvq_attention_with_kv_cache_static_scratch")


def decode_step_workspace_size(num_req: int, heads_q: int, heads_kv: int, head_dim: int,
                               kv_cache_dtype, max_query_len: int = 1,
                               use_alibi: bool = False) -> int:
    dt = parse_kv_cache_dtype(kv_cache_dtype) if isinstance(kv_cache_dtype, str) else kv_cache_dtype
    out = _c.c_size_t()
    _check(lib.kvq_decode_step_workspace_size(num_req, heads_q, heads_kv, head_dim, dt,
                                              max_query_len, int(bool(use_alibi)),
                                              _c.byref(out)), "kvq_decode_step_workspace_size")
    return out.value


class Prepared:
    """One C-ABI call with its arguments marshalled once (pointers, sizes,
    the stream), for a serving loop that calls it every step on the same
    buffers: calling the object only crosses into the library.  The tensors
    behind the pointers must stay alive (and in place) while it is used."""

    def __init__(self, fn, args, what: str):
        self.fn = fn
        self.args = tuple(args)
        self.what = what

    def __call__(self) -> None:
        _check(self.fn(*self.args), self.what)


def _decode_step_args(key, value, slot_mapping, key_cache, value_cache, q, query_start_loc,
                      seq_lens, block_table, max_query_len, sm_scale, window, soft_cap, k_scale,
                      v_scale, out, workspace, kv_cache_dtype, heads_kv, alibi_slopes, sinks,
                      stream, num_blocks):
    dt = parse_kv_cache_dtype(kv_cache_dtype) if isinstance(kv_cache_dtype, str) else kv_cache_dtype
    _, Hq, D = q.shape
    T = key.shape[0]
    nb = key_cache.shape[0] if num_blocks is None else num_blocks
    return (_c.c_int(seq_lens.shape[0]), _c.c_int(Hq), _c.c_int(heads_kv), _c.c_int(D),
            _c.c_int(dt), _ptr(key), _ptr(value), _c.c_int64(T), _c.c_int64(key.stride(0)),
            _c.c_int64(value.stride(0)), _ptr(slot_mapping), _ptr(key_cache), _ptr(value_cache),
            _c.c_int64(nb), _c.c_int(key_cache.shape[1]), _ptr(q), _ptr(query_start_loc),
            _ptr(seq_lens), _ptr(block_table), _c.c_int(block_table.stride(0)),
            _c.c_int(int(max_query_len)), _c.c_float(sm_scale), _c.c_int(int(window)),
            _c.c_float(soft_cap), _ptr(alibi_slopes), _ptr(sinks), _c.c_float(k_scale),
            _c.c_float(v_scale), _ptr(out), _ptr(workspace),
            _c.c_size_t(workspace.numel() * workspace.element_size()), _stream(stream))


def decode_step(key, value, slot_mapping, key_cache, value_cache, q, query_start_loc, seq_lens,
                block_table, max_query_len: int, sm_scale: float, window: int, soft_cap: float,
                k_scale: float, v_scale: float, out, workspace, kv_cache_dtype, heads_kv: int,
                alibi_slopes=None, sinks=None, stream=None, num_blocks=None) -> None:
    """kvq_decode_step: the new rows key/value bf16 [T, Hkv, D] with their
    slot_mapping int64 [T]; q / out bf16 [sum Q, Hq, D]; query_start_loc,
    seq_lens int32 device; workspace: a zero-filled uint8 device tensor of
    >= decode_step_workspace_size(...) bytes."""
    _check(lib.kvq_decode_step(*_decode_step_args(
        key, value, slot_mapping, key_cache, value_cache, q, query_start_loc, seq_lens,
        block_table, max_query_len, sm_scale, window, soft_cap, k_scale, v_scale, out, workspace,
        kv_cache_dtype, heads_kv, alibi_slopes, sinks, stream, num_blocks)), "kvq_decode_step")


def prepare_decode_step(key, value, slot_mapping, key_cache, value_cache, q, query_start_loc,
                        seq_lens, block_table, max_query_len: int, sm_scale: float, window: int,
                        soft_cap: float, k_scale: float, v_scale: float, out, workspace,
                        kv_cache_dtype, heads_kv: int, alibi_slopes=None, sinks=None,
                        stream=None, num_blocks=None) -> Prepared:
    """decode_step with its arguments marshalled once (see Prepared)."""
    return Prepared(lib.kvq_decode_step, _decode_step_args(
        key, value, slot_mapping, key_cache, value_cache, q, query_start_loc, seq_lens,
        block_table, max_query_len, sm_scale, window, soft_cap, k_scale, v_scale, out, workspace,
        kv_cache_dtype, heads_kv, alibi_slopes, sinks, stream, num_blocks), "kvq_decode_step")


def _host_io_args(host_in, dev_in, host_out, out_bytes):
    in_bytes = host_in.numel() * host_in.element_size()
    if dev_in.numel() * dev_in.element_size() < in_bytes:
        raise ValueError("dev_in is smaller than host_in")
    if out_bytes > host_out.numel() * host_out.element_size():
        raise ValueError("out_bytes exceeds host_out")
    return (_ptr(host_in), _ptr(dev_in), _c.c_size_t(in_bytes), _ptr(host_out),
            _c.c_size_t(int(out_bytes)))


def prepare_decode_step_host_io(host_in, dev_in, host_out, out_bytes: int, key, value,
                                slot_mapping, key_cache, value_cache, q, query_start_loc,
                                seq_lens, block_table, max_query_len: int, sm_scale: float,
                                window: int, soft_cap: float, k_scale: float, v_scale: float,
                                out, workspace, kv_cache_dtype, heads_kv: int, alibi_slopes=None,
                                sinks=None, stream=None, num_blocks=None) -> Prepared:
    """kvq_decode_step_host_io, marshalled once (see Prepared): each call
    copies host_in (a pinned uint8 tensor) to dev_in, runs the decode step
    (whose device tensors may be views of dev_in), copies out_bytes of out
    to host_out (pinned) and waits for the stream.  out None: the step
    writes its output straight into host_out (out_bytes ignored)."""
    return Prepared(lib.kvq_decode_step_host_io, _host_io_args(host_in, dev_in, host_out, out_bytes)
                    + _decode_step_args(key, value, slot_mapping, key_cache, value_cache, q,
                                        query_start_loc, seq_lens, block_table, max_query_len,
                                        sm_scale, window, soft_cap, k_scale, v_scale, out,
                                        workspace, kv_cache_dtype, heads_kv, alibi_slopes, sinks,
                                        stream, num_blocks), "kvq_decode_step_host_io")


class DecodeStepGraph:
    """A host-buffer decode step captured once in a CUDA graph
    (kvq_decode_step_graph_create); calling it replays the step on the
    stream it was made for and waits (kvq_decode_step_graph_launch).  The
    buffers behind it must stay alive, in place, until close()."""

    def __init__(self, handle, stream):
        self._h = handle
        self._stream = stream
        self._launch = lib.kvq_decode_step_graph_launch

    def __call__(self) -> None:
        _check(self._launch(self._h, self._stream), "kvq_decode_step_graph_launch")

    def close(self) -> None:
        if self._h:
            lib.kvq_decode_step_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def decode_step_graph(host_in, dev_in, host_out, out_bytes: int, key, value, slot_mapping,
                      key_cache, value_cache, q, query_start_loc, seq_lens, block_table,
                      max_query_len: int, sm_scale: float, window: int, soft_cap: float,
                      k_scale: float, v_scale: float, out, workspace, kv_cache_dtype,
                      heads_kv: int, alibi_slopes=None, sinks=None, stream=None,
                      num_blocks=None) -> DecodeStepGraph:
    """kvq_decode_step_graph_create with the arguments of
    prepare_decode_step_host_io; host_in must be pinned (the fused kernel
    stages it).  Rewrite host_in between calls of the returned object."""
    args = (_host_io_args(host_in, dev_in, host_out, out_bytes)
            + _decode_step_args(key, value, slot_mapping, key_cache, value_cache, q,
                                query_start_loc, seq_lens, block_table, max_query_len, sm_scale,
                                window, soft_cap, k_scale, v_scale, out, workspace,
                                kv_cache_dtype, heads_kv, alibi_slopes, sinks, stream,
                                num_blocks))
    h = _p()
    _check(lib.kvq_decode_step_graph_create(*args[:-1], _c.byref(h)), "kvq_decode_step_graph_create")
    return DecodeStepGraph(h, args[-1])


def decode_step_check(workspace) -> None:
    """Raise KvqError if a decode_step run with this workspace flagged an
    error (synchronises the device)."""
    _check(lib.kvq_decode_step_check(_ptr(workspace)), "kvq_decode_step_check")
