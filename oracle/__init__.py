"""CPU oracle for quantized paged-KV attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product library never does, and this
package imports nothing from it: the oracle is the plain C in
``kvq_oracle.c`` (scalar codecs, one-key-at-a-time binary64 attention),
compiled with gcc and called through ctypes on numpy arrays.

Sources restated (prhub.com.cn summaries of vLLM pull requests):
  * vllm PR 39445 "CPU 后端新增 FP8 KV 缓存量化支持" -- Breakdown item 1 and
    Key files: scalar fp8 e4m3 encode/decode, the reshape into the cache;
  * vllm PR 50194 "修复 CPU FP8 注意力调度器临时缓冲区大小计算错误" -- Key
    source snippet: dtype indices 0/1/2, causal / window / soft_cap options;
  * vllm PR 38378 "为 Triton 注意力后端引入 KV 缓存按令牌头 INT8/FP8 量化" --
    Breakdown item 3 and Risks: per-(token, head) absmax scales stored inline.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against library routines (torch's fp8 casts, torch.round, numpy softmax),
the OCP FP8 definition's printed values (``tests/golden/``), closed forms and
invariants.  Agreement with vLLM's own kernels is unpinned: neither its code
nor model weights are available.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build", platform.machine())
_LIB_PATH = os.path.join(_BUILD_DIR, "libkvq_oracle.so")

AUTO, FP8_E4M3, FP8_E5M2, INT8_PER_TOKEN_HEAD, FP8_PER_TOKEN_HEAD, FP8_E5M2_PER_TOKEN_HEAD = range(6)
E4M3, E5M2 = 0, 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, OpenMP, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        c = ctypes
        p = c.c_void_p
        lib.kvo_fp8_decode.restype = c.c_double
        lib.kvo_fp8_decode.argtypes = [c.c_int, c.c_uint8]
        lib.kvo_fp8_encode.restype = c.c_uint8
        lib.kvo_fp8_encode.argtypes = [c.c_int, c.c_float]
        lib.kvo_int8_encode.restype = c.c_int8
        lib.kvo_int8_encode.argtypes = [c.c_float]
        lib.kvo_row_bytes.restype = c.c_int64
        lib.kvo_row_bytes.argtypes = [c.c_int, c.c_int]
        lib.kvo_reshape_and_cache.restype = c.c_int
        lib.kvo_reshape_and_cache.argtypes = [
            p, p, c.c_int64, c.c_int64, c.c_int64, c.c_int, c.c_int, p, p,
            c.c_int64, c.c_int, p, c.c_int, c.c_float, c.c_float]
        lib.kvo_attention.restype = c.c_int
        lib.kvo_attention.argtypes = [
            c.c_int, c.c_int, c.c_int, c.c_int, p, p, p, c.c_int, c.c_int, p,
            p, p, c.c_int, c.c_double, c.c_int, c.c_int, c.c_double,
            c.c_float, c.c_float, p, p, p, c.c_int64, p]
        lib.kvo_attention_fp32_bound.restype = c.c_int
        lib.kvo_attention_fp32_bound.argtypes = lib.kvo_attention.argtypes
        lib.kvo_attention_probs.restype = c.c_int64
        lib.kvo_attention_probs.argtypes = [
            c.c_int, c.c_int, c.c_int, c.c_int, p, p, c.c_int, c.c_int, p, p,
            p, c.c_int, c.c_double, c.c_int, c.c_int, c.c_double, c.c_float,
            p, p, c.c_int64, c.c_int, p, p]
        lib.kvo_num_threads.restype = c.c_int
        lib.kvo_num_threads.argtypes = []
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def num_threads() -> int:
    return int(_load().kvo_num_threads())


def fp8_decode(fmt: int, code: int) -> float:
    """Value of one fp8 code (fmt: E4M3 or E5M2)."""
    return float(_load().kvo_fp8_decode(fmt, code))


def fp8_encode(fmt: int, y: float) -> int:
    """fp8 code of a binary32 value (RNE, saturating)."""
    return int(_load().kvo_fp8_encode(fmt, float(np.float32(y))))


def fp8_encode_array(fmt: int, y: np.ndarray) -> np.ndarray:
    lib = _load()
    y = _c(y, np.float32).ravel()
    return np.fromiter((lib.kvo_fp8_encode(fmt, float(v)) for v in y),
                       dtype=np.uint8, count=y.size)


def int8_encode(y: float) -> int:
    return int(_load().kvo_int8_encode(float(np.float32(y))))


def row_bytes(dtype: int, head_dim: int) -> int:
    return int(_load().kvo_row_bytes(dtype, head_dim))


def reshape_and_cache(key_bits: np.ndarray, value_bits: np.ndarray,
                      key_cache: np.ndarray, value_cache: np.ndarray,
                      slot_mapping: np.ndarray, dtype: int, k_scale: float,
                      v_scale: float, block_size: int) -> None:
    """Write K/V (bf16 bit patterns, uint16 [T, Hkv, D]) into the uint8 caches
    [NB, B, Hkv, row] in place."""
    key_bits = _c(key_bits, np.uint16)
    value_bits = _c(value_bits, np.uint16)
    slot_mapping = _c(slot_mapping, np.int64)
    assert key_cache.dtype == np.uint8 and key_cache.flags.c_contiguous
    assert value_cache.dtype == np.uint8 and value_cache.flags.c_contiguous
    T, Hkv, D = key_bits.shape
    nb = key_cache.shape[0]
    rc = _load().kvo_reshape_and_cache(
        _ptr(key_bits), _ptr(value_bits), T, Hkv * D, Hkv * D, Hkv, D,
        _ptr(key_cache), _ptr(value_cache), nb, block_size,
        _ptr(slot_mapping), dtype, float(k_scale), float(v_scale))
    if rc != 0:
        raise ValueError("oracle reshape_and_cache rejected its arguments")


def attention(q_bits: np.ndarray, key_cache: np.ndarray,
              value_cache: np.ndarray, query_start_loc, seq_lens, block_table,
              heads_kv: int, block_size: int, dtype: int, sm_scale: float,
              causal: bool, window: int, soft_cap: float, k_scale: float,
              v_scale: float, tokens=None, alibi_slopes=None, sinks=None) -> np.ndarray:
    """float32 [n, Hq, D] attention output for the listed query tokens
    (all tokens when ``tokens`` is None).  alibi_slopes / sinks: float32
    [Hq] per q head, or None."""
    return _attention_call("kvo_attention", q_bits, key_cache, value_cache, query_start_loc,
                           seq_lens, block_table, heads_kv, block_size, dtype, sm_scale, causal,
                           window, soft_cap, k_scale, v_scale, tokens, alibi_slopes, sinks)


def attention_fp32_bound(q_bits: np.ndarray, key_cache: np.ndarray,
                         value_cache: np.ndarray, query_start_loc, seq_lens, block_table,
                         heads_kv: int, block_size: int, dtype: int, sm_scale: float,
                         causal: bool, window: int, soft_cap: float, k_scale: float,
                         v_scale: float, tokens=None, alibi_slopes=None,
                         sinks=None) -> np.ndarray:
    """float32 [n, Hq, D]: first-order bound on how far a binary32
    evaluation (binary32 scores and sums, 11-bit softmax weights) of the
    attention may land from the exact result (kvo_attention_fp32_bound)."""
    return _attention_call("kvo_attention_fp32_bound", q_bits, key_cache, value_cache,
                           query_start_loc, seq_lens, block_table, heads_kv, block_size, dtype,
                           sm_scale, causal, window, soft_cap, k_scale, v_scale, tokens,
                           alibi_slopes, sinks)


def _per_head(x, Hq):
    if x is None:
        return None
    a = _c(x, np.float32).ravel()
    if a.size != Hq:
        raise ValueError("per-head array must have heads_q entries")
    return a


def _attention_call(fn, q_bits, key_cache, value_cache, query_start_loc, seq_lens, block_table,
                    heads_kv, block_size, dtype, sm_scale, causal, window, soft_cap, k_scale,
                    v_scale, tokens, alibi_slopes=None, sinks=None):
    q_bits = _c(q_bits, np.uint16)
    qsl = _c(query_start_loc, np.int32)
    sl = _c(seq_lens, np.int32)
    bt = _c(block_table, np.int32)
    if bt.ndim == 1:
        bt = bt.reshape(len(sl), -1)
    _, Hq, D = q_bits.shape
    tok = None if tokens is None else _c(tokens, np.int64)
    n = int(qsl[-1]) if tok is None else tok.size
    out = np.zeros((n, Hq, D), dtype=np.float32)
    al, sk = _per_head(alibi_slopes, Hq), _per_head(sinks, Hq)
    rc = getattr(_load(), fn)(
        len(sl), Hq, heads_kv, D, _ptr(q_bits), _ptr(key_cache),
        _ptr(value_cache), block_size, dtype, _ptr(qsl), _ptr(sl), _ptr(bt),
        bt.shape[1], float(sm_scale), int(bool(causal)), int(window),
        float(soft_cap), float(k_scale), float(v_scale), _ptr(al), _ptr(sk), _ptr(tok),
        0 if tok is None else tok.size, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle {fn} rejected its arguments")
    return out


def attention_probs(q_bits: np.ndarray, key_cache: np.ndarray,
                    query_start_loc, seq_lens, block_table, heads_kv: int,
                    block_size: int, dtype: int, sm_scale: float, causal: bool,
                    window: int, soft_cap: float, k_scale: float, token: int,
                    head_q: int, alibi_slopes=None, sinks=None, with_sink=False):
    """Softmax weights (float64 [L]) of one query token and q head; with
    ``with_sink`` also the sink's weight (a float)."""
    q_bits = _c(q_bits, np.uint16)
    qsl = _c(query_start_loc, np.int32)
    sl = _c(seq_lens, np.int32)
    bt = _c(block_table, np.int32)
    if bt.ndim == 1:
        bt = bt.reshape(len(sl), -1)
    _, Hq, D = q_bits.shape
    probs = np.zeros(max(1, int(sl.max())), dtype=np.float64)
    sink_w = np.zeros(1, dtype=np.float64)
    al, sk = _per_head(alibi_slopes, Hq), _per_head(sinks, Hq)
    L = _load().kvo_attention_probs(
        len(sl), Hq, heads_kv, D, _ptr(q_bits), _ptr(key_cache), block_size,
        dtype, _ptr(qsl), _ptr(sl), _ptr(bt), bt.shape[1], float(sm_scale),
        int(bool(causal)), int(window), float(soft_cap), float(k_scale),
        _ptr(al), _ptr(sk), int(token), int(head_q), _ptr(probs), _ptr(sink_w))
    if L < 0:
        raise ValueError("oracle attention_probs rejected its arguments")
    return (probs[:L].copy(), float(sink_w[0])) if with_sink else probs[:L].copy()
