"""Seeded synthetic workloads for quantized paged-KV attention.

This module only draws inputs: shapes, seeded random values, block tables,
slot mappings and the harness's per-tensor scale recipe.  It holds none of
the method's arithmetic (no quantisation, no attention), so the oracle and
the CUDA path can both be fed from it.

Every tensor is built on the CPU with ``torch.Generator('cpu')`` seeded by
``1000 + index`` so that the oracle and the GPU see identical bytes.

Workloads (the shapes of the pages' cases):
  1 tiny      2 requests (Q, L) = (1, 37), (8, 8); Hq 4, Hkv 2, D 64, B 16,
              8 physical blocks, fp8_e4m3, k_scale 0.05, v_scale 0.04.
  2 decode    64 requests, Q = 1, L ~ U[1024, 4096]; Hq 32, Hkv 8, D 128,
              B 16, fp8_e4m3, per-tensor scales absmax / 448.
  3 prefill   4 requests, Q = L = 1024, causal; Hq 16, Hkv 2, D 256,
              B 2176, 4 blocks, fp8_e4m3; 1% of elements x20.
  4 mixed     16 prefills Q = L ~ U[128, 2048] + 48 decodes L ~ U[512, 8192];
              Hq 32, Hkv 8, D 128, B 16; int8 / fp8 per-token-head; K/V
              scaled per token by exp(U(ln 0.1, ln 10)).
  5 long      32 requests, Q = 1, L = 32768; Hq 64, Hkv 8, D 128, B 16,
              window 4096, soft_cap 50, fp8_e5m2, scales absmax / 57344.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

E4M3_MAX = 448.0
E5M2_MAX = 57344.0


@dataclass
class Workload:
    name: str
    kv_cache_dtype: str
    heads_q: int
    heads_kv: int
    head_dim: int
    block_size: int
    num_blocks: int
    query_lens: List[int]
    seq_lens: List[int]
    q: torch.Tensor              # bf16 [sum Q, Hq, D]
    key: torch.Tensor            # bf16 [T, Hkv, D]: every context token
    value: torch.Tensor          # bf16 [T, Hkv, D]
    slot_mapping: torch.Tensor   # int64 [T]
    block_table: torch.Tensor    # int32 [R, max_blocks]
    query_start_loc: torch.Tensor  # int32 [R + 1]
    seq_lens_t: torch.Tensor     # int32 [R]
    token_req: torch.Tensor      # int32 [T]: request of each context token
    token_pos: torch.Tensor      # int32 [T]: position of each context token
    sm_scale: float
    causal: bool = True
    window: int = 0
    soft_cap: float = 0.0
    k_scale: float = 1.0
    v_scale: float = 1.0
    meta: dict = field(default_factory=dict)

    @property
    def num_req(self) -> int:
        return len(self.seq_lens)

    @property
    def num_query_tokens(self) -> int:
        return int(sum(self.query_lens))

    @property
    def num_tokens(self) -> int:
        return int(self.key.shape[0])

    def new_token_mask(self) -> torch.Tensor:
        """Context tokens that are this step's queries (the last Q of each
        request): the tokens a serving step writes before attending."""
        qlen = torch.tensor(self.query_lens, dtype=torch.int32)
        slen = torch.tensor(self.seq_lens, dtype=torch.int32)
        start = (slen - qlen)[self.token_req.long()]
        return self.token_pos >= start


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, g: torch.Generator) -> torch.Tensor:
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _paged_layout(seq_lens: List[int], block_size: int, g: torch.Generator,
                  num_blocks: Optional[int] = None, extra_blocks: int = 0):
    """Random physical placement: block_table rows are slices of a random
    permutation of the block pool; slot_mapping follows the table."""
    need = [math.ceil(L / block_size) for L in seq_lens]
    pool = sum(need) + extra_blocks
    if num_blocks is None:
        num_blocks = pool
    assert num_blocks >= sum(need)
    perm = torch.randperm(num_blocks, generator=g)[: sum(need)].to(torch.int32)
    max_blocks = max(1, max(need) if need else 1)
    table = torch.zeros((len(seq_lens), max_blocks), dtype=torch.int32)
    slots, reqs, poss = [], [], []
    off = 0
    for r, (L, n) in enumerate(zip(seq_lens, need)):
        table[r, :n] = perm[off: off + n]
        off += n
        pos = torch.arange(L, dtype=torch.int64)
        blk = table[r, (pos // block_size)].to(torch.int64)
        slots.append(blk * block_size + pos % block_size)
        reqs.append(torch.full((L,), r, dtype=torch.int32))
        poss.append(pos.to(torch.int32))
    cat = (lambda xs, dt: torch.cat(xs) if xs else torch.zeros(0, dtype=dt))
    return (num_blocks, table, cat(slots, torch.int64), cat(reqs, torch.int32),
            cat(poss, torch.int32))


def custom(name: str, query_lens: List[int], seq_lens: List[int],
           heads_q: int, heads_kv: int, head_dim: int, block_size: int,
           kv_cache_dtype: str, seed: int, *, causal: bool = True,
           window: int = 0, soft_cap: float = 0.0, num_blocks=None,
           extra_blocks: int = 0, outlier_p: float = 0.0,
           outlier_mul: float = 20.0, token_scale_range=None,
           k_scale=None, v_scale=None, sm_scale=None,
           scale_max: Optional[float] = None) -> Workload:
    """A seeded workload of any shape.  Per-tensor scales default to
    absmax / scale_max over all K (resp. V) when not given."""
    assert len(query_lens) == len(seq_lens)
    g = _gen(seed)
    R = len(seq_lens)
    T = int(sum(seq_lens))
    nq = int(sum(query_lens))
    q = torch.randn((nq, heads_q, head_dim), generator=g, dtype=torch.float32)
    k = torch.randn((T, heads_kv, head_dim), generator=g, dtype=torch.float32)
    v = torch.randn((T, heads_kv, head_dim), generator=g, dtype=torch.float32)
    if outlier_p > 0:
        for t in (q, k, v):
            mask = torch.rand(t.shape, generator=g) < outlier_p
            t[mask] *= outlier_mul
    if token_scale_range is not None:
        lo, hi = token_scale_range
        u = torch.rand((T,), generator=g, dtype=torch.float64)
        f = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
        f = f.to(torch.float32).view(T, 1, 1)
        k *= f
        v *= f
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    nb, table, slots, treq, tpos = _paged_layout(seq_lens, block_size, g,
                                                 num_blocks, extra_blocks)
    qsl = torch.zeros(R + 1, dtype=torch.int32)
    if R:
        qsl[1:] = torch.cumsum(torch.tensor(query_lens, dtype=torch.int32), 0)
    if scale_max is None:
        scale_max = E5M2_MAX if kv_cache_dtype == "fp8_e5m2" else E4M3_MAX
    if k_scale is None:
        k_scale = float(k.abs().max().float() / scale_max) if T else 1.0
    if v_scale is None:
        v_scale = float(v.abs().max().float() / scale_max) if T else 1.0
    return Workload(
        name=name, kv_cache_dtype=kv_cache_dtype, heads_q=heads_q,
        heads_kv=heads_kv, head_dim=head_dim, block_size=block_size,
        num_blocks=nb, query_lens=list(query_lens), seq_lens=list(seq_lens),
        q=q, key=k, value=v, slot_mapping=slots, block_table=table,
        query_start_loc=qsl,
        seq_lens_t=torch.tensor(seq_lens, dtype=torch.int32),
        token_req=treq, token_pos=tpos,
        sm_scale=(1.0 / math.sqrt(head_dim)) if sm_scale is None else sm_scale,
        causal=causal, window=window, soft_cap=soft_cap,
        k_scale=float(k_scale), v_scale=float(v_scale))


def _uniform_ints(g, lo, hi, n):
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


def config(index: int, kv_cache_dtype: Optional[str] = None) -> Workload:
    """The five workloads of the pages' cases, at full size."""
    seed = 1000 + index
    if index == 1:
        return custom("tiny decode+prefill", [1, 8], [37, 8], 4, 2, 64, 16,
                      "fp8_e4m3", seed, num_blocks=8, k_scale=0.05,
                      v_scale=0.04, sm_scale=1.0 / 8.0)
    if index == 2:
        L = _uniform_ints(_gen(seed + 100), 1024, 4096, 64)
        return custom("decode batch: 64 seqs, L~U[1024,4096], Hq32/Hkv8, "
                      "D128, fp8_e4m3", [1] * 64, L, 32, 8, 128, 16,
                      "fp8_e4m3", seed)
    if index == 3:
        return custom("large prefill: 4x1024 causal, Hq16/Hkv2, D256, "
                      "B2176, fp8_e4m3", [1024] * 4, [1024] * 4, 16, 2, 256,
                      2176, "fp8_e4m3", seed, num_blocks=4, outlier_p=0.01,
                      outlier_mul=20.0)
    if index == 4:
        dt = kv_cache_dtype or "int8_per_token_head"
        g = _gen(seed + 100)
        pre = _uniform_ints(g, 128, 2048, 16)
        dec = _uniform_ints(g, 512, 8192, 48)
        ql = pre + [1] * 48
        sl = pre + dec
        order = torch.randperm(64, generator=g).tolist()
        ql = [ql[i] for i in order]
        sl = [sl[i] for i in order]
        return custom(f"mixed: 16 prefills + 48 decodes, Hq32/Hkv8, D128, {dt}",
                      ql, sl, 32, 8, 128, 16, dt, seed,
                      token_scale_range=(0.1, 10.0))
    if index == 5:
        return custom("long decode: 32 x 32768, window 4096, soft_cap 50, "
                      "Hq64/Hkv8, D128, fp8_e5m2", [1] * 32, [32768] * 32, 64,
                      8, 128, 16, "fp8_e5m2", seed, window=4096,
                      soft_cap=50.0)
    raise ValueError(f"no workload {index}")


def scaled(index: int, seed_offset: int = 0,
           kv_cache_dtype: Optional[str] = None) -> Workload:
    """Smaller cases of each workload's shape that the oracle finishes in
    seconds, still spanning several tiles and a ragged tail."""
    seed = 2000 + index + 10 * seed_offset
    g = _gen(seed + 100)
    if index == 2:
        L = _uniform_ints(g, 100, 700, 6)
        return custom("decode (scaled)", [1] * 6, L, 32, 8, 128, 16,
                      "fp8_e4m3", seed)
    if index == 3:
        return custom("prefill (scaled)", [200, 77], [200, 77], 16, 2, 256,
                      2176, "fp8_e4m3", seed, num_blocks=3, outlier_p=0.01)
    if index == 4:
        dt = kv_cache_dtype or "int8_per_token_head"
        pre = _uniform_ints(g, 20, 150, 3)
        dec = _uniform_ints(g, 30, 400, 5)
        return custom(f"mixed (scaled, {dt})", pre + [1] * 5, pre + dec, 32, 8,
                      128, 16, dt, seed, token_scale_range=(0.1, 10.0))
    if index == 5:
        return custom("long decode (scaled)", [1] * 3, [1500, 777, 2049], 64, 8,
                      128, 16, "fp8_e5m2", seed, window=300, soft_cap=50.0)
    raise ValueError(f"no scaled workload {index}")


def alibi_slopes(heads_q: int):
    """float32 [heads_q] ALiBi slopes, the usual geometric sequence
    2^(-8 (h + 1) / n) over the next power of two n >= heads_q, interleaved
    as in the ALiBi paper for head counts that are not powers of two."""
    n = 1 << max(0, math.ceil(math.log2(max(1, heads_q))))
    base = [2.0 ** (-8.0 * (h + 1) / n) for h in range(n)]
    if n == heads_q:
        return torch.tensor(base, dtype=torch.float32).numpy()
    extra = [2.0 ** (-4.0 * (2 * h + 1) / n) for h in range(heads_q - n // 2)]
    return torch.tensor(base[: n // 2] + extra, dtype=torch.float32).numpy()


def sink_logits(heads_q: int, seed: int):
    """float32 [heads_q] seeded sink logits ~ N(0, 2^2)."""
    return (torch.randn((heads_q,), generator=_gen(seed), dtype=torch.float32) * 2.0).numpy()


def bf16_bits(t: torch.Tensor):
    """uint16 numpy view of a bf16 tensor's bit patterns (CPU copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
