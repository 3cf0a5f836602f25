"""The scheduler's plan against an independent derivation (no GPU).

vllm PR 50194 page, Breakdown item 1 and Key source snippet: the scheduler
is the single source of the tiles and scratch the kernels run with, built
from the host sequence lengths, the causal flag and the window.  These tests
export the plan (kvq_sched_export_plan) for seeded batches and check it
against the tiles and key ranges derived here from the definitions alone:
row tiles of up to 16 packed (query, head) rows per kv head go to the decode
kernel and larger requests to 128-row prefill tiles; a row sees the keys
p - window < j <= p (causal) with p its position; the decode's 16-token
chunks of each tile are streamed exactly once, in contiguous pieces, by
equal warp segments; cut tiles have one merge item with disjoint partial
rows inside the workspace.
"""
import math

import numpy as np
import pytest

from int8_kv_cache_reshape_gb300 import build as kbuild

kbuild.build()
from int8_kv_cache_reshape_gb300 import kvq  # noqa: E402

CHUNK = 16


def derive(seq_lens, query_lens, hq, hkv, causal, window):
    """(decode tiles {(req, h): (nrows, key_lo, key_hi)}, prefill tiles [...])"""
    G = hq // hkv
    decode, prefill = {}, []
    for r, (L, Q) in enumerate(zip(seq_lens, query_lens)):
        if Q == 0:
            continue
        rows = Q * G

        def keys(row0, n):
            p_min = L - Q + row0 // G
            p_max = L - Q + (row0 + n - 1) // G
            hi = p_max + 1 if causal else L
            lo = max(0, p_min - window + 1) if window > 0 else 0
            return lo, hi

        for h in range(hkv):
            if rows > 16:
                for row0 in range(0, rows, 128):
                    n = min(128, rows - row0)
                    prefill.append((r, h, row0, n) + keys(row0, n))
            else:
                decode[(r, h)] = (rows,) + keys(0, rows)
    return decode, prefill


def check_plan(seq_lens, query_lens, hq=32, hkv=8, D=128, causal=True, window=0,
               dtype="fp8_e4m3"):
    qsl = np.concatenate([[0], np.cumsum(query_lens)]).astype(np.int32)
    s = kvq.get_scheduler_metadata(len(seq_lens), hq, hkv, D, np.array(seq_lens, np.int32), qsl,
                                   causal, window, dtype)
    plan, info = s.plan(), s.info()
    s.close()
    decode, prefill = derive(seq_lens, query_lens, hq, hkv, causal, window)
    P = plan["pieces"]

    # prefill tiles: the derived set, longest key range first.  A build with
    # CTA pairs (quantised caches at head_dim >= 128): list entries 2i, 2i + 1
    # are consecutive row tiles of one (request, kv head) (or a last tile and
    # an empty partner, nrows 0), longest key-range union first.
    allt = [tuple(int(x) for x in t) for t in plan["prefill_tiles"]]
    got = [t for t in allt if t[3] > 0]
    assert sorted(got) == sorted(prefill)
    if info["prefill_cta_group"] == 2:
        assert len(allt) % 2 == 0
        spans = []
        for a, b in zip(allt[0::2], allt[1::2]):
            assert (a[0], a[1]) == (b[0], b[1]) and b[2] == a[2] + a[3] and a[3] > 0
            assert a[3] == 128 or b[3] == 0
            if b[3] == 0:
                # the empty partner: the last tile of its (request, kv head)
                assert a[2] + a[3] == query_lens[a[0]] * (hq // hkv) and b[4:] == a[4:]
            spans.append(max(a[5], b[5]) - min(a[4], b[4]))
    else:
        assert len(allt) == len(got)
        spans = [t[5] - t[4] for t in got]
        # equal key ranges keep (request, kv head, first row) order: the deal
        # is deterministic
        for a, b in zip(got, got[1:]):
            if a[5] - a[4] == b[5] - b[4]:
                assert a[:3] < b[:3]
    assert all(a >= b for a, b in zip(spans, spans[1:]))

    # decode tiles: the derived set, each in its launch class
    tiles = {}
    for i, p in enumerate(P):
        key = (int(p["req"]), int(p["kv_head"]))
        tiles.setdefault(key, []).append(i)
        assert p["row0"] == 0
        assert (int(p["nrows"]), int(p["key_lo"]), int(p["key_hi"])) == decode[key]
        assert p["launch"] == (0 if p["nrows"] <= 8 else 1)
    assert set(tiles) == set(decode)

    # each class: pieces end to end over its flat chunk sequence
    for c in (0, 1):
        idx = np.nonzero(P["launch"] == c)[0]
        T = plan["num_chunks"][c]
        assert list(idx) == list(range(idx[0], idx[0] + len(idx))) if len(idx) else T == 0
        flat = P["flat0"][idx].astype(np.int64)
        n = P["nchunks"][idx].astype(np.int64)
        if len(idx):
            assert flat[0] == 0 and np.all(n >= 1)
            assert np.array_equal(flat[1:], flat[:-1] + n[:-1])
            assert flat[-1] + n[-1] == T
        want = sum(math.ceil(hi / CHUNK) - lo // CHUNK for (rows, lo, hi) in decode.values()
                   if (0 if rows <= 8 else 1) == c)
        assert T == want

    # each tile: its pieces cover its chunk range once, in order, adjacent in
    # the flat sequence; cut tiles have one merge item with their partial rows
    used_merges = set()
    intervals = []
    for key, ids in tiles.items():
        rows, lo, hi = decode[key]
        ids = sorted(ids, key=lambda i: P["flat0"][i])
        c0 = [int(P["chunk0"][i]) for i in ids]
        nc = [int(P["nchunks"][i]) for i in ids]
        assert c0[0] == lo // CHUNK and c0[-1] + nc[-1] == math.ceil(hi / CHUNK)
        assert all(c0[k + 1] == c0[k] + nc[k] for k in range(len(ids) - 1))
        assert all(P["flat0"][ids[k + 1]] == P["flat0"][ids[k]] + nc[k] for k in range(len(ids) - 1))
        if len(ids) == 1:
            assert P["part"][ids[0]] == -1 and P["merge"][ids[0]] == -1
            continue
        m = int(P["merge"][ids[0]])
        assert m >= 0 and all(P["merge"][i] == m for i in ids) and m not in used_merges
        used_merges.add(m)
        mi = plan["merges"][m]
        assert (int(mi["req"]), int(mi["kv_head"]), int(mi["row0"]), int(mi["nrows"])) == \
            key + (0, rows)
        assert mi["nsplits"] == len(ids)
        assert [int(P["part"][i]) for i in ids] == [int(mi["part"]) + k * rows for k in range(len(ids))]
        intervals.append((int(mi["part"]), int(mi["part"]) + len(ids) * rows))
    assert used_merges == set(range(len(plan["merges"])))
    intervals.sort()
    assert all(a[1] <= b[0] for a, b in zip(intervals, intervals[1:]))
    if intervals:
        assert info["workspace_bytes"] >= intervals[-1][1] * (D + 1) * 4

    # each warp: its stream-K segment [w T / W, (w + 1) T / W) starts in its
    # first piece.  Head lockstep (head-major tile order, W a multiple of the
    # kv heads): segment w = h * W / Hkv + v runs on warp v * Hkv + h.
    base = 0
    for c in (0, 1):
        W, T = plan["num_warps"][c], plan["num_chunks"][c]
        inter = plan["lockstep"][c] and W % hkv == 0
        for w in range(W):
            lo, hi = w * T // W, (w + 1) * T // W
            phys = (w % (W // hkv)) * hkv + w // (W // hkv) if inter else w
            fp = int(plan["warp_first_piece"][base + phys])
            if hi == lo:
                assert fp == -1
                continue
            assert P["launch"][fp] == c
            assert P["flat0"][fp] <= lo < P["flat0"][fp] + P["nchunks"][fp]
        base += W

    # head lockstep: tiles in head-major order, and, when W is a multiple of
    # the kv head count, every kv head of a request cut at the same chunks
    for c in (0, 1):
        if not plan["lockstep"][c]:
            continue
        idx = np.nonzero(P["launch"] == c)[0]
        heads = P["kv_head"][idx]
        assert np.all(np.diff(heads) >= 0)
        if plan["num_warps"][c] % hkv:
            continue
        cuts = {}
        for key, ids in tiles.items():
            if P["launch"][ids[0]] != c:
                continue
            cut = tuple((int(P["chunk0"][i]), int(P["nchunks"][i]))
                        for i in sorted(ids, key=lambda i: P["flat0"][i]))
            cuts.setdefault(key[0], set()).add(cut)
        assert all(len(v) == 1 for v in cuts.values())
    return plan


def _batch(seed, n, q_max, l_max, mixed):
    rng = np.random.default_rng(seed)
    L = rng.integers(1, l_max + 1, n)
    Q = np.ones(n, np.int64)
    if mixed:
        Q = np.minimum(L, rng.integers(0, q_max + 1, n))
    return [int(x) for x in L], [int(x) for x in Q]


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 8), (16, 2), (64, 4)])
def test_decode_batches(monkeypatch, seed, hq, hkv):
    monkeypatch.delenv("KVQ_DECODE_WARPS", raising=False)
    L, Q = _batch(seed, 48, 1, 5000, mixed=False)
    check_plan(L, Q, hq, hkv)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("window", [0, 1, 37, 1000])
def test_mixed_batches_and_windows(monkeypatch, seed, window):
    monkeypatch.delenv("KVQ_DECODE_WARPS", raising=False)
    L, Q = _batch(100 + seed, 40, 40, 3000, mixed=True)
    check_plan(L, Q, 16, 4, window=window)


@pytest.mark.parametrize("warps", [1, 3, 8, 64, 100000])
def test_forced_warp_counts(monkeypatch, warps):
    monkeypatch.setenv("KVQ_DECODE_WARPS", str(warps))
    L, Q = _batch(7, 30, 3, 2000, mixed=True)
    plan = check_plan(L, Q, 32, 8)
    if warps == 100000:   # one chunk per warp: every multi-chunk tile is cut
        assert all(n == 1 for n in plan["pieces"]["nchunks"])


def test_non_causal_and_head_sizes(monkeypatch):
    monkeypatch.delenv("KVQ_DECODE_WARPS", raising=False)
    L, Q = _batch(9, 20, 3, 700, mixed=True)
    for D in (64, 128, 256):
        check_plan(L, Q, 16, 8, D=D, causal=False, dtype="int8_per_token_head")


def test_empty_plans():
    plan = check_plan([], [])
    assert plan["pieces"].size == 0 and plan["prefill_tiles"].size == 0
    plan = check_plan([50, 0], [0, 0])
    assert plan["num_chunks"] == [0, 0]


def test_export_refuses_small_arrays():
    import ctypes
    s = kvq.get_scheduler_metadata(1, 8, 2, 64, np.array([100], np.int32),
                                   np.array([0, 1], np.int32), True, 0, "fp8_e4m3")
    buf = np.zeros(1, kvq.PLAN_PIECE)
    rc = kvq.lib.kvq_sched_export_plan(s.handle, buf.ctypes.data, 0, None, 0, None, 0, None, 0)
    assert rc == kvq.E_INVALID_ARG
    s.close()


def test_lockstep_follows_the_row_size(monkeypatch):
    """Rows that are whole 128-byte lines (fp8 at head_dim 128) keep the
    request-major order; per-token-head rows (D + 16 bytes) and 64-byte rows
    are laid out head-major with a warp count that is a multiple of the kv
    heads; KVQ_DECODE_LOCKSTEP forces either; one kv head has nothing to lock."""
    monkeypatch.delenv("KVQ_DECODE_WARPS", raising=False)
    L, Q = _batch(11, 40, 1, 4000, mixed=False)
    assert check_plan(L, Q, 32, 8, D=128, dtype="fp8_e4m3")["lockstep"][0] == 0
    for D, dtype in ((128, "int8_per_token_head"), (64, "fp8_e5m2")):
        plan = check_plan(L, Q, 32, 8, D=D, dtype=dtype)
        assert plan["lockstep"][0] == 1 and plan["num_warps"][0] % 8 == 0
    assert check_plan(L, Q, 8, 1, D=64)["lockstep"][0] == 0
    monkeypatch.setenv("KVQ_DECODE_LOCKSTEP", "1")
    assert check_plan(L, Q, 32, 8, D=128, dtype="fp8_e4m3")["lockstep"][0] == 1
    monkeypatch.setenv("KVQ_DECODE_LOCKSTEP", "0")
    plan = check_plan(L, Q, 32, 8, D=128, dtype="int8_per_token_head")
    assert plan["lockstep"][0] == 0
    assert list(plan["pieces"]["req"]) == sorted(plan["pieces"]["req"])


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("hkv", [2, 3, 8])
def test_lockstep_keeps_stream_k_balance(monkeypatch, seed, hkv):
    """Head-major order keeps the equal stream-K segments: no warp streams
    more than one chunk above the mean, on decode batches of mixed lengths."""
    monkeypatch.delenv("KVQ_DECODE_WARPS", raising=False)
    L, Q = _batch(200 + seed, 64, 1, 8192, mixed=False)
    plan = check_plan(L, Q, 4 * hkv, hkv, D=128, dtype="fp8_per_token_head")
    assert plan["lockstep"][0] == 1
    T, W = plan["num_chunks"][0], plan["num_warps"][0]
    assert int(plan["pieces"]["nchunks"].max()) <= math.ceil(T / W)
