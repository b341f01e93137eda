"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test checks the oracle against something it cannot agree with by
construction: hand-derived worked examples, the byte counts printed by the
pages' allocation screen, library routines in special cases, a brute-force
bijection on iota payloads, the permutation invariant, round trips, a virtual
sequence-head exchange, and the second (PyTorch chain) oracle.  The last
group plants plausible mistakes in copies of the chain oracle and shows that
the pins reject every one of them.
"""
import random

import pytest
import torch

from oracle import chain, loops
from sequence_head_relayout_gb300 import workloads as W
from tests import _golden

pytestmark = pytest.mark.usefixtures("oracle_built")


def iota(shape):
    n = 1
    for s in shape:
        n *= s
    return torch.arange(n, dtype=torch.int32).to(torch.int16).view(*shape)


def rand_bits(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(-(1 << 15), 1 << 15, shape, generator=g, dtype=torch.int32).to(torch.int16)


def strided_view(shape, seed, kind):
    """A view of the given logical shape whose strides are not contiguous."""
    g = random.Random(seed)
    if kind == "contiguous":
        return rand_bits(shape, seed)
    if kind == "padded":
        pad = g.randint(1, 9)
        base = rand_bits((shape[0], _prod(shape[1:]) + pad), seed)
        return base[:, :_prod(shape[1:])].unflatten(1, shape[1:])
    if kind == "permuted":
        # allocate with the two middle-ish axes swapped, then view back
        order = list(range(len(shape)))
        order[0], order[-2] = order[-2], order[0]
        alloc = [shape[i] for i in order]
        base = rand_bits(tuple(alloc), seed)
        inv = [order.index(i) for i in range(len(shape))]
        return base.permute(*inv)
    if kind == "dstride":
        base = rand_bits(tuple(shape[:-1]) + (2 * shape[-1],), seed)
        return base[..., ::2]
    raise ValueError(kind)


def _prod(xs):
    n = 1
    for x in xs:
        n *= x
    return n


def bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    return a.shape == b.shape and torch.equal(a.view(torch.int16), b.view(torch.int16))


# --------------------------------------------------------------------------
# 1. Hand-derived worked examples (tests/golden/*.txt)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", _golden.examples("pack"))
def test_golden_pack(name):
    g = _golden.load(name)
    T, H, D, P, C = g["T"], g["H"], g["D"], g["P"], g["C"]
    src = iota((T, 3, H, D))
    assert loops.qkv_pack(src, P, C).tolist() == g["expected"]
    assert chain.qkv_pack(src, P, C).tolist() == g["expected"]


@pytest.mark.parametrize("name", _golden.examples("split"))
def test_golden_split(name):
    g = _golden.load(name)
    T, H, D, P, C = g["T"], g["H"], g["D"], g["P"], g["C"]
    src = iota((T, H, D))
    assert loops.attn_split(src, P, C).tolist() == g["expected"]
    assert chain.attn_split(src, P, C).tolist() == g["expected"]


@pytest.mark.parametrize("name", _golden.examples("merge"))
def test_golden_merge(name):
    g = _golden.load(name)
    T, H, D, P, C = g["T"], g["H"], g["D"], g["P"], g["C"]
    src = iota((T * H * D,))
    assert loops.head_merge(src, T, H, D, P, C).reshape(-1).tolist() == g["expected"]
    assert chain.head_merge(src, T, H, D, P, C).reshape(-1).tolist() == g["expected"]


def test_golden_piece_tables_ragged():
    g = _golden.load("piece_tables_ragged.txt")
    T, H, D, P, C = 55413, 32, 64, 4, 4
    for op, key in ((loops.OP_QKV_PACK, "pack"), (loops.OP_ATTN_SPLIT, "split"),
                    (loops.OP_HEAD_MERGE, "merge")):
        a, b, c = loops.piece_table(op, T, H, D, P, C)
        assert a == g[key + "_tok_start"], key
        assert b == g[key + "_tok_len"], key
        assert c == g[key + "_packed_off"], key


# --------------------------------------------------------------------------
# 2. Byte counts printed on the pages (allocation screen)
# --------------------------------------------------------------------------

def test_page_byte_counts():
    g = _golden.load("page_byte_counts.txt")
    T, H, D, P, C = g["T"], g["H"], g["D"], g["P"], g["C"]
    # zero-stride sources: the oracle reads one element many times, so only the
    # destination has to exist; the element count is the oracle's own cursor.
    one4 = torch.zeros(1, dtype=torch.int16).expand(T, 3, H, D)
    packed = loops.qkv_pack(one4, P, C)
    assert packed.numel() * 2 == g["pack_direct_bytes"]
    assert 2 * packed.numel() * 2 == g["pack_reference_bytes"]
    del packed
    one3 = torch.zeros(1, dtype=torch.int16).expand(T, H, D)
    split = loops.attn_split(one3, P, C)
    merged_src = torch.zeros(T * H * D, dtype=torch.int16)
    merged = loops.head_merge(merged_src, T, H, D, P, C,
                              out=torch.zeros(1, dtype=torch.int16).expand(T, H, D))
    assert merged.numel() * 2 == g["merge_direct_bytes"]
    assert 2 * merged_src.numel() * 2 == g["merge_reference_bytes"]
    # the pages' split output per call is one overlap chunk's quarter
    assert split.numel() * 2 == C * g["split_per_call_bytes"]


# --------------------------------------------------------------------------
# 3. Special cases that reduce to a library routine
# --------------------------------------------------------------------------

@pytest.mark.parametrize("seed", [0, 1])
def test_library_reductions(seed):
    T, H, D = 7, 6, 5
    x4 = rand_bits((T, 3, H, D), seed)
    # one slot, one chunk: the pack is stack(q, k, v) made contiguous
    ref = torch.stack([x4[:, 0], x4[:, 1], x4[:, 2]]).contiguous().reshape(-1)
    assert bits_equal(loops.qkv_pack(x4, 1, 1), ref)
    # one head per slot, one chunk: slot p is head p -> axes (h, s, t, d)
    ref = x4.permute(2, 1, 0, 3).contiguous().reshape(-1)
    assert bits_equal(loops.qkv_pack(x4, H, 1), ref)

    x3 = rand_bits((T, H, D), seed + 10)
    flat = x3.reshape(-1)
    # merge with one slot and one chunk is a reshape of the received buffer
    assert bits_equal(loops.head_merge(flat, T, H, D, 1, 1), x3)
    # merge with one head per slot and one chunk: the buffer is [H][T][D]
    assert bits_equal(loops.head_merge(flat, T, H, D, H, 1),
                      flat.view(H, T, D).permute(1, 0, 2).contiguous())
    # split into consecutive token shards with one chunk, or one shard with
    # any number of chunks, keeps token order: a plain contiguous copy
    for P, C in ((1, 1), (3, 1), (1, 4), (T, 1)):
        assert bits_equal(loops.attn_split(x3, P, C), flat), (P, C)


# --------------------------------------------------------------------------
# 4. Brute force on iota payloads: the map is a bijection
# --------------------------------------------------------------------------

def test_iota_bijection_tiny():
    cfg = W.CONFIGS["tiny"]
    src, _ = W.pack_source(cfg, payload="iota")
    n = 3 * cfg.T * cfg.H * cfg.D
    assert n < (1 << 16)
    out = loops.qkv_pack(src, cfg.P, cfg.C).to(torch.int32) & 0xFFFF
    assert torch.equal(out.sort().values, torch.arange(n, dtype=torch.int32))
    s3, _ = W.split_source(cfg, payload="iota")
    out = loops.attn_split(s3, cfg.P, cfg.C).to(torch.int32) & 0xFFFF
    assert torch.equal(out.sort().values, torch.arange(n // 3, dtype=torch.int32))
    m = W.merge_source(cfg, payload="iota")
    out = loops.head_merge(m, cfg.T, cfg.H, cfg.D, cfg.P, cfg.C).reshape(-1).to(torch.int32) & 0xFFFF
    assert torch.equal(out.sort().values, torch.arange(n // 3, dtype=torch.int32))


@pytest.mark.parametrize("shape", [(5, 4, 3, 2, 3), (9, 6, 4, 3, 4), (3, 2, 8, 2, 5)])
def test_iota_bijection_ragged(shape):
    T, H, D, P, C = shape
    for out, n in ((loops.qkv_pack(iota((T, 3, H, D)), P, C), 3 * T * H * D),
                   (loops.attn_split(iota((T, H, D)), P, C), T * H * D),
                   (loops.head_merge(iota((T * H * D,)), T, H, D, P, C).reshape(-1), T * H * D)):
        assert torch.equal(out.to(torch.int32).sort().values, torch.arange(n, dtype=torch.int32))


# --------------------------------------------------------------------------
# 5. Permutation invariant at the 4k shape
# --------------------------------------------------------------------------

def _hist(t):
    return torch.bincount(t.reshape(-1).to(torch.int32) & 0xFFFF, minlength=1 << 16)


def test_histogram_invariant_4k():
    cfg = W.CONFIGS["4k"]
    src, _ = W.pack_source(cfg)
    assert torch.equal(_hist(loops.qkv_pack(src, cfg.P, cfg.C)), _hist(src))
    s3, _ = W.split_source(cfg)
    assert torch.equal(_hist(loops.attn_split(s3, cfg.P, cfg.C)), _hist(s3))
    m = W.merge_source(cfg)
    assert torch.equal(_hist(loops.head_merge(m, cfg.T, cfg.H, cfg.D, cfg.P, cfg.C)), _hist(m))


# --------------------------------------------------------------------------
# 6. Round trips
# --------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(4096, 32, 128, 2, 4), (13, 6, 3, 3, 4), (2, 4, 2, 4, 5),
                                   (0, 4, 8, 2, 3)])
def test_round_trips(shape):
    T, H, D, P, C = shape
    x4 = rand_bits((T, 3, H, D), 7)
    assert bits_equal(loops.qkv_unpack(loops.qkv_pack(x4, P, C), T, H, D, P, C), x4)
    x3 = rand_bits((T, H, D), 8)
    assert bits_equal(loops.attn_unsplit(loops.attn_split(x3, P, C), T, H, D, P, C), x3)
    assert bits_equal(loops.head_merge(loops.head_split(x3, P, C), T, H, D, P, C), x3)


def virtual_exchange(A: torch.Tensor, P: int, C: int):
    """Ulysses return path on P virtual ranks, on CPU.

    Rank r holds head group r of every token (after attention) and splits it;
    chunk c of rank r's slot q travels to rank q, which stores it at slot r of
    its chunk-c block; rank q then merges and must hold A's token shard q.
    """
    T, H, D = A.shape
    Hp = H // P
    sent = [loops.attn_split(A[:, r * Hp:(r + 1) * Hp], P, C) for r in range(P)]
    tables = loops.piece_table(loops.OP_ATTN_SPLIT, T, Hp, D, P, C)
    results = []
    for q in range(P):
        parts = []
        for c in range(C):
            for r in range(P):
                e = c * P + q
                start, length, off = tables[0][e], tables[1][e], tables[2][e]
                parts.append(sent[r][off:off + length * Hp * D])
        recv = torch.cat(parts)
        n_q = tables[1][q] + sum(tables[1][c * P + q] for c in range(1, C))
        results.append((loops.head_merge(recv, n_q, H, D, P, C), n_q))
    return results


@pytest.mark.parametrize("shape", [(37, 8, 4, 2, 4), (55, 12, 2, 4, 4), (5, 4, 2, 4, 2),
                                   (64, 4, 16, 2, 1)])
def test_virtual_exchange_split_then_merge(shape):
    T, H, D, P, C = shape
    A = rand_bits((T, H, D), 11)
    shard = -(-T // P)
    t0 = 0
    for q, (merged, n_q) in enumerate(virtual_exchange(A, P, C)):
        expect = A[min(T, q * shard):min(T, (q + 1) * shard)]
        assert n_q == expect.shape[0]
        assert bits_equal(merged, expect), q
        t0 += n_q
    assert t0 == T


# --------------------------------------------------------------------------
# 7. The two oracles agree on random shapes, strides and payloads
# --------------------------------------------------------------------------

SHAPES = [(64, 4, 16, 2, 1), (33, 6, 8, 3, 4), (7, 8, 3, 8, 16), (1, 2, 1, 2, 3),
          (100, 12, 2, 4, 7), (0, 4, 4, 2, 2), (9, 1, 5, 1, 2)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("kind", ["contiguous", "padded", "permuted", "dstride"])
def test_loops_agree_with_chain(shape, kind):
    T, H, D, P, C = shape
    seed = hash((shape, kind)) & 0xFFFF
    x4 = strided_view((T, 3, H, D), seed, kind)
    assert bits_equal(loops.qkv_pack(x4, P, C), chain.qkv_pack(x4, P, C))
    x3 = strided_view((T, H, D), seed + 1, kind)
    assert bits_equal(loops.attn_split(x3, P, C), chain.attn_split(x3, P, C))
    flat = rand_bits((T * H * D,), seed + 2)
    out = strided_view((T, H, D), seed + 3, kind)
    got = loops.head_merge(flat, T, H, D, P, C, out=out)
    assert bits_equal(got.contiguous(), chain.head_merge(flat, T, H, D, P, C))


def test_special_patterns_survive():
    vals = [v - 0x10000 if v >= 0x8000 else v for v in W.SPECIAL_BITS]
    x = torch.tensor(vals * 4, dtype=torch.int16).view(2, 3, 2, 2)
    out = loops.qkv_pack(x, 2, 2)
    assert sorted(out.tolist()) == sorted(x.reshape(-1).tolist())


def test_oracle_rejects_bad_arguments():
    lib = loops.lib()
    s = (loops._I64 * 4)(1, 1, 1, 1)
    assert lib.oracle_qkv_pack(None, s, 4, 3, 2, 2, 1, None) < 0      # H % P != 0
    assert lib.oracle_attn_split(None, s, 4, 3, 2, 0, 1, None) < 0    # P < 1
    assert lib.oracle_head_merge(None, 4, 4, 2, 2, 0, None, s) < 0    # C < 1


# --------------------------------------------------------------------------
# 8. Planted mistakes: each plausible slip in the chain fails some pin
# --------------------------------------------------------------------------

def _pack_mutant(kind):
    def f(src, P, C):
        x = src.view(torch.int16)
        T, _, H, D = x.shape
        stacked = torch.stack(x.unbind(1))
        sizes = chain.part_sizes(T, C)
        if kind == "floor_quota":
            q = T // C
            sizes = [q] * (C - 1) + [T - q * (C - 1)]
        blocks = []
        for ch in torch.split(stacked, sizes, dim=1):
            if kind == "round_robin_heads":
                g = ch.unflatten(2, (H // P, P)).permute(3, 0, 1, 2, 4)
            else:
                g = ch.unflatten(2, (P, H // P))
                perm = {"token_outside_qkv": (2, 1, 0, 3, 4),
                        "d_before_head": (2, 0, 1, 4, 3)}.get(kind, (2, 0, 1, 3, 4))
                g = g.permute(*perm)
            blocks.append(g.contiguous().reshape(-1))
        if kind == "slot_outside_chunk":
            n = len(blocks)
            per = [b.view(P, -1) for b in blocks]
            return torch.cat([per[c][p] for p in range(P) for c in range(n)])
        return torch.cat(blocks)
    return f


@pytest.mark.parametrize("kind", ["floor_quota", "round_robin_heads", "token_outside_qkv",
                                  "d_before_head", "slot_outside_chunk"])
def test_pins_catch_planted_pack_mistakes(kind):
    g = _golden.load("pack_T3_H4_D2_P2_C2.txt")
    src = iota((g["T"], 3, g["H"], g["D"]))
    assert _pack_mutant(kind)(src, g["P"], g["C"]).tolist() != g["expected"]
    assert _pack_mutant("none")(src, g["P"], g["C"]).tolist() == g["expected"]


def test_pins_catch_planted_split_mistake():
    # a split that chunks every shard with the global quota ceil(T/C) instead
    # of its own ceil(n_p/C) breaks the hand example and the exchange identity
    def split_global_quota(x, P, C):
        T = x.shape[0]
        q = -(-T // C)
        shards = torch.split(x, chain.part_sizes(T, P), dim=0)
        blocks = []
        for c in range(C):
            for s in shards:
                blocks.append(s[c * q:(c + 1) * q].contiguous().reshape(-1))
        return torch.cat(blocks)
    g = _golden.load("split_T5_H2_D2_P2_C2.txt")
    src = iota((g["T"], g["H"], g["D"]))
    assert split_global_quota(src, g["P"], g["C"]).tolist() != g["expected"]


# --------------------------------------------------------------------------
# 9. Receive-side QKV unpack
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", _golden.examples("unpack"))
def test_golden_unpack(name):
    g = _golden.load(name)
    T, H, D, P, C = g["T"], g["H"], g["D"], g["P"], g["C"]
    recv = iota((3 * T * (H // P) * D,))
    for impl in (loops.qkv_unpack_recv, chain.qkv_unpack_recv):
        q, k, v = impl(recv, T, H, D, P, C)
        assert q.reshape(-1).tolist() == g["expected_q"]
        assert k.reshape(-1).tolist() == g["expected_k"]
        assert v.reshape(-1).tolist() == g["expected_v"]


def forward_exchange(X: torch.Tensor, P: int, C: int):
    """Ulysses forward path on P virtual ranks, on CPU: rank r packs its token
    shard of the global [T,3,H,D] activation; block (c, p) of rank r travels to
    rank p, which stores it at source slot r of its chunk-c block."""
    T, _, H, D = X.shape
    shard = -(-T // P)
    bounds = [(min(T, r * shard), min(T, (r + 1) * shard)) for r in range(P)]
    sent, tables = [], []
    for a, b in bounds:
        sent.append(loops.qkv_pack(X[a:b], P, C))
        tables.append(loops.piece_table(loops.OP_QKV_PACK, b - a, H, D, P, C))
    recv = []
    for p in range(P):
        parts = []
        for c in range(C):
            for r in range(P):
                e = c * P + p
                length, off = tables[r][1][e], tables[r][2][e]
                parts.append(sent[r][off:off + 3 * length * (H // P) * D])
        recv.append(torch.cat(parts))
    return recv


@pytest.mark.parametrize("shape", [(37, 8, 4, 2, 4), (55, 12, 2, 4, 4), (5, 4, 2, 4, 2),
                                   (64, 4, 16, 2, 1), (9, 6, 3, 3, 5)])
def test_virtual_exchange_pack_then_unpack(shape):
    T, H, D, P, C = shape
    X = rand_bits((T, 3, H, D), 21)
    Hp = H // P
    for p, recv in enumerate(forward_exchange(X, P, C)):
        q, k, v = loops.qkv_unpack_recv(recv, T, H, D, P, C)
        for s, out in enumerate((q, k, v)):
            assert bits_equal(out, X[:, s, p * Hp:(p + 1) * Hp].contiguous()), (p, s)


def test_unpack_library_reduction():
    T, H, D = 11, 6, 4
    recv = rand_bits((3 * T * H * D,), 5)
    q, k, v = loops.qkv_unpack_recv(recv, T, H, D, 1, 1)
    ref = recv.view(3, T, H, D)
    for s, out in enumerate((q, k, v)):
        assert bits_equal(out, ref[s])


@pytest.mark.parametrize("shape", SHAPES)
def test_unpack_loops_agree_with_chain(shape):
    T, H, D, P, C = shape
    recv = rand_bits((3 * T * (H // P) * D,), 31)
    want = chain.qkv_unpack_recv(recv, T, H, D, P, C)
    # strided outputs: [H/P, T, D] allocations viewed as [T, H/P, D]
    outs = tuple(torch.zeros((H // P, T, D), dtype=torch.int16).permute(1, 0, 2)
                 for _ in range(3))
    got = loops.qkv_unpack_recv(recv, T, H, D, P, C, outs=outs)
    for a, b in zip(got, want):
        assert bits_equal(a.contiguous(), b)


def test_unpack_iota_bijection():
    T, H, D, P, C = 13, 8, 3, 4, 3
    n = 3 * T * (H // P) * D
    out = torch.cat([o.reshape(-1) for o in loops.qkv_unpack_recv(iota((n,)), T, H, D, P, C)])
    assert torch.equal(out.to(torch.int32).sort().values, torch.arange(n, dtype=torch.int32))


def test_pins_catch_planted_unpack_mistake():
    # chunking every source rank's shard with the global quota ceil(T/C)
    def unpack_global_quota(recv, T, H, D, P, C):
        flat = recv.reshape(-1)
        Hp = H // P
        q = -(-T // C)
        shard = chain.part_sizes(T, P)
        per_rank = [[] for _ in range(P)]
        off = 0
        for c in range(C):
            for r in range(P):
                L = max(0, min(q, shard[r] - c * q))
                n = 3 * L * Hp * D
                per_rank[r].append(flat[off:off + n].view(3, L, Hp, D))
                off += n
        full = torch.cat([torch.cat(b, 1) for b in per_rank], 1)
        return tuple(full[s].contiguous() for s in range(3))
    g = _golden.load("unpack_T5_H4_D1_P2_C2.txt")
    recv = iota((30,))
    q, _, _ = unpack_global_quota(recv, 5, 4, 1, 2, 2)
    assert q.reshape(-1).tolist() != g["expected_q"]


# --------------------------------------------------------------------------
# 10. Slot-major ([p][c]) block order
# --------------------------------------------------------------------------

def test_golden_slot_major_pack():
    g = _golden.load("slotmajor_pack_T3_H4_D2_P2_C2.txt")
    T, H, D, P, C = g["T"], g["H"], g["D"], g["P"], g["C"]
    cp = loops.qkv_pack(iota((T, 3, H, D)), P, C)
    assert loops.to_slot_major(0, cp, T, H, D, P, C).tolist() == g["expected"]
    assert chain.to_slot_major(0, cp, T, H, D, P, C).tolist() == g["expected"]


@pytest.mark.parametrize("shape", [(7, 6, 5, 3, 4), (55, 8, 2, 4, 4), (5, 4, 2, 4, 2),
                                   (1, 2, 3, 2, 5), (0, 2, 2, 2, 2)])
def test_slot_major_library_reductions(shape):
    T, H, D, P, C = shape
    x3 = rand_bits((T, H, D), 3)
    # the split's shards are consecutive token ranges and a shard's chunks are
    # consecutive too: in slot-major order the split is a contiguous copy
    pc = loops.to_slot_major(1, loops.attn_split(x3, P, C), T, H, D, P, C)
    assert bits_equal(pc, x3.reshape(-1))
    # a slot-major merge source holds head group p of every token at slot p:
    # it is a [P][T][H/P][D] tensor and the merge is a permute
    flat = rand_bits((T * H * D,), 4)
    cp = loops.to_chunk_major(2, flat, T, H, D, P, C)
    merged = loops.head_merge(cp, T, H, D, P, C)
    assert bits_equal(merged, flat.view(P, T, H // P, D).permute(1, 0, 2, 3).reshape(T, H, D))


@pytest.mark.parametrize("op", [0, 1, 2, 3])
@pytest.mark.parametrize("shape", [(33, 6, 8, 3, 4), (7, 8, 3, 8, 16), (100, 12, 2, 4, 7),
                                   (9, 4, 5, 2, 1)])
def test_reorder_loops_agree_with_chain_and_invert(op, shape):
    T, H, D, P, C = shape
    n = {0: 3 * T * H * D, 1: T * H * D, 2: T * H * D, 3: 3 * T * (H // P) * D}[op]
    cp = rand_bits((n,), op + 40)
    pc = loops.to_slot_major(op, cp, T, H, D, P, C)
    assert bits_equal(pc, chain.to_slot_major(op, cp, T, H, D, P, C))
    assert bits_equal(loops.to_chunk_major(op, pc, T, H, D, P, C), cp)
    if C == 1 or P == 1:                      # one index: both orders coincide
        assert bits_equal(pc, cp)
