"""The layout contract under a real collective: P = 2 gloo ranks on CPU.

Forward path ("速度、显存与质量", section "剖析单次去噪请求": QKV pack ->
inbound exchange -> QKV unpack): each rank packs its token shard of a seeded
global [T,3,H,D] activation, and for every overlap chunk c exchanges the
chunk's P-slot slab with ``all_to_all_single``; the send and receive split
sizes come only from the library's piece tables (``vf_piece_table`` for the
pack and for the unpack).  Rank p then unpacks and must hold head group p of
every token.  Return path (attention-result pack -> outbound exchange -> final
unpack): each rank splits its head group of the global attention output,
exchanges per chunk, merges, and must hold its token shard with all heads.

The data movement runs in the CPU oracle (no GPU here); what is under test is
that the [chunk][slot] storage and the piece tables are all a real exchange
needs -- also for the opt-in INT8 transport, whose codes and per-head-row
scales travel in the same blocks.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as tmp

pytestmark = pytest.mark.usefixtures("oracle_built", "lib_built")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _bits(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(-(1 << 15), 1 << 15, shape, generator=g, dtype=torch.int32).to(
        torch.int16)


def _exchange(send, send_sizes, recv_sizes):
    """all_to_all_single of 16-bit elements, moved as bytes (bit-exact)."""
    recv = torch.empty(2 * sum(recv_sizes), dtype=torch.uint8)
    dist.all_to_all_single(recv, send.contiguous().view(torch.uint8),
                           [2 * n for n in recv_sizes], [2 * n for n in send_sizes])
    return recv.view(torch.int16)


def _rank_main(rank, world, port, shape, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import sequence_head_relayout_gb300 as vf
        from oracle import loops
        T, H, D, C = shape
        P = world
        Hp = H // P
        shard = -(-T // P)
        a, b = min(T, rank * shard), min(T, (rank + 1) * shard)

        # ---- forward: pack -> per-chunk all-to-all -> unpack
        X = _bits((T, 3, H, D), 1)                       # same seed on every rank
        sent = loops.qkv_pack(X[a:b], P, C)
        ptab = vf.piece_table(vf.OP_QKV_PACK, b - a, H, D, P, C)
        utab = vf.piece_table(vf.OP_QKV_UNPACK, T, H, D, P, C)
        per_tok = 3 * Hp * D
        recv_parts = []
        for c in range(C):
            send_sizes = [ptab[1][c * P + p] * per_tok for p in range(P)]
            lo = ptab[2][c * P]
            send = sent[lo:lo + sum(send_sizes)].contiguous()
            recv_sizes = [utab[1][c * P + r] * per_tok for r in range(P)]
            recv = _exchange(send, send_sizes, recv_sizes)
            assert utab[2][c * P] == sum(p.numel() for p in recv_parts)
            recv_parts.append(recv)
        q, k, v = loops.qkv_unpack_recv(torch.cat(recv_parts), T, H, D, P, C)
        fwd_ok = all(torch.equal(o, X[:, s, rank * Hp:(rank + 1) * Hp])
                     for s, o in enumerate((q, k, v)))

        # ---- return: split -> per-chunk all-to-all -> merge
        A = _bits((T, H, D), 2)
        mine = A[:, rank * Hp:(rank + 1) * Hp]           # head group of this rank
        sent = loops.attn_split(mine, P, C)
        stab = vf.piece_table(vf.OP_ATTN_SPLIT, T, Hp, D, P, C)
        mtab = vf.piece_table(vf.OP_HEAD_MERGE, b - a, H, D, P, C)
        per_tok = Hp * D
        recv_parts = []
        for c in range(C):
            send_sizes = [stab[1][c * P + p] * per_tok for p in range(P)]
            lo = stab[2][c * P]
            send = sent[lo:lo + sum(send_sizes)].contiguous()
            recv_sizes = [mtab[1][c * P + r] * per_tok for r in range(P)]
            recv_parts.append(_exchange(send, send_sizes, recv_sizes))
        merged = loops.head_merge(torch.cat(recv_parts), b - a, H, D, P, C)
        ret_ok = torch.equal(merged, A[a:b])

        # ---- the opt-in lossy transport over the same exchange: INT8 codes and
        # their per-head-row scales travel in the same blocks (a block of n
        # elements carries n / D scales); the receiver's dequantised Q, K, V
        # must equal what the oracle makes of the whole global activation
        # quantised row by row (the quantiser is per head row, so sharding
        # cannot change a code)
        from sequence_head_relayout_gb300 import workloads as W
        Xf = W.finite_rows_(torch.empty((T, 3, H, D), dtype=torch.int16), 5)
        codes, scales = loops.qkv_pack_q(Xf[a:b], P, C, loops.INT8)
        per_tok = 3 * Hp * D
        rc, rs = [], []
        for c in range(C):
            send_sizes = [ptab[1][c * P + p] * per_tok for p in range(P)]
            recv_sizes = [utab[1][c * P + r] * per_tok for r in range(P)]
            lo = ptab[2][c * P]
            send_c = codes[lo:lo + sum(send_sizes)].contiguous()
            recv_c = torch.empty(sum(recv_sizes), dtype=torch.uint8)
            dist.all_to_all_single(recv_c, send_c.view(torch.uint8), recv_sizes, send_sizes)
            rc.append(recv_c)
            send_s = scales[lo // D:(lo + sum(send_sizes)) // D].contiguous()
            recv_s = torch.empty(sum(recv_sizes) // D, dtype=torch.float32)
            dist.all_to_all_single(recv_s, send_s, [n // D for n in recv_sizes],
                                   [n // D for n in send_sizes])
            rs.append(recv_s)
        got = loops.qkv_unpack_q(torch.cat(rc), torch.cat(rs), T, H, D, P, C, loops.INT8)
        # reference: every head row of the global tensor quantised and
        # dequantised alone (P = 1, C = 1 split of a [rows, 1, D] view)
        rows = Xf.view(T * 3 * H, 1, D)
        c1, s1 = loops.attn_split_q(rows, 1, 1, loops.INT8)
        ref = loops.head_merge_q(c1, s1, T * 3 * H, 1, D, 1, 1, loops.INT8).view(T, 3, H, D)
        lossy_ok = all(torch.equal(o, ref[:, s, rank * Hp:(rank + 1) * Hp])
                       for s, o in enumerate(got))
        out[rank] = (bool(fwd_ok), bool(ret_ok), bool(lossy_ok))
    finally:
        dist.destroy_process_group()


def _run(world, shape):
    ctx = tmp.get_context("spawn")
    out = ctx.Manager().dict()
    tmp.start_processes(_rank_main, args=(world, _free_port(), shape, out), nprocs=world,
                        join=True, start_method="spawn")
    return dict(out)


def test_two_rank_exchange_round_trips():
    out = _run(2, (37, 8, 16, 4))                 # T odd: short last shard and chunk
    assert out == {0: (True, True, True), 1: (True, True, True)}


def test_two_rank_exchange_pages_like_geometry():
    out = _run(2, (1001, 28, 8, 4))               # pages' H and P, small T and D
    assert out == {0: (True, True, True), 1: (True, True, True)}
