"""Seeded fuzz of the C ABI's host-side checks, without a GPU.

Every entry point gets thousands of random argument sets mixing ordinary
values with extremes: zero, negative, 2^30 and 2^30 + 1 (the extent limit),
2^31, values near 2^62 and 2^63 - 1 whose products overflow int64, odd and
zero strides, NULL and misaligned pointers, chunk ranges outside [0, C],
unknown ops, orders and formats.  The library must answer each with one of
its documented statuses and never crash; a call may return VF_OK only when it
moves nothing (the header's rule: an empty element count or chunk range
returns without touching the GPU).  Pointers are small fake values: the
library queries pointers but never dereferences them on the host, and no
fake value is a device address, so nothing is ever launched.  The piece
table and the size functions are checked against their documented results
and must never write past the capacity they are given.
"""
import ctypes
import random

import pytest

import sequence_head_relayout_gb300 as vf

I64 = ctypes.c_int64
STATUSES = {0, -1, -2, -3, -4, -5}
EXTREMES = [0, 1, 2, 3, 7, 8, 64, 128, 1 << 20, 1 << 30, (1 << 30) + 1, 1 << 31,
            1 << 40, 1 << 62, (1 << 63) - 1, -1, -7, -(1 << 63)]
FAKE = [None, 0x1000, 0x2000, 0x10000, 0x1001, 0x100008]


@pytest.fixture(scope="module")
def L(lib_built):
    return vf.lib()


def _val(rng, lo=0, hi=300):
    return rng.choice(EXTREMES) if rng.random() < 0.35 else rng.randint(lo, hi)


def _arr(vals):
    return (I64 * len(vals))(*vals)


def _moves_nothing(T, H, D, c_count):
    return T == 0 or H == 0 or D == 0 or c_count == 0


def test_entry_points_fuzz(L):
    rng = random.Random(20261203)
    counts = {}
    for _ in range(6000):
        T, H, D = _val(rng), _val(rng, 1, 64), _val(rng, 1, 256)
        P, C = _val(rng, 1, 8), _val(rng, 1, 8)
        c0, cn = _val(rng, -2, 10), _val(rng, -2, 10)
        st4 = _arr([_val(rng, 0, 1 << 16) for _ in range(4)])
        st3 = _arr([_val(rng, 0, 1 << 16) for _ in range(3)])
        src, dst, q, k, v, sc = (rng.choice(FAKE) for _ in range(6))
        which = rng.randrange(12)
        if which == 0:
            rc, cn = L.vf_qkv_pack(src, st4, T, H, D, P, C, dst, None), C
        elif which == 1:
            rc, cn = L.vf_attn_split(src, st3, T, H, D, P, C, dst, None), C
        elif which == 2:
            rc, cn = L.vf_head_merge(src, rng.choice([st3, None]), T, H, D, P, C, dst,
                                     None), C
        elif which == 3:
            rc, cn = L.vf_qkv_unpack(src, T, H, D, P, C, q, k, v,
                                     rng.choice([st3, None]), None), C
        elif which == 4:
            rc = L.vf_qkv_pack_chunks(src, st4, T, H, D, P, C, c0, cn, dst, None)
        elif which == 5:
            rc = L.vf_attn_split_chunks(src, st3, T, H, D, P, C, c0, cn, dst, None)
        elif which == 6:
            rc = L.vf_head_merge_chunks(src, st3, T, H, D, P, C, c0, cn, dst, None)
        elif which == 7:
            rc = L.vf_qkv_unpack_chunks(src, T, H, D, P, C, c0, cn, q, k, v, st3, None)
        elif which == 8:
            rc = L.vf_qkv_pack3(q, k, v, st3, T, H, D, P, C, c0, cn, dst, None)
        else:
            d = vf._Desc(op=rng.randrange(-1, 6), order=rng.randrange(-1, 3), T=T, H=H, D=D,
                         P=P, C=C, c_begin=c0, c_count=cn, packed=dst)
            for i in range(3):
                d.strided[i] = rng.choice(FAKE)
                d.strides[i] = st3[i]
            if which == 9:
                rc = L.vf_relayout(ctypes.byref(d), None)
            elif which == 10:
                rc = L.vf_relayout_q(ctypes.byref(d), rng.randrange(-1, 4), sc, None)
            else:
                rc = L.vf_relayout_q(None, 1, sc, None)
        assert rc in STATUSES, (which, rc)
        if rc == 0:
            assert _moves_nothing(T, H, D, cn), (which, T, H, D, P, C, c0, cn)
        counts[rc] = counts.get(rc, 0) + 1
    # the fuzz reached the argument checks and the pointer checks alike
    assert counts.get(-1, 0) > 100 and counts.get(-2, 0) > 10
    assert counts.get(0, 0) > 10 and counts.get(-4, 0) + counts.get(-1, 0) > 1000


def test_lossy_named_entry_points_fuzz(L):
    rng = random.Random(7)
    for _ in range(2000):
        T, H, D = _val(rng), _val(rng, 1, 64), _val(rng, 1, 256)
        P, C = _val(rng, 1, 8), _val(rng, 1, 8)
        st4 = _arr([_val(rng, 0, 1 << 16) for _ in range(4)])
        st3 = _arr([_val(rng, 0, 1 << 16) for _ in range(3)])
        a, b, c, q, k, v = (rng.choice(FAKE + [0x1004]) for _ in range(6))
        which = rng.randrange(4)
        if which == 0:
            rc = L.vf_qkv_pack_int8(a, st4, T, H, D, P, C, b, c, None)
        elif which == 1:
            rc = L.vf_qkv_unpack_int8(a, c, T, H, D, P, C, q, k, v, st3, None)
        elif which == 2:
            rc = L.vf_attn_split_fp8(a, st3, T, H, D, P, C, b, c, None)
        else:
            rc = L.vf_head_merge_fp8(a, c, st3, T, H, D, P, C, b, None)
        assert rc in STATUSES
        if rc == 0:
            assert _moves_nothing(T, H, D, C)


def test_sizes_and_piece_tables_fuzz(L):
    rng = random.Random(99)
    guard = -0x5A5A5A5A
    for _ in range(4000):
        op, order = rng.randrange(-1, 5), rng.randrange(-1, 3)
        T, H, D = _val(rng), _val(rng, 1, 64), _val(rng, 1, 256)
        P, C = _val(rng, 1, 12), _val(rng, 1, 12)
        n = L.vf_packed_elems(op, T, H, D, P, C)
        ns = L.vf_scale_count(op, T, H, D, P, C)
        assert n < 0 and n in STATUSES or n >= 0
        assert (n < 0) == (ns < 0)
        if n >= 0:
            slabs = 3 if op in (0, 3) else 1
            heads = H if op in (0, 1, 2) else H // P
            assert n == slabs * T * heads * D
            assert ns == (n // D if D else 0)
        cap = rng.randrange(0, 40)
        arrs = [(I64 * (cap + 4))(*([guard] * (cap + 4))) for _ in range(3)]
        got = L.vf_piece_table_ex(op, order, T, H, D, P, C, *arrs, cap)
        assert got in STATUSES or 0 < got <= cap
        for a in arrs:                                  # nothing written past cap
            assert list(a)[cap:] == [guard] * 4
        if got > 0:
            assert got == P * C and n >= 0
            tok_len = list(arrs[1])[:got]
            assert all(x >= 0 for x in tok_len)
            total = sum(tok_len)
            assert total == (T if op in (1, 3) else T * P)
