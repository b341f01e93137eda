"""The C ABI on the host, without a GPU.

Checks that ``libvf_relayout.so`` loads and exports every function that
``include/*.h`` declares, that its pure-host functions (sizes and piece
tables) agree with the oracle and the hand-derived fixtures, and that every
rejected argument is rejected before the library touches CUDA (fake pointer
values are safe here because nothing is dereferenced or launched).
"""
import ctypes
import glob
import os
import re
import subprocess

import pytest

import sequence_head_relayout_gb300 as vf
from oracle import loops
from tests import _golden

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
I64 = ctypes.c_int64


@pytest.fixture(scope="module")
def L(lib_built):
    return vf.lib()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(vf_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = declared_functions()
    for want in ("vf_qkv_pack", "vf_attn_split", "vf_head_merge", "vf_packed_elems",
                 "vf_piece_table", "vf_status_string", "vf_qkv_unpack", "vf_qkv_pack3",
                 "vf_qkv_pack_chunks", "vf_attn_split_chunks", "vf_head_merge_chunks",
                 "vf_qkv_unpack_chunks"):
        assert want in names


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", vf.LIB_PATH], check=True,
                         capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (vf_[a-z0-9_]+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(L, n)


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "vf_relayout.h"\nint main(void){return VF_OK;}\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-c", str(src), "-o", str(tmp_path / "t.o")], check=True)


def test_status_strings(L):
    for s in (0, -1, -2, -3, -4, -5, 7):
        assert isinstance(L.vf_status_string(s), bytes) and L.vf_status_string(s)


def test_packed_elems_matches_page_byte_counts(L):
    g = _golden.load("page_byte_counts.txt")
    T, H, D, P, C = g["T"], g["H"], g["D"], g["P"], g["C"]
    assert vf.packed_elems(vf.OP_QKV_PACK, T, H, D, P, C) * 2 == g["pack_direct_bytes"]
    assert vf.packed_elems(vf.OP_HEAD_MERGE, T, H, D, P, C) * 2 == g["merge_direct_bytes"]
    assert vf.packed_elems(vf.OP_ATTN_SPLIT, T, H, D, P, C) * 2 == C * g["split_per_call_bytes"]


def test_piece_tables_match_hand_derivation(L):
    g = _golden.load("piece_tables_ragged.txt")
    for op, key in ((vf.OP_QKV_PACK, "pack"), (vf.OP_ATTN_SPLIT, "split"),
                    (vf.OP_HEAD_MERGE, "merge")):
        a, b, c = vf.piece_table(op, 55413, 32, 64, 4, 4)
        assert a == g[key + "_tok_start"]
        assert b == g[key + "_tok_len"]
        assert c == g[key + "_packed_off"]


@pytest.mark.parametrize("shape", [(0, 4, 8, 2, 3), (1, 2, 2, 2, 5), (5, 4, 1, 4, 2),
                                   (55414, 28, 128, 2, 4), (200000, 32, 128, 8, 4),
                                   (37, 6, 16, 3, 7), (4, 6, 2, 6, 16)])
def test_piece_tables_match_oracle(L, shape):
    T, H, D, P, C = shape
    for op in (0, 1, 2, 3):
        if op != 1 and H % P:
            continue
        assert vf.piece_table(op, T, H, D, P, C) == loops.piece_table(op, T, H, D, P, C)


def _call(L, fn, src, strides, T, H, D, P, C, dst):
    arr = None if strides is None else (I64 * len(strides))(*strides)
    return getattr(L, fn)(src, arr, T, H, D, P, C, dst, None)


FAKE_SRC, FAKE_DST = 1 << 40, 1 << 41


@pytest.mark.parametrize("args,status", [
    (("vf_qkv_pack", FAKE_SRC, (96, 32, 8, 1), 4, 4, 8, 3, 1, FAKE_DST), -1),   # H % P
    (("vf_qkv_pack", FAKE_SRC, (96, 32, 8, 1), 4, 4, 8, 0, 1, FAKE_DST), -1),   # P < 1
    (("vf_qkv_pack", FAKE_SRC, (96, 32, 8, 1), 4, 4, 8, 2, 0, FAKE_DST), -1),   # C < 1
    (("vf_qkv_pack", FAKE_SRC, (96, 32, 8, 1), -1, 4, 8, 2, 1, FAKE_DST), -1),  # T < 0
    (("vf_qkv_pack", FAKE_SRC, (96, -32, 8, 1), 4, 4, 8, 2, 1, FAKE_DST), -1),  # negative stride
    (("vf_qkv_pack", FAKE_SRC, None, 4, 4, 8, 2, 1, FAKE_DST), -1),             # no strides
    (("vf_qkv_pack", None, (96, 32, 8, 1), 4, 4, 8, 2, 1, FAKE_DST), -1),       # null src
    (("vf_qkv_pack", FAKE_SRC, (96, 32, 8, 1), 4, 4, 8, 2, 1, None), -1),       # null dst
    (("vf_qkv_pack", FAKE_SRC, (96, 32, 8, 1), (1 << 30) + 1, 4, 8, 2, 1, FAKE_DST), -1),  # T > 2^30
    (("vf_qkv_pack", FAKE_SRC + 1, (96, 32, 8, 1), 4, 4, 8, 2, 1, FAKE_DST), -1),   # odd address
    (("vf_attn_split", FAKE_SRC, (8, 8, 1), 1, 2, (1 << 30) + 8, 2, 1, FAKE_DST), -1),  # D > 2^30
    (("vf_attn_split", FAKE_SRC, (8, 8, 1), 1, (1 << 30) + 8, 1, 2, 1, FAKE_DST), -1),  # H > 2^30
    (("vf_head_merge", FAKE_SRC, None, 4, 4, 8, 2, 1, FAKE_DST + 3), -1),           # odd address
    (("vf_qkv_pack", FAKE_SRC, (96, 32, 8, 1), 4, 4, 8, 2, 1 << 21, FAKE_DST), -1),  # P*C > 2^20
    (("vf_qkv_pack", FAKE_SRC, (1 << 62, 32, 8, 1), 4, 4, 8, 2, 1, FAKE_DST), -2),  # offset overflow
    (("vf_qkv_pack", FAKE_SRC, (96, 32, 8, 1), 1 << 30, 1 << 20, 1 << 12, 2, 1, FAKE_DST), -2),
    (("vf_attn_split", FAKE_SRC, (1 << 40, 8, 1), 1 << 30, 4, 8, 2, 1, FAKE_DST), -2),
    (("vf_qkv_pack", FAKE_SRC, (96, 32, 8, 1), 4, 4, 8, 2, 1, FAKE_SRC + 64), -3),  # alias
    (("vf_attn_split", FAKE_SRC, (32, 8, 1), 4, 4, 8, 3, 1, FAKE_SRC + 10), -3),
    (("vf_attn_split", FAKE_SRC, None, 4, 4, 8, 3, 1, FAKE_DST), -1),
    (("vf_head_merge", FAKE_SRC, (32, 8, 1), 4, 4, 8, 3, 1, FAKE_DST), -1),     # H % P
    (("vf_head_merge", FAKE_SRC, (0, 8, 1), 4, 4, 8, 2, 1, FAKE_DST), -1),      # overlapping dst
    (("vf_head_merge", FAKE_SRC, (8, 8, 1), 4, 4, 8, 2, 1, FAKE_DST), -1),      # overlapping dst
    (("vf_head_merge", FAKE_SRC, None, 4, 4, 8, 2, 1, FAKE_SRC + 2), -3),       # alias
])
def test_rejected_before_cuda(L, args, status):
    assert _call(L, *args) == status


@pytest.mark.parametrize("fn,strides", [("vf_qkv_pack", (0, 0, 0, 0)), ("vf_attn_split", (0, 0, 0)),
                                        ("vf_head_merge", None)])
def test_empty_calls_return_ok_without_cuda(L, fn, strides):
    # T = 0, H = 0 or D = 0: nothing to move, no pointer is needed
    for T, H, D in ((0, 4, 8), (4, 0, 8), (4, 4, 0)):
        assert _call(L, fn, None, strides, T, H, D, 2, 3, None) == 0


def _i64(*xs):
    return (I64 * len(xs))(*xs)


def test_unpack_and_range_rejections(L):
    Q, K, V = FAKE_DST, FAKE_DST + (1 << 20), FAKE_DST + (2 << 20)
    st = _i64(16, 8, 1)
    # H % P, aliasing outputs, output overlapping the received buffer
    assert L.vf_qkv_unpack(FAKE_SRC, 4, 6, 8, 4, 2, Q, K, V, st, None) == -1
    assert L.vf_qkv_unpack(FAKE_SRC, 4, 4, 8, 2, 2, Q, Q, V, st, None) == -3
    assert L.vf_qkv_unpack(FAKE_SRC, 4, 4, 8, 2, 2, Q, K, FAKE_SRC + 8, st, None) == -3
    assert L.vf_qkv_unpack(FAKE_SRC, 4, 4, 8, 2, 2, Q, K, V, _i64(0, 8, 1), None) == -1
    assert L.vf_qkv_unpack(FAKE_SRC, 4, 4, 8, 2, 2, Q + 1, K, V, st, None) == -1
    # chunk ranges
    s4 = _i64(96, 32, 8, 1)
    for c0, cn in ((-1, 1), (0, -1), (2, 1), (1, 2), (3, 0)):
        assert L.vf_qkv_pack_chunks(FAKE_SRC, s4, 4, 4, 8, 2, 2, c0, cn, FAKE_DST, None) == -1
        assert L.vf_attn_split_chunks(FAKE_SRC, _i64(32, 8, 1), 4, 4, 8, 2, 2, c0, cn,
                                      FAKE_DST, None) == -1
        assert L.vf_head_merge_chunks(FAKE_SRC, None, 4, 4, 8, 2, 2, c0, cn, FAKE_DST,
                                      None) == -1
        assert L.vf_qkv_unpack_chunks(FAKE_SRC, 4, 4, 8, 2, 2, c0, cn, Q, K, V, st, None) == -1
    # an empty chunk range moves nothing and needs no GPU
    assert L.vf_qkv_pack_chunks(FAKE_SRC, s4, 4, 4, 8, 2, 2, 1, 0, FAKE_DST, None) == 0
    assert L.vf_qkv_unpack_chunks(FAKE_SRC, 4, 4, 8, 2, 2, 2, 0, Q, K, V, st, None) == 0
    # three-pointer pack: strides required; q, k, v may overlap (read only) but
    # not the destination
    assert L.vf_qkv_pack3(FAKE_SRC, FAKE_SRC, FAKE_SRC, None, 4, 4, 8, 2, 2, 0, 2,
                          FAKE_DST, None) == -1
    assert L.vf_qkv_pack3(FAKE_SRC, FAKE_SRC, FAKE_DST, _i64(32, 8, 1), 4, 4, 8, 2, 2, 0, 2,
                          FAKE_DST + 16, None) == -3


def test_packed_elems_unpack(L):
    assert vf.packed_elems(vf.OP_QKV_UNPACK, 55414, 28, 128, 2, 4) == 3 * 55414 * 14 * 128
    assert L.vf_packed_elems(3, 10, 3, 8, 2, 2) == -1


def test_piece_table_capacity(L):
    a = (I64 * 3)()
    assert L.vf_piece_table(0, 10, 4, 8, 2, 2, a, a, a, 3) == -5
    assert L.vf_piece_table(9, 10, 4, 8, 2, 2, a, a, a, 3) == -1
    assert L.vf_packed_elems(0, 10, 3, 8, 2, 2) == -1
    assert L.vf_packed_elems(1, 10, 3, 8, 2, 2) == 240


def test_binding_refuses_pageable_cpu_tensors(L):
    import torch
    with pytest.raises(ValueError):
        vf.qkv_pack(torch.zeros((4, 3, 2, 8), dtype=torch.int16), 2, 1)
    with pytest.raises(ValueError):
        vf.attn_split(torch.zeros((4, 2, 8), dtype=torch.bfloat16), 2, 1)
    with pytest.raises(ValueError):
        vf.attn_split(torch.zeros((4, 2, 8), dtype=torch.float32), 2, 1)


@pytest.mark.parametrize("shape", [(55413, 32, 64, 4, 4), (37, 6, 16, 3, 7), (5, 4, 2, 4, 2),
                                   (0, 2, 2, 2, 3)])
def test_slot_major_piece_tables(L, shape):
    """Slot-major offsets are the chunk-major blocks (lengths from the oracle's
    table) laid out p outer, c inner."""
    T, H, D, P, C = shape
    for op in (0, 1, 2, 3):
        tok, length, _ = loops.piece_table(op, T, H, D, P, C)
        per = {0: 3 * (H // P) * D, 1: H * D, 2: (H // P) * D, 3: 3 * (H // P) * D}[op]
        want, cur = [0] * (P * C), 0
        for p in range(P):
            for c in range(C):
                want[c * P + p] = cur
                cur += length[c * P + p] * per
        got = vf.piece_table(op, T, H, D, P, C, order="slot_major")
        assert got[0] == tok and got[1] == length and got[2] == want


def test_relayout_descriptor_rejections(L):
    d = vf._Desc(op=0, order=0, T=4, H=4, D=8, P=2, C=2, c_begin=0, c_count=2,
                 packed=FAKE_DST)
    for i in range(3):
        d.strided[i] = FAKE_SRC + 4096 * i
    d.strides[0], d.strides[1], d.strides[2] = 32, 8, 1
    assert L.vf_relayout(None, None) == -1
    d.order = 2
    assert L.vf_relayout(ctypes.byref(d), None) == -1
    d.order, d.op = 1, 7
    assert L.vf_relayout(ctypes.byref(d), None) == -1
    d.op, d.P = 0, 3
    assert L.vf_relayout(ctypes.byref(d), None) == -1            # H % P
    d.P, d.c_count = 2, 0
    assert L.vf_relayout(ctypes.byref(d), None) == 0             # nothing to move
    d.c_count, d.packed = 2, FAKE_SRC + 8
    assert L.vf_relayout(ctypes.byref(d), None) == -3            # packed overlaps q
    d.op, d.packed = 3, FAKE_DST                                 # unpack writes q, k, v
    d.strided[1] = d.strided[0]
    assert L.vf_relayout(ctypes.byref(d), None) == -3            # outputs alias
    assert L.vf_piece_table_ex(0, 5, 4, 4, 8, 2, 2, _i64(0, 0, 0, 0), _i64(0, 0, 0, 0),
                               _i64(0, 0, 0, 0), 4) == -1


def test_piece_tables_random_shapes_against_oracle(L):
    """300 random shapes, every op, both block orders: the library's host
    tables equal the oracle's (chunk-major) and its permutation (slot-major)."""
    import random
    rng = random.Random(1234)
    for _ in range(300):
        P = rng.choice([1, 2, 3, 4, 7, 8, 16])
        C = rng.choice([1, 2, 3, 4, 5, 9, 16])
        H = P * rng.choice([1, 2, 3])
        D = rng.choice([1, 8, 64, 128])
        T = rng.choice([0, 1, 2, 5, rng.randrange(1, 200), rng.randrange(1000, 100000)])
        for op in (0, 1, 2, 3):
            tok, length, off = loops.piece_table(op, T, H, D, P, C)
            assert vf.piece_table(op, T, H, D, P, C) == (tok, length, off)
            per = {0: 3 * (H // P) * D, 1: H * D, 2: (H // P) * D, 3: 3 * (H // P) * D}[op]
            want, cur = [0] * (P * C), 0
            for p in range(P):
                for c in range(C):
                    want[c * P + p] = cur
                    cur += length[c * P + p] * per
            assert vf.piece_table(op, T, H, D, P, C, order="slot_major")[2] == want
            # every token appears once per destination slot (pack, merge: all
            # slots see every token) or once in all (split, unpack: shards)
            assert sum(length) == (T * P if op in (0, 2) else T)
