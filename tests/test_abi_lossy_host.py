"""Host side of the opt-in lossy transport's C ABI, without a GPU.

Sizes (``vf_scale_count``), and every argument rejected before the library
touches CUDA: an unknown format, missing or misaligned scales, scales that
overlap the codes or a strided view.  Fake pointer values are safe: nothing
is dereferenced or launched.  A call that passes every host check reaches the
CUDA pointer query, which fails here (no device) with VF_ERR_CUDA -- that is
how the tests see that, e.g., an odd codes address is accepted.
"""
import ctypes

import pytest

import sequence_head_relayout_gb300 as vf

I64 = ctypes.c_int64
FAKE_SRC, FAKE_CODES, FAKE_SCALES = 1 << 40, 1 << 41, 1 << 42
OK, ERR_ARG, ERR_ALIAS, ERR_CUDA = 0, -1, -3, -4


@pytest.fixture(scope="module")
def L(lib_built):
    return vf.lib()


def _i64(*xs):
    return (I64 * len(xs))(*xs)


def test_scale_count_is_one_per_head_row(L):
    T, H, D, P, C = 37, 8, 16, 4, 3
    for op in (0, 1, 2, 3):
        assert vf.scale_count(op, T, H, D, P, C) * D == vf.packed_elems(op, T, H, D, P, C)
    assert L.vf_scale_count(0, 5, 4, 0, 2, 1) == 0
    assert L.vf_scale_count(0, 5, 3, 8, 2, 1) == ERR_ARG                 # H % P
    assert L.vf_scale_count(9, 5, 4, 8, 2, 1) == ERR_ARG


def _desc(op=1, T=4, H=4, D=8, P=2, C=2, packed=FAKE_CODES):
    d = vf._Desc(op=op, order=0, T=T, H=H, D=D, P=P, C=C, c_begin=0, c_count=C, packed=packed)
    d.strided[0] = FAKE_SRC
    d.strides[0], d.strides[1], d.strides[2] = H * D, D, 1
    return d


def test_relayout_q_rejections(L):
    d = _desc()
    for fmt in (0, 3, -1):
        assert L.vf_relayout_q(ctypes.byref(d), fmt, FAKE_SCALES, None) == ERR_ARG
    assert L.vf_relayout_q(None, 1, FAKE_SCALES, None) == ERR_ARG
    assert L.vf_relayout_q(ctypes.byref(d), 1, None, None) == ERR_ARG       # no scales
    assert L.vf_relayout_q(ctypes.byref(d), 2, FAKE_SCALES + 2, None) == ERR_ARG  # misaligned
    # 4 x 4 x 8 = 128 code bytes, 16 scales (64 bytes)
    assert L.vf_relayout_q(ctypes.byref(d), 1, FAKE_CODES + 124, None) == ERR_ALIAS
    assert L.vf_relayout_q(ctypes.byref(d), 1, FAKE_CODES + 128, None) == ERR_CUDA
    assert L.vf_relayout_q(ctypes.byref(d), 1, FAKE_SRC + 64, None) == ERR_ALIAS   # scales in src
    d2 = _desc(packed=FAKE_SRC + 32)
    assert L.vf_relayout_q(ctypes.byref(d2), 1, FAKE_SCALES, None) == ERR_ALIAS    # codes in src
    # codes need no alignment: an odd address passes the host checks
    d3 = _desc(packed=FAKE_CODES + 1)
    assert L.vf_relayout_q(ctypes.byref(d3), 2, FAKE_SCALES, None) == ERR_CUDA
    # the strided side still holds 16-bit elements
    d4 = _desc()
    d4.strided[0] = FAKE_SRC + 1
    assert L.vf_relayout_q(ctypes.byref(d4), 2, FAKE_SCALES, None) == ERR_ARG
    # nothing to move: no pointer is looked at
    d5 = _desc(T=0, packed=None)
    assert L.vf_relayout_q(ctypes.byref(d5), 1, None, None) == OK
    d6 = _desc()
    d6.c_count = 0
    assert L.vf_relayout_q(ctypes.byref(d6), 1, None, None) == OK


def test_named_lossy_entries_check_their_arguments(L):
    s4 = _i64(96, 32, 8, 1)
    assert L.vf_qkv_pack_int8(FAKE_SRC, s4, 4, 4, 8, 3, 1, FAKE_CODES, FAKE_SCALES,
                              None) == ERR_ARG                            # H % P
    assert L.vf_qkv_pack_int8(FAKE_SRC, s4, 4, 4, 8, 2, 1, FAKE_CODES, None, None) == ERR_ARG
    assert L.vf_qkv_pack_int8(FAKE_SRC, s4, 4, 4, 8, 2, 1, FAKE_CODES, FAKE_SCALES,
                              None) == ERR_CUDA                           # host checks pass
    st = _i64(16, 8, 1)
    assert L.vf_qkv_unpack_int8(FAKE_CODES, FAKE_SCALES, 4, 4, 8, 2, 2, FAKE_SRC,
                                FAKE_SRC, FAKE_SRC + 4096, st, None) == ERR_ALIAS
    assert L.vf_attn_split_fp8(FAKE_SRC, _i64(32, 8, 1), 4, 4, 8, 2, 2, FAKE_CODES,
                               FAKE_CODES + 64, None) == ERR_ALIAS
    assert L.vf_head_merge_fp8(FAKE_CODES, FAKE_SCALES, None, 4, 4, 8, 2, 2, FAKE_SRC,
                               None) == ERR_CUDA
    assert L.vf_head_merge_fp8(FAKE_CODES, FAKE_SCALES, None, 4, 4, 8, 2, 2,
                               FAKE_SCALES + 8, None) == ERR_ALIAS        # dst over scales


def test_binding_refuses_pageable_and_bad_formats(L):
    import torch
    x = torch.zeros((4, 2, 8), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        vf.attn_split_q(x, 2, 1)
    with pytest.raises(ValueError):
        vf.qkv_pack_q(torch.zeros((4, 3, 2, 8), dtype=torch.bfloat16), 2, 1, fmt="fp4")
    # float16 would be read as bfloat16 bit patterns: refused for its dtype
    # (checked before the memory kind)
    with pytest.raises(ValueError, match="bfloat16"):
        vf.attn_split_q(torch.zeros((4, 2, 8), dtype=torch.float16), 2, 1)
