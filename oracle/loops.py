"""ctypes front end of the scalar-loop oracle (``vf_oracle.c``).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Every function takes
and returns PyTorch CPU tensors of 16-bit elements; bf16 tensors are viewed as
int16 so that bit patterns (NaN payloads, -0) are what is compared.  Strided
views are passed as their first element's address plus their element strides,
exactly as the oracle's loops read them.
"""
import ctypes

import torch

from . import build as _build

OP_QKV_PACK, OP_ATTN_SPLIT, OP_HEAD_MERGE, OP_QKV_UNPACK = 0, 1, 2, 3

_lib = None
_I64 = ctypes.c_int64
_P = ctypes.c_void_p
_INT = ctypes.c_int


def lib():
    global _lib
    if _lib is None:
        l = ctypes.CDLL(_build.build())
        arr4 = ctypes.POINTER(_I64)
        for name, args in {
            "oracle_qkv_pack": [_P, arr4, _I64, _I64, _I64, _I64, _I64, _P],
            "oracle_qkv_unpack": [_P, _I64, _I64, _I64, _I64, _I64, _P, arr4],
            "oracle_attn_split": [_P, arr4, _I64, _I64, _I64, _I64, _I64, _P],
            "oracle_attn_unsplit": [_P, _I64, _I64, _I64, _I64, _I64, _P, arr4],
            "oracle_head_merge": [_P, _I64, _I64, _I64, _I64, _I64, _P, arr4],
            "oracle_head_split": [_P, arr4, _I64, _I64, _I64, _I64, _I64, _P],
            "oracle_qkv_unpack_recv": [_P, _I64, _I64, _I64, _I64, _I64, _P, _P, _P, arr4],
            "oracle_piece_table": [ctypes.c_int, _I64, _I64, _I64, _I64, _I64,
                                   arr4, arr4, arr4, _I64],
            "oracle_reorder_blocks": [ctypes.c_int, _I64, _I64, _I64, _I64, _I64, _P, _P,
                                      ctypes.c_int],
            "oracle_qkv_pack_q": [_P, arr4, _I64, _I64, _I64, _I64, _I64, _INT, _P, _P],
            "oracle_qkv_unpack_q": [_P, _P, _I64, _I64, _I64, _I64, _I64, _INT, _P, _P, _P,
                                    arr4],
            "oracle_attn_split_q": [_P, arr4, _I64, _I64, _I64, _I64, _I64, _INT, _P, _P],
            "oracle_head_merge_q": [_P, _P, _I64, _I64, _I64, _I64, _I64, _INT, _P, arr4],
        }.items():
            f = getattr(l, name)
            f.argtypes = args
            f.restype = _I64
        l.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        l.oracle_e4m3_encode.restype = ctypes.c_uint8
        l.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        l.oracle_e4m3_decode.restype = ctypes.c_float
        l.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        l.oracle_f32_to_bf16.restype = ctypes.c_uint16
        _lib = l
    return _lib


def _bits(t: torch.Tensor) -> torch.Tensor:
    if t.device.type != "cpu":
        raise ValueError("the oracle runs on CPU tensors only")
    if t.element_size() != 2:
        raise ValueError("the oracle moves 16-bit elements")
    return t if t.dtype == torch.int16 else t.view(torch.int16)


def _strides(t: torch.Tensor):
    return (_I64 * t.dim())(*t.stride())


def _check(n, expect, what):
    if n != expect:
        raise RuntimeError("%s: oracle moved %d elements, expected %d" % (what, n, expect))


def qkv_pack(src: torch.Tensor, P: int, C: int) -> torch.Tensor:
    """QKV destination pack of a [T,3,H,D] view; returns flat packed storage."""
    s = _bits(src)
    T, three, H, D = s.shape
    assert three == 3
    out = torch.empty(3 * T * H * D, dtype=torch.int16)
    n = lib().oracle_qkv_pack(s.data_ptr(), _strides(s), T, H, D, P, C, out.data_ptr())
    _check(n, out.numel(), "qkv_pack")
    return out


def qkv_unpack(packed: torch.Tensor, T: int, H: int, D: int, P: int, C: int) -> torch.Tensor:
    """Inverse of ``qkv_pack``: flat packed storage back to contiguous [T,3,H,D]."""
    p = _bits(packed).contiguous()
    out = torch.empty((T, 3, H, D), dtype=torch.int16)
    n = lib().oracle_qkv_unpack(p.data_ptr(), T, H, D, P, C, out.data_ptr(), _strides(out))
    _check(n, p.numel(), "qkv_unpack")
    return out


def attn_split(src: torch.Tensor, P: int, C: int) -> torch.Tensor:
    """Attention-result split of a [T,H,D] view; returns flat packed storage."""
    s = _bits(src)
    T, H, D = s.shape
    out = torch.empty(T * H * D, dtype=torch.int16)
    n = lib().oracle_attn_split(s.data_ptr(), _strides(s), T, H, D, P, C, out.data_ptr())
    _check(n, out.numel(), "attn_split")
    return out


def attn_unsplit(packed: torch.Tensor, T: int, H: int, D: int, P: int, C: int) -> torch.Tensor:
    """Inverse of ``attn_split``: flat packed storage back to contiguous [T,H,D]."""
    p = _bits(packed).contiguous()
    out = torch.empty((T, H, D), dtype=torch.int16)
    n = lib().oracle_attn_unsplit(p.data_ptr(), T, H, D, P, C, out.data_ptr(), _strides(out))
    _check(n, p.numel(), "attn_unsplit")
    return out


def head_merge(packed: torch.Tensor, T: int, H: int, D: int, P: int, C: int,
               out: torch.Tensor = None) -> torch.Tensor:
    """Returned-head merge of flat packed storage into a [T,H,D] tensor.

    ``out`` may be any non-overlapping strided [T,H,D] int16 view; a
    contiguous one is allocated when it is omitted.
    """
    p = _bits(packed).contiguous()
    if out is None:
        out = torch.empty((T, H, D), dtype=torch.int16)
    o = _bits(out)
    assert tuple(o.shape) == (T, H, D)
    n = lib().oracle_head_merge(p.data_ptr(), T, H, D, P, C, o.data_ptr(), _strides(o))
    _check(n, T * H * D, "head_merge")
    return out


def head_split(src: torch.Tensor, P: int, C: int) -> torch.Tensor:
    """Inverse of ``head_merge``: a [T,H,D] view into the merge's packed storage."""
    s = _bits(src)
    T, H, D = s.shape
    out = torch.empty(T * H * D, dtype=torch.int16)
    n = lib().oracle_head_split(s.data_ptr(), _strides(s), T, H, D, P, C, out.data_ptr())
    _check(n, out.numel(), "head_split")
    return out


def qkv_unpack_recv(recv: torch.Tensor, T: int, H: int, D: int, P: int, C: int,
                    outs=None):
    """Receive-side QKV unpack: flat received storage of 3*T*(H/P)*D elements
    into (Q, K, V), each a [T, H/P, D] tensor.  ``outs`` may give three
    strided [T, H/P, D] int16 views sharing one stride tuple."""
    r = _bits(recv).contiguous()
    Hp = H // P
    if outs is None:
        outs = tuple(torch.empty((T, Hp, D), dtype=torch.int16) for _ in range(3))
    q, k, v = (_bits(o) for o in outs)
    assert q.stride() == k.stride() == v.stride()
    n = lib().oracle_qkv_unpack_recv(r.data_ptr(), T, H, D, P, C, q.data_ptr(), k.data_ptr(),
                                     v.data_ptr(), _strides(q))
    _check(n, 3 * T * Hp * D, "qkv_unpack_recv")
    return outs


def piece_table(op: int, T: int, H: int, D: int, P: int, C: int):
    """(tok_start, tok_len, packed_off) lists over (c, p) in storage order."""
    m = P * C
    a, b, c = (_I64 * m)(), (_I64 * m)(), (_I64 * m)()
    n = lib().oracle_piece_table(op, T, H, D, P, C, a, b, c, m)
    if n != m:
        raise ValueError("oracle_piece_table rejected its arguments")
    return list(a), list(b), list(c)


def to_slot_major(op: int, packed: torch.Tensor, T: int, H: int, D: int, P: int,
                  C: int) -> torch.Tensor:
    """[c][p] packed storage of ``op`` re-ordered into [p][c] block order."""
    src = _bits(packed).contiguous()
    out = torch.empty_like(src)
    n = lib().oracle_reorder_blocks(op, T, H, D, P, C, src.data_ptr(), out.data_ptr(), 1)
    _check(n, src.numel(), "reorder_blocks")
    return out


def to_chunk_major(op: int, packed: torch.Tensor, T: int, H: int, D: int, P: int,
                   C: int) -> torch.Tensor:
    """[p][c] packed storage of ``op`` re-ordered into [c][p] block order."""
    src = _bits(packed).contiguous()
    out = torch.empty_like(src)
    n = lib().oracle_reorder_blocks(op, T, H, D, P, C, src.data_ptr(), out.data_ptr(), 0)
    _check(n, src.numel(), "reorder_blocks")
    return out


# ---- lossy transport (opt-in) ---------------------------------------------
# fmt: INT8 = 1, E4M3 = 2.  Codes are one byte per element (int8 or uint8
# bits), scales one float32 per head row, both in the exact op's layout.

INT8, E4M3 = 1, 2


def _code_dtype(fmt):
    return torch.int8 if fmt == INT8 else torch.uint8


def qkv_pack_q(src: torch.Tensor, P: int, C: int, fmt: int):
    """Quantising QKV pack of a [T,3,H,D] view -> (codes, scales)."""
    s = _bits(src)
    T, _, H, D = s.shape
    codes = torch.empty(3 * T * H * D, dtype=_code_dtype(fmt))
    scales = torch.empty(3 * T * H, dtype=torch.float32)
    n = lib().oracle_qkv_pack_q(s.data_ptr(), _strides(s), T, H, D, P, C, fmt,
                                codes.data_ptr(), scales.data_ptr())
    _check(n, codes.numel(), "qkv_pack_q")
    return codes, scales


def attn_split_q(src: torch.Tensor, P: int, C: int, fmt: int):
    """Quantising attention-result split of a [T,H,D] view -> (codes, scales)."""
    s = _bits(src)
    T, H, D = s.shape
    codes = torch.empty(T * H * D, dtype=_code_dtype(fmt))
    scales = torch.empty(T * H, dtype=torch.float32)
    n = lib().oracle_attn_split_q(s.data_ptr(), _strides(s), T, H, D, P, C, fmt,
                                  codes.data_ptr(), scales.data_ptr())
    _check(n, codes.numel(), "attn_split_q")
    return codes, scales


def head_merge_q(codes, scales, T, H, D, P, C, fmt):
    """Dequantising merge -> [T,H,D] bf16 bits (int16)."""
    out = torch.empty((T, H, D), dtype=torch.int16)
    n = lib().oracle_head_merge_q(codes.contiguous().data_ptr(), scales.contiguous().data_ptr(),
                                  T, H, D, P, C, fmt, out.data_ptr(), _strides(out))
    _check(n, T * H * D, "head_merge_q")
    return out


def qkv_unpack_q(codes, scales, T, H, D, P, C, fmt):
    """Dequantising receive-side unpack -> Q, K, V as [T,H/P,D] bf16 bits."""
    Hp = H // P
    outs = tuple(torch.empty((T, Hp, D), dtype=torch.int16) for _ in range(3))
    n = lib().oracle_qkv_unpack_q(codes.contiguous().data_ptr(), scales.contiguous().data_ptr(),
                                  T, H, D, P, C, fmt, outs[0].data_ptr(), outs[1].data_ptr(),
                                  outs[2].data_ptr(), _strides(outs[0]))
    _check(n, 3 * T * Hp * D, "qkv_unpack_q")
    return outs


def e4m3_encode(x: float) -> int:
    return int(lib().oracle_e4m3_encode(x))


def e4m3_decode(c: int) -> float:
    return float(lib().oracle_e4m3_decode(c))


def f32_to_bf16(x: float) -> int:
    return int(lib().oracle_f32_to_bf16(x))
