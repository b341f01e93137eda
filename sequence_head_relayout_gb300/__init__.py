"""GB300-native exact destination-major relayouts around sequence-head attention.

Thin ctypes binding over ``libvf_relayout.so`` (C ABI in
``include/vf_relayout.h``): the functions here only marshal tensor pointers,
strides and the current CUDA stream; every element is moved by the library's
sm_103a kernels.  PyTorch provides device memory and streams.  There is no
CPU path: the library must be built (``__graft_entry__.build()``) and the
tensors must be addressable by the GPU -- CUDA memory, or pinned host memory
that the kernels read or write directly over the host link -- otherwise the
calls raise.

Operations ("Sol-Engine alignment on SM86 and SM89", section "What is
enabled"):

* :func:`qkv_pack`   -- fused [T,3,H,D] QKV view -> destination-major send buffer;
* :func:`attn_split` -- attention output [T,H,D] view -> per-destination token shards;
* :func:`head_merge` -- received destination-major buffer -> token-major [T,H,D];
* :func:`qkv_unpack` -- received QKV buffer -> Q, K, V [T,H/P,D] views ("速度、显存与
  质量", section "剖析单次去噪请求": the QKV unpack before Flash-SDPA);
* :func:`qkv_pack3`  -- the pack from three separate Q, K, V views.

Every function takes ``chunks=(c_begin, c_count)`` to move only those overlap
chunks (the packed buffer is always the full one) and ``order`` for the block
order of the packed storage: ``"chunk_major"`` ([c][p], the four-chunk overlap
layout, default) or ``"slot_major"`` ([p][c]).

Opt-in lossy transport (same page, table "Upstream gap and disposition", row
"INT8 QKV and FP8 output transport"): :func:`qkv_pack_q`, :func:`attn_split_q`,
:func:`head_merge_q` and :func:`qkv_unpack_q` quantise each head row to
8-bit codes (``fmt="int8"`` -> int8 codes, ``fmt="e4m3"`` -> float8_e4m3fn
codes) plus one float32 scale per head row, in the exact ops' layout, and
dequantise to bfloat16 on the receive side.  The format is stated in
``include/vf_relayout.h``.
"""
import ctypes
import os

import torch

__all__ = ["qkv_pack", "qkv_pack3", "attn_split", "head_merge", "qkv_unpack", "packed_elems",
           "piece_table", "VFError", "lib", "OP_QKV_PACK", "OP_ATTN_SPLIT", "OP_HEAD_MERGE",
           "OP_QKV_UNPACK", "qkv_pack_q", "attn_split_q", "head_merge_q", "qkv_unpack_q",
           "scale_count", "FORMATS"]

OP_QKV_PACK, OP_ATTN_SPLIT, OP_HEAD_MERGE, OP_QKV_UNPACK = 0, 1, 2, 3
ORDERS = {"chunk_major": 0, "slot_major": 1}
FORMATS = {"int8": 1, "e4m3": 2}

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libvf_relayout.so")

_lib = None
_I64 = ctypes.c_int64
_P = ctypes.c_void_p
_I64P = ctypes.POINTER(_I64)


class _Desc(ctypes.Structure):
    """vf_relayout_desc of the C ABI."""
    _fields_ = [("op", ctypes.c_int32), ("order", ctypes.c_int32),
                ("T", _I64), ("H", _I64), ("D", _I64), ("P", _I64), ("C", _I64),
                ("c_begin", _I64), ("c_count", _I64), ("packed", _P),
                ("strided", _P * 3), ("strides", _I64 * 3)]


class VFError(RuntimeError):
    """A negative status returned by the library."""

    def __init__(self, fn, status):
        self.status = status
        msg = lib().vf_status_string(status).decode()
        super().__init__("%s failed: %s (status %d)" % (fn, msg, status))


def lib():
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libvf_relayout.so is not built; run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        l = ctypes.CDLL(LIB_PATH)
        sig = {
            "vf_qkv_pack": [_P, _I64P] + [_I64] * 5 + [_P, _P],
            "vf_attn_split": [_P, _I64P] + [_I64] * 5 + [_P, _P],
            "vf_head_merge": [_P, _I64P] + [_I64] * 5 + [_P, _P],
            "vf_qkv_unpack": [_P] + [_I64] * 5 + [_P, _P, _P, _I64P, _P],
            "vf_qkv_pack_chunks": [_P, _I64P] + [_I64] * 7 + [_P, _P],
            "vf_attn_split_chunks": [_P, _I64P] + [_I64] * 7 + [_P, _P],
            "vf_head_merge_chunks": [_P, _I64P] + [_I64] * 7 + [_P, _P],
            "vf_qkv_unpack_chunks": [_P] + [_I64] * 7 + [_P, _P, _P, _I64P, _P],
            "vf_qkv_pack3": [_P, _P, _P, _I64P] + [_I64] * 7 + [_P, _P],
        }
        for name, args in sig.items():
            f = getattr(l, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        l.vf_packed_elems.argtypes = [ctypes.c_int, _I64, _I64, _I64, _I64, _I64]
        l.vf_packed_elems.restype = _I64
        l.vf_piece_table.argtypes = [ctypes.c_int, _I64, _I64, _I64, _I64, _I64,
                                     _I64P, _I64P, _I64P, _I64]
        l.vf_piece_table.restype = _I64
        l.vf_piece_table_ex.argtypes = [ctypes.c_int, ctypes.c_int, _I64, _I64, _I64, _I64,
                                        _I64, _I64P, _I64P, _I64P, _I64]
        l.vf_piece_table_ex.restype = _I64
        l.vf_relayout.argtypes = [ctypes.POINTER(_Desc), _P]
        l.vf_relayout.restype = ctypes.c_int
        l.vf_relayout_q.argtypes = [ctypes.POINTER(_Desc), ctypes.c_int, _P, _P]
        l.vf_relayout_q.restype = ctypes.c_int
        for name, args in {
            "vf_qkv_pack_int8": [_P, _I64P] + [_I64] * 5 + [_P, _P, _P],
            "vf_qkv_unpack_int8": [_P, _P] + [_I64] * 5 + [_P, _P, _P, _I64P, _P],
            "vf_attn_split_fp8": [_P, _I64P] + [_I64] * 5 + [_P, _P, _P],
            "vf_head_merge_fp8": [_P, _P, _I64P] + [_I64] * 5 + [_P, _P],
        }.items():
            f = getattr(l, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        l.vf_scale_count.argtypes = [ctypes.c_int, _I64, _I64, _I64, _I64, _I64]
        l.vf_scale_count.restype = _I64
        l.vf_status_string.argtypes = [ctypes.c_int]
        l.vf_status_string.restype = ctypes.c_char_p
        _lib = l
    return _lib


def _check16(t: torch.Tensor, what: str):
    """A 16-bit tensor the GPU can address: CUDA memory, or pinned (page-locked,
    mapped) host memory, which the kernels read and write directly over the
    host link.  Pageable host memory is refused: there is no CPU path."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % what)
    if t.device.type != "cuda" and not (t.device.type == "cpu" and t.is_pinned()):
        raise ValueError("%s must be a CUDA tensor or pinned host memory "
                         "(there is no CPU path)" % what)
    if t.element_size() != 2:
        raise ValueError("%s must hold 16-bit elements (bf16/fp16/int16)" % what)


def _strides(t: torch.Tensor):
    return (_I64 * t.dim())(*t.stride())


def _stream(stream, device):
    """The stream to enqueue on: the given one, else the current stream of the
    tensor's device (of the current device for pinned host tensors)."""
    if stream is None:
        stream = torch.cuda.current_stream(device if device.type == "cuda" else None)
    return ctypes.c_void_p(stream.cuda_stream)


def _call(fn, *args):
    rc = getattr(_lib or lib(), fn)(*args)
    if rc != 0:
        raise VFError(fn, rc)


def _n_packed(op, T, H, D, P):
    """Packed element count for sizing outputs (the library validates the
    shape again on every call); odd shapes go through the library's check."""
    if P < 1 or min(T, H, D) < 0:
        return packed_elems(op, T, H, D, P, 1)            # raises VFError
    if op == OP_QKV_PACK:
        return 3 * T * H * D
    if op == OP_QKV_UNPACK:
        return 3 * T * (H // P) * D
    return T * H * D


def packed_elems(op: int, T: int, H: int, D: int, P: int, C: int) -> int:
    """Elements of the packed side of ``op`` (3*T*H*D for the pack, T*H*D for the
    split and the merge, 3*T*(H/P)*D for the unpack)."""
    n = lib().vf_packed_elems(op, T, H, D, P, C)
    if n < 0:
        raise VFError("vf_packed_elems", n)
    return n


def _order(order) -> int:
    o = ORDERS.get(order)
    if o is None:
        raise ValueError("order must be one of %s" % sorted(ORDERS))
    return o


def piece_table(op: int, T: int, H: int, D: int, P: int, C: int, order="chunk_major"):
    """(tok_start, tok_len, packed_off) lists; entry c*P + p is block (c, p),
    packed_off places the blocks in the given storage order."""
    m = P * C
    a, b, c = (_I64 * m)(), (_I64 * m)(), (_I64 * m)()
    n = lib().vf_piece_table_ex(op, _order(order), T, H, D, P, C, a, b, c, m)
    if n < 0:
        raise VFError("vf_piece_table", n)
    return list(a), list(b), list(c)


def _range(chunks, C):
    return (0, C) if chunks is None else (int(chunks[0]), int(chunks[1]))


def _relayout(op, order, T, H, D, P, C, chunks, packed, strided, strides, stream,
              fmt=0, scales=None):
    """vf_relayout (or vf_relayout_q with a format) with a descriptor: the
    general entry, any block order."""
    c0, cn = _range(chunks, C)
    d = _Desc(op=op, order=order, T=T, H=H, D=D, P=P, C=C, c_begin=c0, c_count=cn,
              packed=packed)
    for i, ptr in enumerate(strided):
        d.strided[i] = ptr
    for i, st in enumerate(strides):
        d.strides[i] = st
    if fmt:
        rc = lib().vf_relayout_q(ctypes.byref(d), fmt, scales, stream)
        if rc != 0:
            raise VFError("vf_relayout_q", rc)
        return
    rc = lib().vf_relayout(ctypes.byref(d), stream)
    if rc != 0:
        raise VFError("vf_relayout", rc)


def _flat_out(out, n, like):
    if out is None:
        out = torch.empty(n, dtype=like.dtype, device=like.device,
                          pin_memory=like.device.type == "cpu")
    _check16(out, "out")
    if not out.is_contiguous() or out.numel() != n:
        raise ValueError("out must be contiguous with %d elements" % n)
    return out


def qkv_pack(src: torch.Tensor, P: int, C: int, out: torch.Tensor = None,
             stream: torch.cuda.Stream = None, chunks=None,
             order="chunk_major") -> torch.Tensor:
    """QKV destination pack of a [T,3,H,D] CUDA view (any strides).

    Returns (or fills) a flat tensor of 3*T*H*D elements: blocks (c, p) in
    order, each head group p of chunk c as q, k, v slabs [L_c][H/P][D].
    """
    _check16(src, "src")
    if src.dim() != 4 or src.shape[1] != 3:
        raise ValueError("src must be a [T,3,H,D] view")
    T, _, H, D = src.shape
    out = _flat_out(out, _n_packed(OP_QKV_PACK, T, H, D, P), src)
    o = _order(order)
    if o:
        st = src.stride()
        bases = [src.data_ptr() + s * st[1] * src.element_size() for s in range(3)]
        _relayout(OP_QKV_PACK, o, T, H, D, P, C, chunks, out.data_ptr(), bases,
                  (st[0], st[2], st[3]), _stream(stream, src.device))
        return out
    c0, cn = _range(chunks, C)
    _call("vf_qkv_pack_chunks", src.data_ptr(), _strides(src), T, H, D, P, C, c0, cn,
          out.data_ptr(), _stream(stream, src.device))
    return out


def qkv_pack3(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, P: int, C: int,
              out: torch.Tensor = None, stream: torch.cuda.Stream = None,
              chunks=None, order="chunk_major") -> torch.Tensor:
    """QKV destination pack from three [T,H,D] CUDA views with equal strides."""
    for t, name in ((q, "q"), (k, "k"), (v, "v")):
        _check16(t, name)
    if q.dim() != 3 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must be [T,H,D] views of one shape")
    if q.stride() != k.stride() or q.stride() != v.stride():
        raise ValueError("q, k, v must share their strides")
    T, H, D = q.shape
    out = _flat_out(out, _n_packed(OP_QKV_PACK, T, H, D, P), q)
    o = _order(order)
    if o:
        _relayout(OP_QKV_PACK, o, T, H, D, P, C, chunks, out.data_ptr(),
                  [q.data_ptr(), k.data_ptr(), v.data_ptr()], q.stride(),
                  _stream(stream, q.device))
        return out
    c0, cn = _range(chunks, C)
    _call("vf_qkv_pack3", q.data_ptr(), k.data_ptr(), v.data_ptr(), _strides(q), T, H, D, P,
          C, c0, cn, out.data_ptr(), _stream(stream, q.device))
    return out


def attn_split(src: torch.Tensor, P: int, C: int, out: torch.Tensor = None,
               stream: torch.cuda.Stream = None, chunks=None,
               order="chunk_major") -> torch.Tensor:
    """Attention-result split of a [T,H,D] CUDA view (any strides).

    Returns (or fills) a flat tensor of T*H*D elements: blocks (c, p) in
    order, each chunk c of token shard p as [L][H][D].
    """
    _check16(src, "src")
    if src.dim() != 3:
        raise ValueError("src must be a [T,H,D] view")
    T, H, D = src.shape
    out = _flat_out(out, _n_packed(OP_ATTN_SPLIT, T, H, D, P), src)
    o = _order(order)
    if o:
        _relayout(OP_ATTN_SPLIT, o, T, H, D, P, C, chunks, out.data_ptr(), [src.data_ptr()],
                  src.stride(), _stream(stream, src.device))
        return out
    c0, cn = _range(chunks, C)
    _call("vf_attn_split_chunks", src.data_ptr(), _strides(src), T, H, D, P, C, c0, cn,
          out.data_ptr(), _stream(stream, src.device))
    return out


def head_merge(src: torch.Tensor, T: int, H: int, D: int, P: int, C: int,
               out: torch.Tensor = None, stream: torch.cuda.Stream = None,
               chunks=None, order="chunk_major") -> torch.Tensor:
    """Returned-head merge of a flat received buffer into a [T,H,D] view.

    ``out`` may be any non-overlapping strided [T,H,D] CUDA view; a
    contiguous tensor is allocated when it is omitted.
    """
    _check16(src, "src")
    n = _n_packed(OP_HEAD_MERGE, T, H, D, P)
    if not src.is_contiguous() or src.numel() != n:
        raise ValueError("src must be contiguous with %d elements" % n)
    if out is None:
        out = torch.empty((T, H, D), dtype=src.dtype, device=src.device,
                          pin_memory=src.device.type == "cpu")
    _check16(out, "out")
    if tuple(out.shape) != (T, H, D):
        raise ValueError("out must have shape [T,H,D]")
    o = _order(order)
    if o:
        _relayout(OP_HEAD_MERGE, o, T, H, D, P, C, chunks, src.data_ptr(), [out.data_ptr()],
                  out.stride(), _stream(stream, src.device))
        return out
    c0, cn = _range(chunks, C)
    _call("vf_head_merge_chunks", src.data_ptr(), _strides(out), T, H, D, P, C, c0, cn,
          out.data_ptr(), _stream(stream, src.device))
    return out


def qkv_unpack(recv: torch.Tensor, T: int, H: int, D: int, P: int, C: int, outs=None,
               stream: torch.cuda.Stream = None, chunks=None, order="chunk_major"):
    """Receive-side QKV unpack: flat received buffer of 3*T*(H/P)*D elements
    into (Q, K, V), each a [T, H/P, D] view (global token order).

    ``outs`` may give three non-overlapping [T, H/P, D] CUDA views sharing one
    stride tuple; contiguous tensors are allocated when it is omitted.
    """
    _check16(recv, "recv")
    n = _n_packed(OP_QKV_UNPACK, T, H, D, P)
    if not recv.is_contiguous() or recv.numel() != n:
        raise ValueError("recv must be contiguous with %d elements" % n)
    Hp = H // P
    if outs is None:
        outs = tuple(torch.empty((T, Hp, D), dtype=recv.dtype, device=recv.device,
                                 pin_memory=recv.device.type == "cpu") for _ in range(3))
    q, k, v = outs
    for t, name in ((q, "q"), (k, "k"), (v, "v")):
        _check16(t, name)
        if tuple(t.shape) != (T, Hp, D):
            raise ValueError("%s must have shape [T,H/P,D]" % name)
    if q.stride() != k.stride() or q.stride() != v.stride():
        raise ValueError("q, k, v must share their strides")
    o = _order(order)
    if o:
        _relayout(OP_QKV_UNPACK, o, T, H, D, P, C, chunks, recv.data_ptr(),
                  [q.data_ptr(), k.data_ptr(), v.data_ptr()], q.stride(),
                  _stream(stream, recv.device))
        return outs
    c0, cn = _range(chunks, C)
    _call("vf_qkv_unpack_chunks", recv.data_ptr(), T, H, D, P, C, c0, cn, q.data_ptr(),
          k.data_ptr(), v.data_ptr(), _strides(q), _stream(stream, recv.device))
    return outs


# ---- opt-in lossy transport --------------------------------------------------

def _fmt(fmt) -> int:
    f = FORMATS.get(fmt)
    if f is None:
        raise ValueError("fmt must be one of %s" % sorted(FORMATS))
    return f


def _code_dtype(f):
    return torch.int8 if f == 1 else torch.float8_e4m3fn


def _gpu_addressable(t, what):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % what)
    if t.device.type != "cuda" and not (t.device.type == "cpu" and t.is_pinned()):
        raise ValueError("%s must be a CUDA tensor or pinned host memory "
                         "(there is no CPU path)" % what)


def scale_count(op: int, T: int, H: int, D: int, P: int, C: int) -> int:
    """Scales (one per head row) of the packed side of ``op``."""
    n = lib().vf_scale_count(op, T, H, D, P, C)
    if n < 0:
        raise VFError("vf_scale_count", n)
    return n


def _codes_scales(codes, scales, n, rows, f, like, what):
    """Check (or allocate) the flat codes and scales buffers."""
    if codes is None:
        codes = torch.empty(n, dtype=_code_dtype(f), device=like.device,
                            pin_memory=like.device.type == "cpu")
    if scales is None:
        scales = torch.empty(rows, dtype=torch.float32, device=like.device,
                             pin_memory=like.device.type == "cpu")
    _gpu_addressable(codes, what + " codes")
    _gpu_addressable(scales, what + " scales")
    if codes.element_size() != 1 or not codes.is_contiguous() or codes.numel() != n:
        raise ValueError("codes must be a contiguous 8-bit tensor of %d elements" % n)
    if scales.dtype != torch.float32 or not scales.is_contiguous() or scales.numel() != rows:
        raise ValueError("scales must be a contiguous float32 tensor of %d elements" % rows)
    return codes, scales


def _rows(n, D):
    return n // D if D > 0 else 0


def _check_bf16(t: torch.Tensor, what: str):
    """The lossy transport reads and writes BF16 values (int16 views of BF16
    bit patterns are accepted too); float16 would be misread."""
    if isinstance(t, torch.Tensor) and t.dtype not in (torch.bfloat16, torch.int16):
        raise ValueError("%s must hold bfloat16 values (or their int16 bit patterns)" % what)
    _check16(t, what)


def qkv_pack_q(src: torch.Tensor, P: int, C: int, fmt="int8", codes=None, scales=None,
               stream: torch.cuda.Stream = None, chunks=None, order="chunk_major"):
    """Quantising QKV pack of a [T,3,H,D] bf16 view -> (codes, scales): the
    layout of :func:`qkv_pack`, one byte per element, one scale per head row."""
    _check_bf16(src, "src")
    if src.dim() != 4 or src.shape[1] != 3:
        raise ValueError("src must be a [T,3,H,D] view")
    f = _fmt(fmt)
    T, _, H, D = src.shape
    n = _n_packed(OP_QKV_PACK, T, H, D, P)
    codes, scales = _codes_scales(codes, scales, n, _rows(n, D), f, src, "pack")
    st = src.stride()
    bases = [src.data_ptr() + s * st[1] * src.element_size() for s in range(3)]
    _relayout(OP_QKV_PACK, _order(order), T, H, D, P, C, chunks, codes.data_ptr(), bases,
              (st[0], st[2], st[3]), _stream(stream, src.device), f, scales.data_ptr())
    return codes, scales


def attn_split_q(src: torch.Tensor, P: int, C: int, fmt="e4m3", codes=None, scales=None,
                 stream: torch.cuda.Stream = None, chunks=None, order="chunk_major"):
    """Quantising attention-result split of a [T,H,D] bf16 view -> (codes, scales)."""
    _check_bf16(src, "src")
    if src.dim() != 3:
        raise ValueError("src must be a [T,H,D] view")
    f = _fmt(fmt)
    T, H, D = src.shape
    n = _n_packed(OP_ATTN_SPLIT, T, H, D, P)
    codes, scales = _codes_scales(codes, scales, n, _rows(n, D), f, src, "split")
    _relayout(OP_ATTN_SPLIT, _order(order), T, H, D, P, C, chunks, codes.data_ptr(),
              [src.data_ptr()], src.stride(), _stream(stream, src.device), f,
              scales.data_ptr())
    return codes, scales


def head_merge_q(codes: torch.Tensor, scales: torch.Tensor, T: int, H: int, D: int, P: int,
                 C: int, fmt="e4m3", out: torch.Tensor = None,
                 stream: torch.cuda.Stream = None, chunks=None, order="chunk_major"):
    """Dequantising returned-head merge -> [T,H,D] bfloat16 (or into ``out``)."""
    f = _fmt(fmt)
    n = _n_packed(OP_HEAD_MERGE, T, H, D, P)
    codes, scales = _codes_scales(codes, scales, n, _rows(n, D), f, codes, "merge")
    if out is None:
        out = torch.empty((T, H, D), dtype=torch.bfloat16, device=codes.device,
                          pin_memory=codes.device.type == "cpu")
    _check_bf16(out, "out")
    if tuple(out.shape) != (T, H, D):
        raise ValueError("out must have shape [T,H,D]")
    _relayout(OP_HEAD_MERGE, _order(order), T, H, D, P, C, chunks, codes.data_ptr(),
              [out.data_ptr()], out.stride(), _stream(stream, codes.device), f,
              scales.data_ptr())
    return out


def qkv_unpack_q(codes: torch.Tensor, scales: torch.Tensor, T: int, H: int, D: int, P: int,
                 C: int, fmt="int8", outs=None, stream: torch.cuda.Stream = None,
                 chunks=None, order="chunk_major"):
    """Dequantising receive-side unpack -> (Q, K, V), each [T,H/P,D] bfloat16."""
    f = _fmt(fmt)
    n = _n_packed(OP_QKV_UNPACK, T, H, D, P)
    codes, scales = _codes_scales(codes, scales, n, _rows(n, D), f, codes, "unpack")
    Hp = H // P
    if outs is None:
        outs = tuple(torch.empty((T, Hp, D), dtype=torch.bfloat16, device=codes.device,
                                 pin_memory=codes.device.type == "cpu") for _ in range(3))
    q, k, v = outs
    for t, name in ((q, "q"), (k, "k"), (v, "v")):
        _check_bf16(t, name)
        if tuple(t.shape) != (T, Hp, D):
            raise ValueError("%s must have shape [T,H/P,D]" % name)
    if q.stride() != k.stride() or q.stride() != v.stride():
        raise ValueError("q, k, v must share their strides")
    _relayout(OP_QKV_UNPACK, _order(order), T, H, D, P, C, chunks, codes.data_ptr(),
              [q.data_ptr(), k.data_ptr(), v.data_ptr()], q.stride(),
              _stream(stream, codes.device), f, scales.data_ptr())
    return outs
