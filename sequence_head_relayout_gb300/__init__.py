"""GB300-native exact destination-major relayouts around sequence-head attention.

Thin ctypes binding over ``libvf_relayout.so`` (C ABI in
``include/vf_relayout.h``): the functions here only marshal tensor pointers,
strides and the current CUDA stream; every element is moved by the library's
sm_103a kernels.  PyTorch provides device memory and streams.  There is no
CPU path: the library must be built (``__graft_entry__.build()``) and the
tensors must live on a CUDA device, otherwise the calls raise.

Operations ("Sol-Engine alignment on SM86 and SM89", section "What is
enabled"):

* :func:`qkv_pack`   -- fused [T,3,H,D] QKV view -> destination-major send buffer;
* :func:`attn_split` -- attention output [T,H,D] view -> per-destination token shards;
* :func:`head_merge` -- received destination-major buffer -> token-major [T,H,D].
"""
import ctypes
import os

import torch

__all__ = ["qkv_pack", "attn_split", "head_merge", "packed_elems", "piece_table",
           "VFError", "lib", "OP_QKV_PACK", "OP_ATTN_SPLIT", "OP_HEAD_MERGE"]

OP_QKV_PACK, OP_ATTN_SPLIT, OP_HEAD_MERGE = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libvf_relayout.so")

_lib = None
_I64 = ctypes.c_int64
_P = ctypes.c_void_p
_I64P = ctypes.POINTER(_I64)


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
        for name in ("vf_qkv_pack", "vf_attn_split"):
            f = getattr(l, name)
            f.argtypes = [_P, _I64P, _I64, _I64, _I64, _I64, _I64, _P, _P]
            f.restype = ctypes.c_int
        l.vf_head_merge.argtypes = [_P, _I64P, _I64, _I64, _I64, _I64, _I64, _P, _P]
        l.vf_head_merge.restype = ctypes.c_int
        l.vf_packed_elems.argtypes = [ctypes.c_int, _I64, _I64, _I64, _I64, _I64]
        l.vf_packed_elems.restype = _I64
        l.vf_piece_table.argtypes = [ctypes.c_int, _I64, _I64, _I64, _I64, _I64,
                                     _I64P, _I64P, _I64P, _I64]
        l.vf_piece_table.restype = _I64
        l.vf_status_string.argtypes = [ctypes.c_int]
        l.vf_status_string.restype = ctypes.c_char_p
        _lib = l
    return _lib


def _check16(t: torch.Tensor, what: str):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % what)
    if t.device.type != "cuda":
        raise ValueError("%s must be a CUDA tensor (there is no CPU path)" % what)
    if t.element_size() != 2:
        raise ValueError("%s must hold 16-bit elements (bf16/fp16/int16)" % what)


def _strides(t: torch.Tensor):
    return (_I64 * t.dim())(*t.stride())


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _call(fn, *args):
    rc = getattr(lib(), fn)(*args)
    if rc != 0:
        raise VFError(fn, rc)


def packed_elems(op: int, T: int, H: int, D: int, P: int, C: int) -> int:
    """Elements of the packed side of ``op`` (3*T*H*D for the pack, else T*H*D)."""
    n = lib().vf_packed_elems(op, T, H, D, P, C)
    if n < 0:
        raise VFError("vf_packed_elems", n)
    return n


def piece_table(op: int, T: int, H: int, D: int, P: int, C: int):
    """(tok_start, tok_len, packed_off) lists over (c, p) blocks in storage order."""
    m = P * C
    a, b, c = (_I64 * m)(), (_I64 * m)(), (_I64 * m)()
    n = lib().vf_piece_table(op, T, H, D, P, C, a, b, c, m)
    if n < 0:
        raise VFError("vf_piece_table", n)
    return list(a), list(b), list(c)


def qkv_pack(src: torch.Tensor, P: int, C: int, out: torch.Tensor = None,
             stream: torch.cuda.Stream = None) -> torch.Tensor:
    """QKV destination pack of a [T,3,H,D] CUDA view (any strides).

    Returns (or fills) a flat tensor of 3*T*H*D elements: blocks (c, p) in
    order, each head group p of chunk c as q, k, v slabs [L_c][H/P][D].
    """
    _check16(src, "src")
    if src.dim() != 4 or src.shape[1] != 3:
        raise ValueError("src must be a [T,3,H,D] view")
    T, _, H, D = src.shape
    n = packed_elems(OP_QKV_PACK, T, H, D, P, C)
    if out is None:
        out = torch.empty(n, dtype=src.dtype, device=src.device)
    _check16(out, "out")
    if not out.is_contiguous() or out.numel() != n:
        raise ValueError("out must be contiguous with %d elements" % n)
    _call("vf_qkv_pack", src.data_ptr(), _strides(src), T, H, D, P, C, out.data_ptr(),
          _stream(stream, src.device))
    return out


def attn_split(src: torch.Tensor, P: int, C: int, out: torch.Tensor = None,
               stream: torch.cuda.Stream = None) -> torch.Tensor:
    """Attention-result split of a [T,H,D] CUDA view (any strides).

    Returns (or fills) a flat tensor of T*H*D elements: blocks (c, p) in
    order, each chunk c of token shard p as [L][H][D].
    """
    _check16(src, "src")
    if src.dim() != 3:
        raise ValueError("src must be a [T,H,D] view")
    T, H, D = src.shape
    n = packed_elems(OP_ATTN_SPLIT, T, H, D, P, C)
    if out is None:
        out = torch.empty(n, dtype=src.dtype, device=src.device)
    _check16(out, "out")
    if not out.is_contiguous() or out.numel() != n:
        raise ValueError("out must be contiguous with %d elements" % n)
    _call("vf_attn_split", src.data_ptr(), _strides(src), T, H, D, P, C, out.data_ptr(),
          _stream(stream, src.device))
    return out


def head_merge(src: torch.Tensor, T: int, H: int, D: int, P: int, C: int,
               out: torch.Tensor = None, stream: torch.cuda.Stream = None) -> torch.Tensor:
    """Returned-head merge of a flat received buffer into a [T,H,D] view.

    ``out`` may be any non-overlapping strided [T,H,D] CUDA view; a
    contiguous tensor is allocated when it is omitted.
    """
    _check16(src, "src")
    n = packed_elems(OP_HEAD_MERGE, T, H, D, P, C)
    if not src.is_contiguous() or src.numel() != n:
        raise ValueError("src must be contiguous with %d elements" % n)
    if out is None:
        out = torch.empty((T, H, D), dtype=src.dtype, device=src.device)
    _check16(out, "out")
    if tuple(out.shape) != (T, H, D):
        raise ValueError("out must have shape [T,H,D]")
    _call("vf_head_merge", src.data_ptr(), _strides(out), T, H, D, P, C, out.data_ptr(),
          _stream(stream, src.device))
    return out
