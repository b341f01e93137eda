"""Seeded random search for the opt-in lossy transport: every op, both
formats, both block orders, random shapes, strided-side layouts and element
offsets (which select the vector path), random code-buffer offsets -- the
CUDA kernels against the lossy oracle, bit for bit (codes, scale bits,
dequantised bfloat16 bits)."""
import random

import pytest
import torch

import sequence_head_relayout_gb300 as vf
from oracle import chain, loops
from sequence_head_relayout_gb300 import workloads as W

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("oracle_built")]

DEV = torch.device("cuda:0")
FMT = {"int8": loops.INT8, "e4m3": loops.E4M3}


def strided_view(shape, layout, offset):
    """A CUDA int16 view of the logical shape (token axis first)."""
    n = 1
    for s in shape:
        n *= s
    if layout == "contiguous":
        return torch.empty(offset + n, dtype=torch.int16, device=DEV)[offset:].view(*shape)
    if layout == "padded":
        T, inner = shape[0], n // shape[0]
        base = torch.empty(offset + T * (inner + 5), dtype=torch.int16, device=DEV)[offset:]
        return base.view(T, inner + 5)[:, :inner].unflatten(1, shape[1:])
    if layout == "head_major":
        perm = (shape[-2], shape[0]) + tuple(shape[1:-2]) + (shape[-1],)
        base = torch.empty(offset + n, dtype=torch.int16, device=DEV)[offset:].view(*perm)
        return base.permute(1, 0, 2) if len(shape) == 3 else base.permute(1, 2, 0, 3)
    full = shape[:-1] + (2 * shape[-1],)                  # d-stride 2
    return torch.empty(offset + 2 * n, dtype=torch.int16, device=DEV)[offset:].view(
        *full)[..., ::2]


def slot_major(op, flat, T, H, D, P, C, per):
    lens = [x // per for row in chain.block_lengths(op, T, H, D, P, C) for x in row]
    blocks = list(torch.split(flat, lens))
    return torch.cat([blocks[c * P + p] for p in range(P) for c in range(C)])


def chunk_major(op, flat, T, H, D, P, C, per):
    lens = [x // per for row in chain.block_lengths(op, T, H, D, P, C) for x in row]
    sm = [lens[c * P + p] for p in range(P) for c in range(C)]
    blocks = list(torch.split(flat, sm))
    at = {}
    i = 0
    for p in range(P):
        for c in range(C):
            at[(c, p)] = blocks[i]
            i += 1
    return torch.cat([at[(c, p)] for c in range(C) for p in range(P)])


def codes_buffer(n, fmt, offset):
    dt = torch.int8 if fmt == "int8" else torch.uint8
    base = torch.empty(offset + n, dtype=dt, device=DEV)[offset:]
    return base if fmt == "int8" else base.view(torch.float8_e4m3fn)


@pytest.mark.parametrize("seed", range(40))
def test_lossy_fuzz(seed):
    rng = random.Random(1000 + seed)
    P = rng.choice([1, 2, 3, 4])
    H = P * rng.choice([1, 2, 3])
    D = rng.choice([8, 16, 24, 64, 96, 128, 136])
    T = rng.choice([1, 2, 7, 33, 100, 257])
    C = rng.choice([1, 2, 3, 4, 6])
    fmt = rng.choice(["int8", "e4m3"])
    order = rng.choice(["chunk_major", "slot_major"])
    layout = rng.choice(["contiguous", "padded", "head_major", "dstride2"])
    offset = rng.choice([0, 1, 2, 4, 8])
    coff = rng.choice([0, 1, 3, 8])
    f = FMT[fmt]

    # quantising pack
    x4 = strided_view((T, 3, H, D), layout, offset)
    W.finite_rows_(x4, seed)
    n = 3 * T * H * D
    codes, scales = codes_buffer(n, fmt, coff), torch.empty(n // D, device=DEV)
    vf.qkv_pack_q(x4, P, C, fmt=fmt, codes=codes, scales=scales, order=order)
    wc, ws = loops.qkv_pack_q(x4.cpu(), P, C, f)
    wc, ws = wc.view(torch.uint8), ws
    if order == "slot_major":
        wc = slot_major(0, wc, T, H, D, P, C, 1)
        ws = slot_major(0, ws, T, H, D, P, C, D)
    assert torch.equal(codes.view(torch.uint8).cpu(), wc), (seed, "pack codes")
    assert torch.equal(scales.cpu().view(torch.int32), ws.view(torch.int32)), (seed, "pack scales")

    # quantising split
    x3 = strided_view((T, H, D), layout, offset)
    W.finite_rows_(x3, seed + 1)
    n = T * H * D
    codes, scales = codes_buffer(n, fmt, coff), torch.empty(n // D, device=DEV)
    vf.attn_split_q(x3, P, C, fmt=fmt, codes=codes, scales=scales, order=order)
    mc, ms = loops.attn_split_q(x3.cpu(), P, C, f)             # the oracle's, chunk-major
    mc = mc.view(torch.uint8)
    wc, ws = mc, ms
    if order == "slot_major":
        wc = slot_major(1, wc, T, H, D, P, C, 1)
        ws = slot_major(1, ws, T, H, D, P, C, D)
    assert torch.equal(codes.view(torch.uint8).cpu(), wc), (seed, "split codes")
    assert torch.equal(scales.cpu().view(torch.int32), ws.view(torch.int32)), (seed, "split scales")

    # dequantising merge of the oracle's split storage (a full-head view at P),
    # given to the kernel in the block order under test, at a code offset
    out = strided_view((T, H, D), layout if layout != "dstride2" else "contiguous", offset)
    rc = codes_buffer(n, fmt, coff)
    rc.view(torch.uint8).copy_(wc)
    vf.head_merge_q(rc, ws.to(DEV), T, H, D, P, C, fmt=fmt, out=out.view(torch.bfloat16),
                    order=order)
    if order == "slot_major":          # the same bytes read as the merge's (c, p) blocks
        mc = chunk_major(2, wc, T, H, D, P, C, 1)
        ms = chunk_major(2, ws, T, H, D, P, C, D)
    want = loops.head_merge_q(mc, ms, T, H, D, P, C, f)
    assert torch.equal(out.cpu(), want), (seed, "merge")

    # dequantising unpack of the pack's first 3*T*(H/P)*D codes
    Hp = H // P
    m = 3 * T * Hp * D
    rc = codes_buffer(m, fmt, coff)
    rc.view(torch.uint8).copy_(torch.randint(0, 256, (m,), dtype=torch.int32).to(torch.uint8))
    if fmt == "e4m3":
        u = rc.view(torch.uint8)
        u.copy_(torch.where((u & 0x7F) == 0x7F, torch.zeros_like(u), u))
    rs = torch.rand(m // D, device=DEV) * 2.0 ** rng.randrange(-20, 10)
    outs = tuple(strided_view((T, Hp, D), "contiguous" if layout == "dstride2" else layout,
                              offset).view(torch.bfloat16) for _ in range(3))
    vf.qkv_unpack_q(rc, rs, T, H, D, P, C, fmt=fmt, outs=outs, order=order)
    uc, us = rc.view(torch.uint8).cpu(), rs.cpu()
    if order == "slot_major":
        uc = chunk_major(3, uc, T, H, D, P, C, 1)
        us = chunk_major(3, us, T, H, D, P, C, D)
    want = loops.qkv_unpack_q(uc, us, T, H, D, P, C, f)
    for o, w in zip(outs, want):
        assert torch.equal(o.view(torch.int16).cpu(), w), (seed, "unpack")
