"""GPU parity of the shared-memory staged path (tiled_kernel.cuh): 16- and
32-byte head rows (D = 8, 16) with a head-major strided side, where moving
whole head rows would leave DRAM sectors half used.

Every op in both block orders, ragged token and head tiles (T not a multiple
of the tile's 64 / 32 tokens, H not a multiple of its 32 heads), chunk ranges,
guard bands around the strided side, and the same shapes with a token-major
strided side (which stays on the row-block kernel) -- all bit for bit
against the oracle."""
import pytest
import torch

import sequence_head_relayout_gb300 as vf
from oracle import loops

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("oracle_built")]

DEV = torch.device("cuda:0")


def rand_bits(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(-(1 << 15), 1 << 15, shape, generator=g, dtype=torch.int32).to(
        torch.int16)


def head_major(x_thd):
    """[T,H,D] values stored as an [H,T,D] buffer, viewed as [T,H,D]."""
    return x_thd.permute(1, 0, 2).contiguous().to(DEV).permute(1, 0, 2)


SHAPES = [
    # T, H, D, P, C
    (1000, 40, 8, 2, 4),      # 40 heads: a full and a partial head tile
    (777, 32, 16, 4, 3),
    (65, 6, 8, 2, 2),         # one token past a tile, few heads
    (33, 64, 16, 8, 1),       # one token past a 32-token tile
    (5, 2, 8, 1, 4),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_split_head_major_source(shape):
    T, H, D, P, C = shape
    x = rand_bits((T, H, D), 1)
    got = vf.attn_split(head_major(x), P, C)
    assert torch.equal(got.cpu(), loops.attn_split(x, P, C))
    got = vf.attn_split(head_major(x), P, C, order="slot_major")
    want = loops.to_slot_major(vf.OP_ATTN_SPLIT, loops.attn_split(x, P, C), T, H, D, P, C)
    assert torch.equal(got.cpu(), want)


@pytest.mark.parametrize("shape", SHAPES)
def test_merge_head_major_destination(shape):
    T, H, D, P, C = shape
    if H % P:
        pytest.skip("merge needs H % P == 0")
    flat = rand_bits((T * H * D,), 2)
    base = torch.full((H + 2, T, D), 0x7FA5, dtype=torch.int16, device=DEV)   # guard heads
    out = base[1:H + 1].permute(1, 0, 2)
    vf.head_merge(flat.to(DEV), T, H, D, P, C, out=out)
    assert torch.equal(out.cpu(), loops.head_merge(flat, T, H, D, P, C))
    assert bool((base[0] == 0x7FA5).all()) and bool((base[H + 1] == 0x7FA5).all())


@pytest.mark.parametrize("shape", SHAPES)
def test_pack3_and_unpack_head_major(shape):
    T, H, D, P, C = shape
    if H % P:
        pytest.skip("pack and unpack need H % P == 0")
    Hp = H // P
    x = rand_bits((T, 3, H, D), 3)
    q, k, v = (head_major(x[:, s].contiguous()) for s in range(3))
    got = vf.qkv_pack3(q, k, v, P, C)
    assert torch.equal(got.cpu(), loops.qkv_pack(x, P, C))
    # chunk by chunk equals one call
    part = torch.zeros_like(got)
    for c in reversed(range(C)):
        vf.qkv_pack3(q, k, v, P, C, out=part, chunks=(c, 1))
    assert torch.equal(part, got)
    recv = rand_bits((3 * T * Hp * D,), 4)
    outs = tuple(torch.empty((Hp, T, D), dtype=torch.int16, device=DEV).permute(1, 0, 2)
                 for _ in range(3))
    vf.qkv_unpack(recv.to(DEV), T, H, D, P, C, outs=outs)
    for o, w in zip(outs, loops.qkv_unpack_recv(recv, T, H, D, P, C)):
        assert torch.equal(o.cpu(), w)


@pytest.mark.parametrize("D", [8, 16])
def test_token_major_views_unchanged(D):
    # the same short head rows with a token-major strided side (row-block kernel)
    T, H, P, C = 300, 24, 4, 3
    x = rand_bits((T, H, D), 5)
    got = vf.attn_split(x.to(DEV), P, C)
    assert torch.equal(got.cpu(), loops.attn_split(x, P, C))


def test_misaligned_head_major_view_falls_back():
    # a view starting 2 bytes into its buffer cannot use 16-byte vectors: the
    # row-block kernel's narrow path takes it, with the same result
    T, H, D, P, C = 200, 8, 8, 2, 2
    x = rand_bits((T, H, D), 6)
    buf = torch.empty(H * T * D + 1, dtype=torch.int16, device=DEV)
    view = buf[1:].view(H, T, D)
    view.copy_(x.permute(1, 0, 2).to(DEV))
    got = vf.attn_split(view.permute(1, 0, 2), P, C)
    assert torch.equal(got.cpu(), loops.attn_split(x, P, C))
