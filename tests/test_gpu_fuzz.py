"""Seeded random search over shapes, strides, offsets and chunk ranges: every
op of the CUDA library against the CPU oracle, bit for bit.

Each case draws T, H, D, P, C (including empty shards and chunks), a layout
for the strided side (contiguous, padded rows, head-major, d-stride 2, or a
broadcast source), an element offset into the allocations (which selects the
vector width), and a chunk range; the chunk-range result is compared with
the full oracle output on the range's blocks or tokens only.
"""
import random

import pytest
import torch

import sequence_head_relayout_gb300 as vf
from oracle import loops

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("oracle_built")]

DEV = torch.device("cuda:0")
SENT = -23131            # 0xA5A5 as int16


def rand_bits(n, rng):
    g = torch.Generator().manual_seed(rng.randrange(1 << 30))
    return torch.randint(-(1 << 15), 1 << 15, (n,), generator=g, dtype=torch.int32).to(
        torch.int16)


def view_of(shape, layout, offset, rng, read_only=True, pad=None):
    """A CUDA view of the logical shape (token axis first) with the layout."""
    T = shape[0]
    inner = 1
    for s in shape[1:]:
        inner *= s
    if layout == "contiguous":
        base = rand_bits(offset + T * inner, rng).to(DEV)
        return base[offset:offset + T * inner].view(*shape)
    if layout == "padded":
        pad = pad or rng.randrange(1, 24)
        base = rand_bits(offset + T * (inner + pad), rng).to(DEV)
        return base[offset:offset + T * (inner + pad)].view(T, inner + pad)[:, :inner].unflatten(
            1, shape[1:])
    if layout == "head_major":           # token axis second in memory
        perm_shape = (shape[-2], T) + tuple(shape[1:-2]) + (shape[-1],)
        n = T * inner
        base = rand_bits(offset + n, rng).to(DEV)[offset:offset + n].view(*perm_shape)
        # memory order (h, t, [3], d) -> logical (t, [3], h, d)
        if len(shape) == 3:
            return base.permute(1, 0, 2)
        return base.permute(1, 2, 0, 3)
    if layout == "dstride2":
        full = shape[:-1] + (2 * shape[-1],)
        n = 1
        for s in full:
            n *= s
        base = rand_bits(offset + n, rng).to(DEV)
        return base[offset:offset + n].view(*full)[..., ::2]
    if layout == "broadcast" and read_only:
        one = rand_bits(offset + inner, rng).to(DEV)[offset:offset + inner].view(1, *shape[1:])
        return one.expand(*shape)
    return view_of(shape, "contiguous", offset, rng)


def case(seed):
    rng = random.Random(seed)
    P = rng.choice([1, 2, 3, 4, 5])
    H = P * rng.choice([1, 2, 3, 4])
    D = rng.choice([1, 3, 8, 16, 24, 40, 64])
    T = rng.choice([0, 1, 2, 7, 33, 100, 257])
    C = rng.choice([1, 2, 3, 4, 6])
    layout = rng.choice(["contiguous", "padded", "head_major", "dstride2", "broadcast"])
    offset = rng.choice([0, 0, 1, 2, 4, 8])
    c0 = rng.randrange(0, C + 1)
    cn = rng.randrange(0, C - c0 + 1)
    return rng, T, H, D, P, C, layout, offset, c0, cn


@pytest.mark.parametrize("seed", range(48))
def test_fuzz_all_ops(seed):
    rng, T, H, D, P, C, layout, offset, c0, cn = case(seed)
    Hp = H // P

    # pack: full, and a chunk range against the full oracle on those blocks
    x4 = view_of((T, 3, H, D), layout, offset, rng)
    want = loops.qkv_pack(x4.cpu(), P, C)
    assert torch.equal(vf.qkv_pack(x4, P, C).cpu(), want)
    got = torch.full((3 * T * H * D,), SENT, dtype=torch.int16, device=DEV)
    vf.qkv_pack(x4, P, C, out=got, chunks=(c0, cn))
    tok, length, off = vf.piece_table(vf.OP_QKV_PACK, T, H, D, P, C)
    mask = torch.zeros(got.numel(), dtype=torch.bool)
    for c in range(c0, c0 + cn):
        for p in range(P):
            e = c * P + p
            mask[off[e]:off[e] + length[e] * 3 * Hp * D] = True
    got = got.cpu()
    assert torch.equal(got[mask], want[mask])
    assert bool((got[~mask] == SENT).all())

    # three-pointer pack from the slabs of the same view
    assert torch.equal(vf.qkv_pack3(x4[:, 0], x4[:, 1], x4[:, 2], P, C).cpu(), want)

    # split, in both block orders
    x3 = view_of((T, H, D), layout, offset, rng)
    want3 = loops.attn_split(x3.cpu(), P, C)
    assert torch.equal(vf.attn_split(x3, P, C).cpu(), want3)
    assert torch.equal(vf.attn_split(x3, P, C, order="slot_major").cpu(),
                       loops.to_slot_major(1, want3, T, H, D, P, C))
    assert torch.equal(vf.qkv_pack(x4, P, C, order="slot_major").cpu(),
                       loops.to_slot_major(0, want, T, H, D, P, C))

    # merge into a strided destination (never broadcast)
    flat = rand_bits(T * H * D, rng).to(DEV)
    out = view_of((T, H, D), layout if layout != "broadcast" else "padded", offset, rng,
                  read_only=False)
    out.fill_(SENT)
    vf.head_merge(flat, T, H, D, P, C, out=out)
    assert torch.equal(out.cpu(), loops.head_merge(flat.cpu(), T, H, D, P, C))

    # unpack into three strided outputs
    recv = rand_bits(3 * T * Hp * D, rng).to(DEV)
    lay = layout if layout not in ("broadcast", "dstride2") else "contiguous"
    pad = rng.randrange(1, 24)
    outs = [view_of((T, Hp, D), lay, offset, rng, read_only=False, pad=pad) for _ in range(3)]
    assert len({o.stride() for o in outs}) == 1 or T <= 1
    if len({o.stride() for o in outs}) == 1:
        vf.qkv_unpack(recv, T, H, D, P, C, outs=tuple(outs))
        for a, b in zip(outs, loops.qkv_unpack_recv(recv.cpu(), T, H, D, P, C)):
            assert torch.equal(a.cpu(), b)
