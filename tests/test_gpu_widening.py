"""GPU parity of the widened entry points against the CPU oracle, bit for bit:
the receive-side QKV unpack, the chunk-range entry points, the three-pointer
pack, and both directions of a virtual sequence-head exchange run entirely
with the CUDA relayouts (the exchange itself is emulated by device copies,
test-only)."""
import pytest
import torch

import sequence_head_relayout_gb300 as vf
from oracle import loops
from sequence_head_relayout_gb300 import workloads as W

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("oracle_built")]

DEV = torch.device("cuda:0")
CONFIG_NAMES = ["tiny", "4k", "pages", "ragged", "large"]


def rand_bits(shape, seed, device=DEV):
    g = torch.Generator(device="cpu").manual_seed(seed)
    t = torch.randint(-(1 << 15), 1 << 15, shape, generator=g, dtype=torch.int32)
    return t.to(torch.int16).to(device)


def same_bits(a, b):
    a = a.view(torch.int16)
    b = b.view(torch.int16).to(a.device)
    return a.shape == b.shape and torch.equal(a, b)


# --------------------------------------------------------------------------
# Receive-side QKV unpack
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", CONFIG_NAMES)
def test_qkv_unpack_config(name):
    cfg = W.CONFIGS[name]
    T, H, D, P, C = cfg.T, cfg.H, cfg.D, cfg.P, cfg.C
    Hp = H // P
    recv = torch.empty(3 * T * Hp * D, dtype=torch.int16, device=DEV)
    W.fill_(recv, cfg.payload, cfg.seed + 3000)
    if cfg.merge_dst == "head_major":
        outs = tuple(torch.empty((Hp, T, D), dtype=torch.int16, device=DEV).permute(1, 0, 2)
                     for _ in range(3))
    else:
        outs = None
    got = vf.qkv_unpack(recv, T, H, D, P, C, outs=outs)
    want = loops.qkv_unpack_recv(recv.cpu(), T, H, D, P, C)
    for g, w in zip(got, want):
        assert same_bits(g.contiguous(), w)


@pytest.mark.parametrize("shape", [(0, 4, 8, 2, 3), (1, 4, 8, 2, 4), (5, 4, 16, 4, 2),
                                   (37, 6, 5, 3, 4), (29, 8, 24, 2, 8), (13, 16, 8, 16, 8)])
def test_qkv_unpack_edges(shape):
    T, H, D, P, C = shape
    recv = rand_bits((3 * T * (H // P) * D,), 7)
    got = vf.qkv_unpack(recv, T, H, D, P, C)
    want = loops.qkv_unpack_recv(recv.cpu(), T, H, D, P, C)
    for g, w in zip(got, want):
        assert same_bits(g, w)


@pytest.mark.parametrize("offset", [0, 1, 2, 4])
def test_qkv_unpack_alignment_classes(offset):
    T, H, D, P, C = 23, 8, 32, 2, 3
    Hp = H // P
    n = 3 * T * Hp * D
    buf = rand_bits((n + 16,), 9)
    recv = buf[offset:offset + n]
    big = torch.zeros((3, T * Hp * D + 16), dtype=torch.int16, device=DEV)
    outs = tuple(big[s, offset:offset + T * Hp * D].view(T, Hp, D) for s in range(3))
    vf.qkv_unpack(recv, T, H, D, P, C, outs=outs)
    want = loops.qkv_unpack_recv(recv.cpu(), T, H, D, P, C)
    for g, w in zip(outs, want):
        assert same_bits(g, w)
    assert not bool(big[:, :offset].any()) and not bool(big[:, offset + T * Hp * D:].any())


# --------------------------------------------------------------------------
# Chunk ranges: chunk by chunk (any order) equals the full call, and a
# single chunk touches only its own blocks and tokens
# --------------------------------------------------------------------------

SENT = W._as_i16(0x7FA5)


@pytest.mark.parametrize("shape", [(4096, 32, 128, 2, 4), (55413 // 8, 32, 64, 4, 4),
                                   (17, 4, 8, 2, 8)])
def test_chunk_ranges_compose(shape):
    T, H, D, P, C = shape
    x4 = rand_bits((T, 3, H, D), 1)
    x3 = rand_bits((T, H, D), 2)
    flat = rand_bits((T * H * D,), 3)
    recv = rand_bits((3 * T * (H // P) * D,), 4)
    full = (vf.qkv_pack(x4, P, C), vf.attn_split(x3, P, C), vf.head_merge(flat, T, H, D, P, C),
            vf.qkv_unpack(recv, T, H, D, P, C))
    parts = [torch.full_like(full[0], SENT), torch.full_like(full[1], SENT),
             torch.full_like(full[2], SENT)] + [torch.full_like(full[3][0], SENT)
                                                for _ in range(3)]
    for c in reversed(range(C)):
        vf.qkv_pack(x4, P, C, out=parts[0], chunks=(c, 1))
        vf.attn_split(x3, P, C, out=parts[1], chunks=(c, 1))
        vf.head_merge(flat, T, H, D, P, C, out=parts[2], chunks=(c, 1))
        vf.qkv_unpack(recv, T, H, D, P, C, outs=tuple(parts[3:]), chunks=(c, 1))
    assert same_bits(parts[0], full[0])
    assert same_bits(parts[1], full[1])
    assert same_bits(parts[2], full[2])
    for a, b in zip(parts[3:], full[3]):
        assert same_bits(a, b)


def test_single_chunk_touches_only_its_blocks():
    T, H, D, P, C = 41, 8, 16, 2, 4
    x4 = rand_bits((T, 3, H, D), 5)
    full = vf.qkv_pack(x4, P, C)
    tok, length, off = vf.piece_table(vf.OP_QKV_PACK, T, H, D, P, C)
    c = 2
    out = torch.full_like(full, SENT)
    vf.qkv_pack(x4, P, C, out=out, chunks=(c, 1))
    mask = torch.zeros(out.numel(), dtype=torch.bool, device=DEV)
    per = 3 * (H // P) * D
    for p in range(P):
        e = c * P + p
        mask[off[e]:off[e] + length[e] * per] = True
    assert same_bits(out[mask], full[mask])
    assert bool((out[~mask] == SENT).all())

    # merge of chunk c writes exactly chunk c's tokens
    flat = rand_bits((T * H * D,), 6)
    fullm = vf.head_merge(flat, T, H, D, P, C)
    outm = torch.full_like(fullm, SENT)
    vf.head_merge(flat, T, H, D, P, C, out=outm, chunks=(c, 1))
    t0, t1 = tok[c * P], tok[c * P] + length[c * P]
    assert same_bits(outm[t0:t1], fullm[t0:t1])
    assert bool((outm[:t0] == SENT).all()) and bool((outm[t1:] == SENT).all())


def test_empty_chunk_range_is_a_no_op():
    x4 = rand_bits((9, 3, 4, 8), 1)
    out = torch.full((3 * 9 * 4 * 8,), SENT, dtype=torch.int16, device=DEV)
    vf.qkv_pack(x4, 2, 3, out=out, chunks=(1, 0))
    torch.cuda.synchronize()
    assert bool((out == SENT).all())


# --------------------------------------------------------------------------
# Three-pointer pack
# --------------------------------------------------------------------------

@pytest.mark.parametrize("layout", ["separate", "head_major", "same_tensor"])
def test_qkv_pack3_equals_fused_pack(layout):
    T, H, D, P, C = 333, 8, 64, 4, 4
    if layout == "separate":
        q, k, v = (rand_bits((T, H, D), s) for s in (1, 2, 3))
    elif layout == "head_major":
        q, k, v = (rand_bits((H, T, D), s).permute(1, 0, 2) for s in (1, 2, 3))
    else:
        q = k = v = rand_bits((T, H, D), 4)
    got = vf.qkv_pack3(q, k, v, P, C)
    fused = torch.stack([q, k, v], dim=1)            # [T,3,H,D]
    assert same_bits(got, loops.qkv_pack(fused.cpu(), P, C))


def test_qkv_pack3_pages_shape():
    cfg = W.CONFIGS["pages"]
    src, _ = W.pack_source(cfg, device=DEV)
    got = vf.qkv_pack3(src[:, 0], src[:, 1], src[:, 2], cfg.P, cfg.C)
    assert same_bits(got, vf.qkv_pack(src, cfg.P, cfg.C))


# --------------------------------------------------------------------------
# Virtual exchanges on the GPU
# --------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(4096, 32, 128, 2, 4), (3001, 16, 64, 4, 4),
                                   (55413, 8, 64, 8, 4), (5, 4, 16, 4, 2)])
def test_gpu_forward_exchange_pack_unpack(shape):
    """Rank r packs its token shard; block (c, p) of rank r goes to rank p's
    chunk-c block at slot r; rank p unpacks and holds head group p of every
    token."""
    T, H, D, P, C = shape
    Hp = H // P
    X = rand_bits((T, 3, H, D), 11)
    shard = -(-T // P)
    bounds = [(min(T, r * shard), min(T, (r + 1) * shard)) for r in range(P)]
    sent = [vf.qkv_pack(X[a:b], P, C) for a, b in bounds]
    tables = [vf.piece_table(vf.OP_QKV_PACK, b - a, H, D, P, C) for a, b in bounds]
    for p in range(P):
        parts = []
        for c in range(C):
            for r in range(P):
                e = c * P + p
                length, off = tables[r][1][e], tables[r][2][e]
                parts.append(sent[r][off:off + 3 * length * Hp * D])
        recv = torch.cat(parts)
        q, k, v = vf.qkv_unpack(recv, T, H, D, P, C)
        for s, out in enumerate((q, k, v)):
            assert same_bits(out, X[:, s, p * Hp:(p + 1) * Hp].contiguous()), (p, s)


@pytest.mark.parametrize("shape", [(4096, 32, 128, 2, 4), (3001, 16, 64, 4, 4),
                                   (55413, 8, 64, 8, 4), (5, 4, 16, 4, 2)])
def test_gpu_return_exchange_split_merge(shape):
    """Rank r splits its head group r of the attention output (a strided view
    of the global tensor); rank q merges what it receives and holds token
    shard q with all heads."""
    T, H, D, P, C = shape
    Hp = H // P
    A = rand_bits((T, H, D), 12)
    sent = [vf.attn_split(A[:, r * Hp:(r + 1) * Hp], P, C) for r in range(P)]
    tok, length, off = vf.piece_table(vf.OP_ATTN_SPLIT, T, Hp, D, P, C)
    shard = -(-T // P)
    for q in range(P):
        parts = []
        for c in range(C):
            for r in range(P):
                e = c * P + q
                parts.append(sent[r][off[e]:off[e] + length[e] * Hp * D])
        recv = torch.cat(parts)
        n_q = sum(length[c * P + q] for c in range(C))
        merged = vf.head_merge(recv, n_q, H, D, P, C)
        assert same_bits(merged, A[min(T, q * shard):min(T, (q + 1) * shard)].contiguous())


# --------------------------------------------------------------------------
# Pinned host memory: the kernels read and write it directly
# --------------------------------------------------------------------------

def test_pinned_host_zero_copy_all_ops():
    T, H, D, P, C = 1001, 8, 64, 2, 4
    Hp = H // P
    base4 = rand_bits((T, 3 * H * D + 16), 1, device="cpu").pin_memory()   # padded rows
    hx4 = base4[:, :3 * H * D].unflatten(1, (3, H, D))
    got = vf.qkv_pack(hx4, P, C)                         # pinned in, pinned out
    torch.cuda.synchronize()
    assert got.device.type == "cpu" and got.is_pinned()
    assert same_bits(got, loops.qkv_pack(hx4, P, C))

    hx3 = rand_bits((H, T, D), 2, device="cpu").pin_memory().permute(1, 0, 2)
    dev_out = torch.empty(T * H * D, dtype=torch.int16, device=DEV)
    vf.attn_split(hx3, P, C, out=dev_out)               # pinned in, device out
    assert same_bits(dev_out, loops.attn_split(hx3, P, C))

    flat = rand_bits((T * H * D,), 3)                   # device in, pinned out
    hout = torch.zeros((T, H, D), dtype=torch.int16).pin_memory()
    vf.head_merge(flat, T, H, D, P, C, out=hout)
    torch.cuda.synchronize()
    assert same_bits(hout, loops.head_merge(flat.cpu(), T, H, D, P, C))

    recv = rand_bits((3 * T * Hp * D,), 4, device="cpu").pin_memory()
    q, k, v = vf.qkv_unpack(recv, T, H, D, P, C)
    torch.cuda.synchronize()
    for a, b in zip((q, k, v), loops.qkv_unpack_recv(recv, T, H, D, P, C)):
        assert a.is_pinned() and same_bits(a, b)
