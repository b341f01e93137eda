"""Second, independent oracle: the pages' own reference materialisation.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

"Sol-Engine alignment on SM86 and SM89", section "What is enabled": before the
direct kernels, the sequence-head path built its exchange buffers with
stack/permute/contiguous (QKV pack) and cat/permute/contiguous (returned-head
merge) chains, and every direct output must equal those element for element.
This module is that chain written with PyTorch CPU view and copy operations,
one overlap chunk at a time.  It never computes a flat offset: the layout
comes out of ``stack``/``unflatten``/``permute``/``contiguous``/``cat``.

The chunk and shard partitions follow the same reading as the C oracle
(quota ceil(n/parts), short tail), restated here on purpose rather than shared.
"""
import torch


def _bits(t: torch.Tensor) -> torch.Tensor:
    if t.device.type != "cpu":
        raise ValueError("the chain oracle runs on CPU tensors only")
    return t if t.dtype == torch.int16 else t.view(torch.int16)


def part_sizes(n: int, parts: int):
    """Sizes of the pieces when n items are cut with quota ceil(n/parts)."""
    q = -(-n // parts)
    return [max(0, min(q, n - i * q)) for i in range(parts)]


def qkv_pack(src: torch.Tensor, P: int, C: int) -> torch.Tensor:
    """stack(q,k,v) -> per chunk: group heads by slot, permute slot outermost,
    contiguous -> cat.  ``src`` is any [T,3,H,D] view."""
    x = _bits(src)
    T, _, H, D = x.shape
    stacked = torch.stack(x.unbind(1))                      # [3, T, H, D]
    blocks = []
    for chunk in torch.split(stacked, part_sizes(T, C), dim=1):
        L = chunk.shape[1]
        grouped = chunk.unflatten(2, (P, H // P))           # [3, L, P, Hp, D]
        blocks.append(grouped.permute(2, 0, 1, 3, 4).contiguous().reshape(-1))
        assert blocks[-1].numel() == 3 * L * H * D
    return torch.cat(blocks) if blocks else torch.empty(0, dtype=torch.int16)


def attn_split(src: torch.Tensor, P: int, C: int) -> torch.Tensor:
    """Token shards per destination, each cut into overlap chunks; storage
    is chunk-outer, destination-inner.  ``src`` is any [T,H,D] view."""
    x = _bits(src)
    T = x.shape[0]
    shards = torch.split(x, part_sizes(T, P), dim=0)
    chunks = [torch.split(s, part_sizes(s.shape[0], C), dim=0) for s in shards]
    blocks = [chunks[p][c].contiguous().reshape(-1) for c in range(C) for p in range(P)]
    return torch.cat(blocks) if blocks else torch.empty(0, dtype=torch.int16)


def head_merge(packed: torch.Tensor, T: int, H: int, D: int, P: int, C: int) -> torch.Tensor:
    """Per chunk: view the received slab as [slot, token, head-in-group, d],
    permute token outermost, concatenate the chunks -> contiguous [T,H,D]."""
    flat = _bits(packed).reshape(-1)
    Hp = H // P
    pieces, off = [], 0
    for L in part_sizes(T, C):
        n = P * L * Hp * D
        slab = flat[off:off + n].view(P, L, Hp, D)
        pieces.append(slab.permute(1, 0, 2, 3).reshape(L, H, D))
        off += n
    assert off == flat.numel()
    return torch.cat(pieces, 0).contiguous()


def qkv_unpack_recv(recv: torch.Tensor, T: int, H: int, D: int, P: int, C: int):
    """Receive side of the forward exchange: cut the received storage into
    (chunk, source rank) blocks, view each as [3, tokens, Hp, D], concatenate
    each rank's chunks, then the ranks in order -> (Q, K, V) as [T, Hp, D]."""
    flat = _bits(recv).reshape(-1)
    Hp = H // P
    shard = part_sizes(T, P)
    per_rank = [[] for _ in range(P)]
    off = 0
    for c in range(C):
        for r in range(P):
            L = part_sizes(shard[r], C)[c]
            n = 3 * L * Hp * D
            per_rank[r].append(flat[off:off + n].view(3, L, Hp, D))
            off += n
    assert off == flat.numel()
    full = torch.cat([torch.cat(blocks, 1) for blocks in per_rank], 1)   # [3, T, Hp, D]
    return tuple(full[s].contiguous() for s in range(3))


def block_lengths(op: int, T: int, H: int, D: int, P: int, C: int):
    """Element count of every (c, p) block, c outer: a chunk of T (pack,
    merge) or a chunk of token shard p (split, unpack), times the elements
    per token."""
    per_token = {0: 3 * (H // P) * D, 1: H * D, 2: (H // P) * D, 3: 3 * (H // P) * D}[op]
    if op in (1, 3):
        shards = part_sizes(T, P)
        return [[part_sizes(shards[p], C)[c] * per_token for p in range(P)] for c in range(C)]
    return [[part_sizes(T, C)[c] * per_token for _ in range(P)] for c in range(C)]


def to_slot_major(op: int, packed: torch.Tensor, T: int, H: int, D: int, P: int, C: int):
    """Cut [c][p] storage into its blocks and concatenate them p outer."""
    flat = _bits(packed).reshape(-1)
    lens = block_lengths(op, T, H, D, P, C)
    blocks = list(torch.split(flat, [n for row in lens for n in row]))
    return torch.cat([blocks[c * P + p] for p in range(P) for c in range(C)]) if blocks \
        else flat.clone()
