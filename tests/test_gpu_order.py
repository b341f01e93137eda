"""GPU parity of the slot-major ([p][c]) block order against the oracle: the
same blocks as the chunk-major layout, placed destination by destination."""
import pytest
import torch

import sequence_head_relayout_gb300 as vf
from oracle import loops
from sequence_head_relayout_gb300 import workloads as W

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("oracle_built")]

DEV = torch.device("cuda:0")
SM = "slot_major"


def same(a, b):
    return torch.equal(a.reshape(-1).view(torch.int16).cpu(), b.reshape(-1).view(torch.int16))


@pytest.mark.parametrize("name", ["tiny", "4k", "pages", "ragged", "large"])
def test_slot_major_all_ops(name):
    cfg = W.CONFIGS[name]
    T, H, D, P, C = cfg.T, cfg.H, cfg.D, cfg.P, cfg.C
    Hp = H // P
    src4, _ = W.pack_source(cfg, device=DEV)
    want = loops.to_slot_major(0, loops.qkv_pack(src4.cpu(), P, C), T, H, D, P, C)
    assert same(vf.qkv_pack(src4, P, C, order=SM), want)
    assert same(vf.qkv_pack3(src4[:, 0], src4[:, 1], src4[:, 2], P, C, order=SM), want)
    del want

    src3, _ = W.split_source(cfg, device=DEV)
    want = loops.to_slot_major(1, loops.attn_split(src3.cpu(), P, C), T, H, D, P, C)
    assert same(vf.attn_split(src3, P, C, order=SM), want)

    cp = W.merge_source(cfg)                                   # chunk-major bits, CPU
    pc = loops.to_slot_major(2, cp, T, H, D, P, C).to(DEV)
    out, _ = W.merge_destination(cfg, device=DEV)
    vf.head_merge(pc, T, H, D, P, C, out=out, order=SM)
    assert same(out.contiguous(), loops.head_merge(cp, T, H, D, P, C))

    recv = torch.empty(3 * T * Hp * D, dtype=torch.int16)
    W.fill_(recv, cfg.payload, cfg.seed + 3000)
    pcr = loops.to_slot_major(3, recv, T, H, D, P, C).to(DEV)
    got = vf.qkv_unpack(pcr, T, H, D, P, C, order=SM)
    for a, b in zip(got, loops.qkv_unpack_recv(recv, T, H, D, P, C)):
        assert same(a, b)


def test_slot_major_chunk_ranges_compose():
    T, H, D, P, C = 1001, 8, 32, 4, 4
    g = torch.Generator().manual_seed(3)
    x4 = torch.randint(-(1 << 15), 1 << 15, (T, 3, H, D), generator=g, dtype=torch.int32).to(
        torch.int16).to(DEV)
    full = vf.qkv_pack(x4, P, C, order=SM)
    part = torch.zeros_like(full)
    for c in (2, 0, 3, 1):
        vf.qkv_pack(x4, P, C, out=part, chunks=(c, 1), order=SM)
    assert torch.equal(part, full)
    # destination p's span is contiguous in slot-major order
    tok, length, off = vf.piece_table(vf.OP_QKV_PACK, T, H, D, P, C, order=SM)
    per = 3 * (H // P) * D
    for p in range(P):
        assert off[p] + sum(length[c * P + p] for c in range(C)) * per == (
            off[p + 1] if p + 1 < P else full.numel())


def test_split_slot_major_is_a_contiguous_copy():
    cfg = W.CONFIGS["pages"]
    src3, _ = W.split_source(cfg, device=DEV)
    got = vf.attn_split(src3, cfg.P, cfg.C, order=SM)
    assert torch.equal(got, src3.contiguous().reshape(-1))
