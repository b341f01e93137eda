"""GPU parity of the opt-in lossy transport on rows that hold NaN or infinity.

"Sol-Engine alignment on SM86 and SM89", table "Upstream gap and
disposition", row "INT8 QKV and FP8 output transport", names the variant and
gives no format.  The reading for values the format cannot carry: a head row
holding a NaN or an infinity is sent as a lost row (scale = the float32 quiet
NaN 0x7FC00000, every code 0) and leaves every other row alone; the receive
side writes the bfloat16 quiet NaN 0x7FC0 into every element of a row whose
scale is not finite.  The oracle states the same reading and is pinned on
hand-worked rows; here the kernels are compared with it bit for bit (code
bytes, scale bit patterns, bfloat16 patterns) at the 4k and the ragged
workloads, with NaN and infinity planted into about one head row in 97, and
on uniform 16-bit patterns (row maxima across the whole bfloat16 range,
subnormals, about one row in five lost) through every op.

Every expected value is the oracle's, computed from the same seeded inputs;
the receive side is fed the oracle's own codes and scales.
"""
import pytest
import torch

import sequence_head_relayout_gb300 as vf
from oracle import loops
from sequence_head_relayout_gb300 import workloads as W

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("oracle_built")]

DEV = torch.device("cuda:0")
LOST_SCALE = 0x7FC00000
LOST_VALUE = 0x7FC0


def u8(t):
    return t.reshape(-1).view(torch.uint8).cpu()


def u32(t):
    return t.reshape(-1).view(torch.int32).cpu().to(torch.int64) & 0xFFFFFFFF


def u16(t):
    return t.reshape(-1).view(torch.int16).cpu().to(torch.int32) & 0xFFFF


def first_diff(a, b):
    bad = (a != b).nonzero()
    return None if bad.numel() == 0 else (int(bad[0]), int(a[bad[0]]), int(b[bad[0]]))


def _planted(view, seed):
    """Finite rows of widely varying magnitude, then NaN and infinities
    planted into about one row in 97."""
    W.finite_rows_(view, seed)
    W.plant_non_finite_(view, seed + 1)
    return view


@pytest.mark.parametrize("name", ["4k", "ragged"])
def test_int8_pack_and_unpack_with_lost_rows(name):
    cfg = W.CONFIGS[name]
    T, H, D, P, C = cfg.T, cfg.H, cfg.D, cfg.P, cfg.C
    x, _ = W.pack_source(cfg, device=DEV)
    _planted(x, cfg.seed + 40)
    codes, scales = vf.qkv_pack_q(x, P, C, fmt="int8")
    wc, ws = loops.qkv_pack_q(x.cpu(), P, C, loops.INT8)
    lost = int((u32(ws) == LOST_SCALE).sum())
    assert lost >= 3 * T * H // 97 - 1                 # the planted rows are lost rows
    assert torch.equal(u8(codes), u8(wc)), first_diff(u8(codes), u8(wc))
    assert torch.equal(u32(scales), u32(ws)), first_diff(u32(scales), u32(ws))

    # receive side: one head group's worth of the oracle's codes and scales
    Hp = H // P
    nu = 3 * T * Hp * D
    rc, rs = wc[:nu].contiguous(), ws[:nu // D].contiguous()
    assert int((u32(rs) == LOST_SCALE).sum()) > 0
    outs = vf.qkv_unpack_q(rc.to(DEV), rs.to(DEV), T, H, D, P, C, fmt="int8")
    want = loops.qkv_unpack_q(rc, rs, T, H, D, P, C, loops.INT8)
    for got, exp in zip(outs, want):
        assert torch.equal(u16(got), u16(exp)), first_diff(u16(got), u16(exp))


@pytest.mark.parametrize("name", ["4k", "ragged"])
def test_e4m3_split_and_merge_with_lost_rows(name):
    cfg = W.CONFIGS[name]
    T, H, D, P, C = cfg.T, cfg.H, cfg.D, cfg.P, cfg.C
    x, _ = W.split_source(cfg, device=DEV)
    _planted(x, cfg.seed + 50)
    codes, scales = vf.attn_split_q(x, P, C, fmt="e4m3")
    wc, ws = loops.attn_split_q(x.cpu(), P, C, loops.E4M3)
    assert int((u32(ws) == LOST_SCALE).sum()) >= T * H // 97 - 1
    assert torch.equal(u8(codes), u8(wc)), first_diff(u8(codes), u8(wc))
    assert torch.equal(u32(scales), u32(ws)), first_diff(u32(scales), u32(ws))

    dst, base = W.merge_destination(cfg, device=DEV, fill=0x1234)
    out = dst.view(torch.bfloat16)
    vf.head_merge_q(wc.view(torch.float8_e4m3fn).to(DEV), ws.to(DEV), T, H, D, P, C,
                    fmt="e4m3", out=out)
    want = loops.head_merge_q(wc, ws, T, H, D, P, C, loops.E4M3)
    assert torch.equal(u16(dst.contiguous()), u16(want)), \
        first_diff(u16(dst.contiguous()), u16(want))
    assert int((u16(want) == LOST_VALUE).sum()) >= D * (T * H // 97 - 1)


@pytest.mark.parametrize("fmt", ["int8", "e4m3"])
@pytest.mark.parametrize("D", [8, 64, 128, 520])
def test_non_finite_scales_on_the_receive_side(fmt, D):
    # scales +inf, -inf, NaNs with payloads and huge finite values (products
    # that overflow to infinity) among ordinary ones; every dequantiser path:
    # D = 8 and 64, 128 on the 8-element path, D = 520 on the per-lane loop
    T, H, P, C = 301, 4, 2, 3
    n = T * H * D
    g = torch.Generator().manual_seed(D + len(fmt))
    c = torch.randint(0, 256, (n,), generator=g, dtype=torch.int32)
    if fmt == "e4m3":
        c = torch.where((c & 0x7F) == 0x7F, torch.zeros_like(c), c)
    codes = c.to(torch.uint8)
    rows = n // D
    s = torch.rand(rows, generator=g) * 2.0 ** -10
    bits = s.view(torch.int32).clone()
    special = torch.tensor([0x7F800000, 0xFF800000, 0x7FC00000, 0xFFC00001, 0x7F800001,
                            0x7F000000, 0x7E800000], dtype=torch.int64).to(torch.int32)
    pick = torch.arange(0, rows, 11)
    bits[pick] = special[torch.arange(pick.numel()) % special.numel()]
    s = bits.view(torch.float32)
    dt = torch.int8 if fmt == "int8" else torch.float8_e4m3fn
    f = loops.INT8 if fmt == "int8" else loops.E4M3
    got = vf.head_merge_q(codes.view(dt).to(DEV), s.to(DEV), T, H, D, P, C, fmt=fmt)
    want = loops.head_merge_q(codes.view(dt) if fmt == "int8" else codes, s, T, H, D, P, C, f)
    assert torch.equal(u16(got), u16(want)), first_diff(u16(got), u16(want))
    assert int((u16(want) == LOST_VALUE).sum()) >= 5 * D * (pick.numel() // 7)


def test_e4m3_nan_codes_arrive_as_nan():
    # the quantiser never writes the E4M3 NaN codes 0x7F and 0xFF; a receive
    # side given them writes a NaN there (payload unspecified) and leaves
    # every other element exact
    T, H, D, P, C = 64, 2, 64, 2, 2
    n = T * H * D
    g = torch.Generator().manual_seed(77)
    c = torch.randint(0, 256, (n,), generator=g, dtype=torch.int32)
    c[::13] = 0x7F
    c[5::17] = 0xFF
    codes = c.to(torch.uint8)
    s = torch.rand(n // D, generator=g) + 0.5
    got = vf.head_merge_q(codes.view(torch.float8_e4m3fn).to(DEV), s.to(DEV), T, H, D, P, C,
                          fmt="e4m3")
    want = loops.head_merge_q(codes, s, T, H, D, P, C, loops.E4M3)
    gf = got.float().cpu().reshape(-1)
    wf = want.view(torch.bfloat16).float().reshape(-1)
    assert torch.equal(gf.isnan(), wf.isnan())
    ok = ~wf.isnan()
    assert torch.equal(u16(got)[ok], u16(want)[ok])
    # the merge writes the chunk layout's codes to token-major order: every
    # NaN code becomes exactly one NaN element
    assert int(wf.isnan().sum()) == int(((c & 0x7F) == 0x7F).sum())


@pytest.mark.parametrize("fmt", ["int8", "e4m3"])
@pytest.mark.parametrize("T,H,D,P,C", [(1500, 8, 64, 4, 3), (700, 6, 128, 2, 4),
                                       (333, 4, 32, 2, 2)])
def test_random_bit_patterns_every_op(fmt, T, H, D, P, C):
    # uniform 16-bit patterns: magnitudes over the whole bfloat16 range (row
    # maxima up to 2^128, where 1/amax is subnormal), subnormals, and about
    # one row in five holding a NaN or an infinity; every op, bit for bit
    f = loops.INT8 if fmt == "int8" else loops.E4M3
    x4 = W.fill_(torch.empty(T * 3 * H * D, dtype=torch.int16, device=DEV), "bits",
                 T + D).view(T, 3, H, D)
    codes, scales = vf.qkv_pack_q(x4, P, C, fmt=fmt)
    wc, ws = loops.qkv_pack_q(x4.cpu(), P, C, f)
    assert int((u32(ws) == LOST_SCALE).sum()) > 0
    assert torch.equal(u8(codes), u8(wc)), first_diff(u8(codes), u8(wc))
    assert torch.equal(u32(scales), u32(ws)), first_diff(u32(scales), u32(ws))
    x3 = W.fill_(torch.empty(H * T * D, dtype=torch.int16, device=DEV), "bits",
                 2 * T + D).view(H, T, D).permute(1, 0, 2)
    codes, scales = vf.attn_split_q(x3, P, C, fmt=fmt)
    sc, ss = loops.attn_split_q(x3.cpu(), P, C, f)
    assert torch.equal(u8(codes), u8(sc)), first_diff(u8(codes), u8(sc))
    assert torch.equal(u32(scales), u32(ss)), first_diff(u32(scales), u32(ss))
    # receive sides fed the oracle's own codes and scales
    dt = torch.int8 if fmt == "int8" else torch.float8_e4m3fn
    got = vf.head_merge_q(sc.view(dt).to(DEV), ss.to(DEV), T, H, D, P, C, fmt=fmt)
    want = loops.head_merge_q(sc, ss, T, H, D, P, C, f)
    assert torch.equal(u16(got), u16(want)), first_diff(u16(got), u16(want))
    nu = 3 * T * (H // P) * D
    rc, rs = wc[:nu].contiguous(), ws[:nu // D].contiguous()
    outs = vf.qkv_unpack_q(rc.view(dt).to(DEV), rs.to(DEV), T, H, D, P, C, fmt=fmt)
    for g, w in zip(outs, loops.qkv_unpack_q(rc, rs, T, H, D, P, C, f)):
        assert torch.equal(u16(g), u16(w)), first_diff(u16(g), u16(w))
