"""GPU parity of the opt-in lossy transport: codes, scales and dequantised
outputs bit for bit against the CPU oracle.

"Sol-Engine alignment on SM86 and SM89", table "Upstream gap and
disposition", row "INT8 QKV and FP8 output transport".  The quantiser's
decisions are integer (a code per element) and both sides take them in
float32 with one rounding per step, so the bar is exact equality: every code
byte, every scale's 32-bit pattern, every dequantised bfloat16 pattern.

Inputs: finite bf16 rows of widely varying magnitude with planted zero,
signed-zero, below-floor, at-floor and denormal rows (quantising side); valid
codes (no E4M3 NaN code) with seeded non-negative scales, some zero
(dequantising side).  Shapes cover every vector width (D % 8, D % 4, D % 2,
odd strides), a group size that is not a power of two's worth of vectors
(D = 96), the per-lane loops (D = 520, 1040), ragged chunks and shards, empty
chunks, chunk ranges, both block orders, pinned host memory, the named C
entry points, the pages' full workload in full and the large workload on
sampled rows.
"""
import ctypes

import pytest
import torch

import sequence_head_relayout_gb300 as vf
from oracle import chain, loops
from sequence_head_relayout_gb300 import workloads as W

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("oracle_built")]

DEV = torch.device("cuda:0")
FMT = {"int8": loops.INT8, "e4m3": loops.E4M3}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    vf.lib()
    yield
    torch.cuda.synchronize()


def u8(t):
    return t.reshape(-1).view(torch.uint8).cpu()


def i32(t):
    return t.reshape(-1).view(torch.int32).cpu()


def first_diff(a, b):
    bad = (a != b).nonzero()
    return None if bad.numel() == 0 else (int(bad[0]), int(a[bad[0]]), int(b[bad[0]]))


def pack_view(T, H, D, layout, seed, device=DEV):
    """A finite [T,3,H,D] 16-bit view: contiguous, head-major or padded rows
    (an odd pad makes every stride odd: the 1-element vector path)."""
    if layout == "contiguous":
        base = torch.empty(T * 3 * H * D, dtype=torch.int16, device=device)
        v = base.view(T, 3, H, D)
    elif layout == "head_major":
        base = torch.empty(T * H * 3 * D, dtype=torch.int16, device=device)
        v = base.view(T, H, 3, D).permute(0, 2, 1, 3)
    else:
        pad = int(layout.split(":")[1])
        base = torch.full((T * (3 * H * D + pad),), W._as_i16(W.PAD_SENTINEL),
                          dtype=torch.int16, device=device)
        v = base.view(T, 3 * H * D + pad)[:, :3 * H * D].unflatten(1, (3, H, D))
    W.finite_rows_(v, seed)
    return v


def split_view(T, H, D, layout, seed, device=DEV):
    if layout == "contiguous":
        v = torch.empty((T, H, D), dtype=torch.int16, device=device)
    elif layout == "bhtd":
        v = torch.empty((H, T, D), dtype=torch.int16, device=device).permute(1, 0, 2)
    else:                                             # odd row stride
        v = torch.empty((T, H * D + 1), dtype=torch.int16, device=device)[:, :H * D]
        v = v.unflatten(1, (H, D))
    W.finite_rows_(v, seed)
    return v


def random_codes(n, rows, fmt, seed, device=DEV):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    c = torch.randint(0, 256, (n,), generator=g, device=device, dtype=torch.int32)
    if fmt == "e4m3":
        c = torch.where((c & 0x7F) == 0x7F, torch.zeros_like(c), c)
    codes = c.to(torch.uint8)
    s = torch.randn(rows, generator=g, device=device).abs()
    s = s * torch.pow(2.0, torch.randint(-30, 10, (rows,), generator=g, device=device).float())
    s[::7] = 0.0
    if fmt == "int8":
        codes = codes.view(torch.int8)
    else:
        codes = codes.view(torch.float8_e4m3fn)
    return codes, s.contiguous()


SHAPES = [
    # T, H, D, P, C
    (64, 4, 16, 2, 1),
    (257, 8, 128, 2, 4),
    (1001, 6, 96, 3, 4),      # 12 vectors per row, groups of 16 lanes
    (300, 4, 512, 2, 3),      # 64 vectors per row: the per-lane loop
    (123, 4, 6, 2, 2),        # D % 8 != 0: 2-element vectors
    (77, 4, 12, 4, 5),        # 4-element vectors, empty trailing chunks
    (9, 2, 8, 1, 16),         # more chunks than tokens
    (3, 8, 64, 8, 2),         # fewer tokens than destinations
    (40, 2, 520, 2, 3),       # 65 vectors: quantise on the 8-element path, the
                              # dequantiser's per-lane loop
    (21, 2, 1040, 2, 2),      # 130 vectors: the quantiser's per-lane loop
    (100, 64, 8, 64, 64),     # 12,288 pack pieces: many launches of 120
]


@pytest.mark.parametrize("fmt", ["int8", "e4m3"])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("layout", ["contiguous", "head_major", "pad:3"])
def test_pack_q_parity(fmt, shape, layout):
    T, H, D, P, C = shape
    x = pack_view(T, H, D, layout, seed=T + D)
    codes, scales = vf.qkv_pack_q(x, P, C, fmt=fmt)
    wc, ws = loops.qkv_pack_q(x.cpu(), P, C, FMT[fmt])
    assert torch.equal(u8(codes), u8(wc)), first_diff(u8(codes), u8(wc))
    assert torch.equal(i32(scales), i32(ws)), first_diff(i32(scales), i32(ws))


@pytest.mark.parametrize("fmt", ["int8", "e4m3"])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("layout", ["contiguous", "bhtd", "odd_rows"])
def test_split_q_parity(fmt, shape, layout):
    T, H, D, P, C = shape
    x = split_view(T, H, D, layout, seed=2 * T + D)
    codes, scales = vf.attn_split_q(x, P, C, fmt=fmt)
    wc, ws = loops.attn_split_q(x.cpu(), P, C, FMT[fmt])
    assert torch.equal(u8(codes), u8(wc)), first_diff(u8(codes), u8(wc))
    assert torch.equal(i32(scales), i32(ws)), first_diff(i32(scales), i32(ws))


@pytest.mark.parametrize("fmt", ["int8", "e4m3"])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("dst", ["contiguous", "head_major"])
def test_merge_q_parity(fmt, shape, dst):
    T, H, D, P, C = shape
    n = T * H * D
    codes, scales = random_codes(n, T * H, fmt, seed=T + 5)
    if dst == "contiguous":
        out = torch.full((T, H, D), 0x7FA5, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    else:
        out = torch.full((H, T, D), 0x7FA5, dtype=torch.int16,
                         device=DEV).view(torch.bfloat16).permute(1, 0, 2)
    vf.head_merge_q(codes, scales, T, H, D, P, C, fmt=fmt, out=out)
    want = loops.head_merge_q(u8(codes), scales.cpu(), T, H, D, P, C, FMT[fmt])
    got = out.contiguous().view(torch.int16).reshape(-1).cpu()
    assert torch.equal(got, want.reshape(-1)), first_diff(got, want.reshape(-1))


@pytest.mark.parametrize("fmt", ["int8", "e4m3"])
@pytest.mark.parametrize("shape", SHAPES)
def test_unpack_q_parity(fmt, shape):
    T, H, D, P, C = shape
    Hp = H // P
    codes, scales = random_codes(3 * T * Hp * D, 3 * T * Hp, fmt, seed=T + 9)
    outs = vf.qkv_unpack_q(codes, scales, T, H, D, P, C, fmt=fmt)
    want = loops.qkv_unpack_q(u8(codes), scales.cpu(), T, H, D, P, C, FMT[fmt])
    for o, w in zip(outs, want):
        got = o.view(torch.int16).reshape(-1).cpu()
        assert torch.equal(got, w.reshape(-1)), first_diff(got, w.reshape(-1))


@pytest.mark.parametrize("fmt", ["int8", "e4m3"])
def test_strided_unpack_outputs(fmt):
    # Q, K, V as padded-row slices of one [3, T, Hp, D + 8] allocation
    T, H, D, P, C = 517, 8, 64, 2, 4
    Hp = H // P
    codes, scales = random_codes(3 * T * Hp * D, 3 * T * Hp, fmt, seed=3)
    big = torch.zeros((3, T, Hp, D + 8), dtype=torch.bfloat16, device=DEV)
    outs = tuple(big[s, :, :, :D] for s in range(3))
    vf.qkv_unpack_q(codes, scales, T, H, D, P, C, fmt=fmt, outs=outs)
    want = loops.qkv_unpack_q(u8(codes), scales.cpu(), T, H, D, P, C, FMT[fmt])
    for s in range(3):
        assert torch.equal(outs[s].contiguous().view(torch.int16).cpu(), want[s])
    assert bool((big[:, :, :, D:] == 0).all())                # padding untouched


# ------------------------------------------------------------ chunk ranges, orders

def _reorder_slot_major(op, flat, T, H, D, P, C, per):
    """[c][p] blocks -> [p][c]; ``per`` = items per element (1 for codes,
    1/D for scales, given as a divisor)."""
    lens = [n // per for row in chain.block_lengths(op, T, H, D, P, C) for n in row]
    blocks = list(torch.split(flat, lens))
    return torch.cat([blocks[c * P + p] for p in range(P) for c in range(C)])


@pytest.mark.parametrize("fmt", ["int8", "e4m3"])
def test_slot_major_and_chunk_ranges(fmt):
    T, H, D, P, C = 777, 8, 64, 4, 4
    x = split_view(T, H, D, "bhtd", seed=41)
    # slot-major split: the chunk-major result with blocks reordered
    codes, scales = vf.attn_split_q(x, P, C, fmt=fmt, order="slot_major")
    wc, ws = loops.attn_split_q(x.cpu(), P, C, FMT[fmt])
    assert torch.equal(u8(codes), _reorder_slot_major(1, u8(wc), T, H, D, P, C, 1))
    assert torch.equal(i32(scales), _reorder_slot_major(1, i32(ws), T, H, D, P, C, D))
    # the pack one chunk per call equals one full call
    xp = pack_view(T, H, D, "contiguous", seed=42)
    full_c, full_s = vf.qkv_pack_q(xp, P, C, fmt=fmt)
    part_c = torch.zeros_like(full_c.view(torch.uint8)).view(full_c.dtype)
    part_s = torch.zeros_like(full_s)
    for c in range(C):
        vf.qkv_pack_q(xp, P, C, fmt=fmt, codes=part_c, scales=part_s, chunks=(c, 1))
    assert torch.equal(u8(part_c), u8(full_c)) and torch.equal(i32(part_s), i32(full_s))
    # a chunk range touches only its own blocks
    blank_c = torch.full_like(full_c.view(torch.uint8), 0xA5).view(full_c.dtype)
    blank_s = torch.full_like(full_s, -1.0)
    vf.qkv_pack_q(xp, P, C, fmt=fmt, codes=blank_c, scales=blank_s, chunks=(1, 2))
    _, lengths, offs = vf.piece_table(vf.OP_QKV_PACK, T, H, D, P, C)
    lo, hi = offs[1 * P], offs[3 * P] if 3 < C else full_c.numel()
    got, ref = u8(blank_c), u8(full_c)
    assert torch.equal(got[lo:hi], ref[lo:hi])
    assert bool((got[:lo] == 0xA5).all()) and bool((got[hi:] == 0xA5).all())
    assert bool((blank_s[:lo // D] == -1).all()) and bool((blank_s[hi // D:] == -1).all())
    # merge and unpack, slot-major input: equal to the chunk-major result of
    # the reordered-back storage
    n = T * H * D
    mc, ms = random_codes(n, T * H, fmt, seed=43)
    out_s = vf.head_merge_q(mc, ms, T, H, D, P, C, fmt=fmt, order="slot_major")
    lens = [n_ for row in chain.block_lengths(2, T, H, D, P, C) for n_ in row]
    cm_codes = _to_chunk_major(u8(mc), lens, P, C, 1)
    cm_scales = _to_chunk_major(ms.cpu(), lens, P, C, D)
    want = loops.head_merge_q(cm_codes, cm_scales, T, H, D, P, C, FMT[fmt])
    assert torch.equal(out_s.view(torch.int16).cpu(), want)


def _to_chunk_major(flat, lens, P, C, per):
    """Inverse of the slot-major reorder: blocks stored p outer -> c outer."""
    lens_sm = [lens[c * P + p] // per for p in range(P) for c in range(C)]
    blocks = list(torch.split(flat, lens_sm))
    by_cp = {}
    i = 0
    for p in range(P):
        for c in range(C):
            by_cp[(c, p)] = blocks[i]
            i += 1
    return torch.cat([by_cp[(c, p)] for c in range(C) for p in range(P)])


def test_pinned_host_buffers():
    # codes and scales written straight into pinned host memory
    T, H, D, P, C = 300, 8, 128, 2, 4
    x = pack_view(T, H, D, "contiguous", seed=51)
    n = 3 * T * H * D
    codes = torch.empty(n, dtype=torch.int8, pin_memory=True)
    scales = torch.empty(n // D, dtype=torch.float32, pin_memory=True)
    vf.qkv_pack_q(x, P, C, fmt="int8", codes=codes, scales=scales)
    torch.cuda.synchronize()
    wc, ws = loops.qkv_pack_q(x.cpu(), P, C, loops.INT8)
    assert torch.equal(u8(codes), u8(wc)) and torch.equal(i32(scales), i32(ws))


# ------------------------------------------------------------ named C entry points

def _i64(*xs):
    return (ctypes.c_int64 * len(xs))(*xs)


def _s():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_named_entry_points():
    L = vf.lib()
    T, H, D, P, C = 333, 8, 64, 2, 4
    Hp = H // P
    x = pack_view(T, H, D, "head_major", seed=61)
    n = 3 * T * H * D
    codes = torch.empty(n, dtype=torch.int8, device=DEV)
    scales = torch.empty(n // D, dtype=torch.float32, device=DEV)
    assert L.vf_qkv_pack_int8(x.data_ptr(), _i64(*x.stride()), T, H, D, P, C, codes.data_ptr(),
                              scales.data_ptr(), _s()) == 0
    wc, ws = loops.qkv_pack_q(x.cpu(), P, C, loops.INT8)
    assert torch.equal(u8(codes), u8(wc)) and torch.equal(i32(scales), i32(ws))

    rc, rs = random_codes(3 * T * Hp * D, 3 * T * Hp, "int8", seed=62)
    q, k, v = (torch.empty((T, Hp, D), dtype=torch.bfloat16, device=DEV) for _ in range(3))
    assert L.vf_qkv_unpack_int8(rc.data_ptr(), rs.data_ptr(), T, H, D, P, C, q.data_ptr(),
                                k.data_ptr(), v.data_ptr(), None, _s()) == 0
    want = loops.qkv_unpack_q(u8(rc), rs.cpu(), T, H, D, P, C, loops.INT8)
    for o, w in zip((q, k, v), want):
        assert torch.equal(o.view(torch.int16).cpu(), w)

    a = split_view(T, H, D, "bhtd", seed=63)
    fc = torch.empty(T * H * D, dtype=torch.uint8, device=DEV)
    fs = torch.empty(T * H, dtype=torch.float32, device=DEV)
    assert L.vf_attn_split_fp8(a.data_ptr(), _i64(*a.stride()), T, H, D, P, C, fc.data_ptr(),
                               fs.data_ptr(), _s()) == 0
    wc, ws = loops.attn_split_q(a.cpu(), P, C, loops.E4M3)
    assert torch.equal(u8(fc), u8(wc)) and torch.equal(i32(fs), i32(ws))

    mc, ms = random_codes(T * H * D, T * H, "e4m3", seed=64)
    out = torch.empty((T, H, D), dtype=torch.bfloat16, device=DEV)
    assert L.vf_head_merge_fp8(mc.data_ptr(), ms.data_ptr(), None, T, H, D, P, C,
                               out.data_ptr(), _s()) == 0
    want = loops.head_merge_q(u8(mc), ms.cpu(), T, H, D, P, C, loops.E4M3)
    assert torch.equal(out.view(torch.int16).cpu(), want)


# ------------------------------------------------------------ full-size workloads

def test_pages_workload_in_full():
    """The pages' shape (T*H = 55,414*28, D = 128, two destinations, four
    overlap chunks) in the benchmark's layouts: INT8 pack and unpack, E4M3
    split and merge, every output compared in full."""
    cfg = W.CONFIGS["pages"]
    T, H, D, P, C = cfg.T, cfg.H, cfg.D, cfg.P, cfg.C
    x = pack_view(T, H, D, "pad:64", seed=71)
    codes, scales = vf.qkv_pack_q(x, P, C, fmt="int8")
    wc, ws = loops.qkv_pack_q(x.cpu(), P, C, loops.INT8)
    assert torch.equal(u8(codes), u8(wc)) and torch.equal(i32(scales), i32(ws))
    del x, codes, scales
    # the receive side takes the oracle's own codes and scales (one rank's worth)
    Hp = H // P
    rc, rs = wc[:3 * T * Hp * D].contiguous(), ws[:3 * T * Hp].contiguous()
    outs = vf.qkv_unpack_q(rc.to(DEV), rs.to(DEV), T, H, D, P, C, fmt="int8")
    want = loops.qkv_unpack_q(rc, rs, T, H, D, P, C, loops.INT8)
    for o, w in zip(outs, want):
        assert torch.equal(o.view(torch.int16).cpu(), w)
    del outs, want, wc, ws, rc, rs

    a = split_view(T, H, D, "bhtd", seed=72)
    fc, fs = vf.attn_split_q(a, P, C, fmt="e4m3")
    wc, ws = loops.attn_split_q(a.cpu(), P, C, loops.E4M3)
    assert torch.equal(u8(fc), u8(wc)) and torch.equal(i32(fs), i32(ws))
    del fc, fs
    out = vf.head_merge_q(wc.to(DEV), ws.to(DEV), T, H, D, P, C, fmt="e4m3")
    want = loops.head_merge_q(wc, ws, T, H, D, P, C, loops.E4M3)
    assert torch.equal(out.view(torch.int16).cpu(), want)


def test_large_workload_sampled_rows():
    """The large shape (200,000 tokens, 32 heads, 8 destinations): the GPU
    pack in full, checked on 4,000 sampled head rows, each quantised alone by
    the oracle and located through the oracle's piece table."""
    cfg = W.CONFIGS["large"]
    T, H, D, P, C = cfg.T, cfg.H, cfg.D, cfg.P, cfg.C
    Hp = H // P
    x = pack_view(T, H, D, "contiguous", seed=81)
    for fmt in ("int8", "e4m3"):
        codes, scales = vf.qkv_pack_q(x, P, C, fmt=fmt)
        tok, lens, offs = loops.piece_table(vf.OP_QKV_PACK, T, H, D, P, C)
        g = torch.Generator().manual_seed(82)
        ts = torch.randint(0, T, (4000,), generator=g).tolist()
        ss = torch.randint(0, 3, (4000,), generator=g).tolist()
        hs = torch.randint(0, H, (4000,), generator=g).tolist()
        rows = x[ts, ss, hs].cpu().view(4000, 1, D)
        wc, ws = loops.attn_split_q(rows, 1, 1, FMT[fmt])       # each row alone
        wc = u8(wc).view(4000, D)
        cu, sc = u8(codes), i32(scales)
        wsb = i32(ws)
        for i, (t, s, h) in enumerate(zip(ts, ss, hs)):
            c = next(c for c in range(C) if tok[c * P] <= t < tok[c * P] + lens[c * P])
            p, hh = divmod(h, Hp)
            L = lens[c * P + p]
            e = offs[c * P + p] + ((s * L + (t - tok[c * P])) * Hp + hh) * D
            assert torch.equal(cu[e:e + D], wc[i]), (fmt, t, s, h)
            assert int(sc[e // D]) == int(wsb[i]), (fmt, t, s, h)


# ------------------------------------------------------------ accuracy gate

def test_transport_accuracy_gate():
    """The lossy transport's quality gate on seeded N(0,1) activations at the
    pages' head count and head dim (the benchmark reports the same figures):
    INT8 Q/K/V through pack -> unpack, then attention; E4M3 attention output
    through split -> merge.  Expected from the format: INT8 steps are
    amax/127 (about 0.6% RMS of a unit-variance row), E4M3 keeps 3 mantissa
    bits (a few % RMS)."""
    import bench
    q = bench.lossy_quality(DEV, T=2048)
    assert 0.002 < q["int8_qkv_rel_err"] < 0.015, q
    assert 0.0 < q["int8_qkv_attention_out_rel_err"] < 0.02, q
    assert 0.01 < q["e4m3_attention_out_rel_err"] < 0.05, q


# ------------------------------------------------------------ rounding ties on the device

def _e4m3_positive_grid():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).float()
    return sorted({v for v in vals.tolist() if v == v and v >= 0})


@pytest.mark.parametrize("fmt", ["int8", "e4m3"])
def test_rounding_ties_on_device(fmt):
    """Rows whose scale factor is exactly 1 (amax = 127 or 448), so that
    q = x: every half-integer (INT8) and every midpoint between neighbouring
    E4M3 values (all exact in bfloat16) is a tie, which the device must round
    to even exactly as the oracle does; both signs, on both vector paths."""
    if fmt == "int8":
        top = 127.0
        ties = [k + 0.5 for k in range(0, 127)]
    else:
        top = 448.0
        grid = _e4m3_positive_grid()
        ties = [(a + b) / 2 for a, b in zip(grid, grid[1:])]
    vals = ties + [-t for t in ties]
    D = 128
    rows = -(-len(vals) // (D - 1))
    x = torch.zeros(rows, D)
    flat = torch.tensor(vals + [0.0] * (rows * (D - 1) - len(vals)))
    x[:, 1:] = flat.view(rows, D - 1)
    x[:, 0] = top
    xb = x.to(torch.bfloat16)
    assert torch.equal(xb.float(), x)                      # every tie exact in bfloat16
    bits = xb.view(torch.int16).view(rows, 1, D)
    for D_used, sl in ((D, bits), (6, bits[:, :, :6].contiguous())):
        codes, scales = vf.attn_split_q(sl.to(DEV), 1, 1, fmt=fmt)
        wc, ws = loops.attn_split_q(sl, 1, 1, FMT[fmt])
        assert torch.equal(u8(codes), u8(wc)), first_diff(u8(codes), u8(wc))
        assert torch.equal(i32(scales), i32(ws))
