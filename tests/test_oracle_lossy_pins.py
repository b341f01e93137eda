"""Pins of the lossy-transport oracle (opt-in INT8 / FP8 E4M3 transport).

"Sol-Engine alignment on SM86 and SM89", table "Upstream gap and
disposition", row "INT8 QKV and FP8 output transport", names the variant and
gives no format; the oracle's reading (per head row absmax scaling, float32
decisions, round half to even, E4M3 saturating at 448, dequantisation to
bfloat16) is pinned here against things other than itself:

  * the scalar conversions against PyTorch's own float8_e4m3fn and bfloat16
    conversions (library routines), over every code and every tie;
  * a row worked by hand;
  * rows built on the exact grid (integer codes times a power of two), where
    quantisation is exact: the codes must then be the exact oracle's layout of
    the integer codes and the round trip must reproduce the input bit for bit
    -- this ties the lossy layout to the exact one, itself pinned by golden
    examples;
  * closed-form error bounds on random rows (rounding to nearest, not
    truncation; the right scale);
  * the degenerate rows: all zero, below the 2^-96 floor, signed zero.
"""
import math

import pytest
import torch

from oracle import loops

pytestmark = pytest.mark.usefixtures("oracle_built")

INT8, E4M3 = loops.INT8, loops.E4M3


def _bf16_bits(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16).view(torch.int16)


def _bits_to_f32(b: torch.Tensor) -> torch.Tensor:
    return b.view(torch.bfloat16).float()


# ---------------------------------------------------------------- scalar pins

def test_e4m3_decode_every_code_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float()
    for c in range(256):
        if c in (0x7F, 0xFF):                # the format's two NaN codes (never written)
            assert math.isnan(loops.e4m3_decode(c)) and math.isnan(ref[c].item())
            continue
        assert loops.e4m3_decode(c) == ref[c].item(), hex(c)


def _e4m3_grid():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).float()
    return sorted({v for v in vals.tolist() if not math.isnan(v) and v >= 0})


def test_e4m3_encode_matches_torch_on_codes_ties_and_random():
    grid = _e4m3_grid()
    mids = [(a + b) / 2 for a, b in zip(grid, grid[1:])]          # exact ties, all in float32
    g = torch.Generator().manual_seed(11)
    rnd = (torch.rand(20000, generator=g) * 2 - 1) * 463.0
    tiny = torch.rand(4000, generator=g) * 2 ** -5               # subnormal range and below
    vals = torch.tensor(grid + mids + [-v for v in grid + mids], dtype=torch.float32)
    vals = torch.cat([vals, rnd, tiny, -tiny])
    ref = vals.to(torch.float8_e4m3fn).view(torch.uint8).tolist()
    got = [loops.e4m3_encode(v) for v in vals.tolist()]
    bad = [(v, r, o) for v, r, o in zip(vals.tolist(), ref, got) if r != o]
    assert not bad, bad[:5]


def test_e4m3_encode_saturates_at_448():
    # E4M3 has no infinities; its largest finite value is 1.75 * 2^8 = 448
    # (code 0x7E): with saturation every larger magnitude maps there.
    for v in (448.0, 450.0, 464.0, 480.0, 1e4, 3e38):
        assert loops.e4m3_encode(v) == 0x7E
        assert loops.e4m3_encode(-v) == 0xFE
    assert loops.e4m3_encode(0.0) == 0x00 and loops.e4m3_encode(-0.0) == 0x80


def test_f32_to_bf16_matches_torch_including_ties():
    g = torch.Generator().manual_seed(12)
    bits = torch.randint(0, 1 << 31, (20000,), generator=g, dtype=torch.int64)
    sign = torch.randint(0, 2, (20000,), generator=g, dtype=torch.int64) << 31
    u = (bits | sign) & 0xFFFFFFFF
    u = u[((u >> 23) & 0xFF) != 0xFF]                            # finite only
    ties = (u & ~0xFFFF) | 0x8000                                 # exactly half-way
    u = torch.cat([u, ties, torch.tensor([0, 1 << 31, 0x7F7FFFFF, 0x00000001])])
    f = u.to(torch.int32).view(torch.float32)
    ref = f.to(torch.bfloat16).view(torch.int16).tolist()
    got = [loops.f32_to_bf16(v) for v in f.tolist()]
    got = [x - (1 << 16) if x >= 1 << 15 else x for x in got]     # as int16
    bad = [(hex(int(a)), r, o) for a, r, o in zip(u.tolist(), ref, got) if r != o]
    assert not bad, bad[:5]


# ---------------------------------------------------------------- a row by hand

def test_row_worked_by_hand():
    # row (1, -1/2, 1/4, 0, 3/4, -1, 1/8, 3/8): amax = 1.
    # INT8: inv = 127, q = (127, -63.5, 31.75, 0, 95.25, -127, 15.875, 47.625);
    #   half to even sends -63.5 to -64; scale = 1/127 (float32).
    # E4M3: inv = 448, q = (448, -224, 112, 0, 336, -448, 56, 168);
    #   336 = 1.3125 * 2^8 and 168 = 1.3125 * 2^7 are ties between mantissas
    #   2 and 3 and go to the even 2: 320 and 160.
    row = torch.tensor([1.0, -0.5, 0.25, 0.0, 0.75, -1.0, 0.125, 0.375])
    x = _bf16_bits(row).view(1, 1, 8)
    codes, scales = loops.attn_split_q(x, 1, 1, INT8)
    assert codes.tolist() == [127, -64, 32, 0, 95, -127, 16, 48]
    assert scales.tolist() == [torch.tensor(1.0 / 127, dtype=torch.float32).item()]
    codes, scales = loops.attn_split_q(x, 1, 1, E4M3)
    assert codes.tolist() == [0x7E, 0xF6, 0x6E, 0x00, 0x7A, 0xFE, 0x66, 0x72]
    assert scales.tolist() == [torch.tensor(1.0 / 448, dtype=torch.float32).item()]
    # dequantised: 320/448 and 160/448 become 0.714285.. and 0.357142..,
    # which round to bfloat16 as 0.71484375 and 0.357421875
    y = loops.head_merge_q(codes, scales, 1, 1, 8, 1, 1, E4M3)
    assert _bits_to_f32(y).flatten().tolist() == [1.0, -0.5, 0.25, 0.0, 0.71484375, -1.0, 0.125,
                                                  0.357421875]


def test_int8_ties_go_to_even():
    # amax = 127 makes inv = 1 and q = x exactly: every half-integer is a tie
    row = torch.tensor([127.0, 0.5, 1.5, 2.5, -0.5, -2.5, 3.5, 126.5])
    codes, scales = loops.attn_split_q(_bf16_bits(row).view(1, 1, 8), 1, 1, INT8)
    assert scales.tolist() == [1.0]
    assert codes.tolist() == [127, 0, 2, 2, 0, -2, 4, 126]


# ------------------------------------------------- exact grid: layout and round trip

def _grid_rows(shape, fmt, seed):
    """Rows whose quantisation is exact: per head row an exponent e, codes
    from the format's grid with one element at the full-scale magnitude; the
    value is code * 2^e.  Returns (bf16 bits, codes as 16-bit patterns,
    exponent per row)."""
    g = torch.Generator().manual_seed(seed)
    *lead, D = shape
    if fmt == INT8:
        codes = torch.randint(-127, 128, shape, generator=g, dtype=torch.int32)
        full = 127
        val = codes.float()
    else:
        codes = torch.randint(0, 256, shape, generator=g, dtype=torch.int32)
        codes[(codes & 0x7F) == 0x7F] = 0x00                       # no NaN codes
        full = 0x7E
        val = codes.to(torch.uint8).view(torch.float8_e4m3fn).float()
    where = torch.randint(0, D, tuple(lead) + (1,), generator=g)
    sgn = torch.randint(0, 2, tuple(lead) + (1,), generator=g)
    if fmt == INT8:
        top = torch.where(sgn == 0, 127, -127).to(torch.int32)
        codes.scatter_(-1, where, top)
        val = codes.float()
    else:
        top = torch.where(sgn == 0, full, full | 0x80).to(torch.int32)
        codes.scatter_(-1, where, top)
        val = codes.to(torch.uint8).view(torch.float8_e4m3fn).float()
    e = torch.randint(-20, 21, tuple(lead) + (1,), generator=g)
    x = val * torch.pow(2.0, e.float())
    bits = _bf16_bits(x)
    assert torch.equal(_bits_to_f32(bits), x)                      # exact in bfloat16
    return bits, codes.to(torch.int16), e.squeeze(-1)


@pytest.mark.parametrize("fmt", [INT8, E4M3])
@pytest.mark.parametrize("T,H,D,P,C", [(13, 4, 8, 2, 3), (7, 6, 16, 3, 4), (5, 2, 24, 1, 2)])
def test_pack_codes_are_exact_layout_and_round_trip(fmt, T, H, D, P, C):
    x, codes16, e = _grid_rows((T, 3, H, D), fmt, 100 + T + fmt)
    codes, scales = loops.qkv_pack_q(x, P, C, fmt)
    expect = loops.qkv_pack(codes16, P, C)                          # exact layout of the codes
    assert torch.equal(codes.to(torch.int16) & 0xFF, expect & 0xFF)
    # scale = amax / top = 2^e exactly, one per head row, in the pack's row order
    srow = torch.pow(2.0, e.float()).unsqueeze(-1).expand(T, 3, H, D).contiguous()
    expect_s = _bits_to_f32(loops.qkv_pack(_bf16_bits(srow), P, C)[::D])
    assert torch.equal(scales, expect_s)


@pytest.mark.parametrize("fmt", [INT8, E4M3])
@pytest.mark.parametrize("T,H,D,P,C", [(13, 4, 8, 2, 3), (11, 3, 16, 4, 2)])
def test_split_merge_round_trip_on_exact_grid(fmt, T, H, D, P, C):
    # split of a head group, then the merge of the full-head view: with one
    # destination (P=1) the merge reads exactly the split's storage
    x, codes16, _ = _grid_rows((T, H, D), fmt, 200 + T + fmt)
    codes, scales = loops.attn_split_q(x, P, C, fmt)
    assert torch.equal(codes.to(torch.int16) & 0xFF, loops.attn_split(codes16, P, C) & 0xFF)
    c1, s1 = loops.attn_split_q(x, 1, C, fmt)
    y = loops.head_merge_q(c1, s1, T, H, D, 1, C, fmt)
    assert torch.equal(y, x)


@pytest.mark.parametrize("fmt", [INT8, E4M3])
def test_unpack_inverts_pack_on_exact_grid(fmt):
    # receive side at P ranks, simulated: rank r's pack of its token shard,
    # chunk by chunk, laid out as the unpack receives it for head group g
    T, H, D, P, C = 17, 6, 8, 3, 2
    Hp = H // P
    x, _, _ = _grid_rows((T, 3, H, D), fmt, 300 + fmt)
    shard = -(-T // P)
    packs = [loops.qkv_pack_q(x[min(T, r * shard):min(T, (r + 1) * shard)], P, C, fmt)
             for r in range(P)]
    for g in range(P):
        codes, scales = [], []
        for c in range(C):
            for r in range(P):
                n_r = min(T, (r + 1) * shard) - min(T, r * shard)
                q = -(-n_r // C)
                L = max(0, min(n_r, (c + 1) * q) - min(n_r, c * q))
                # rank r's block (c, g): offset of chunk c, then slot g
                c_lo = sum(max(0, min(n_r, (cc + 1) * q) - min(n_r, cc * q))
                           for cc in range(c)) * 3 * H * D
                lo = c_lo + g * 3 * L * Hp * D
                n = 3 * L * Hp * D
                codes.append(packs[r][0][lo:lo + n])
                scales.append(packs[r][1][lo // D:(lo + n) // D])
        outs = loops.qkv_unpack_q(torch.cat(codes), torch.cat(scales), T, H, D, P, C, fmt)
        for s, o in enumerate(outs):
            assert torch.equal(o, x[:, s, g * Hp:(g + 1) * Hp])


# ---------------------------------------------------------------- error bounds

def _random_rows(T, H, D, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, D, generator=g) * torch.exp(torch.randn(T, H, 1, generator=g) * 2)
    return _bf16_bits(x)


def test_int8_error_bound_and_full_scale_code():
    T, H, D = 64, 8, 64
    xb = _random_rows(T, H, D, 21)
    codes, scales = loops.attn_split_q(xb, 1, 1, INT8)
    y = _bits_to_f32(loops.head_merge_q(codes, scales, T, H, D, 1, 1, INT8))
    x = _bits_to_f32(xb).double()
    s = scales.view(T, H, 1).double()
    amax = x.abs().amax(-1, keepdim=True)
    err = (y.double() - x).abs()
    # rounding to nearest: half a step of `scale`, plus float32 and bfloat16
    # rounding of the product (at most 2^-8 of |y|: bfloat16 keeps 8
    # significant bits) and of inv and scale
    bound = 0.5 * s + 2.0 ** -8 * y.double().abs() + 2.0 ** -20 * amax
    assert bool((err <= bound).all())
    assert float((err / s).max()) > 0.45            # the bound is nearly reached
    # the row's largest magnitude takes the full-scale code +-127
    c = codes.view(T, H, D).to(torch.int32)
    arg = x.abs().argmax(-1, keepdim=True)
    assert bool((c.gather(-1, arg).abs() == 127).all())
    assert int(c.abs().max()) == 127
    assert torch.allclose(s.squeeze(-1), (amax / 127).squeeze(-1), rtol=2 ** -23, atol=0)


def test_e4m3_error_bound_and_full_scale_code():
    T, H, D = 64, 8, 64
    xb = _random_rows(T, H, D, 22)
    codes, scales = loops.attn_split_q(xb, 1, 1, E4M3)
    y = _bits_to_f32(loops.head_merge_q(codes, scales, T, H, D, 1, 1, E4M3))
    x = _bits_to_f32(xb).double()
    s = scales.view(T, H, 1).double()
    err = (y.double() - x).abs()
    # three mantissa bits: half a unit in the last place is at most 2^-4 of
    # the magnitude in the normal range, 2^-10 (times scale) below it
    bound = (2.0 ** -4 * x.abs() + 2.0 ** -10 * s) * (1 + 2.0 ** -20) + 2.0 ** -8 * y.double().abs()
    assert bool((err <= bound).all())
    c = codes.view(T, H, D).to(torch.int32)
    arg = x.abs().argmax(-1, keepdim=True)
    assert bool(((c.gather(-1, arg) & 0x7F) == 0x7E).all())
    assert int((c & 0x7F).max()) <= 0x7E


# ---------------------------------------------------------------- degenerate rows

@pytest.mark.parametrize("fmt", [INT8, E4M3])
def test_zero_and_floor_rows_send_zero(fmt):
    rows = torch.tensor([[0.0] * 8, [-0.0] * 8, [1e-30, -2e-30, 0, 0, 0, 0, 0, 3e-31],
                         [2.0 ** -96] + [0.0] * 7])
    x = _bf16_bits(rows).view(4, 1, 8)
    codes, scales = loops.attn_split_q(x, 1, 1, fmt)
    assert scales[:3].tolist() == [0.0, 0.0, 0.0]
    assert codes[:24].to(torch.int32).tolist() == [0] * 24
    # at the floor itself the row is live: its element takes the full-scale code
    assert scales[3].item() > 0
    assert (int(codes[24]) & 0xFF) == (127 if fmt == INT8 else 0x7E)
    y = loops.head_merge_q(codes, scales, 4, 1, 8, 1, 1, fmt)
    assert y[:3].flatten().tolist() == [0] * 24                    # +0 bits


def test_signed_zero_in_a_live_row():
    x = _bf16_bits(torch.tensor([-0.0, 1.0, 0.0, -1.0])).view(1, 1, 4)
    c8, s8 = loops.attn_split_q(x, 1, 1, INT8)
    assert c8.tolist() == [0, 127, 0, -127]
    cf, sf = loops.attn_split_q(x, 1, 1, E4M3)
    assert (cf.to(torch.int32) & 0xFF).tolist() == [0x80, 0x7E, 0x00, 0xFE]
    y = loops.head_merge_q(cf, sf, 1, 1, 4, 1, 1, E4M3)
    assert (y.to(torch.int32) & 0xFFFF).flatten().tolist() == [0x8000, 0x3F80, 0x0000, 0xBF80]


# ---------------------------------------------------------------- non-finite rows
#
# Reading of the variant for values the pages' format cannot carry: a head
# row holding a NaN or an infinity is sent as a lost row (scale = the float32
# quiet NaN 0x7FC00000, every code 0); the receive side writes the bfloat16
# quiet NaN 0x7FC0 into every element of a row whose scale is not finite.

QNAN32, QNAN16 = 0x7FC00000, 0x7FC0
HAND_BITS = [0x3F80, 0xBF00, 0x3E80, 0x0000, 0x3F40, 0xBF80, 0x3E00, 0x3EC0]   # the hand row


def _u32(t: torch.Tensor):
    return [v & 0xFFFFFFFF for v in t.contiguous().view(torch.int32).tolist()]


def _u16(t: torch.Tensor):
    return [v & 0xFFFF for v in t.contiguous().view(torch.int16).flatten().tolist()]


def _as_i16(rows):
    return torch.tensor([[v - 0x10000 if v >= 0x8000 else v for v in r] for r in rows],
                        dtype=torch.int16)


@pytest.mark.parametrize("fmt", [INT8, E4M3])
def test_nonfinite_rows_are_sent_as_lost_rows(fmt):
    rows = [[0x3F80, 0x7FC0, 0x4000, 0, 0, 0, 0, 0],          # 1, quiet NaN, 2
            [0x3F80, 0x7F80, 0x4000, 0, 0, 0, 0, 0],          # +inf beside finite values
            [0xFF80, 0, 0, 0, 0, 0, 0, 0],                    # -inf alone
            [0, 0, 0, 0, 0, 0, 0, 0xFFC1],                    # a negative NaN with payload
            [0x7F81, 0x7F80, 0xFF80, 0x7FC0, 0, 0, 0, 0],     # several kinds at once
            HAND_BITS]                                        # finite: as if it were alone
    x = _as_i16(rows).view(len(rows), 1, 8)
    codes, scales = loops.attn_split_q(x, 1, 1, fmt)
    assert _u32(scales)[:5] == [QNAN32] * 5
    assert [v & 0xFF for v in codes[:40].view(torch.int8).tolist()] == [0] * 40
    hand_c, hand_s = loops.attn_split_q(_as_i16([HAND_BITS]).view(1, 1, 8), 1, 1, fmt)
    assert torch.equal(codes[40:].view(torch.int8), hand_c.view(torch.int8))
    assert _u32(scales[5:]) == _u32(hand_s)
    # the receive side: lost rows arrive as NaN, the finite row unchanged
    y = loops.head_merge_q(codes, scales, len(rows), 1, 8, 1, 1, fmt)
    assert _u16(y)[:40] == [QNAN16] * 40
    assert _u16(y[5:]) == _u16(loops.head_merge_q(hand_c, hand_s, 1, 1, 8, 1, 1, fmt))


@pytest.mark.parametrize("fmt", [INT8, E4M3])
def test_non_finite_scales_dequantise_to_nan_rows(fmt):
    # codes 1, -1, 0, full scale, ... under scales +inf, -inf, a NaN with a
    # payload and the sign set, and 2^127 (finite; its products overflow)
    full = 127 if fmt == INT8 else 0x7E                       # 127 or 448
    one = 1 if fmt == INT8 else 0x38                          # 1.0
    neg_full = (-127) & 0xFF if fmt == INT8 else 0xFE
    c = torch.tensor([one, full, 0, neg_full] * 4, dtype=torch.uint8)
    s = torch.tensor([0x7F800000, 0xFF800000, 0xFFC00001, 0x7F000000],
                     dtype=torch.int64).to(torch.int32).view(torch.float32)
    if fmt == INT8:
        c = c.view(torch.int8)
    y = _u16(loops.head_merge_q(c, s, 4, 1, 4, 1, 1, fmt))
    assert y[:12] == [QNAN16] * 12
    # 1 * 2^127 = 0x7F00 in bfloat16; 127 * 2^127 and 448 * 2^127 overflow
    # float32 and round to +inf (0x7F80); 0 stays +0; the negative full scale
    # goes to -inf (0xFF80)
    assert y[12:] == [0x7F00, 0x7F80, 0x0000, 0xFF80]


def test_e4m3_nan_codes_dequantise_to_nan():
    c = torch.tensor([0x7F, 0xFF, 0x38, 0xB8], dtype=torch.uint8)
    s = torch.tensor([1.0], dtype=torch.float32)
    y = loops.head_merge_q(c, s, 1, 1, 4, 1, 1, E4M3)
    v = y.view(torch.bfloat16).float().flatten()
    assert math.isnan(v[0].item()) and math.isnan(v[1].item())
    assert v[2:].tolist() == [1.0, -1.0]


@pytest.mark.parametrize("fmt", [INT8, E4M3])
def test_lost_rows_leave_the_other_rows_alone(fmt):
    # planting NaN or infinity into some rows changes exactly those rows'
    # codes and scales; every other row is what it was without them
    T, H, D = 24, 5, 16
    xb = _random_rows(T, H, D, 31).clone()
    ref_c, ref_s = loops.attn_split_q(xb, 2, 3, fmt)
    g = torch.Generator().manual_seed(32)
    lost = torch.zeros(T, H, dtype=torch.bool)
    for i in range(12):
        t, h, d = (int(torch.randint(0, n, (1,), generator=g)) for n in (T, H, D))
        xb[t, h, d] = (0x7FC0, 0x7F80, -0x80, -0x3F)[i % 4]    # NaN, +inf, -inf, NaN 0xFFC1
        lost[t, h] = True
    c, s = loops.attn_split_q(xb, 2, 3, fmt)
    # the split's layout of the lost-row mask (as 16-bit ones), one per head row
    mask = loops.attn_split(lost.to(torch.int16).unsqueeze(-1).expand(T, H, D).contiguous(),
                            2, 3)[::D].bool()
    assert int(mask.sum()) == int(lost.sum())
    sb, rb = torch.tensor(_u32(s)), torch.tensor(_u32(ref_s))
    assert bool((sb[mask] == QNAN32).all()) and torch.equal(sb[~mask], rb[~mask])
    cc, rc = c.view(torch.uint8).view(-1, D), ref_c.view(torch.uint8).view(-1, D)
    assert int(cc[mask].sum()) == 0 and torch.equal(cc[~mask], rc[~mask])


def test_bad_format_is_rejected():
    x = _bf16_bits(torch.ones(2, 1, 8))
    with pytest.raises(Exception):
        loops.attn_split_q(x, 1, 1, 3)


# ---------------------------------------------------------------- planted mistakes

def _mutant_split_codes(x_bits, fmt, kind):
    """A restated per-head-row quantiser with one planted mistake (kind), on a
    [T,H,D] bf16 view with P = C = 1 (the split's layout is then the identity).
    Returns (codes as int list, scales as float list)."""
    import numpy as np
    x = _bits_to_f32(x_bits.contiguous()).numpy().astype(np.float32)
    T, H, D = x.shape
    top = np.float32(127.0 if fmt == INT8 else 448.0)
    if kind == "per_token_amax":
        amax = np.abs(x).reshape(T, H * D).max(axis=1).repeat(H).reshape(T, H, 1)
    else:
        amax = np.abs(x).max(axis=2, keepdims=True)
    live = amax >= np.float32(2.0 ** -96) if kind != "no_floor" else amax > 0
    if kind == "scale_128":
        top_q = np.float32(128.0)
    else:
        top_q = top
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = np.where(live, top_q / amax, np.float32(0)).astype(np.float32)
        scale = np.where(live, amax / top, np.float32(0)).astype(np.float32)
    q = (x * inv).astype(np.float32)
    if fmt == INT8:
        if kind == "truncate":
            r = np.trunc(q)
        elif kind == "half_away":
            r = np.sign(q) * np.floor(np.abs(q) + np.float32(0.5))
        else:
            r = np.rint(q)
        c = np.clip(r, -127, 127).astype(np.int64)
        c = np.where(live, c, 0)
        codes = [int(v) for v in c.reshape(-1)]
    else:
        t = torch.from_numpy(q.reshape(-1))
        if kind == "truncate":                  # round toward zero onto the E4M3 grid
            rn = t.clamp(-448, 448).to(torch.float8_e4m3fn).float()
            over = rn.abs() > t.abs()
            # step back one code where rounding went away from zero
            cb = rn.to(torch.float8_e4m3fn).view(torch.uint8).to(torch.int32)
            cb = torch.where(over & (cb & 0x7F > 0), cb - 1, cb)
            cc = cb
        else:
            cc = t.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).to(torch.int32)
        cc = torch.where(torch.from_numpy(np.broadcast_to(live, q.shape).reshape(-1).copy()),
                         cc, torch.zeros_like(cc))
        codes = [int(v) for v in cc]
    return codes, [float(v) for v in scale.reshape(-1)]


def _pin_inputs():
    """The pinned rows: the hand row, the INT8 ties row, exact-grid rows with
    per-row exponents, a below-floor row (as [T,H,D] bf16 bits)."""
    hand = _bf16_bits(torch.tensor([1.0, -0.5, 0.25, 0.0, 0.75, -1.0, 0.125, 0.375])).view(1, 1, 8)
    ties = _bf16_bits(torch.tensor([127.0, 0.5, 1.5, 2.5, -0.5, -2.5, 3.5, 126.5])).view(1, 1, 8)
    floor = _bf16_bits(torch.tensor([1e-30, -2e-30, 0, 0, 0, 0, 0, 3e-31])).view(1, 1, 8)
    return [hand, ties, floor] + [_grid_rows((5, 4, 8), f, 900 + f)[0] for f in (INT8, E4M3)]


# Half-away rounding is planted in the INT8 path only: the restated E4M3
# encoder is PyTorch's conversion, against which the oracle's E4M3 rounding is
# pinned directly above.
MUTANTS = [(f, k) for f in (INT8, E4M3)
           for k in ("truncate", "half_away", "scale_128", "per_token_amax", "no_floor")
           if not (f == E4M3 and k == "half_away")]


@pytest.mark.parametrize("fmt,kind", MUTANTS)
def test_pins_catch_planted_lossy_mistakes(fmt, kind):
    """The unmutated restatement reproduces the oracle on every pinned input;
    each planted mistake changes a code or a scale on at least one of them."""
    caught = False
    for x in _pin_inputs():
        c_ok, s_ok = loops.attn_split_q(x, 1, 1, fmt)
        want = ([int(v) for v in c_ok.tolist()] if fmt == INT8 else
                [int(v) for v in c_ok.view(torch.uint8).tolist()], s_ok.tolist())
        assert _mutant_split_codes(x, fmt, "none") == want
        caught = caught or _mutant_split_codes(x, fmt, kind) != want
    assert caught, kind
