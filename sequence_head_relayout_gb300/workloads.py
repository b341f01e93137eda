"""Seeded synthetic workloads for the three relayouts.

This module builds inputs only: shapes, strides, allocations and seeded bit
patterns.  It holds none of the relayouts' arithmetic (no chunk, shard or
destination offset is computed here), so the tests may feed the same tensors
to the CUDA library and to the CPU oracle.

The named configurations follow the shapes of the pages' measurements
("Sol-Engine alignment on SM86 and SM89", section "What is enabled": the
representative 55,413-token Base16 shape, whose allocation-screen byte counts
fix T*H = 55,414*28 at D = 128 and BF16) plus a tiny, a 4k, a ragged and a
large case.  The pages measured on private video requests; these seeded
tensors stand in for those activations at the stated shapes.

All tensors hold 16-bit elements as ``torch.int16`` bit patterns; bf16 values
are produced by rounding seeded N(0,1) float32 draws to bf16 and viewing the
result as int16.
"""
from dataclasses import dataclass

import torch

# Bit patterns planted into random payloads: -0, a quiet NaN, a negative NaN
# with payload, a signalling-NaN payload, +inf and the smallest denormal.
SPECIAL_BITS = (0x8000, 0x7FC0, 0xFFC1, 0x7F81, 0x7F80, 0x0001)
# Fill value for source padding that a relayout must never read.  A NaN
# payload that rounding N(0,1) draws to bf16 can never produce.
PAD_SENTINEL = 0x7FA5


def _as_i16(v: int) -> int:
    return v - 0x10000 if v >= 0x8000 else v


@dataclass(frozen=True)
class Config:
    """One workload.

    pack_src:  "contiguous"  -- [T,3,H,D] allocation;
               "padded_rows" -- [T, 3*H*D + pad] allocation, first 3*H*D
                                columns viewed as [T,3,H,D];
               "head_major"  -- [T,H,3,D] allocation viewed as [T,3,H,D].
    split_src: "contiguous"  -- [T,H,D];  "bhtd" -- [H,T,D] allocation viewed
               as [T,H,D] (an attention output in head-major layout).
    merge_dst: "contiguous"  -- [T,H,D];  "head_major" -- [H,T,D] allocation
               viewed as [T,H,D].
    payload:   "normal" (bf16 of N(0,1)), "bits" (uniform 16-bit patterns with
               the special patterns planted), "iota" (logical element i holds
               i mod 2**16).
    """
    name: str
    T: int
    H: int
    D: int
    P: int
    C: int
    pack_src: str = "contiguous"
    split_src: str = "contiguous"
    merge_dst: str = "contiguous"
    payload: str = "normal"
    seed: int = 0
    pad: int = 0


CONFIGS = {
    "tiny": Config("tiny", T=64, H=4, D=16, P=2, C=1, payload="bits", seed=1),
    "4k": Config("4k", T=4096, H=32, D=128, P=2, C=4, payload="normal", seed=2),
    "pages": Config("pages", T=55414, H=28, D=128, P=2, C=4, pack_src="padded_rows",
                    split_src="bhtd", payload="normal", seed=3, pad=64),
    "ragged": Config("ragged", T=55413, H=32, D=64, P=4, C=4, pack_src="head_major",
                     split_src="bhtd", merge_dst="head_major", payload="bits", seed=4),
    "large": Config("large", T=200000, H=32, D=128, P=8, C=4, payload="normal", seed=5),
}

_FILL_CHUNK = 1 << 26


def fill_(buf: torch.Tensor, payload: str, seed: int) -> torch.Tensor:
    """Fill a flat int16 tensor in place with a seeded payload."""
    assert buf.dtype == torch.int16 and buf.dim() == 1
    n = buf.numel()
    g = torch.Generator(device=buf.device)
    g.manual_seed(seed)
    for a in range(0, n, _FILL_CHUNK):
        b = min(n, a + _FILL_CHUNK)
        if payload == "iota":
            v = torch.arange(a, b, device=buf.device, dtype=torch.int64).remainder_(1 << 16)
            buf[a:b].copy_(torch.where(v >= (1 << 15), v - (1 << 16), v).to(torch.int16))
        elif payload == "bits":
            buf[a:b].copy_(torch.randint(-(1 << 15), 1 << 15, (b - a,), generator=g,
                                         device=buf.device, dtype=torch.int32).to(torch.int16))
        elif payload == "normal":
            x = torch.randn(b - a, generator=g, device=buf.device, dtype=torch.float32)
            buf[a:b].copy_(x.to(torch.bfloat16).view(torch.int16))
        else:
            raise ValueError(payload)
    if payload == "bits" and n:
        step = max(1, n // 97)
        idx = torch.arange(0, n, step, device=buf.device)[:len(SPECIAL_BITS) * 16]
        vals = torch.tensor([_as_i16(SPECIAL_BITS[i % len(SPECIAL_BITS)])
                             for i in range(idx.numel())], dtype=torch.int16, device=buf.device)
        buf[idx] = vals
        buf[-1] = _as_i16(SPECIAL_BITS[0])
    return buf


def _fill_view(view: torch.Tensor, payload: str, seed: int) -> None:
    """Fill the logical elements of a view (row-major logical order)."""
    flat = torch.empty(view.numel(), dtype=torch.int16, device=view.device)
    fill_(flat, payload, seed)
    view.copy_(flat.view(view.shape))


def pack_source(cfg: Config, device="cpu", payload: str = None, seed: int = None):
    """Return (view [T,3,H,D] int16, backing allocation)."""
    payload = payload or cfg.payload
    seed = cfg.seed if seed is None else seed
    T, H, D = cfg.T, cfg.H, cfg.D
    if cfg.pack_src == "contiguous":
        base = torch.empty(T * 3 * H * D, dtype=torch.int16, device=device)
        view = base.view(T, 3, H, D)
    elif cfg.pack_src == "padded_rows":
        base = torch.empty(T * (3 * H * D + cfg.pad), dtype=torch.int16, device=device)
        base.fill_(_as_i16(PAD_SENTINEL))
        view = base.view(T, 3 * H * D + cfg.pad)[:, :3 * H * D].unflatten(1, (3, H, D))
    elif cfg.pack_src == "head_major":
        base = torch.empty(T * H * 3 * D, dtype=torch.int16, device=device)
        view = base.view(T, H, 3, D).permute(0, 2, 1, 3)
    else:
        raise ValueError(cfg.pack_src)
    if cfg.pack_src == "padded_rows" or payload == "iota":
        _fill_view(view, payload, seed)
    else:
        fill_(base, payload, seed)
    return view, base


def split_source(cfg: Config, device="cpu", payload: str = None, seed: int = None):
    """Return (view [T,H,D] int16, backing allocation)."""
    payload = payload or cfg.payload
    seed = (cfg.seed if seed is None else seed) + 1000
    T, H, D = cfg.T, cfg.H, cfg.D
    base = torch.empty(T * H * D, dtype=torch.int16, device=device)
    if cfg.split_src == "contiguous":
        view = base.view(T, H, D)
    elif cfg.split_src == "bhtd":
        view = base.view(H, T, D).permute(1, 0, 2)
    else:
        raise ValueError(cfg.split_src)
    if payload == "iota":
        _fill_view(view, payload, seed)
    else:
        fill_(base, payload, seed)
    return view, base


def merge_source(cfg: Config, device="cpu", payload: str = None, seed: int = None):
    """Return the flat received (packed) storage of T*H*D elements."""
    payload = payload or cfg.payload
    seed = (cfg.seed if seed is None else seed) + 2000
    base = torch.empty(cfg.T * cfg.H * cfg.D, dtype=torch.int16, device=device)
    return fill_(base, payload, seed)


def merge_destination(cfg: Config, device="cpu", fill: int = None):
    """Return (view [T,H,D] int16, backing allocation) for the merge output."""
    T, H, D = cfg.T, cfg.H, cfg.D
    base = torch.empty(T * H * D, dtype=torch.int16, device=device)
    if fill is not None:
        base.fill_(_as_i16(fill))
    if cfg.merge_dst == "contiguous":
        view = base.view(T, H, D)
    elif cfg.merge_dst == "head_major":
        view = base.view(H, T, D).permute(1, 0, 2)
    else:
        raise ValueError(cfg.merge_dst)
    return view, base


def finite_rows_(view: torch.Tensor, seed: int) -> torch.Tensor:
    """Fill a 16-bit view [..., D] in place with finite bf16 rows for the
    lossy transport: each D-element row is N(0,1) draws times 2^k, k a seeded
    integer in [-24, 24] (rows of very different magnitude), with planted
    rows: all +0, all -0 and +0 mixed, a row scaled by 2^-100 (below the
    quantiser's 2^-96 floor), a row whose largest magnitude is exactly 2^-96,
    and rows mixing bf16 denormals with normal values."""
    D = view.shape[-1]
    rows = view.numel() // D if D else 0
    if rows == 0:
        return view
    g = torch.Generator(device=view.device)
    g.manual_seed(seed)
    x = torch.randn((rows, D), generator=g, device=view.device, dtype=torch.float32)
    k = torch.randint(-24, 25, (rows, 1), generator=g, device=view.device)
    x = x * torch.pow(2.0, k.to(torch.float32))
    step = max(1, rows // 53)
    for j, r in enumerate(range(0, rows, step)):
        kind = j % 5
        if kind == 0:
            x[r] = 0.0
        elif kind == 1:
            x[r] = torch.where(torch.arange(D, device=view.device) % 2 == 0, -0.0, 0.0)
        elif kind == 2:
            x[r] = x[r] / x[r].abs().max().clamp_min(1e-30) * 2.0 ** -100
        elif kind == 3:
            x[r] = x[r] / x[r].abs().max().clamp_min(1e-30) * 2.0 ** -97
            x[r, 0] = 2.0 ** -96
        else:
            x[r, ::3] = 2.0 ** -130                       # bf16 denormal
    view.copy_(x.to(torch.bfloat16).view(torch.int16).view(view.shape))
    return view


# Non-finite 16-bit patterns planted by plant_non_finite_: a quiet NaN, +inf,
# -inf, a negative NaN with payload, a signalling-NaN payload.
NON_FINITE_BITS = (0x7FC0, 0x7F80, 0xFF80, 0xFFC1, 0x7F81)


def plant_non_finite_(view: torch.Tensor, seed: int, every: int = 97) -> torch.Tensor:
    """Overwrite one element in every `every`-th D-element row of a 16-bit view
    [..., D] (rows in logical order, starting at a seeded row) with a
    non-finite pattern (NON_FINITE_BITS in turn), at a seeded position in the
    row.  Returns the view."""
    D = view.shape[-1]
    rows = view.numel() // D if D else 0
    if rows == 0:
        return view
    g = torch.Generator()
    g.manual_seed(seed)
    first = int(torch.randint(0, min(every, rows), (1,), generator=g))
    idx = torch.arange(first, rows, every)
    pos = torch.randint(0, D, (idx.numel(),), generator=g)
    vals = torch.tensor([_as_i16(NON_FINITE_BITS[i % len(NON_FINITE_BITS)])
                         for i in range(idx.numel())], dtype=torch.int16)
    flat = view.reshape(rows, D) if view.is_contiguous() else None
    if flat is not None:
        flat[idx.to(view.device), pos.to(view.device)] = vals.to(view.device)
    else:
        lead = view.shape[:-1]
        coords = torch.unravel_index(idx, lead)
        view[tuple(c.to(view.device) for c in coords) + (pos.to(view.device),)] = \
            vals.to(view.device)
    return view
