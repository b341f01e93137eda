"""The relayouts inside a captured CUDA graph: the library allocates nothing
and never synchronises, so a whole sequence-head step (pack, split, merge,
unpack, and chunk ranges) can be captured once and replayed; replays read the
inputs' current contents."""
import pytest
import torch

import sequence_head_relayout_gb300 as vf
from oracle import loops
from sequence_head_relayout_gb300 import workloads as W

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("oracle_built")]

DEV = torch.device("cuda:0")


def test_capture_and_replay_step():
    cfg = W.CONFIGS["4k"]
    T, H, D, P, C = cfg.T, cfg.H, cfg.D, cfg.P, cfg.C
    Hp = H // P
    src4, _ = W.pack_source(cfg, device=DEV)
    src3, _ = W.split_source(cfg, device=DEV)
    msrc = W.merge_source(cfg, device=DEV)
    recv = torch.empty(3 * T * Hp * D, dtype=torch.int16, device=DEV)
    W.fill_(recv, "bits", 7)
    packed = torch.empty(3 * T * H * D, dtype=torch.int16, device=DEV)
    split = torch.empty(T * H * D, dtype=torch.int16, device=DEV)
    merged = torch.empty((T, H, D), dtype=torch.int16, device=DEV)
    qkv = tuple(torch.empty((T, Hp, D), dtype=torch.int16, device=DEV) for _ in range(3))
    chunk1 = torch.zeros(3 * T * H * D, dtype=torch.int16, device=DEV)

    def step():
        vf.qkv_pack(src4, P, C, out=packed)
        vf.attn_split(src3, P, C, out=split)
        vf.head_merge(msrc, T, H, D, P, C, out=merged)
        vf.qkv_unpack(recv, T, H, D, P, C, outs=qkv)
        vf.qkv_pack(src4, P, C, out=chunk1, chunks=(1, 1))

    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(side):
        step()                                   # warm-up outside the capture
    torch.cuda.current_stream(DEV).wait_stream(side)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()

    for trial in range(2):
        # new input contents, then replay
        src4.copy_(torch.randint(-(1 << 15), 1 << 15, src4.shape, dtype=torch.int32,
                                 device=DEV).to(torch.int16))
        msrc.random_(-(1 << 15), 1 << 15)
        recv.random_(-(1 << 15), 1 << 15)
        packed.zero_()
        merged.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(packed.cpu(), loops.qkv_pack(src4.cpu(), P, C))
        assert torch.equal(split.cpu(), loops.attn_split(src3.cpu(), P, C))
        assert torch.equal(merged.cpu(), loops.head_merge(msrc.cpu(), T, H, D, P, C))
        for a, b in zip(qkv, loops.qkv_unpack_recv(recv.cpu(), T, H, D, P, C)):
            assert torch.equal(a.cpu(), b)
        tok, length, off = vf.piece_table(vf.OP_QKV_PACK, T, H, D, P, C)
        a = off[1 * P]
        b = off[2 * P]
        assert torch.equal(chunk1[a:b].cpu(), packed[a:b].cpu())


def test_capture_and_replay_lossy_transport():
    """The opt-in INT8 / E4M3 transport in a captured graph: quantising pack
    and split, dequantising unpack and merge of the captured codes."""
    T, H, D, P, C = 1500, 8, 128, 2, 4
    Hp = H // P
    x = torch.empty((T, 3, H, D), dtype=torch.int16, device=DEV)
    a = torch.empty((T, H, D), dtype=torch.int16, device=DEV)
    codes = torch.empty(3 * T * H * D, dtype=torch.int8, device=DEV)
    scales = torch.empty(3 * T * H, dtype=torch.float32, device=DEV)
    fcodes = torch.empty(T * H * D, dtype=torch.float8_e4m3fn, device=DEV)
    fscales = torch.empty(T * H, dtype=torch.float32, device=DEV)
    qkv = tuple(torch.empty((T, Hp, D), dtype=torch.bfloat16, device=DEV) for _ in range(3))
    merged = torch.empty((T, H, D), dtype=torch.bfloat16, device=DEV)
    n_recv = 3 * T * Hp * D

    def step():
        vf.qkv_pack_q(x, P, C, fmt="int8", codes=codes, scales=scales)
        vf.attn_split_q(a, P, C, fmt="e4m3", codes=fcodes, scales=fscales)
        vf.qkv_unpack_q(codes[:n_recv], scales[:n_recv // D], T, H, D, P, C, fmt="int8",
                        outs=qkv)
        vf.head_merge_q(fcodes, fscales, T, H, D, P, C, fmt="e4m3", out=merged)

    W.finite_rows_(x, 1)
    W.finite_rows_(a, 2)
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream(DEV).wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()

    for trial in range(2):
        W.finite_rows_(x, 10 + trial)
        W.finite_rows_(a, 20 + trial)
        g.replay()
        torch.cuda.synchronize()
        wc, ws = loops.qkv_pack_q(x.cpu(), P, C, loops.INT8)
        assert torch.equal(codes.cpu(), wc) and torch.equal(scales.cpu(), ws)
        fc, fs = loops.attn_split_q(a.cpu(), P, C, loops.E4M3)
        assert torch.equal(fcodes.cpu().view(torch.uint8), fc) and torch.equal(fscales.cpu(), fs)
        want = loops.qkv_unpack_q(wc[:n_recv], ws[:n_recv // D], T, H, D, P, C, loops.INT8)
        for o, w in zip(qkv, want):
            assert torch.equal(o.cpu().view(torch.int16), w)
        wm = loops.head_merge_q(fc, fs, T, H, D, P, C, loops.E4M3)
        assert torch.equal(merged.cpu().view(torch.int16), wm)
