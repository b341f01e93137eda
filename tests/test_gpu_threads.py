"""Concurrent calls: the library keeps no global state, so several host
threads may enqueue relayouts on their own streams at once (the ctypes calls
release the interpreter lock, so the C calls really overlap)."""
import threading

import pytest
import torch

import sequence_head_relayout_gb300 as vf
from oracle import loops

pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("oracle_built")]

DEV = torch.device("cuda:0")


def test_threads_on_separate_streams():
    shapes = [(1001 + 37 * i, 8, 64, (2, 4, 8)[i % 3], 1 + i % 4) for i in range(8)]
    jobs = []
    for i, (T, H, D, P, C) in enumerate(shapes):
        g = torch.Generator().manual_seed(i)
        x = torch.randint(-(1 << 15), 1 << 15, (T, 3, H, D), generator=g,
                          dtype=torch.int32).to(torch.int16)
        jobs.append((x, x.to(DEV), P, C))
    torch.cuda.synchronize()              # inputs are ready before any thread's stream reads
    results = [None] * len(jobs)
    errors = []

    def work(i):
        try:
            x, xd, P, C = jobs[i]
            s = torch.cuda.Stream(DEV)
            with torch.cuda.stream(s):
                outs = [vf.qkv_pack(xd, P, C) for _ in range(20)]
                results[i] = outs[-1]
            s.synchronize()
        except Exception as e:            # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for (x, _, P, C), got in zip(jobs, results):
        assert torch.equal(got.cpu(), loops.qkv_pack(x, P, C))


def test_lossy_threads_on_separate_streams():
    """The same for the opt-in lossy transport: concurrent quantising packs
    (INT8) and splits (E4M3) from eight host threads."""
    from sequence_head_relayout_gb300 import workloads as W
    shapes = [(777 + 53 * i, 8, 128, (2, 4, 8)[i % 3], 1 + i % 4) for i in range(8)]
    jobs = []
    for i, (T, H, D, P, C) in enumerate(shapes):
        x4 = W.finite_rows_(torch.empty((T, 3, H, D), dtype=torch.int16), 100 + i)
        x3 = W.finite_rows_(torch.empty((T, H, D), dtype=torch.int16), 200 + i)
        jobs.append((x4, x3, x4.to(DEV), x3.to(DEV), P, C))
    torch.cuda.synchronize()
    results = [None] * len(jobs)
    errors = []

    def work(i):
        try:
            _, _, x4d, x3d, P, C = jobs[i]
            s = torch.cuda.Stream(DEV)
            with torch.cuda.stream(s):
                for _ in range(10):
                    packed = vf.qkv_pack_q(x4d, P, C, fmt="int8")
                    split = vf.attn_split_q(x3d, P, C, fmt="e4m3")
                results[i] = (packed, split)
            s.synchronize()
        except Exception as e:            # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for (x4, x3, _, _, P, C), ((pc, ps), (sc, ss)) in zip(jobs, results):
        wc, ws = loops.qkv_pack_q(x4, P, C, loops.INT8)
        assert torch.equal(pc.cpu(), wc) and torch.equal(ps.cpu(), ws)
        wc, ws = loops.attn_split_q(x3, P, C, loops.E4M3)
        assert torch.equal(sc.cpu().view(torch.uint8), wc) and torch.equal(ss.cpu(), ws)
