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
