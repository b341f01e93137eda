"""The bench's PyTorch materialisation chains (the pages' "reference" arm of
the A/B/A comparison) compute the same relayouts as the oracle, on CPU."""
import pytest
import torch

import bench
from oracle import loops
from sequence_head_relayout_gb300 import workloads as W

pytestmark = pytest.mark.usefixtures("oracle_built", "lib_built")


@pytest.mark.parametrize("name", ["tiny", "4k"])
def test_torch_chain_equals_oracle(name):
    cfg = W.CONFIGS[name]
    ch = bench.TorchChain(cfg)
    src, _ = W.pack_source(cfg)
    s3, _ = W.split_source(cfg)
    m = W.merge_source(cfg)
    assert torch.equal(ch.qkv_pack(src), loops.qkv_pack(src, cfg.P, cfg.C))
    assert torch.equal(ch.attn_split(s3), loops.attn_split(s3, cfg.P, cfg.C))
    assert torch.equal(ch.head_merge(m),
                       loops.head_merge(m, cfg.T, cfg.H, cfg.D, cfg.P, cfg.C))
