"""A head split of one problem over ranks, as `bench.py --split heads` runs it, computes
exactly what one launch over all heads computes: KDA heads are independent recurrences,
so each rank's launch over its own head range must reproduce that range of the full
launch bit for bit (prefill outputs, final states and checkpoints; decode outputs and
states).  One GPU runs every rank's share in turn."""
import pytest
import torch

import bench
from kimi_delta_attention_06_gb300 import kda, workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kimi_delta_attention_06_gb300 import build
    build.build()


def _prefill(c, out_dtype):
    return kda.prefill(c.q, c.k, c.v, c.log_alpha, c.beta, c.cu_seqlens, init_state=c.init_state,
                       ckpt_stride=c.ckpt_stride, out_dtype=out_dtype)


@pytest.mark.parametrize("world", [2, 4])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_prefill_head_split_matches_the_full_launch(world, out_dtype):
    # ragged sequences with initial states and checkpoints, 8 heads of 128
    full = workloads.prefill_case([700, 333, 64, 1], H=8, D=128, seed=21, device=DEV, ckpt_stride=256)
    out, fin, ck = _prefill(full, out_dtype)
    for rank in range(world):
        h0, h1 = bench.head_range(full.H, world, rank)
        o_r, f_r, c_r = _prefill(workloads.head_slice(full, h0, h1), out_dtype)
        assert torch.equal(o_r, out[:, h0:h1])
        assert torch.equal(f_r, fin[:, h0:h1])
        assert torch.equal(c_r, ck[:, h0:h1])
    assert kda.kda_device_status() == 0


def test_decode_head_split_matches_the_full_launch():
    dc = workloads.decode_case(N=96, H=8, D=128, steps=2, seed=22, device=DEV)
    parts = [workloads.head_slice(dc, *bench.head_range(8, 2, r)) for r in range(2)]
    state = dc.state.clone()
    for i, st in enumerate(dc.steps):
        out = kda.decode_step(st["q"], st["k"], st["v"], st["log_alpha"], st["beta"], state)
        for r, p in enumerate(parts):
            h0, h1 = bench.head_range(8, 2, r)
            s = p.steps[i]
            o_r = kda.decode_step(s["q"], s["k"], s["v"], s["log_alpha"], s["beta"], p.state)
            assert torch.equal(o_r, out[:, h0:h1])
            assert torch.equal(p.state, state[:, h0:h1])
    assert kda.kda_device_status() == 0


def test_segmented_head_split_matches_the_full_launch():
    """A head-split rank that runs the segmented prefill (as `bench.py --split heads` does when
    a rank holds few heads) gives its heads of the full plain launch within the parity
    tolerances (not bit for bit: the segment start states are formed through the segment
    transitions and offsets)."""
    from tests import _parity as P
    full = workloads.prefill_case([20000], H=8, D=128, seed=23, device=DEV, ckpt_stride=4096)
    out, fin, ck = kda.prefill(full.q, full.k, full.v, full.log_alpha, full.beta, full.cu_seqlens,
                               init_state=full.init_state, ckpt_stride=4096, out_dtype=torch.float32)
    for rank in range(2):
        h0, h1 = bench.head_range(8, 2, rank)
        c = workloads.head_slice(full, h0, h1)
        o_r, f_r, c_r = kda.prefill(c.q, c.k, c.v, c.log_alpha, c.beta, c.cu_seqlens, init_state=c.init_state,
                                    ckpt_stride=4096, out_dtype=torch.float32, segments=8)
        P.check_out(o_r, out[:, h0:h1], torch.float32)
        P.check_state(f_r, fin[:, h0:h1])
        P.check_state(c_r, ck[:, h0:h1])
    assert kda.kda_device_status() == 0
