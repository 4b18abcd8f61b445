"""kda_chunk_prefill_noalloc against kda_chunk_prefill on the GPU.

The allocation-free entry point runs the same kernel with its hand-off ring in
the library's fixed device array instead of pool memory, so two calls in a row
must reproduce the pool-backed call bit for bit (outputs, final states and
checkpoints).  This file is collected last on purpose.
"""
import pytest
import torch

from kimi_delta_attention_06_gb300 import kda, workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kimi_delta_attention_06_gb300 import build
    build.build()


def _outputs(case, n_ck):
    T, H, D = case.q.shape
    N = case.cu_seqlens.numel() - 1
    return (torch.full((T, H, D), float("nan"), device=DEV, dtype=torch.bfloat16),
            torch.full((N, H, D, D), float("nan"), device=DEV),
            torch.full((n_ck, H, D, D), float("nan"), device=DEV))


def _call(fn, case, dev_in, outs, stride):
    q, k, v, la, beta, s0, cu = dev_in
    T, H, D = case.q.shape
    out, fin, ck = outs
    fn(q, k, v, la, beta, s0, cu, case.cu_seqlens, case.cu_seqlens.numel() - 1, T, H, D, D,
       out, kda.KDA_OUT_BF16, fin, ck, stride)


@pytest.mark.parametrize("lens", [[700, 64, 1130], [700, 64, 1130, 391]],
                         ids=["24_pairs", "32_pairs_full_array"])
def test_noalloc_matches_pool_entry_point_twice(lens):
    """3 or 4 sequences x 8 heads, ragged lengths, nonzero initial states.  The 4-sequence case
    fills every one of the KDA_NOALLOC_MAX_SEQ_HEADS rings, up to the array's end."""
    stride = 256
    case = workloads.prefill_case(lens, H=8, D=128, seed=21, ckpt_stride=stride)
    assert len(lens) * 8 <= kda.KDA_NOALLOC_MAX_SEQ_HEADS
    dev_in = tuple(None if x is None else x.to(DEV) for x in
                   (case.q, case.k, case.v, case.log_alpha, case.beta, case.init_state, case.cu_seqlens))
    n_ck = kda.kda_ckpt_count(case.cu_seqlens, stride)
    ref = _outputs(case, n_ck)
    _call(kda.kda_chunk_prefill, case, dev_in, ref, stride)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == kda.KDA_OK
    assert all(torch.isfinite(t).all() for t in ref)
    for _ in range(2):
        got = _outputs(case, n_ck)
        _call(kda.kda_chunk_prefill_noalloc, case, dev_in, got, stride)
        torch.cuda.synchronize()
        assert kda.kda_device_status() == kda.KDA_OK
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


def test_noalloc_refuses_more_pairs_than_its_scratch():
    case = workloads.prefill_case([128, 128], H=kda.KDA_NOALLOC_MAX_SEQ_HEADS, D=64, seed=2, s0_std=None)
    dev_in = tuple(None if x is None else x.to(DEV) for x in
                   (case.q, case.k, case.v, case.log_alpha, case.beta, case.init_state, case.cu_seqlens))
    outs = _outputs(case, 0)
    with pytest.raises(kda.KdaError) as e:
        _call(kda.kda_chunk_prefill_noalloc, case, dev_in, (outs[0], outs[1], None), 0)
    assert e.value.status == kda.KDA_ERR_UNSUPPORTED
    assert torch.isnan(outs[0].float()).all()          # nothing was launched
