"""GPU parity of kda_chunk_prefill_segmented (one prompt, its chunks split into segments
that run side by side) against the fp64 oracle, through the C ABI.

The segmented call must give the one-sequence prefill's results: every output row, the
final state and the prompt's own checkpoints (not the extra segment ends), with the chunk
grid and checkpoint grid placed by the prompt's absolute start position.  Cases cover
3, 5 and 8 segments, start positions on and off the 64-token grid (off it, the run that
forms the transitions starts with a short leading sequence), all three decay layouts,
head dims 64 and 128, both output dtypes, the fused output norm, the fallbacks to one
plain prefill, the empty prompt, and the full 145408-token prompt at 4 heads (one GPU's
share of 32 heads split over 8)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import prep as oprep
from kimi_delta_attention_06_gb300 import kda, workloads
from tests import _parity as P

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kimi_delta_attention_06_gb300 import build
    build.build()
    oracle.build()


def _la(c, decay):
    return {kda.KDA_DECAY_CHANNEL: c.log_alpha, kda.KDA_DECAY_HEAD: c.log_alpha[:, :, 0].contiguous(),
            kda.KDA_DECAY_NONE: None}[decay]


def _oracle_la(c, decay):
    """The decay the oracle sees for a layout: per channel, the head's value on every
    channel, or zero."""
    if decay == kda.KDA_DECAY_CHANNEL:
        return c.log_alpha.cpu()
    if decay == kda.KDA_DECAY_HEAD:
        return c.log_alpha[:, :, :1].expand_as(c.log_alpha).cpu()
    return torch.zeros_like(c.log_alpha).cpu()


def _seg(c, decay, segments, start_pos, out_dtype, gamma=None):
    return kda.prefill(c.q, c.k, c.v, _la(c, decay), c.beta, c.cu_seqlens, init_state=c.init_state,
                       ckpt_stride=c.ckpt_stride, out_dtype=out_dtype, decay=decay,
                       start_pos_host=torch.tensor([start_pos], dtype=torch.int32), segments=segments,
                       norm_gamma=gamma)


def _ref(c, decay, start_pos):
    return oracle.prefill(c.q.cpu(), c.k.cpu(), c.v.cpu(), _oracle_la(c, decay), c.beta.cpu(), c.cu_seqlens,
                          None if c.init_state is None else c.init_state.cpu(), ckpt_stride=c.ckpt_stride,
                          start_pos=[start_pos])


@pytest.mark.parametrize("segments,start_pos", [(3, 0), (5, 37), (8, 128), (8, 4133)])
@pytest.mark.parametrize("decay", [kda.KDA_DECAY_CHANNEL, kda.KDA_DECAY_HEAD, kda.KDA_DECAY_NONE])
def test_segmented_matches_oracle(segments, start_pos, decay):
    c = workloads.prefill_case([5000], H=4, D=128, seed=31, device=DEV, la_shift=-1.0, s0_std=0.05,
                               ckpt_stride=1024)
    ro, rf, rc = _ref(c, decay, start_pos)
    for od in (torch.float32, torch.bfloat16):
        out, fin, ck = _seg(c, decay, segments, start_pos, od)
        assert ck.shape[0] == rc.shape[0] == kda.kda_ckpt_count_ex(
            c.cu_seqlens, torch.tensor([start_pos], dtype=torch.int32), c.ckpt_stride)
        P.check_out(out, ro, od)
        P.check_state(fin, rf)
        P.check_state(ck, rc, "checkpoints")
    assert kda.kda_device_status() == 0


def test_segmented_head_dim_64_no_initial_state():
    c = workloads.prefill_case([3000], H=8, D=64, seed=32, device=DEV, la_shift=0.0, s0_std=None, ckpt_stride=512)
    ro, rf, rc = _ref(c, kda.KDA_DECAY_CHANNEL, 0)
    out, fin, ck = _seg(c, kda.KDA_DECAY_CHANNEL, 6, 0, torch.float32)
    P.check_out(out, ro, torch.float32)
    P.check_state(fin, rf)
    P.check_state(ck, rc, "checkpoints")
    assert kda.kda_device_status() == 0


def test_segmented_agrees_with_the_plain_prefill():
    """Same prompt, plain one-sequence call against 4 and 7 segments: the states agree to the
    state tolerance and the outputs to the output tolerance."""
    c = workloads.prefill_case([20000], H=4, D=128, seed=33, device=DEV, ckpt_stride=4096)
    sp = torch.tensor([64], dtype=torch.int32)
    o0, f0, k0 = kda.prefill(c.q, c.k, c.v, c.log_alpha, c.beta, c.cu_seqlens, init_state=c.init_state,
                             ckpt_stride=c.ckpt_stride, out_dtype=torch.float32, start_pos_host=sp)
    for segments in (4, 7):
        o, f, k = _seg(c, kda.KDA_DECAY_CHANNEL, segments, 64, torch.float32)
        P.check_out(o, o0, torch.float32)
        P.check_state(f, f0)
        P.check_state(k, k0)
    assert kda.kda_device_status() == 0


def test_segmented_fused_output_norm():
    c = workloads.prefill_case([4000], H=4, D=128, seed=34, device=DEV, ckpt_stride=0)
    g = torch.Generator(device=DEV).manual_seed(35)
    gamma = torch.rand(4, 128, generator=g, device=DEV) + 0.5
    ro, _, _ = _ref(c, kda.KDA_DECAY_CHANNEL, 0)
    y_ref = oprep.output_norm(ro, gamma.cpu().double().numpy(), 1e-6)
    y, _, _ = _seg(c, kda.KDA_DECAY_CHANNEL, 5, 0, torch.float32, gamma=gamma)
    d = (y.double().cpu().numpy() - y_ref)
    assert np.abs(d).max() <= 3e-2 * np.sqrt((y_ref ** 2).mean())
    assert kda.kda_device_status() == 0


@pytest.mark.parametrize("segments,T", [(1, 3000), (2, 3000), (8, 100), (8, 120)])
def test_segmented_falls_back_to_one_plain_prefill(segments, T):
    """Fewer than 3 segments (asked for, or a prompt of under 3 chunks): one plain launch,
    bit-identical to the one-sequence kda_chunk_prefill_ex."""
    c = workloads.prefill_case([T], H=4, D=128, seed=36, device=DEV, ckpt_stride=128)
    sp = torch.tensor([5], dtype=torch.int32)
    o0, f0, k0 = kda.prefill(c.q, c.k, c.v, c.log_alpha, c.beta, c.cu_seqlens, init_state=c.init_state,
                             ckpt_stride=c.ckpt_stride, out_dtype=torch.float32, start_pos_host=sp)
    o, f, k = _seg(c, kda.KDA_DECAY_CHANNEL, segments, 5, torch.float32)
    assert torch.equal(o, o0) and torch.equal(f, f0) and torch.equal(k, k0)


def test_segmented_empty_prompt_returns_the_initial_state():
    c = workloads.prefill_case([0], H=4, D=128, seed=37, device=DEV, ckpt_stride=64)
    out, fin, ck = _seg(c, kda.KDA_DECAY_CHANNEL, 8, 0, torch.float32)
    assert out.numel() == 0 and ck.shape[0] == 0
    assert torch.equal(fin, c.init_state)


def test_segmented_long_prompt_4_heads_every_row():
    """The 145408-token prompt at 4 heads (32 heads split over 8 GPUs), 8 segments,
    checkpoints every 32768 tokens: every output row, the final state and the five
    checkpoints against the oracle, in the bf16 mode and under the strict fp32 bound."""
    c = workloads.single_case(145408, seed=2, device=DEV, ckpt_stride=32768)
    c = workloads.head_slice(c, 12, 16)
    ro, rf, rc = _ref(c, kda.KDA_DECAY_CHANNEL, 0)
    out, fin, ck = _seg(c, kda.KDA_DECAY_CHANNEL, 8, 0, torch.bfloat16)
    assert ck.shape[0] == 5
    P.check_out(out, ro, torch.bfloat16)
    P.check_state(fin, rf)
    P.check_state(ck, rc, "checkpoints")
    del out
    out32, fin32, _ = _seg(c, kda.KDA_DECAY_CHANNEL, 8, 0, torch.float32)
    P.check_out(out32, ro, torch.float32)
    assert torch.equal(fin32, fin)
    assert kda.kda_device_status() == 0


def test_segmented_skips_only_transitions_that_cannot_matter():
    """Heads 0 and 1 decay strongly (their transition over a segment is far below fp32
    rounding, so it is not formed), heads 2 and 3 weakly (it is formed and applied): every
    head must match the oracle, and a prompt whose decays are all weak must match too."""
    c = workloads.prefill_case([6000], H=4, D=128, seed=38, device=DEV, la_shift=-1.0, s0_std=0.05,
                               ckpt_stride=1024)
    # log-decays in [-0.15, -0.05] per token and channel on heads 0-1 (a 1000-token segment
    # decays by at least e^-50), in [-0.002, 0] on heads 2-3; both well inside the prefill's
    # per-chunk domain
    g = torch.Generator(device=DEV).manual_seed(40)
    u = torch.rand(c.log_alpha.shape, generator=g, device=DEV)
    strong, weak = -0.05 - 0.1 * u, -0.002 * u
    c.log_alpha = torch.where(torch.arange(4, device=DEV).view(1, 4, 1) < 2, strong, weak).contiguous()
    for start_pos in (0, 77):
        ro, rf, rc = _ref(c, kda.KDA_DECAY_CHANNEL, start_pos)
        out, fin, ck = _seg(c, kda.KDA_DECAY_CHANNEL, 6, start_pos, torch.float32)
        P.check_out(out, ro, torch.float32)
        P.check_state(fin, rf)
        P.check_state(ck, rc, "checkpoints")
    weak = workloads.prefill_case([6000], H=4, D=128, seed=39, device=DEV, la_shift=-8.0, s0_std=0.05,
                                  ckpt_stride=0)
    ro, rf, _ = _ref(weak, kda.KDA_DECAY_CHANNEL, 0)
    out, fin, _ = _seg(weak, kda.KDA_DECAY_CHANNEL, 6, 0, torch.float32)
    P.check_out(out, ro, torch.float32)
    P.check_state(fin, rf)
    assert kda.kda_device_status() == 0


@pytest.mark.parametrize("decay", [kda.KDA_DECAY_CHANNEL, kda.KDA_DECAY_HEAD])
def test_segmented_varlen_matches_oracle(decay):
    """kda_chunk_prefill_segmented_ex over seven sequences: split ones (3, 4 and 5 segments)
    beside whole ones, an empty one, initial states on every other sequence, start positions
    on and off the chunk grid, checkpoints every 512 tokens.  Per-channel decay forms every
    transition here; per-head decay has them dropped by the bound."""
    lens = [3000, 200, 5000, 64, 0, 1500, 7000]
    sp = [0, 10, 4133, 0, 7, 64, 99]
    c = workloads.prefill_case(lens, H=4, D=128, seed=41, device=DEV, la_shift=-1.0, s0_std=0.05,
                               s0_every_other=True, ckpt_stride=512)
    ro, rf, rc = oracle.prefill(c.q.cpu(), c.k.cpu(), c.v.cpu(), _oracle_la(c, decay), c.beta.cpu(), c.cu_seqlens,
                                c.init_state.cpu(), ckpt_stride=512, start_pos=sp)
    spt = torch.tensor(sp, dtype=torch.int32)
    for od in (torch.float32, torch.bfloat16):
        out, fin, ck = kda.prefill(c.q, c.k, c.v, _la(c, decay), c.beta, c.cu_seqlens, init_state=c.init_state,
                                   ckpt_stride=512, out_dtype=od, decay=decay, start_pos_host=spt, segments=12)
        assert ck.shape[0] == rc.shape[0]
        P.check_out(out, ro, od)
        P.check_state(fin, rf)
        P.check_state(ck, rc, "checkpoints")
    assert kda.kda_device_status() == 0


def test_segmented_varlen_plain_when_nothing_splits():
    """More than 32 sequences, or sequences too short to split: one plain prefill, bit for bit
    the kda_chunk_prefill_ex result."""
    c = workloads.prefill_case([100] * 40, H=4, D=128, seed=42, device=DEV, ckpt_stride=64)
    o0, f0, k0 = kda.prefill(c.q, c.k, c.v, c.log_alpha, c.beta, c.cu_seqlens, init_state=c.init_state,
                             ckpt_stride=64, out_dtype=torch.float32,
                             start_pos_host=torch.zeros(40, dtype=torch.int32))
    o, f, k = kda.prefill(c.q, c.k, c.v, c.log_alpha, c.beta, c.cu_seqlens, init_state=c.init_state,
                          ckpt_stride=64, out_dtype=torch.float32, start_pos_host=torch.zeros(40, dtype=torch.int32),
                          segments=16)
    assert torch.equal(o, o0) and torch.equal(f, f0) and torch.equal(k, k0)
