"""GPU parity of the lineage specialisations of the kernels: Gated DeltaNet (one
log-decay per head and token) and DeltaNet (no decay), for the prefill
(kda_chunk_prefill_ex) and the serving decode (kda_decode_multi).

Each layout is checked against the oracle, which takes the decay broadcast to every
channel (or zero).  The prefill's scalar layouts have arithmetic of their own (the
intra-chunk products in bf16 straight from the staged inputs, the decay applied per
token pair), so they are compared with the oracle, and with the per-channel kernel fed
the broadcast decay only within the parity bounds.  The decode's layouts change where the
decay comes from, not the arithmetic, so they match the per-channel decode bit for bit."""
import pytest
import torch

import oracle
from kimi_delta_attention_06_gb300 import kda, workloads
from tests import _parity as P

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kimi_delta_attention_06_gb300 import build
    build.build()
    oracle.build()


def _head_decay(T, H, seed):
    g = torch.Generator().manual_seed(seed)
    return -torch.nn.functional.softplus(torch.randn(T, H, generator=g) - 2.0)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("decay", [kda.KDA_DECAY_HEAD, kda.KDA_DECAY_NONE])
def test_prefill_layouts(D, decay):
    lens = [1, 63, 200, 64, 130]
    case = workloads.prefill_case(lens, H=4, D=D, seed=80 + D + decay, ckpt_stride=128)
    T, H = case.T, case.H
    if decay == kda.KDA_DECAY_HEAD:
        la_small = _head_decay(T, H, seed=5 + D)
        la_full = la_small[:, :, None].expand(T, H, D).contiguous()
    else:
        la_small = None
        la_full = torch.zeros(T, H, D)
    dev = lambda x: None if x is None else x.to(DEV)
    args = (dev(case.q), dev(case.k), dev(case.v))
    o1, f1, c1 = kda.prefill(*args, dev(la_small), dev(case.beta), case.cu_seqlens, init_state=dev(case.init_state),
                             ckpt_stride=128, out_dtype=torch.float32, decay=decay)
    o0, f0, c0 = kda.prefill(*args, dev(la_full), dev(case.beta), case.cu_seqlens, init_state=dev(case.init_state),
                             ckpt_stride=128, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == kda.KDA_OK
    ro, rf, rc = oracle.prefill(case.q, case.k, case.v, la_full, case.beta, case.cu_seqlens, case.init_state,
                                ckpt_stride=128)
    for o, f, c in ((o1, f1, c1), (o0, f0, c0)):
        P.check_out(o, ro, torch.float32)
        P.check_state(f, rf)
        P.check_state(c, rc)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("decay", [kda.KDA_DECAY_HEAD, kda.KDA_DECAY_NONE])
def test_prefill_layouts_prefix_continuations(D, decay):
    """Sequences that start mid-chunk (prefix continuations) and end mid-chunk: the staged
    q, k tiles then hold neighbouring sequences' tokens, which the scalar layouts' G1 must
    mask out.  Checked against the oracle with start positions."""
    lens = [200, 1, 130, 23, 256, 300]
    start = [0, 40, 63, 1000, 64, 7]
    stride = 128
    case = workloads.prefill_case(lens, H=4, D=D, seed=140 + D + decay, ckpt_stride=stride)
    T, H = case.T, case.H
    if decay == kda.KDA_DECAY_HEAD:
        la_small = _head_decay(T, H, seed=9 + D)
        la_full = la_small[:, :, None].expand(T, H, D).contiguous()
    else:
        la_small, la_full = None, torch.zeros(T, H, D)
    dev = lambda x: None if x is None else x.to(DEV)
    o, f, c = kda.prefill(dev(case.q), dev(case.k), dev(case.v), dev(la_small), dev(case.beta), case.cu_seqlens,
                          init_state=dev(case.init_state), ckpt_stride=stride, out_dtype=torch.float32, decay=decay,
                          start_pos_host=torch.tensor(start, dtype=torch.int32))
    torch.cuda.synchronize()
    assert kda.kda_device_status() == kda.KDA_OK
    ro, rf, rc = oracle.prefill(case.q, case.k, case.v, la_full, case.beta, case.cu_seqlens, case.init_state,
                                ckpt_stride=stride, start_pos=start)
    P.check_out(o, ro, torch.float32)
    P.check_state(f, rf)
    P.check_state(c, rc)


@pytest.mark.parametrize("decay", [kda.KDA_DECAY_HEAD, kda.KDA_DECAY_NONE])
def test_decode_multi_layouts(decay):
    N, K, H, D = 4, 3, 4, 128
    c = workloads.decode_case(N=N, H=H, D=D, steps=K, seed=90 + decay)
    st = lambda key: torch.stack([s[key] for s in c.steps], dim=1).contiguous()
    q, k, v, beta = st("q"), st("k"), st("v"), st("beta")
    if decay == kda.KDA_DECAY_HEAD:
        la_small = -torch.nn.functional.softplus(torch.randn(N, K, H, generator=torch.Generator().manual_seed(3)) - 2)
        la_full = la_small[..., None].expand(N, K, H, D).contiguous()
    else:
        la_small, la_full = None, torch.zeros(N, K, H, D)
    pools = [c.state.clone().to(DEV), c.state.clone().to(DEV)]
    outs = [torch.empty(N, K, H, D, device=DEV) for _ in range(2)]
    for pool, out, la, dk in ((pools[0], outs[0], la_small, decay), (pools[1], outs[1], la_full, kda.KDA_DECAY_CHANNEL)):
        kda.kda_decode_multi(q.to(DEV), k.to(DEV), v.to(DEV), None if la is None else la.to(DEV), beta.to(DEV),
                             pool, N, None, None, 1, out, kda.KDA_OUT_F32, N, K, H, D, D, decay=dk)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == kda.KDA_OK
    assert torch.equal(outs[0], outs[1]) and torch.equal(pools[0], pools[1])
    ref = c.state.double().numpy()
    for j in range(K):
        ro, ref = oracle.decode(q[:, j], k[:, j], v[:, j], la_full[:, j], beta[:, j], ref)
        P.check_out(outs[0][:, j], ro, torch.float32)
    P.check_state(pools[0], ref)


@pytest.mark.parametrize("decay", [kda.KDA_DECAY_HEAD, kda.KDA_DECAY_NONE])
def test_prefill_layouts_32768_sampled_heads(decay):
    """One 32768-token prompt, H=32, D=128, checkpoints every 8192 tokens; the oracle
    replays two heads (outputs on every token, all checkpoints, the end state)."""
    T, H, D, stride = 32768, 32, 128, 8192
    case = workloads.prefill_case([T], H=H, D=D, seed=131 + decay, device=DEV, ckpt_stride=stride)
    la_small = _head_decay(T, H, seed=7).to(DEV) if decay == kda.KDA_DECAY_HEAD else None
    o, f, c = kda.prefill(case.q, case.k, case.v, la_small, case.beta, case.cu_seqlens, init_state=case.init_state,
                          ckpt_stride=stride, out_dtype=torch.bfloat16, decay=decay)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == kda.KDA_OK
    heads = [2, 29]
    la_full = (la_small.cpu()[:, heads, None].expand(T, 2, D) if la_small is not None else torch.zeros(T, 2, D))
    sel = lambda x: x[:, heads].cpu()
    ro, rf, rc = oracle.prefill(sel(case.q), sel(case.k), sel(case.v), la_full.contiguous(), sel(case.beta),
                                case.cu_seqlens, case.init_state[:, heads].cpu(), ckpt_stride=stride)
    P.check_out(o[:, heads], ro, torch.bfloat16)
    P.check_state(f[:, heads], rf)
    P.check_state(c[:, heads], rc)
