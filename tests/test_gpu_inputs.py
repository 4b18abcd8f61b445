"""GPU parity of kda_prepare_inputs and kda_output_norm against the fp64 reference in
oracle/prep.py, and of the whole module path (prepare -> prefill -> output norm) against
the oracle recurrence fed the reference's prepared inputs."""
import numpy as np
import pytest
import torch

import oracle
from oracle import prep
from kimi_delta_attention_06_gb300 import kda, workloads
from tests import _parity as P

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF16_REL = 2.0 ** -8          # one bf16 rounding of the stored result


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kimi_delta_attention_06_gb300 import build
    build.build()
    oracle.build()


def _raw(lens, H, D, seed, with_state):
    g = torch.Generator().manual_seed(seed)
    T = sum(lens)
    xq, xk, xv = (torch.randn(T, H, D, generator=g).to(torch.bfloat16) for _ in range(3))
    w = (torch.randn(3, H, D, 4, generator=g) * 0.5).float()
    a = (torch.randn(T, H, D, generator=g) - 2.0).float()
    b = torch.randn(T, H, generator=g).to(torch.bfloat16)
    cs = torch.randn(len(lens), 3, 3, H, D, generator=g).to(torch.bfloat16) if with_state else None
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens), 0).to(torch.int32)
    return xq, xk, xv, w, a, b, cs, cu


def _gpu_prepare(xq, xk, xv, w, a, b, cs, cu, act):
    T, H, D = xq.shape
    N = cu.numel() - 1
    outs = [torch.empty(T, H, D, device=DEV, dtype=torch.bfloat16) for _ in range(3)]
    la = torch.empty(T, H, D, device=DEV)
    beta = torch.empty(T, H, device=DEV, dtype=torch.bfloat16)
    d = lambda x: None if x is None else x.to(DEV)
    kda.kda_prepare_inputs(d(xq), d(xk), d(xv), d(w), d(cs), d(a), d(b), d(cu), cu, N, T, H, D, act,
                           outs[0], outs[1], outs[2], la, beta)
    return outs[0], outs[1], outs[2], la, beta


def _close_bf16(got, ref, what, scale=None):
    g = got.float().cpu().double().numpy()
    err = np.abs(g - ref)
    bound = BF16_REL * np.abs(ref) + 1e-6 * (np.abs(ref).max() if scale is None else scale)
    assert (err <= bound).all(), f"{what}: max excess {(err - bound).max():.3e}"


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("act", [0, 1])
@pytest.mark.parametrize("with_state", [False, True])
def test_prepare_inputs_against_reference(D, act, with_state):
    lens = [1, 2, 3, 40, 0, 97, 33]                 # sequences shorter than the conv window, empty, ragged
    xq, xk, xv, w, a, b, cs, cu = _raw(lens, 3, D, seed=D + 2 * act + int(with_state), with_state=with_state)
    q, k, v, la, beta = _gpu_prepare(xq, xk, xv, w, a, b, cs, cu, act)
    torch.cuda.synchronize()
    rq, rk, rv, rla, rb = prep.prepare_inputs(xq, xk, xv, w, a, b, cu, conv_state=cs, act=act)
    # q, k are unit vectors; fp32 conv + norm, then one bf16 rounding (plus fp32 rounding slack)
    for got, ref, nm in ((q, rq, "q"), (k, rk, "k")):
        err = np.abs(got.float().cpu().double().numpy() - ref)
        assert (err <= BF16_REL * np.abs(ref) + 2e-5).all(), nm
    _close_bf16(v, rv, "v")
    np.testing.assert_allclose(la.cpu().double().numpy(), rla, rtol=2e-6, atol=1e-7)
    _close_bf16(beta, rb, "beta", scale=1.0)


def test_prepare_inputs_boundaries_at_every_group_offset():
    """16 sequences whose starts fall at every offset inside the 16-token groups a warp
    takes (so groups mix whole-window and boundary tokens), several 64-token tiles each,
    D = 128 with SiLU and carried-in conv state."""
    lens = [16 * (i % 5 + 2) + 1 for i in range(16)]  # 33 .. 97 tokens, each 1 mod 16: starts at offsets 0..15
    xq, xk, xv, w, a, b, cs, cu = _raw(lens, 2, 128, seed=77, with_state=True)
    q, k, v, la, beta = _gpu_prepare(xq, xk, xv, w, a, b, cs, cu, 1)
    torch.cuda.synchronize()
    rq, rk, rv, rla, rb = prep.prepare_inputs(xq, xk, xv, w, a, b, cu, conv_state=cs, act=1)
    starts = cu[:-1].numpy() % 16
    assert sorted(set(starts.tolist())) == list(range(16))
    for got, ref, nm in ((q, rq, "q"), (k, rk, "k")):
        err = np.abs(got.float().cpu().double().numpy() - ref)
        assert (err <= BF16_REL * np.abs(ref) + 2e-5).all(), nm
    _close_bf16(v, rv, "v")
    np.testing.assert_allclose(la.cpu().double().numpy(), rla, rtol=2e-6, atol=1e-7)
    _close_bf16(beta, rb, "beta", scale=1.0)


@pytest.mark.parametrize("o_f32", [False, True])
def test_output_norm_against_reference(o_f32):
    g = torch.Generator().manual_seed(5)
    T, H, D = 77, 4, 128
    o = torch.randn(T, H, D, generator=g) * 3.0
    o = o if o_f32 else o.to(torch.bfloat16)
    gamma = torch.rand(H, D, generator=g) + 0.5
    y = torch.empty(T, H, D, device=DEV, dtype=torch.bfloat16)
    kda.kda_output_norm(o.to(DEV), kda.KDA_OUT_F32 if o_f32 else kda.KDA_OUT_BF16, gamma.to(DEV), 1e-6, y, T, H, D)
    torch.cuda.synchronize()
    _close_bf16(y, prep.output_norm(o, gamma, eps=1e-6), "y", scale=1.0)


def test_module_path_prepare_prefill_norm():
    """prepare -> prefill -> output norm on the GPU, against the same three steps in fp64."""
    lens = [300, 1, 129]
    H, D = 4, 128
    xq, xk, xv, w, a, b, cs, cu = _raw(lens, H, D, seed=9, with_state=False)
    q, k, v, la, beta = _gpu_prepare(xq, xk, xv, w, a, b, None, cu, 1)
    o, fin, _ = kda.prefill(q, k, v, la, beta, cu, out_dtype=torch.float32)
    gamma = (torch.rand(H, D, generator=torch.Generator().manual_seed(1)) + 0.5)
    y = torch.empty_like(o, dtype=torch.bfloat16)
    kda.kda_output_norm(o, kda.KDA_OUT_F32, gamma.to(DEV), 1e-6, y, o.shape[0], H, D)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == kda.KDA_OK
    # the oracle recurrence on exactly the inputs the GPU prefill consumed (its bf16 prep output)
    ro, rf, _ = oracle.prefill(q.cpu(), k.cpu(), v.cpu(), la.cpu(), beta.cpu(), cu)
    P.check_out(o, ro, torch.float32)
    P.check_state(fin, rf)
    yr = prep.output_norm(ro, gamma, eps=1e-6)
    rel = np.abs(y.float().cpu().double().numpy() - yr).max() / np.sqrt((yr ** 2).mean())
    assert rel < 3e-2


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("D", [64, 128])
def test_prefill_with_fused_output_norm(out_dtype, D):
    """The per-head output norm fused into the prefill's output epilogue, against the fp64
    recurrence followed by the fp64 norm, on ragged sequences (full chunks leave through
    the TMA store, partial ones through plain stores) and a prefix continuation."""
    lens = [300, 1, 129, 64]
    H = 4
    case = workloads.prefill_case(lens, H=H, D=D, seed=30 + D, ckpt_stride=0)
    gamma = torch.rand(H, D, generator=torch.Generator().manual_seed(3)) + 0.5
    start = torch.tensor([0, 5, 100, 64], dtype=torch.int32)
    dev = lambda x: None if x is None else x.to(DEV)
    y, fin, _ = kda.prefill(dev(case.q), dev(case.k), dev(case.v), dev(case.log_alpha), dev(case.beta),
                            case.cu_seqlens, init_state=dev(case.init_state), out_dtype=out_dtype,
                            start_pos_host=start, norm_gamma=gamma.to(DEV), norm_eps=1e-6)
    o, fin2, _ = kda.prefill(dev(case.q), dev(case.k), dev(case.v), dev(case.log_alpha), dev(case.beta),
                             case.cu_seqlens, init_state=dev(case.init_state), out_dtype=torch.float32,
                             start_pos_host=start)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == kda.KDA_OK
    assert torch.equal(fin, fin2)                        # the norm touches only the output
    ro, rf, _ = oracle.prefill(case.q, case.k, case.v, case.log_alpha, case.beta, case.cu_seqlens,
                               case.init_state, start_pos=start.tolist())
    P.check_state(fin, rf)
    yr = prep.output_norm(ro, gamma, eps=1e-6)
    yg = y.float().cpu().double().numpy()
    rel = np.abs(yg - yr).max() / np.sqrt((yr ** 2).mean())
    assert rel < 3e-2, rel
    # the separate norm pass applied to the fp32 output gives the same up to its bf16 rounding
    # (half an ulp, 2^-8 |y|, on each side) and the rsqrt's few ulps
    ys = torch.empty(o.shape, device=DEV, dtype=torch.bfloat16)
    kda.kda_output_norm(o, kda.KDA_OUT_F32, gamma.to(DEV), 1e-6, ys, o.shape[0], H, D)
    torch.cuda.synchronize()
    yf, ysf = y.float(), ys.float()
    rms = ysf.pow(2).mean().sqrt()
    assert ((yf - ysf).abs() <= 2.0 ** -7 * ysf.abs() + 1e-3 * rms).all()
