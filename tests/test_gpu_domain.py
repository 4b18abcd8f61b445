"""The prefill's numeric domain on the GPU (include/kda.h, "Decay domain" and "Value range").

Inside the domain the results must meet the usual parity bounds against the fp64 oracle,
including decays close to the stated limit (summed |log_alpha| of a channel below about 174
over one 64-token chunk) and large magnitudes.  Outside it the outputs are undefined, but
the call must say so: kda_device_status returns KDA_ERR_RANGE instead of the caller finding
NaNs later.  None of these inputs can fault the GPU: out-of-range arithmetic only produces
inf / NaN values, which the kernel detects.
"""
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


def _prefill(case, la, out_dtype=torch.float32, v=None, s0=None):
    dev = lambda x: None if x is None else x.to(DEV)
    return kda.prefill(dev(case.q), dev(case.k), dev(case.v if v is None else v), dev(la), dev(case.beta),
                       case.cu_seqlens, init_state=dev(case.init_state if s0 is None else s0),
                       ckpt_stride=case.ckpt_stride, out_dtype=out_dtype)


def _parity(case, la, out, fin, ck, v=None, s0=None):
    ro, rf, rc = oracle.prefill(case.q, case.k, case.v if v is None else v, la, case.beta, case.cu_seqlens,
                                case.init_state if s0 is None else s0, ckpt_stride=case.ckpt_stride)
    P.check_out(out, ro, out.dtype)
    P.check_state(fin, rf)
    if ck is not None:
        P.check_state(ck, rc, "checkpoints")


def test_strong_decay_up_to_the_limit():
    """log_alpha = -softplus(N(0,1) + 1) (about 1.3 nats per token, ~85 per chunk), plus
    planted chunks where 16 channels of one head decay by 2.6 nats on every token: 166 nats
    over the chunk, close to the 174-nat limit.  Every token is compared."""
    T, H, D = 8192, 4, 128
    case = workloads.prefill_case([T], H=H, D=D, seed=41, la_shift=1.0, ckpt_stride=2048)
    la = case.log_alpha.clone()
    for c in (5, 77, 127):
        la[64 * c:64 * c + 64, 1, 32:48] = -2.6
    out, fin, ck = _prefill(case, la)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == kda.KDA_OK
    _parity(case, la, out, fin, ck)
    out16, fin16, _ = _prefill(case, la, torch.bfloat16)
    assert kda.kda_device_status() == kda.KDA_OK
    _parity(case, la, out16, fin16, None)


@pytest.mark.parametrize("scale", [100.0, 1000.0])
def test_large_values_and_states(scale):
    """v and the initial states scaled by 100 and 1000 (|v| up to ~4e3, states of the same
    order), which the fp16 operand copies must carry without overflow or loss."""
    T, H, D = 4096, 4, 128
    case = workloads.prefill_case([3000, 1096], H=H, D=D, seed=43, ckpt_stride=1024)
    v = (case.v.float() * scale).to(torch.bfloat16)
    s0 = case.init_state * scale
    out, fin, ck = _prefill(case, case.log_alpha, v=v, s0=s0)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == kda.KDA_OK
    _parity(case, case.log_alpha, out, fin, ck, v=v, s0=s0)


def _ok_after():
    """The context stays usable: a small in-domain prefill afterwards is correct."""
    c = workloads.tiny_case()
    out, fin, _ = kda.prefill(c.q.to(DEV), c.k.to(DEV), c.v.to(DEV), c.log_alpha.to(DEV), c.beta.to(DEV),
                              c.cu_seqlens, out_dtype=torch.float32)
    assert kda.kda_device_status() == kda.KDA_OK
    ro, rf, _ = oracle.prefill(c.q, c.k, c.v, c.log_alpha, c.beta, c.cu_seqlens, None)
    P.check_out(out, ro, torch.float32)
    P.check_state(fin, rf)


def test_decay_beyond_the_limit_is_reported():
    """One channel of one head decays by 3 nats per token over a whole chunk (192 nats):
    beyond the domain, so the call reports KDA_ERR_RANGE."""
    case = workloads.prefill_case([1000, 300], H=4, D=64, seed=44, ckpt_stride=0)
    la = case.log_alpha.clone()
    la[640:704, 2, 7] = -3.0                      # chunk 10 of the first sequence
    _prefill(case, la)
    assert kda.kda_device_status() == kda.KDA_ERR_RANGE
    assert kda.kda_device_status() == kda.KDA_OK  # reading the status clears it
    _ok_after()


def test_values_beyond_fp16_are_reported():
    """v of order 1e5 overflows the fp16 operand copies; the non-finite state this leaves is
    reported as KDA_ERR_RANGE."""
    case = workloads.prefill_case([500], H=4, D=128, seed=45, ckpt_stride=0)
    v = (case.v.float() * 1e5).to(torch.bfloat16)
    _prefill(case, case.log_alpha, v=v)
    assert kda.kda_device_status() == kda.KDA_ERR_RANGE
    _ok_after()
