"""GPU parity of kda_decode_step against the fp64 oracle (through the C ABI)."""
import numpy as np
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


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_decode_small_multi_step(D, out_dtype):
    c = workloads.decode_case(N=6, H=3, D=D, steps=5, seed=2 + D)
    state = c.state.to(DEV)
    ref = c.state.double().numpy()
    for s in c.steps:
        o = kda.decode_step(s["q"].to(DEV), s["k"].to(DEV), s["v"].to(DEV), s["log_alpha"].to(DEV),
                            s["beta"].to(DEV), state, out_dtype=out_dtype)
        ro, ref = oracle.decode(s["q"], s["k"], s["v"], s["log_alpha"], s["beta"], ref)
        P.check_out(o, ro, out_dtype)
        P.check_state(state, ref)
    assert kda.kda_device_status() == 0


def test_decode_zero_beta_is_pure_decay():
    """beta = 0: the state only decays, S <- Diag(alpha) S, exactly per row."""
    c = workloads.decode_case(N=2, H=2, D=128, steps=1, seed=9)
    s = c.steps[0]
    state = c.state.to(DEV)
    zero = torch.zeros_like(s["beta"])
    kda.decode_step(s["q"].to(DEV), s["k"].to(DEV), s["v"].to(DEV), s["log_alpha"].to(DEV),
                    zero.to(DEV), state, out_dtype=torch.float32)
    expect = c.state.double() * torch.exp(s["log_alpha"].double())[..., None]
    P.check_state(state, expect)


def test_decode_full_config_64_steps():
    """512 sequences x 32 heads x 128 x 128 fp32 states (1.07 GB) in place, 64 steps.
    The oracle follows 8 sampled sequences (all heads) through all 64 steps; after
    step 1 every (sequence, head) checksum is compared against the oracle."""
    N, H, D, steps = 512, 32, 128, 64
    g = torch.Generator(device=DEV).manual_seed(4)
    state = torch.randn(N, H, D, D, generator=g, device=DEV) * 0.02
    sample = [0, 77, 128, 255, 300, 411, 500, 511]
    ref = state[sample].double().cpu().numpy()
    full0 = state.double().cpu().numpy()
    cs = workloads.decode_case(N=N, H=H, D=D, steps=steps, seed=5, device=DEV)
    for i, s in enumerate(cs.steps):
        o = kda.decode_step(s["q"], s["k"], s["v"], s["log_alpha"], s["beta"], state, out_dtype=torch.bfloat16)
        sub = {k: v[sample].cpu() for k, v in s.items()}
        ro, ref = oracle.decode(sub["q"], sub["k"], sub["v"], sub["log_alpha"], sub["beta"], ref)
        P.check_out(o[sample], ro, torch.bfloat16, what=f"step {i} o")
        if i == 0:
            full_o, full_ref = oracle.decode(s["q"].cpu(), s["k"].cpu(), s["v"].cpu(), s["log_alpha"].cpu(),
                                             s["beta"].cpu(), full0)
            got = state.double().cpu().numpy()
            # per-(sequence, head) checksums: sum and Frobenius norm
            np.testing.assert_allclose(got.sum(axis=(2, 3)), full_ref.sum(axis=(2, 3)), rtol=1e-3, atol=1e-3)
            np.testing.assert_allclose(np.linalg.norm(got, axis=(2, 3)), np.linalg.norm(full_ref, axis=(2, 3)),
                                       rtol=1e-4)
            P.check_state(got, full_ref, what="step 1 full state")
            del full0, full_ref, got
    P.check_state(state[sample], ref, what="step 64 sampled states")
    assert kda.kda_device_status() == 0
