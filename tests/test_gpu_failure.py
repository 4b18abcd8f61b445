"""Failure detection on the GPU without a fault: a bounded device-side wait that
nothing satisfies expires, the kernel records KDA_ERR_TIMEOUT and returns, the
host reads it through kda_device_status, and the context stays usable."""
import pytest
import torch

import oracle
from kimi_delta_attention_06_gb300 import kda, workloads
from tests import _parity as P

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_context_survives():
    from kimi_delta_attention_06_gb300 import build
    build.build()
    assert kda.kda_device_status() == kda.KDA_OK
    kda.kda_debug_expire_wait(2_000_000)               # 2 ms bound on a wait nothing completes
    assert kda.kda_device_status() == kda.KDA_ERR_TIMEOUT
    assert kda.kda_device_status() == kda.KDA_OK       # reading clears the word
    # the context is intact: a normal prefill still runs and matches the oracle
    c = workloads.prefill_case([130], H=2, D=64, seed=21, ckpt_stride=64)
    out, fin, ck = kda.prefill(c.q.cuda(), c.k.cuda(), c.v.cuda(), c.log_alpha.cuda(), c.beta.cuda(),
                               c.cu_seqlens, init_state=c.init_state.cuda(), ckpt_stride=64,
                               out_dtype=torch.float32)
    assert kda.kda_device_status() == kda.KDA_OK
    ro, rf, rc = oracle.prefill(c.q, c.k, c.v, c.log_alpha, c.beta, c.cu_seqlens, c.init_state, ckpt_stride=64)
    P.check_out(out, ro, torch.float32)
    P.check_state(fin, rf)
