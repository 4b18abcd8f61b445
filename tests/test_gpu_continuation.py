"""GPU parity of prefix continuations: kda_chunk_prefill_ex with start
positions, whose chunk grid and checkpoints sit on each prompt's absolute grid."""
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


def _dev(x):
    return None if x is None else x.to(DEV)


def _run(case, start_pos, stride, out_dtype=torch.float32):
    return kda.prefill(_dev(case.q), _dev(case.k), _dev(case.v), _dev(case.log_alpha), _dev(case.beta),
                       case.cu_seqlens, init_state=_dev(case.init_state), ckpt_stride=stride, out_dtype=out_dtype,
                       start_pos_host=None if start_pos is None else torch.tensor(start_pos, dtype=torch.int32))


def test_zero_start_positions_equal_the_plain_entry_point():
    case = workloads.prefill_case([300, 64, 1], H=4, D=128, seed=101, ckpt_stride=128)
    a = _run(case, [0, 0, 0], 128)
    b = _run(case, None, 128)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("D", [64, 128])
def test_start_positions_against_oracle(D):
    # offsets 0 (mod 64), 40, 63, 1, 0 and 7; lengths chosen to end mid-chunk, on a chunk
    # end, exactly on a checkpoint, and inside the first partial chunk
    lens = [200, 1, 130, 23, 256, 300]
    start = [0, 40, 63, 1000, 64, 7]
    stride = 128
    case = workloads.prefill_case(lens, H=4, D=D, seed=110 + D, ckpt_stride=stride)
    o, f, c = _run(case, start, stride)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == kda.KDA_OK
    ro, rf, rc = oracle.prefill(case.q, case.k, case.v, case.log_alpha, case.beta, case.cu_seqlens,
                                case.init_state, ckpt_stride=stride, start_pos=start)
    assert c.shape[0] == rc.shape[0] == oracle.ckpt_count(case.cu_seqlens, stride, start)
    P.check_out(o, ro, torch.float32)
    P.check_state(f, rf)
    P.check_state(c, rc)


def test_continuation_matches_one_call():
    """A 1000-token prompt in one call, and the same prompt as a 333-token prefix plus a
    continuation from the prefix's end state: same outputs and end state (to rounding), and
    the continuation's checkpoints are the one-call checkpoints after token 333."""
    T, P_len, stride = 1000, 333, 128
    case = workloads.prefill_case([T], H=4, D=128, seed=120, ckpt_stride=stride)
    o_all, f_all, c_all = _run(case, None, stride)
    pre = workloads.PrefillCase("pre", case.q[:P_len], case.k[:P_len], case.v[:P_len], case.log_alpha[:P_len],
                                case.beta[:P_len], case.init_state, torch.tensor([0, P_len], dtype=torch.int32), stride)
    o_a, f_a, c_a = _run(pre, None, stride)
    cont = workloads.PrefillCase("cont", case.q[P_len:], case.k[P_len:], case.v[P_len:], case.log_alpha[P_len:],
                                 case.beta[P_len:], f_a.cpu(), torch.tensor([0, T - P_len], dtype=torch.int32), stride)
    o_b, f_b, c_b = _run(cont, [P_len], stride)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == kda.KDA_OK
    # one call: 128, 256, ..., 896 and the end (8 slots); prefix: 128, 256, end 333; continuation:
    # 384, ..., 896 and the end 1000 (6 slots)
    assert c_all.shape[0] == 8 and c_a.shape[0] == 3 and c_b.shape[0] == 6
    P.check_out(torch.cat([o_a, o_b]), o_all.cpu().double().numpy(), torch.float32)
    P.check_state(f_b, f_all.cpu().double().numpy())
    P.check_state(c_b, c_all[2:].cpu().double().numpy())
    P.check_state(c_a[:2], c_all[:2].cpu().double().numpy())


def test_continuation_70000_tokens_sampled_head():
    """A 70000-token prompt served as a 40000-token prefix and a 30000-token continuation
    (start position 40000, checkpoints every 32768 absolute tokens): H=32, D=128, one head
    replayed by the oracle over the whole prompt; the continuation's checkpoints sit at
    absolute 65536 and its end, equal to the one-call states there."""
    T, P_len, H, D, stride = 70000, 40000, 32, 128, 32768
    case = workloads.prefill_case([T], H=H, D=D, seed=140, device=DEV, ckpt_stride=stride)
    cu_p = torch.tensor([0, P_len], dtype=torch.int32)
    cu_c = torch.tensor([0, T - P_len], dtype=torch.int32)
    _, f_a, c_a = kda.prefill(case.q[:P_len], case.k[:P_len], case.v[:P_len], case.log_alpha[:P_len],
                              case.beta[:P_len], cu_p, init_state=case.init_state, ckpt_stride=stride)
    o_b, f_b, c_b = kda.prefill(case.q[P_len:], case.k[P_len:], case.v[P_len:], case.log_alpha[P_len:],
                                case.beta[P_len:], cu_c, init_state=f_a, ckpt_stride=stride,
                                start_pos_host=torch.tensor([P_len], dtype=torch.int32))
    torch.cuda.synchronize()
    assert kda.kda_device_status() == kda.KDA_OK
    assert c_a.shape[0] == 2 and c_b.shape[0] == 2          # prefix: 32768, end 40000; continuation: 65536, end
    heads = [11]
    sel = lambda x: x[:, heads].cpu()
    ro, rf, rc = oracle.prefill(sel(case.q), sel(case.k), sel(case.v), sel(case.log_alpha), sel(case.beta),
                                torch.tensor([0, T], dtype=torch.int32), case.init_state[:, heads].cpu(),
                                ckpt_stride=stride)
    # one-call checkpoints: 32768, 65536, end 70000
    assert rc.shape[0] == 3
    rows = np.arange(0, T - P_len, 300)
    P.check_out(o_b[rows][:, heads], ro[P_len + rows], torch.bfloat16)
    P.check_state(c_b[:, heads], rc[1:])
    P.check_state(f_b[:, heads], rf)
