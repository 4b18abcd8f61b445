"""GPU parity of kda_chunk_prefill against the fp64 oracle (through the C ABI)."""
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


def _run(case, out_dtype=torch.float32, ckpt_stride=None, device_inputs=False):
    stride = case.ckpt_stride if ckpt_stride is None else ckpt_stride
    to = (lambda x: x) if device_inputs else (lambda x: None if x is None else x.to(DEV))
    return kda.prefill(to(case.q), to(case.k), to(case.v), to(case.log_alpha), to(case.beta),
                       case.cu_seqlens, init_state=to(case.init_state), ckpt_stride=stride,
                       out_dtype=out_dtype)


def _oracle(case, heads=None, ckpt_stride=None, seqs=None):
    """Oracle on a subset of heads (and optionally sequences); inputs copied to the host."""
    stride = case.ckpt_stride if ckpt_stride is None else ckpt_stride
    hs = slice(None) if heads is None else list(heads)
    cu = case.cu_seqlens
    if seqs is None:
        sel = lambda x: x[:, hs].cpu()
        s0 = None if case.init_state is None else case.init_state[:, hs].cpu()
        return oracle.prefill(sel(case.q), sel(case.k), sel(case.v), sel(case.log_alpha), sel(case.beta),
                              cu, s0, ckpt_stride=stride)
    raise NotImplementedError


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_tiny_case(out_dtype):
    """B=1, H=2, T=256, D=64, zero initial state (the case the oracle finishes instantly)."""
    c = workloads.tiny_case()
    out, fin, _ = _run(c, out_dtype)
    ro, rf, _ = _oracle(c)
    P.check_out(out, ro, out_dtype)
    P.check_state(fin, rf)
    assert kda.kda_device_status() == 0


@pytest.mark.parametrize("D", [64, 128])
def test_ragged_varlen_with_checkpoints(D):
    """Lengths around the chunk size (1, 63, 64, 65, 127, 200, 0, 130): partial chunks,
    empty and length-1 sequences, nonzero initial states, checkpoints every 64 tokens."""
    lens = [1, 63, 64, 65, 127, 200, 0, 130]
    c = workloads.prefill_case(lens, H=3, D=D, seed=11, la_shift=-1.0, s0_std=0.05, ckpt_stride=64)
    for od in (torch.float32, torch.bfloat16):
        out, fin, ck = _run(c, od)
        ro, rf, rc = _oracle(c)
        P.check_out(out, ro, od)
        P.check_state(fin, rf, "final")
        P.check_state(ck, rc, "checkpoints")
    # the empty sequence hands back its initial state unchanged
    torch.testing.assert_close(fin[6].cpu(), c.init_state[6], rtol=0, atol=0)


def test_value_blocks_are_independent_bitwise():
    """Dv=128 runs as two 64-column blocks; each block equals a Dv=64 run on its columns."""
    c = workloads.prefill_case([300, 77], H=2, D=128, seed=12, ckpt_stride=64)
    out, fin, ck = _run(c)
    for jb in range(2):
        sl = slice(64 * jb, 64 * jb + 64)
        o2, f2, c2 = kda.prefill(c.q.to(DEV), c.k.to(DEV), c.v[..., sl].contiguous().to(DEV),
                                 c.log_alpha.to(DEV), c.beta.to(DEV), c.cu_seqlens,
                                 init_state=c.init_state[..., sl].contiguous().to(DEV), ckpt_stride=64,
                                 out_dtype=torch.float32)
        assert torch.equal(o2, out[..., sl])
        assert torch.equal(f2, fin[..., sl])
        assert torch.equal(c2, ck[..., sl])


def test_deterministic_and_resume_from_checkpoint():
    c = workloads.prefill_case([640], H=2, D=128, seed=13, ckpt_stride=256)
    out, fin, ck = _run(c)
    out2, fin2, _ = _run(c)
    assert torch.equal(out, out2) and torch.equal(fin, fin2)
    # resume at token 256 from the first checkpoint: identical chunk grid => identical bits
    cut = 256
    c2 = workloads.PrefillCase("tail", c.q[cut:].contiguous(), c.k[cut:].contiguous(), c.v[cut:].contiguous(),
                               c.log_alpha[cut:].contiguous(), c.beta[cut:].contiguous(), ck[0:1].cpu(),
                               torch.tensor([0, 640 - cut], dtype=torch.int32), 0)
    out3, fin3, _ = _run(c2)
    assert torch.equal(out3, out[cut:])
    assert torch.equal(fin3, fin)


def test_decode_steps_equal_prefill():
    """n decode steps from a state == prefill of the same n tokens from that state."""
    n, H, D = 40, 4, 128
    c = workloads.prefill_case([n], H=H, D=D, seed=14)
    out, fin, _ = _run(c)
    state = c.init_state.to(DEV).clone()
    for t in range(n):
        sl = slice(t, t + 1)
        o = kda.decode_step(c.q[sl].to(DEV), c.k[sl].to(DEV), c.v[sl].to(DEV), c.log_alpha[sl].to(DEV),
                            c.beta[sl].to(DEV), state, out_dtype=torch.float32)
        P.check_out(o[0], out[t], torch.float32, what=f"token {t}")
    P.check_state(state, fin)


def test_single_sequence_8192_sampled_heads():
    """B=1, T=8192, H=32, D=128 (bf16 output); oracle on three sampled heads, every token."""
    c = workloads.single_case(8192, seed=1, device=DEV)
    out, fin, _ = _run(c, torch.bfloat16, device_inputs=True)
    heads = [0, 17, 31]
    ro, rf, _ = _oracle(c, heads)
    P.check_out(out[:, heads], ro, torch.bfloat16)
    P.check_state(fin[:, heads], rf)
    # fp32 output mode on the same inputs meets the strict bound
    out32, _, _ = _run(c, torch.float32, device_inputs=True)
    P.check_out(out32[:, heads], ro, torch.float32)


def test_long_prompt_145408_checkpoints_sampled_head():
    """T=145408 (about 142k), H=32, D=128, checkpoints every 32768 tokens + the end (5 per head).
    The oracle replays one head over the whole prompt; that head's outputs are compared on
    every token (all 64 rows of every chunk), together with all five checkpoints, in the
    bf16 output mode the bench times and, under the strict bound, in the fp32 output mode."""
    c = workloads.single_case(145408, seed=2, device=DEV, ckpt_stride=32768)
    out, fin, ck = _run(c, torch.bfloat16, device_inputs=True)
    assert ck.shape[0] == 5
    heads = [5]
    ro, rf, rc = _oracle(c, heads)
    P.check_out(out[:, heads], ro, torch.bfloat16)
    P.check_state(fin[:, heads], rf)
    P.check_state(ck[:, heads], rc)
    torch.testing.assert_close(ck[4], fin[0], rtol=0, atol=0)
    del out
    out32, fin32, _ = _run(c, torch.float32, device_inputs=True)
    P.check_out(out32[:, heads], ro, torch.float32)
    assert torch.equal(fin32, fin)          # the output dtype changes only the final store
    assert kda.kda_device_status() == 0


def test_varlen_16_sequences_sampled():
    """16 packed sequences, log-uniform lengths in [1k, 64k] (~280k tokens), half with an
    initial state, checkpoints every 32768 tokens; oracle on two heads of all sequences,
    compared on every token, in the bf16 and (strict bound) fp32 output modes."""
    c = workloads.varlen_case(device=DEV)
    out, fin, ck = _run(c, torch.bfloat16, device_inputs=True)
    heads = [3, 30]
    ro, rf, rc = _oracle(c, heads)
    P.check_out(out[:, heads], ro, torch.bfloat16)
    P.check_state(fin[:, heads], rf)
    P.check_state(ck[:, heads], rc)
    del out
    out32, _, _ = _run(c, torch.float32, device_inputs=True)
    P.check_out(out32[:, heads], ro, torch.float32)
    assert kda.kda_device_status() == 0
