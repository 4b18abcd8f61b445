"""GPU parity of kda_decode_multi (state pool + several tokens per pass) against the
fp64 oracle, which steps each token with its single-token decode."""
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


def _tokens(N, K, H, D, seed):
    """K decode tokens for N sequences, stacked as [N, K, H, ...] (same draws as K decode steps)."""
    c = workloads.decode_case(N=N, H=H, D=D, steps=K, seed=seed)
    st = lambda key: torch.stack([s[key] for s in c.steps], dim=1).contiguous()
    return {key: st(key) for key in ("q", "k", "v", "log_alpha", "beta")}, c.steps


def _oracle_run(steps, state0, ntok):
    """Oracle outputs [N, K, H, D] (NaN where not applied) and the state after ntok[n] tokens."""
    N = state0.shape[0]
    K = len(steps)
    st = state0.double().numpy().copy()
    outs = np.full((N, K) + tuple(steps[0]["v"].shape[1:]), np.nan)
    for j, s in enumerate(steps):
        o, nxt = oracle.decode(s["q"], s["k"], s["v"], s["log_alpha"], s["beta"], st)
        for n in range(N):
            if j < ntok[n]:
                outs[n, j] = o[n]
                st[n] = nxt[n]
    return outs, st


def _call(tok, pool, slots, ntok, commit, out, N, K, H, D):
    kda.kda_decode_multi(tok["q"], tok["k"], tok["v"], tok["log_alpha"], tok["beta"], pool, pool.shape[0],
                         slots, ntok, commit, out,
                         kda.KDA_OUT_F32 if out.dtype == torch.float32 else kda.KDA_OUT_BF16, N, K, H, D, D)


@pytest.mark.parametrize("D", [64, 128])
def test_verify_leaves_pool_untouched_and_matches_oracle(D):
    N, K, H, P_slots = 5, 4, 3, 9
    tok_cpu, steps = _tokens(N, K, H, D, seed=30 + D)
    tok = {k: v.to(DEV) for k, v in tok_cpu.items()}
    g = torch.Generator().manual_seed(7)
    pool0 = torch.randn(P_slots, H, D, D, generator=g) * 0.02
    slots_cpu = torch.tensor([7, 2, 0, 5, 8], dtype=torch.int32)
    pool = pool0.to(DEV)
    out = torch.full((N, K, H, D), float("nan"), device=DEV)
    _call(tok, pool, slots_cpu.to(DEV), None, 0, out, N, K, H, D)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == kda.KDA_OK
    assert torch.equal(pool.cpu(), pool0)                      # verify writes no state
    ro, _ = _oracle_run(steps, pool0[slots_cpu.long()], [K] * N)
    P.check_out(out.cpu().reshape(N * K, H, D), ro.reshape(N * K, H, D), torch.float32)


def test_commit_accepted_prefixes():
    N, K, H, D, P_slots = 6, 4, 4, 128, 8
    tok_cpu, steps = _tokens(N, K, H, D, seed=41)
    tok = {k: v.to(DEV) for k, v in tok_cpu.items()}
    g = torch.Generator().manual_seed(8)
    pool0 = torch.randn(P_slots, H, D, D, generator=g) * 0.02
    slots_cpu = torch.tensor([3, 0, 6, 1, 7, 4], dtype=torch.int32)
    ntok_cpu = torch.tensor([4, 0, 1, 3, 2, 4], dtype=torch.int32)
    pool = pool0.to(DEV)
    out = torch.full((N, K, H, D), float("nan"), device=DEV, dtype=torch.float32)
    _call(tok, pool, slots_cpu.to(DEV), ntok_cpu.to(DEV), 1, out, N, K, H, D)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == kda.KDA_OK
    ro, rs = _oracle_run(steps, pool0[slots_cpu.long()], ntok_cpu.tolist())
    got = out.cpu()
    for n in range(N):
        nt = int(ntok_cpu[n])
        assert torch.isnan(got[n, nt:]).all()                   # tokens past the accepted count: untouched
        if nt:
            P.check_out(got[n, :nt], ro[n, :nt], torch.float32)
    pool_after = pool.cpu()
    for n in range(N):
        sl = int(slots_cpu[n])
        if int(ntok_cpu[n]) == 0:
            assert torch.equal(pool_after[sl], pool0[sl])
        else:
            P.check_state(pool_after[sl][None], rs[n][None])
    for sl in set(range(P_slots)) - set(slots_cpu.tolist()):
        assert torch.equal(pool_after[sl], pool0[sl])            # slots nobody names are untouched


def test_one_token_commit_equals_decode_step():
    N, H, D = 7, 5, 128
    tok_cpu, steps = _tokens(N, 1, H, D, seed=52)
    g = torch.Generator().manual_seed(9)
    s0 = torch.randn(N, H, D, D, generator=g) * 0.02
    a, b = s0.to(DEV), s0.to(DEV)
    o1 = kda.decode_step(*(steps[0][x].to(DEV) for x in ("q", "k", "v", "log_alpha", "beta")), a,
                         out_dtype=torch.float32)
    o2 = torch.empty(N, 1, H, D, device=DEV)
    _call({k: v.to(DEV) for k, v in tok_cpu.items()}, b, None, None, 1, o2, N, 1, H, D)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2[:, 0]) and torch.equal(a, b)


def test_two_calls_equal_one_pass():
    """Committing tokens 0..1 then 2..3 (two calls) equals one 4-token commit."""
    N, K, H, D = 4, 4, 2, 128
    tok_cpu, _ = _tokens(N, K, H, D, seed=63)
    g = torch.Generator().manual_seed(10)
    s0 = torch.randn(N, H, D, D, generator=g) * 0.02
    one, two = s0.to(DEV), s0.to(DEV)
    full = {k: v.to(DEV) for k, v in tok_cpu.items()}
    o_one = torch.empty(N, K, H, D, device=DEV)
    _call(full, one, None, None, 1, o_one, N, K, H, D)
    o_two = torch.empty(N, K, H, D, device=DEV)
    for half in range(2):
        part = {k: v[:, 2 * half:2 * half + 2].contiguous() for k, v in full.items()}
        oo = torch.empty(N, 2, H, D, device=DEV)
        _call(part, two, None, None, 1, oo, N, 2, H, D)
        o_two[:, 2 * half:2 * half + 2] = oo
    torch.cuda.synchronize()
    assert torch.equal(o_one, o_two) and torch.equal(one, two)


def test_bad_slot_is_reported_and_skipped():
    N, K, H, D = 3, 2, 2, 64
    tok_cpu, _ = _tokens(N, K, H, D, seed=70)
    pool = torch.zeros(4, H, D, D, device=DEV)
    slots = torch.tensor([1, 9, 2], dtype=torch.int32, device=DEV)       # 9 is out of range
    out = torch.full((N, K, H, D), float("nan"), device=DEV)
    _call({k: v.to(DEV) for k, v in tok_cpu.items()}, pool, slots, None, 0, out, N, K, H, D)
    assert kda.kda_device_status() == kda.KDA_ERR_INVALID_ARG
    assert torch.isnan(out[1]).all() and not torch.isnan(out[0]).any() and not torch.isnan(out[2]).any()
    assert kda.kda_device_status() == kda.KDA_OK                     # the word was cleared


def test_full_pool_512x32_four_token_commit_sampled():
    """512 sequences x 32 heads x 128 x 128 states (1.07 GB) in a shuffled pool, 4 tokens
    each with mixed accepted counts; the oracle follows 6 sampled sequences (all heads)."""
    N, K, H, D = 512, 4, 32, 128
    c = workloads.decode_case(N=N, H=H, D=D, steps=K, seed=77, device=DEV)
    tok = {key: torch.stack([s[key] for s in c.steps], dim=1).contiguous()
           for key in ("q", "k", "v", "log_alpha", "beta")}
    g = torch.Generator().manual_seed(5)
    slots = torch.randperm(N, generator=g).to(torch.int32)
    ntok = torch.randint(0, K + 1, (N,), generator=g).to(torch.int32)
    pool = c.state                              # [N, H, D, D] on the device; slot s is row s
    sample = [0, 100, 255, 300, 411, 511]
    pool0 = pool[slots[sample].long()].double().cpu().numpy()
    out = torch.full((N, K, H, D), float("nan"), device=DEV)
    _call(tok, pool, slots.to(DEV), ntok.to(DEV), 1, out, N, K, H, D)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == kda.KDA_OK
    steps = [{key: tok[key][sample, j].cpu() for key in tok} for j in range(K)]
    ro, rs = _oracle_run(steps, torch.from_numpy(pool0), ntok[sample].tolist())
    got = out[sample].cpu()
    for i, n in enumerate(sample):
        nt = int(ntok[n])
        if nt:
            P.check_out(got[i, :nt], ro[i, :nt], torch.float32)
        P.check_state(pool[int(slots[n])][None], rs[i][None])
