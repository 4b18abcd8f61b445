"""Host-only checks of the C ABI: the library builds, loads and exports every
entry point declared in include/kda.h, and invalid calls are rejected on the
host before anything touches a GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest
import torch

from kimi_delta_attention_06_gb300 import build as kbuild
from kimi_delta_attention_06_gb300 import kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kda.load()


def _declared_functions():
    names = set()
    for hdr in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if hdr.endswith(".h"):
            src = open(os.path.join(ROOT, "include", hdr)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names.update(re.findall(r"\b(kda_\w+)\s*\(", src))
    return sorted(names)


def test_header_declares_expected_entry_points():
    names = _declared_functions()
    for n in ["kda_chunk_prefill", "kda_chunk_prefill_noalloc", "kda_decode_step", "kda_decode_multi", "kda_ckpt_count",
              "kda_chunk_prefill_ex", "kda_ckpt_count_ex", "kda_prepare_inputs", "kda_output_norm",
              "kda_device_status", "kda_status_string", "kda_chunk_size", "kda_debug_expire_wait",
              "kda_chunk_prefill_segmented"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_status_strings_and_chunk_size(lib):
    assert kda.kda_status_string(0) == "ok"
    assert "invalid" in kda.kda_status_string(-1)
    assert "timed out" in kda.kda_status_string(-4)
    assert "numeric domain" in kda.kda_status_string(-5)
    assert kda.KDA_ERR_RANGE == -5
    assert kda.kda_chunk_size() == 64


def test_ckpt_count_matches_policy(lib):
    cu = torch.tensor([0, 145408], dtype=torch.int32)
    assert kda.kda_ckpt_count(cu, 32768) == 5          # 4 interior + the sequence end
    cu = torch.tensor([0, 32768, 32768, 32769], dtype=torch.int32)
    assert kda.kda_ckpt_count(cu, 32768) == 2          # exact multiple: 1; empty: 0; length 1: 1
    assert kda.kda_ckpt_count(cu, 0) == 0
    with pytest.raises(kda.KdaError):
        kda.kda_ckpt_count(torch.tensor([0, 5, 3], dtype=torch.int32), 64)


def _prefill_raw(lib, fn="kda_chunk_prefill", **over):
    """Call a prefill entry point with fake (never dereferenced) aligned pointers."""
    cu = (ctypes.c_int32 * 3)(0, 64, 100)
    a = dict(q=0x1000, k=0x2000, v=0x3000, la=0x4000, beta=0x5000, s0=None, cu=0x6000,
             cu_host=ctypes.cast(cu, ctypes.c_void_p), N=2, T=100, H=2, Dk=64, Dv=64,
             out=0x7000, out_dtype=0, fin=None, ck=None, stride=0, stream=None)
    a.update(over)
    return getattr(lib, fn)(a["q"], a["k"], a["v"], a["la"], a["beta"], a["s0"], a["cu"],
                                 a["cu_host"], a["N"], a["T"], a["H"], a["Dk"], a["Dv"], a["out"],
                                 a["out_dtype"], a["fin"], a["ck"], a["stride"], a["stream"])


def test_prefill_rejects_bad_arguments_on_host(lib):
    bad = ctypes.c_int32 * 3
    assert _prefill_raw(lib, q=None) == kda.KDA_ERR_INVALID_ARG
    assert _prefill_raw(lib, Dk=96) == kda.KDA_ERR_UNSUPPORTED
    assert _prefill_raw(lib, Dv=32) == kda.KDA_ERR_UNSUPPORTED
    assert _prefill_raw(lib, T=99) == kda.KDA_ERR_INVALID_ARG
    assert _prefill_raw(lib, stride=100) == kda.KDA_ERR_INVALID_ARG
    assert _prefill_raw(lib, stride=-64) == kda.KDA_ERR_INVALID_ARG
    assert _prefill_raw(lib, ck=0x8000, stride=0) == kda.KDA_ERR_INVALID_ARG
    assert _prefill_raw(lib, out_dtype=7) == kda.KDA_ERR_INVALID_ARG
    assert _prefill_raw(lib, q=0x1008) == kda.KDA_ERR_INVALID_ARG        # misaligned
    dec = bad(0, 70, 60)
    assert _prefill_raw(lib, cu_host=ctypes.cast(dec, ctypes.c_void_p), T=60) == kda.KDA_ERR_INVALID_ARG
    start = bad(5, 70, 100)
    assert _prefill_raw(lib, cu_host=ctypes.cast(start, ctypes.c_void_p)) == kda.KDA_ERR_INVALID_ARG
    assert _prefill_raw(lib, N=-1) == kda.KDA_ERR_INVALID_ARG
    assert _prefill_raw(lib, N=0, T=0) == kda.KDA_OK                     # nothing to do


def test_noalloc_prefill_rejects_on_host(lib):
    f = "kda_chunk_prefill_noalloc"
    # more (sequence, head) pairs than its fixed scratch holds: refused before any device call
    assert _prefill_raw(lib, fn=f, H=kda.KDA_NOALLOC_MAX_SEQ_HEADS) == kda.KDA_ERR_UNSUPPORTED   # 2 x 32 pairs
    assert _prefill_raw(lib, fn=f, q=None) == kda.KDA_ERR_INVALID_ARG
    assert _prefill_raw(lib, fn=f, stride=100) == kda.KDA_ERR_INVALID_ARG
    assert _prefill_raw(lib, fn=f, N=0, T=0) == kda.KDA_OK


def test_decode_rejects_bad_arguments_on_host(lib):
    f = lib.kda_decode_step
    args = [0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0, 4, 2, 128, 128, None]
    a = list(args); a[0] = None
    assert f(*a) == kda.KDA_ERR_INVALID_ARG
    a = list(args); a[10] = 96; a[11] = 96
    assert f(*a) == kda.KDA_ERR_UNSUPPORTED
    a = list(args); a[10] = 64
    assert f(*a) == kda.KDA_ERR_UNSUPPORTED                                # Dk != Dv
    a = list(args); a[5] = 0x6004
    assert f(*a) == kda.KDA_ERR_INVALID_ARG
    a = list(args); a[8] = 0
    assert f(*a) == kda.KDA_OK                                             # N = 0: nothing to do


def test_decode_multi_rejects_bad_arguments_on_host(lib):
    f = lib.kda_decode_multi
    #       q       k       v       la      beta    pool    slots  sl    ntok  commit out  dt  N  K  H  Dk   Dv decay stream
    args = [0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 8, None, None, 0, 0x7000, 0, 4, 3, 2, 128, 128, 0, None]
    def call(**kw):
        a = list(args)
        for i, val in kw.items():
            a[int(i[1:])] = val
        return f(*a)
    assert call(a0=None) == kda.KDA_ERR_INVALID_ARG
    assert call(a6=3) == kda.KDA_ERR_INVALID_ARG          # identity slots need num_slots >= N
    assert call(a9=2) == kda.KDA_ERR_INVALID_ARG          # commit is 0 or 1
    assert call(a15=64) == kda.KDA_ERR_UNSUPPORTED        # Dk != Dv
    assert call(a15=96, a16=96) == kda.KDA_ERR_UNSUPPORTED
    assert call(a5=0x6004) == kda.KDA_ERR_INVALID_ARG     # misaligned pool
    assert call(a7=0x8002) == kda.KDA_ERR_INVALID_ARG     # misaligned slot array
    assert call(a12=0) == kda.KDA_OK and call(a13=0) == kda.KDA_OK   # nothing to do
    assert call(a17=3) == kda.KDA_ERR_INVALID_ARG         # unknown decay layout
    assert call(a17=2) == kda.KDA_ERR_INVALID_ARG         # no decay: log_alpha must be NULL
    assert call(a3=None) == kda.KDA_ERR_INVALID_ARG       # a decay layout needs log_alpha


def test_prefill_ex_decay_rules_on_host(lib):
    f = "kda_chunk_prefill_ex"
    def raw(decay, **over):
        cu = (ctypes.c_int32 * 3)(0, 64, 100)
        a = dict(q=0x1000, k=0x2000, v=0x3000, la=0x4000, beta=0x5000, s0=None, cu=0x6000,
                 cu_host=ctypes.cast(cu, ctypes.c_void_p), N=2, T=100, H=4, Dk=64, Dv=64,
                 out=0x7000, out_dtype=0, fin=None, ck=None, stride=0, sp=None, sp_host=None, gamma=None, eps=1e-6,
                 stream=None)
        a.update(over)
        return getattr(lib, f)(a["q"], a["k"], a["v"], a["la"], a["beta"], a["s0"], a["cu"], a["cu_host"], a["N"],
                               a["T"], a["H"], a["Dk"], a["Dv"], a["out"], a["out_dtype"], a["fin"], a["ck"],
                               a["stride"], decay, a["sp"], a["sp_host"], a["gamma"], a["eps"], a["stream"])
    assert raw(kda.KDA_DECAY_HEAD, H=6) == kda.KDA_ERR_UNSUPPORTED     # per-head rows need H % 4 == 0
    assert raw(kda.KDA_DECAY_NONE) == kda.KDA_ERR_INVALID_ARG          # log_alpha given but unused
    assert raw(kda.KDA_DECAY_CHANNEL, la=None) == kda.KDA_ERR_INVALID_ARG
    assert raw(7) == kda.KDA_ERR_INVALID_ARG
    assert raw(kda.KDA_DECAY_NONE, la=None, N=0, T=0) == kda.KDA_OK
    sp = (ctypes.c_int32 * 2)(5, -1)
    assert raw(kda.KDA_DECAY_CHANNEL, sp=0x9000) == kda.KDA_ERR_INVALID_ARG       # device copy without host copy
    assert raw(kda.KDA_DECAY_CHANNEL, sp=0x9000,
               sp_host=ctypes.cast(sp, ctypes.c_void_p)) == kda.KDA_ERR_INVALID_ARG   # negative position
    # the fused output norm: gamma 16-byte aligned, eps finite and >= 0
    assert raw(kda.KDA_DECAY_CHANNEL, gamma=0xA004) == kda.KDA_ERR_INVALID_ARG
    assert raw(kda.KDA_DECAY_CHANNEL, gamma=0xA000, eps=-1.0) == kda.KDA_ERR_INVALID_ARG
    assert raw(kda.KDA_DECAY_CHANNEL, gamma=0xA000, eps=float("nan")) == kda.KDA_ERR_INVALID_ARG
    assert raw(kda.KDA_DECAY_CHANNEL, gamma=0xA000, eps=float("inf")) == kda.KDA_ERR_INVALID_ARG


def test_segmented_prefill_rejects_on_host(lib):
    f = lib.kda_chunk_prefill_segmented

    def raw(**over):
        a = dict(q=0x1000, k=0x2000, v=0x3000, la=0x4000, beta=0x5000, s0=None, T=1000, H=4, Dk=128, Dv=128,
                 out=0x7000, out_dtype=0, fin=None, ck=None, stride=0, decay=kda.KDA_DECAY_CHANNEL, sp=0, P=8,
                 gamma=None, eps=1e-6, stream=None)
        a.update(over)
        return f(a["q"], a["k"], a["v"], a["la"], a["beta"], a["s0"], a["T"], a["H"], a["Dk"], a["Dv"], a["out"],
                 a["out_dtype"], a["fin"], a["ck"], a["stride"], a["decay"], a["sp"], a["P"], a["gamma"], a["eps"],
                 a["stream"])
    assert raw(P=0) == kda.KDA_ERR_INVALID_ARG
    assert raw(P=65) == kda.KDA_ERR_INVALID_ARG                        # at most KDA_MAX_SEGMENTS
    assert raw(sp=-1) == kda.KDA_ERR_INVALID_ARG
    assert raw(sp=2 ** 31 - 10) == kda.KDA_ERR_INVALID_ARG             # positions past int32
    assert raw(T=-1) == kda.KDA_ERR_INVALID_ARG
    assert raw(Dv=64) == kda.KDA_ERR_UNSUPPORTED                       # Phi is carried as a Dk x Dv state
    assert raw(Dk=96, Dv=96) == kda.KDA_ERR_UNSUPPORTED
    assert raw(q=None) == kda.KDA_ERR_INVALID_ARG
    assert raw(q=0x1008) == kda.KDA_ERR_INVALID_ARG                    # 16-byte alignment
    assert raw(decay=kda.KDA_DECAY_NONE) == kda.KDA_ERR_INVALID_ARG    # log_alpha given but unused
    assert raw(decay=kda.KDA_DECAY_HEAD, H=6) == kda.KDA_ERR_UNSUPPORTED
    assert raw(ck=0x8000, stride=0) == kda.KDA_ERR_INVALID_ARG
    assert raw(stride=100) == kda.KDA_ERR_INVALID_ARG                   # multiple of 64
    assert raw(gamma=0xA004) == kda.KDA_ERR_INVALID_ARG
    assert raw(gamma=0xA000, eps=float("nan")) == kda.KDA_ERR_INVALID_ARG


def test_segmented_ex_rejects_on_host(lib):
    f = lib.kda_chunk_prefill_segmented_ex
    cu = (ctypes.c_int32 * 4)(0, 3000, 3000, 7000)
    sp = (ctypes.c_int32 * 3)(0, 64, 5)

    def raw(**over):
        a = dict(q=0x1000, k=0x2000, v=0x3000, la=0x4000, beta=0x5000, s0=None, cu=ctypes.cast(cu, ctypes.c_void_p),
                 N=3, T=7000, H=4, Dk=128, Dv=128, out=0x7000, out_dtype=0, fin=None, ck=None, stride=0,
                 decay=kda.KDA_DECAY_CHANNEL, sp=ctypes.cast(sp, ctypes.c_void_p), P=8, gamma=None, eps=1e-6,
                 stream=None)
        a.update(over)
        return f(a["q"], a["k"], a["v"], a["la"], a["beta"], a["s0"], a["cu"], a["N"], a["T"], a["H"], a["Dk"],
                 a["Dv"], a["out"], a["out_dtype"], a["fin"], a["ck"], a["stride"], a["decay"], a["sp"], a["P"],
                 a["gamma"], a["eps"], a["stream"])
    assert raw(P=0) == kda.KDA_ERR_INVALID_ARG
    assert raw(P=65) == kda.KDA_ERR_INVALID_ARG
    assert raw(N=129) == kda.KDA_ERR_UNSUPPORTED                  # at most KDA_MAX_SEGMENTED_SEQS
    assert raw(T=6999) == kda.KDA_ERR_INVALID_ARG                 # cu_seqlens must end at total_tokens
    assert raw(cu=None) == kda.KDA_ERR_INVALID_ARG
    bad = (ctypes.c_int32 * 3)(0, -1, 5)
    assert raw(sp=ctypes.cast(bad, ctypes.c_void_p)) == kda.KDA_ERR_INVALID_ARG
    assert raw(Dv=64) == kda.KDA_ERR_UNSUPPORTED
    assert raw(stride=100) == kda.KDA_ERR_INVALID_ARG
    assert raw(N=0, T=0) == kda.KDA_OK                            # nothing to do, nothing launched


def test_ckpt_count_with_start_positions(lib):
    cu = torch.tensor([0, 9, 9, 100], dtype=torch.int32)
    # s = 6, len 9, stride 4: absolute 8, 12 and the end; empty: none; s = 0, len 91: ceil(91/4) = 23
    assert kda.kda_ckpt_count_ex(cu, torch.tensor([6, 3, 0], dtype=torch.int32), 4) == 3 + 0 + 23
    assert kda.kda_ckpt_count_ex(cu, None, 4) == kda.kda_ckpt_count(cu, 4) == 3 + 0 + 23
    # 145408 tokens continuing a 40000-token prefix: absolute 65536, 98304, 131072, 163840 and the end
    assert kda.kda_ckpt_count_ex(torch.tensor([0, 145408], dtype=torch.int32),
                                 torch.tensor([40000], dtype=torch.int32), 32768) == 5
    with pytest.raises(kda.KdaError):
        kda.kda_ckpt_count_ex(cu, torch.tensor([0, -1, 0], dtype=torch.int32), 4)


def test_prepare_and_norm_reject_on_host(lib):
    cu = (ctypes.c_int32 * 2)(0, 10)
    cuh = ctypes.cast(cu, ctypes.c_void_p)
    f = lib.kda_prepare_inputs
    base = [0x1000, 0x2000, 0x3000, 0x4000, None, 0x5000, 0x6000, 0x7000, cuh, 1, 10, 2, 128, 1,
            0x8000, 0x9000, 0xA000, 0xB000, 0xC000, None]
    def call(**kw):
        a = list(base)
        for i, val in kw.items():
            a[int(i[1:])] = val
        return f(*a)
    assert call(a12=96) == kda.KDA_ERR_UNSUPPORTED
    assert call(a13=2) == kda.KDA_ERR_INVALID_ARG          # conv_act is 0 or 1
    assert call(a0=None) == kda.KDA_ERR_INVALID_ARG
    assert call(a3=0x4004) == kda.KDA_ERR_INVALID_ARG      # misaligned taps
    assert call(a6=0x6001) == kda.KDA_ERR_INVALID_ARG      # misaligned beta pre-activation
    assert call(a10=9) == kda.KDA_ERR_INVALID_ARG          # cu_seqlens end != total_tokens
    g = lib.kda_output_norm
    assert g(0x1000, 0, 0x2000, ctypes.c_float(-1.0), 0x3000, 5, 2, 128, None) == kda.KDA_ERR_INVALID_ARG
    assert g(0x1000, 0, 0x2000, ctypes.c_float(1e-6), 0x3000, 5, 2, 96, None) == kda.KDA_ERR_UNSUPPORTED
    assert g(0x1000, 0, 0x2000, ctypes.c_float(1e-6), 0x3000, 0, 2, 128, None) == kda.KDA_OK


def test_binding_refuses_non_bf16(lib):
    with pytest.raises(TypeError):
        kda.kda_decode_step(torch.zeros(1, 1, 64), torch.zeros(1, 1, 64), torch.zeros(1, 1, 64),
                            torch.zeros(1, 1, 64), torch.zeros(1, 1), torch.zeros(1, 1, 64, 64),
                            torch.zeros(1, 1, 64), 1, 1, 1, 64, 64)


def _slot_positions(bounds, start_pos, stride):
    """Absolute positions of the checkpoint slots the segmented prefill's runs A and F write:
    both cover every segment, so each writes, per segment in order, the stride multiples
    strictly inside it, then its end; run A's slots come first, then run F's."""
    pos = []
    for a, e in zip(bounds[:-1], bounds[1:]):
        a, e = start_pos + a, start_pos + e
        m = (a // stride + 1) * stride
        while m < e:
            pos.append(m)
            m += stride
        pos.append(e)
    return pos + pos


def test_segment_plan_properties(lib):
    """kda_segment_plan on a seeded sweep of prompt lengths, start positions, segment counts
    and strides: bounds on the absolute chunk grid with equal chunk counts, and the kept
    checkpoint slots sit exactly at the prompt's own checkpoint positions (the oracle's
    count and the stride grid)."""
    import random
    import oracle
    oracle.build()
    rng = random.Random(7)
    cases = [(145408, 0, 9, 32768), (5000, 4133, 8, 1024), (5000, 37, 5, 1024), (192, 0, 3, 64),
             (193, 0, 64, 64), (64 * 200, 63, 64, 128)]
    for _ in range(300):
        cases.append((rng.randint(0, 40000), rng.choice([0, rng.randint(0, 100000)]), rng.randint(1, 64),
                      rng.choice([0, 64, 128, 4096, 32768])))
    for T, s0, seg, stride in cases:
        bounds, slots = kda.kda_segment_plan(T, s0, seg, stride)
        P = len(bounds) - 1
        n_chunks = 0 if T == 0 else (s0 + T + 63) // 64 - s0 // 64
        if seg < 3 or n_chunks < 3:
            assert P == 1, (T, s0, seg)
        else:
            per = -(-n_chunks // seg)
            assert P == (1 if -(-n_chunks // per) < 3 else -(-n_chunks // per))
        assert bounds[0] == 0 and bounds[-1] == T
        assert all(x < y for x, y in zip(bounds, bounds[1:])) or T == 0
        if P >= 3:
            assert all((s0 + x) % 64 == 0 for x in bounds[1:-1])
            chunks = [(s0 + y + 63) // 64 - (s0 + x) // 64 for x, y in zip(bounds, bounds[1:])]
            assert len(set(chunks[:-1])) == 1 and 1 <= chunks[-1] <= chunks[0]
        if stride and P >= 3:
            got = [_slot_positions(bounds, s0, stride)[i] for i in slots]
            want = [m for m in range((s0 // stride + 1) * stride, s0 + T, stride)] + [s0 + T]
            assert got == want, (T, s0, seg, stride)
            assert len(slots) == oracle.ckpt_count([0, T], stride, [s0])
            n_run = len(_slot_positions(bounds, s0, stride)) // 2
            # the first segment's checkpoints come from run A, every later one from run F
            assert all((i < n_run) == (pos < s0 + bounds[1]) for i, pos in
                       zip(slots, [_slot_positions(bounds, s0, stride)[i] for i in slots]) if pos != s0 + bounds[1])
        else:
            assert slots == []


def test_segment_plan_rejects(lib):
    b = (ctypes.c_int32 * 65)()
    f = lib.kda_segment_plan
    vp = ctypes.cast(b, ctypes.c_void_p)
    assert f(1000, 0, 0, 0, vp, None, 0) == kda.KDA_ERR_INVALID_ARG
    assert f(1000, 0, 65, 0, vp, None, 0) == kda.KDA_ERR_INVALID_ARG
    assert f(1000, -1, 8, 0, vp, None, 0) == kda.KDA_ERR_INVALID_ARG
    assert f(-1, 0, 8, 0, vp, None, 0) == kda.KDA_ERR_INVALID_ARG
    assert f(1000, 0, 8, 100, vp, None, 0) == kda.KDA_ERR_INVALID_ARG       # stride: multiple of 64
    assert f(1000, 0, 8, 0, None, None, 0) == kda.KDA_ERR_INVALID_ARG        # bounds required
    slots = (ctypes.c_int32 * 1)()
    assert f(145408, 0, 9, 32768, vp, ctypes.cast(slots, ctypes.c_void_p), 1) == kda.KDA_ERR_INVALID_ARG  # 5 > 1
    assert f(145408, 0, 9, 32768, vp, None, 0) == 9
