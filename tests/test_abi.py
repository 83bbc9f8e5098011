"""The C-ABI library without a GPU: it builds, loads, exports every symbol
include/ssd.h declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

from state_space_sequence_ssd_gb300 import _ffi, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssd.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _ffi.lib()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"SSD_API\s+[\w\s\*]+?\b(ssd_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = set(declared_symbols())
    for required in ("ssd_chunk_cumsum", "ssd_chunk_state", "ssd_state_passing", "ssd_chunk_scan",
                     "ssd_forward", "ssd_status_string", "ssd_get_device_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in _ffi.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    for s in range(0, 8):
        msg = lib.ssd_status_string(s)
        assert msg is not None and len(msg) > 0
    assert b"INVALID_ARG" in lib.ssd_status_string(1)
    assert b"RANGE" in lib.ssd_status_string(_ffi.SSD_ERR_RANGE)


def test_debug_hooks_without_launches(lib):
    """The failure-path hooks only set host state: they succeed and restore cleanly without a GPU."""
    assert lib.ssd_debug_set_wait_limit_ns(2_000_000) == 0
    assert lib.ssd_debug_stall(1 << 3) == 0
    assert lib.ssd_debug_stall(0) == 0
    assert lib.ssd_debug_set_wait_limit_ns(0) == 0


FAKE = 4096  # a 16-byte aligned non-null address: validation must fail before it is used


def fwd(lib, **kw):
    a = dict(x=FAKE, dt=FAKE, A=FAKE, B=FAKE, C=FAKE, D=FAKE, init=FAKE, batch=1, seqlen=512, nheads=4,
             headdim=64, ngroups=1, dstate=64, chunk_size=64, y=FAKE, final=FAKE)
    a.update(kw)
    return lib.ssd_forward(a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["init"], a["batch"], a["seqlen"],
                           a["nheads"], a["headdim"], a["ngroups"], a["dstate"], a["chunk_size"], a["y"],
                           a["final"], None)


@pytest.mark.parametrize("kw", [dict(x=None), dict(dt=None), dict(A=None), dict(B=None), dict(C=None),
                                dict(y=None), dict(batch=0), dict(seqlen=0), dict(nheads=-1), dict(dstate=0),
                                dict(chunk_size=0), dict(ngroups=3), dict(x=FAKE + 2), dict(y=FAKE + 8),
                                dict(init=FAKE + 4), dict(final=FAKE + 4)])
def test_forward_rejects_invalid(lib, kw):
    assert fwd(lib, **kw) == _ffi.SSD_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(headdim=128), dict(dstate=96), dict(dstate=1024), dict(chunk_size=32),
                                dict(chunk_size=512)])
def test_forward_rejects_unsupported(lib, kw):
    assert fwd(lib, **kw) == _ffi.SSD_ERR_UNSUPPORTED


def test_stage_entry_points_validate(lib):
    assert lib.ssd_chunk_cumsum(None, FAKE, 1, 64, 4, 64, FAKE, FAKE, None) == _ffi.SSD_ERR_INVALID_ARG
    assert lib.ssd_chunk_cumsum(FAKE, FAKE, 1, 64, 4, 96, FAKE, FAKE, None) == _ffi.SSD_ERR_UNSUPPORTED
    assert lib.ssd_chunk_state(FAKE, FAKE, FAKE, FAKE, 1, 64, 4, 64, 1, 64, 64, None, None) == _ffi.SSD_ERR_INVALID_ARG
    assert lib.ssd_chunk_state(FAKE, FAKE, FAKE, FAKE, 1, 64, 4, 32, 1, 64, 64, FAKE, None) == _ffi.SSD_ERR_UNSUPPORTED
    assert lib.ssd_state_passing(FAKE, FAKE, None, 1, 0, 4, 64, 64, 64, FAKE, None, None) == _ffi.SSD_ERR_INVALID_ARG
    assert lib.ssd_state_passing(FAKE, FAKE, None, 1, 4, 4, 64, 64, 64, FAKE + 4, None, None) == _ffi.SSD_ERR_INVALID_ARG
    assert lib.ssd_chunk_scan(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 1, 64, 4, 64, 1, 64, 64, FAKE, None) \
        == _ffi.SSD_ERR_INVALID_ARG
    assert lib.ssd_chunk_scan(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1, 64, 6, 64, 4, 64, 64, FAKE, None) \
        == _ffi.SSD_ERR_INVALID_ARG


def test_profiling_counters_without_launches(lib):
    assert lib.ssd_profile_reset() == 0
    ms = (ctypes.c_float * 8)()
    cnt = (ctypes.c_int * 8)()
    n = ctypes.c_int(0)
    assert lib.ssd_profile_read(ms, cnt, 8, ctypes.byref(n)) == 0
    assert n.value >= 4
    assert all(cnt[k] == 0 for k in range(n.value))
    assert lib.ssd_kernel_name(3) == b"chunk_scan"
    assert lib.ssd_launch_count() >= 0


def test_binding_requires_cuda_tensors():
    import torch

    import state_space_sequence_ssd_gb300 as ssd
    x = torch.zeros((1, 64, 4, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        ssd.ssd_forward(x, torch.zeros((1, 64, 4)), torch.zeros(4), torch.zeros((1, 64, 1, 64), dtype=torch.bfloat16),
                        torch.zeros((1, 64, 1, 64), dtype=torch.bfloat16), None, None, 64)


def fwd_noalloc(lib, **kw):
    a = dict(x=FAKE, dt=FAKE, A=FAKE, B=FAKE, C=FAKE, D=FAKE, init=FAKE, batch=1, seqlen=512, nheads=4,
             headdim=64, ngroups=1, dstate=64, chunk_size=64, y=FAKE, final=FAKE)
    a.update(kw)
    return lib.ssd_forward_noalloc(a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["init"], a["batch"],
                                   a["seqlen"], a["nheads"], a["headdim"], a["ngroups"], a["dstate"],
                                   a["chunk_size"], a["y"], a["final"], None)


def test_noalloc_validates_before_the_device(lib):
    """Bad arguments and workloads larger than the fixed scratch are refused
    before any CUDA call (the fake pointers are never touched)."""
    assert fwd_noalloc(lib, x=None) == _ffi.SSD_ERR_INVALID_ARG
    assert fwd_noalloc(lib, y=FAKE + 8) == _ffi.SSD_ERR_INVALID_ARG
    assert fwd_noalloc(lib, dstate=96) == _ffi.SSD_ERR_UNSUPPORTED
    assert fwd_noalloc(lib, seqlen=65536, nheads=32, dstate=128, chunk_size=256) == _ffi.SSD_ERR_SCRATCH_TOO_SMALL
    assert b"SCRATCH_TOO_SMALL" in lib.ssd_status_string(_ffi.SSD_ERR_SCRATCH_TOO_SMALL)


def plan(lib, b, L, H, N, G, Q, P=64):
    span, step, nb = ctypes.c_int(-1), ctypes.c_int(-1), ctypes.c_ulonglong(0)
    r = lib.ssd_forward_plan(b, L, H, P, G, N, Q, ctypes.addressof(span), ctypes.addressof(step),
                             ctypes.addressof(nb))
    return r, span.value, step.value, nb.value


@pytest.mark.parametrize("b,L,H,N,G,Q", [(1, 512, 4, 64, 1, 64), (2, 4096, 64, 128, 1, 256),
                                         (1, 65536, 32, 128, 1, 256), (1, 16384, 32, 512, 1, 256),
                                         (1, 262144, 32, 256, 8, 256), (3, 1000, 6, 128, 2, 128)])
def test_forward_plan_is_consistent(lib, b, L, H, N, G, Q):
    """The plan agrees with the workspace the no-allocation entry point accepts or refuses, and its
    spans tile the sequence."""
    r, span, step, nb = plan(lib, b, L, H, N, G, Q)
    assert r == _ffi.SSD_OK
    nc = -(-L // Q)
    assert 1 <= span <= min(64, nc) and step in (1, 2, 4) and span * step <= max(nc, span)
    nspans = -(-nc // span)
    # the parts listed for ssd_forward_noalloc in include/ssd.h, each rounded up to 256 bytes
    parts = 8 * b * H * nc * Q + 4 * b * nspans * H * 64 * N + 4 * b * H * nspans + 4 * b * L * G * N
    assert parts <= nb <= parts + 6 * 256
    fits = nb <= _ffi.SSD_NOALLOC_SCRATCH_BYTES
    got = fwd_noalloc(lib, batch=b, seqlen=L, nheads=H, dstate=N, ngroups=G, chunk_size=Q, x=None)
    assert got == _ffi.SSD_ERR_INVALID_ARG  # null x: refused before the size check either way
    if not fits:
        assert fwd_noalloc(lib, batch=b, seqlen=L, nheads=H, dstate=N, ngroups=G, chunk_size=Q) == \
            _ffi.SSD_ERR_SCRATCH_TOO_SMALL


def test_forward_plan_known_shapes(lib):
    # the shortest span whose chunk_state grid (batch, heads / 4, spans) fits one CTA per SM of a 152-SM
    # device: L 65536 x 32 heads -> 8 x 19 = 152 CTAs of 14 chunks
    assert plan(lib, 1, 65536, 32, 128, 1, 256)[1] == 14
    assert plan(lib, 2, 4096, 64, 128, 1, 256)[1] == 4      # 2 x 16 x 4 = 128 CTAs
    assert plan(lib, 1, 16384, 32, 256, 1, 256)[1] == 8     # two heads per CTA at N 256: 16 x 8 = 128
    # no span of at most 64 chunks fits: ~1216 (batch, head, chunk) units per span wave
    assert plan(lib, 8, 65536, 32, 128, 1, 256)[1] == 54
    assert plan(lib, 1, 262144, 32, 256, 8, 256)[1] == 27
    assert plan(lib, 1, 512, 4, 64, 1, 64)[1:3] == (1, 1)  # 32 CTAs: nothing to merge
    assert plan(lib, 2, 4096, 64, 128, 1, 256)[3] <= _ffi.SSD_NOALLOC_SCRATCH_BYTES  # 40 MiB fits
    assert plan(lib, 1, 65536, 32, 128, 1, 256)[3] > _ffi.SSD_NOALLOC_SCRATCH_BYTES  # 85 MiB does not
    assert plan(lib, 1, 512, 4, 96, 1, 64)[0] == _ffi.SSD_ERR_UNSUPPORTED
    assert plan(lib, 1, 512, 6, 64, 4, 64)[0] == _ffi.SSD_ERR_INVALID_ARG
    assert lib.ssd_forward_plan(1, 512, 4, 64, 1, 64, 64, None, None, None) == _ffi.SSD_OK


def test_forward_plan_run_lengths(lib):
    """compute_out's run length (span x step, in chunks) on a 152-SM device (the value used when no device
    can be queried): long runs where the waves are few and a longer run saves pipeline fills -- even when
    the longer runs leave SMs idle in one wave (2 x 4096, 64 heads: 128 CTAs of two heads in one wave beat
    256 in two, 88.0 against 94.7 us measured on GB300); one span when the batch is large enough that the
    fills are spread over many waves anyway."""
    def run(*a):
        r = plan(lib, *a)
        return r[1] * r[2]
    assert run(1, 65536, 32, 128, 1, 256) == 28   # 10 runs per head pair: 9 of 28 chunks and one of 4
    assert run(2, 4096, 64, 128, 1, 256) == 8
    assert run(1, 16384, 32, 64, 1, 256) == 8
    assert plan(lib, 8, 65536, 32, 128, 1, 256)[2] == 1       # 54-chunk spans, eight waves of CTAs
    assert plan(lib, 1, 512, 4, 64, 1, 64)[2] == 1            # 16 one-chunk CTAs: longer runs only serialize them


def test_step_validation(lib):
    def step(**kw):
        a = dict(x=FAKE, dt=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, state=FAKE, batch=2, nheads=4, headdim=64,
                 ngroups=1, dstate=128, y=FAKE)
        a.update(kw)
        return lib.ssd_step(a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["state"], a["batch"], a["nheads"],
                            a["headdim"], a["ngroups"], a["dstate"], a["y"], None)
    assert step(x=None) == _ffi.SSD_ERR_INVALID_ARG
    assert step(state=None) == _ffi.SSD_ERR_INVALID_ARG
    assert step(y=None) == _ffi.SSD_ERR_INVALID_ARG
    assert step(batch=0) == _ffi.SSD_ERR_INVALID_ARG
    assert step(ngroups=3) == _ffi.SSD_ERR_INVALID_ARG
    assert step(state=FAKE + 4) == _ffi.SSD_ERR_INVALID_ARG
    assert step(x=FAKE + 1) == _ffi.SSD_ERR_INVALID_ARG
    assert step(headdim=32) == _ffi.SSD_ERR_UNSUPPORTED
    assert step(dstate=96) == _ffi.SSD_ERR_UNSUPPORTED


def test_step_multi_validation(lib):
    def multi(**kw):
        a = dict(x=FAKE, dt=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, state=FAKE, batch=2, ntokens=8, nheads=4,
                 headdim=64, ngroups=1, dstate=128, y=FAKE)
        a.update(kw)
        return lib.ssd_step_multi(a["x"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["state"], a["batch"],
                                  a["ntokens"], a["nheads"], a["headdim"], a["ngroups"], a["dstate"], a["y"], None)
    assert multi(x=None) == _ffi.SSD_ERR_INVALID_ARG
    assert multi(state=None) == _ffi.SSD_ERR_INVALID_ARG
    assert multi(ntokens=0) == _ffi.SSD_ERR_INVALID_ARG
    assert multi(ntokens=-3) == _ffi.SSD_ERR_INVALID_ARG
    assert multi(ngroups=3) == _ffi.SSD_ERR_INVALID_ARG
    assert multi(state=FAKE + 8) == _ffi.SSD_ERR_INVALID_ARG
    assert multi(dt=FAKE + 2) == _ffi.SSD_ERR_INVALID_ARG
    assert multi(headdim=128) == _ffi.SSD_ERR_UNSUPPORTED
    assert multi(dstate=32) == _ffi.SSD_ERR_UNSUPPORTED


def test_options_validation(lib):
    """Bad input-side options are rejected before any launch (each case keeps every other argument valid)."""
    def fwd_ex(**kw):
        o = _ffi.InputOptions()
        for k, v in kw.items():
            setattr(o, k, v)
        return lib.ssd_forward_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 512, 4, 64, 1, 64, 64,
                                  ctypes.addressof(o), FAKE, FAKE, None)

    def step_ex(**kw):
        o = _ffi.InputOptions()
        for k, v in kw.items():
            setattr(o, k, v)
        return lib.ssd_step_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 64, 1, 128, ctypes.addressof(o),
                               FAKE, None)
    bad = _ffi.SSD_ERR_INVALID_ARG
    assert fwd_ex(dt_limit=1, dt_min=0.5, dt_max=0.1) == bad
    assert fwd_ex(dt_limit=1, dt_min=float("nan"), dt_max=0.1) == bad
    assert fwd_ex(dt_bias=FAKE + 2) == bad
    assert fwd_ex(z=FAKE + 8) == bad
    assert step_ex(z=FAKE + 1) == bad
    assert step_ex(dt_limit=1, dt_min=1.0, dt_max=0.0) == bad
    # a per-channel D is read in 16-byte pieces by the forward pass
    o = _ffi.InputOptions()
    o.D_per_channel = 1
    assert lib.ssd_forward_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 4, FAKE, 1, 512, 4, 64, 1, 64, 64,
                              ctypes.addressof(o), FAKE, FAKE, None) == bad
