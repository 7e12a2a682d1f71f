"""The C ABI: libla.so builds, loads, exports every symbol include/la.h
declares, and its host-side logic (sizes, status strings, argument
validation) behaves as documented.  No call here reaches a GPU: every
validation case is rejected before the library touches the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from fixed_state_recurrent_gb300 import build, api
    build.build()
    return api.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "la.h"), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("la_prefill", "la_prefill_workspace_bytes", "la_decode_step",
              "delta_prefill", "la_state_bytes", "la_status_string",
              "la_read_device_status", "delta_read_device_status",
              "la_prefill_variant", "la_prefill_variant_workspace_bytes",
              "gated_delta_prefill", "la_prefill_backward",
              "la_prefill_backward_workspace_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared_functions():
        assert hasattr(lib, n), f"libla.so does not export {n}"


def test_state_bytes(lib):
    assert lib.la_state_bytes(64, 64) == 16640   # 64x64 fp32 S plus 64 fp32 z
    assert lib.la_state_bytes(128, 128) == (128 * 128 + 128) * 4
    assert lib.la_state_bytes(0, 64) == 0


def test_status_strings(lib):
    for s in range(5):
        assert lib.la_status_string(s).startswith(b"LA_")
    assert b"TIMEOUT" in lib.la_status_string(4)


def test_workspace_bytes(lib):
    assert lib.la_prefill_workspace_bytes(1, 1, 256, 64, 64, 0, 0) >= 256
    assert lib.la_prefill_workspace_bytes(4, 8, 4096, 64, 64, 1, 0) >= 256
    assert lib.la_prefill_workspace_bytes(0, 1, 256, 64, 64, 0, 0) == 0
    assert lib.la_prefill_workspace_bytes(1, 1, 256, 129, 64, 0, 0) == 0
    assert lib.la_prefill_workspace_bytes(1, 1, 256, 64, 64, 7, 0) == 0
    assert lib.la_prefill_workspace_bytes(1, 1, 256, 64, 64, 1, 96) == 0


def _fake(addr):
    return ctypes.c_void_p(addr)


BASE = 1 << 40  # fake device addresses: never dereferenced, rejected first


def _prefill(lib, **kw):
    a = dict(q=BASE, k=BASE + (1 << 30), v=BASE + (2 << 30), dt=1, B=1, H=1, N=16,
             dk=64, dv=64, eps=1e-6, S0=None, z0=None, o=BASE + (3 << 30),
             SN=BASE + (4 << 30), zN=BASE + (5 << 30), chunk=0,
             ws=BASE + (6 << 30), wsb=1 << 20)
    a.update(kw)
    p = lambda x: None if x is None else _fake(x)
    return lib.la_prefill(p(a["q"]), p(a["k"]), p(a["v"]), a["dt"], a["B"], a["H"],
                          a["N"], a["dk"], a["dv"], a["eps"], p(a["S0"]), p(a["z0"]),
                          p(a["o"]), p(a["SN"]), p(a["zN"]), a["chunk"], p(a["ws"]),
                          a["wsb"], None)


@pytest.mark.parametrize("kw", [
    dict(B=0), dict(H=-1), dict(N=-1), dict(dk=0), dict(dv=129), dict(dk=200),
    dict(eps=-1.0), dict(eps=float("nan")), dict(eps=float("inf")), dict(dt=2),
    dict(q=None), dict(o=None), dict(SN=None), dict(zN=None), dict(ws=None),
    dict(wsb=16), dict(chunk=64),
    dict(q=BASE + 8), dict(o=BASE + (3 << 30) + 4), dict(ws=BASE + (6 << 30) + 2),
    dict(o=BASE + 64),                       # o overlaps q
    dict(SN=BASE + (3 << 30) + 1024),       # S_N overlaps o
    dict(S0=BASE + (7 << 30), SN=BASE + (7 << 30) + 16),  # partial S0/S_N overlap
    dict(zN=BASE + (4 << 30)),              # z_N overlaps S_N
])
def test_prefill_rejects_invalid_arguments(lib, kw):
    assert _prefill(lib, **kw) == 1  # LA_ERR_INVALID_ARG


def test_decode_and_delta_reject_invalid_arguments(lib):
    p = _fake
    # decode: null state, misaligned o, o overlapping S
    assert lib.la_decode_step(p(BASE), p(BASE + 4096), p(BASE + 8192), 1, 1, 1, 64, 64,
                              1e-6, None, p(BASE + (1 << 20)), p(BASE + (2 << 20)), None) == 1
    assert lib.la_decode_step(p(BASE), p(BASE + 4096), p(BASE + 8192), 1, 1, 1, 64, 64,
                              1e-6, p(BASE + (1 << 24)), p(BASE + (1 << 20)),
                              p(BASE + (2 << 20) + 4), None) == 1
    assert lib.la_decode_step(p(BASE), p(BASE + 4096), p(BASE + 8192), 1, 1, 1, 64, 64,
                              1e-6, p(BASE + (1 << 24)), p(BASE + (1 << 20)),
                              p(BASE + (1 << 24) + 256), None) == 1
    assert lib.la_decode_step(p(BASE), p(BASE + 4096), p(BASE + 8192), 1, 1, 1, 0, 64,
                              1e-6, p(BASE + (1 << 24)), p(BASE + (1 << 20)),
                              p(BASE + (2 << 20)), None) == 1
    # delta: bad dims, null beta, reads overlapping k
    assert lib.delta_prefill(p(BASE), p(BASE + (1 << 24)), 1, p(BASE + (2 << 24)), 1, 1, 8,
                             130, 64, None, p(BASE + (3 << 24)), p(BASE + (4 << 24)), None) == 1
    assert lib.delta_prefill(p(BASE), p(BASE + (1 << 24)), 1, None, 1, 1, 8,
                             64, 64, None, p(BASE + (3 << 24)), p(BASE + (4 << 24)), None) == 1
    assert lib.delta_prefill(p(BASE), p(BASE + (1 << 24)), 1, p(BASE + (2 << 24)), 1, 1, 8,
                             64, 64, None, p(BASE + 16), p(BASE + (4 << 24)), None) == 1
    assert lib.la_read_device_status(None, None) == 1


def _variant(lib, **kw):
    a = dict(q=BASE, k=BASE + (1 << 30), v=BASE + (2 << 30), dt=1, B=1, H=1, N=16,
             dk=64, dv=64, eps=1e-6, alpha=BASE + (8 << 30), mode=0, S0=None, z0=None,
             o=BASE + (3 << 30), SN=BASE + (4 << 30), zN=BASE + (5 << 30), ws=None, wsb=0)
    a.update(kw)
    p = lambda x: None if x is None else _fake(x)
    return lib.la_prefill_variant(p(a["q"]), p(a["k"]), p(a["v"]), a["dt"], a["B"], a["H"],
                                  a["N"], a["dk"], a["dv"], ctypes.c_float(a["eps"]),
                                  p(a["alpha"]), a["mode"], p(a["S0"]), p(a["z0"]), p(a["o"]),
                                  p(a["SN"]), p(a["zN"]), p(a["ws"]), a["wsb"], None)


@pytest.mark.parametrize("kw", [
    dict(mode=3), dict(mode=-1),
    dict(mode=2),                           # non-causal takes no decay
    dict(alpha=BASE + (8 << 30) + 4),       # misaligned alpha
    dict(o=BASE + (8 << 30)),               # o overlaps alpha
    dict(eps=-1.0), dict(dk=129), dict(zN=None), dict(q=None),
    dict(ws=BASE + (9 << 30), wsb=16),          # workspace smaller than asked for
    dict(ws=BASE + (9 << 30) + 8, wsb=1 << 26),  # misaligned workspace
    dict(ws=BASE + (3 << 30), wsb=1 << 26),      # workspace overlaps o
])
def test_prefill_variant_rejects_invalid_arguments(lib, kw):
    assert _variant(lib, **kw) == 1  # LA_ERR_INVALID_ARG


def test_prefill_variant_workspace_bytes(lib):
    # bf16 at d = 64 with a decay, write then read or read before write: the
    # tensor-core split over the SMs (the same workspace for both orders);
    # without a decay in causal order, and fp32, the CUDA-core chunk slots
    # (dk dv + dk + 1 floats per chunk), when its heads are few enough to be
    # worth cutting
    assert lib.la_prefill_variant_workspace_bytes(4, 8, 4096, 64, 64, 1, 0, 1) > 0
    assert (lib.la_prefill_variant_workspace_bytes(4, 8, 4096, 64, 64, 1, 1, 1) ==
            lib.la_prefill_variant_workspace_bytes(4, 8, 4096, 64, 64, 1, 0, 1))
    slots = 32 * 10 * (64 * 64 + 64 + 1) * 4  # 32 heads: 10 chunks each fill ~2 blocks per SM
    assert lib.la_prefill_variant_workspace_bytes(4, 8, 4096, 64, 64, 1, 0, 0) == slots
    assert lib.la_prefill_variant_workspace_bytes(4, 8, 4096, 64, 64, 0, 0, 1) == slots
    assert lib.la_prefill_variant_workspace_bytes(4, 8, 4096, 64, 64, 0, 1, 1) == slots
    assert lib.la_prefill_variant_workspace_bytes(1, 1, 256, 64, 64, 0, 2, 0) == 32 * (64 * 64 + 64 + 1) * 4
    assert lib.la_prefill_variant_workspace_bytes(4, 8, 4096, 128, 128, 1, 0, 1) > 0
    assert lib.la_prefill_variant_workspace_bytes(1, 1, 8, 64, 64, 0, 0, 0) == 0   # one chunk
    assert lib.la_prefill_variant_workspace_bytes(8, 64, 4096, 64, 64, 0, 0, 0) == 0  # 512 heads
    assert lib.la_prefill_variant_workspace_bytes(0, 8, 4096, 64, 64, 1, 0, 1) == 0
    # la_prefill's CUDA-core path: the same slots after the 256-byte header
    assert lib.la_prefill_workspace_bytes(1, 1, 256, 64, 64, 0, 0) == 256 + 32 * (64 * 64 + 64 + 1) * 4
    # the backward splits its heads over the SMs on the tensor-core form and,
    # elsewhere, into the CUDA-core prefill's chunks: the state before every
    # chunk, the gradient state after it, and one scratch state per head
    assert lib.la_prefill_backward_workspace_bytes(4, 8, 4096, 64, 64, 1) > 0
    slot = 64 * 64 + 64  # 32 heads: 19 chunks each make about four blocks per SM
    assert lib.la_prefill_backward_workspace_bytes(4, 8, 4096, 64, 64, 0) == 32 * (2 * 19 + 1) * slot * 4
    slot = 128 * 128 + 128
    assert lib.la_prefill_backward_workspace_bytes(4, 8, 4096, 128, 128, 1) == 32 * (2 * 19 + 1) * slot * 4
    assert lib.la_prefill_backward_workspace_bytes(8, 128, 4096, 128, 128, 1) == 0  # 1024 heads: whole heads
    assert lib.la_prefill_backward_workspace_bytes(4, 8, 0, 64, 64, 1) == 0
    assert lib.la_prefill_backward_workspace_bytes(4, 8, 4096, 129, 64, 1) == 0
    # it grows with the tokens (the parked phi(K) rows) and covers at least them
    small = lib.la_prefill_backward_workspace_bytes(1, 1, 256, 64, 64, 1)
    big = lib.la_prefill_backward_workspace_bytes(1, 1, 8192, 64, 64, 1)
    assert big > small and big >= 8192 * 64 * 2


def test_gated_delta_rejects_invalid_arguments(lib):
    p = _fake
    # reads overlapping alpha; misaligned alpha; bad dims
    assert lib.gated_delta_prefill(p(BASE), p(BASE + (1 << 24)), 1, p(BASE + (2 << 24)),
                                   p(BASE + (5 << 24)), 1, 1, 8, 64, 64, None,
                                   p(BASE + (5 << 24)), p(BASE + (4 << 24)), None) == 1
    assert lib.gated_delta_prefill(p(BASE), p(BASE + (1 << 24)), 1, p(BASE + (2 << 24)),
                                   p(BASE + (5 << 24) + 8), 1, 1, 8, 64, 64, None,
                                   p(BASE + (3 << 24)), p(BASE + (4 << 24)), None) == 1
    assert lib.gated_delta_prefill(p(BASE), p(BASE + (1 << 24)), 1, p(BASE + (2 << 24)),
                                   p(BASE + (5 << 24)), 1, 1, 8, 0, 64, None,
                                   p(BASE + (3 << 24)), p(BASE + (4 << 24)), None) == 1


def test_backward_rejects_invalid_arguments(lib):
    p = _fake
    MB = 1 << 24
    def call(**kw):
        a = dict(q=BASE, k=BASE + MB, v=BASE + 2 * MB, dt=1, B=1, H=1, N=16, dk=64, dv=64,
                 eps=1e-6, S0=None, z0=None, dO=BASE + 3 * MB, dSN=None, dzN=None,
                 dq=BASE + 4 * MB, dk_=BASE + 5 * MB, dv_=BASE + 6 * MB, dS0=None, dz0=None,
                 ws=None, wsb=0)
        a.update(kw)
        f = lambda x: None if x is None else p(x)
        return lib.la_prefill_backward(f(a["q"]), f(a["k"]), f(a["v"]), a["dt"], a["B"], a["H"],
                                       a["N"], a["dk"], a["dv"], ctypes.c_float(a["eps"]),
                                       f(a["S0"]), f(a["z0"]), f(a["dO"]), f(a["dSN"]), f(a["dzN"]),
                                       f(a["dq"]), f(a["dk_"]), f(a["dv_"]), f(a["dS0"]),
                                       f(a["dz0"]), f(a["ws"]), a["wsb"], None)
    assert call(dO=None) == 1                    # dO required
    assert call(dq=BASE + 3 * MB) == 1           # dq overlaps dO
    assert call(dk_=BASE + 4 * MB + 64) == 1     # dk overlaps dq
    assert call(dv_=BASE + 6 * MB + 4) == 1      # misaligned
    assert call(dS0=BASE + 2 * MB) == 1          # dS0 overlaps v
    assert call(dk=129) == 1
    assert call(eps=-1.0) == 1
    need = lib.la_prefill_backward_workspace_bytes(1, 1, 16, 64, 64, 1)
    assert need > 0
    assert call(ws=BASE + 8 * MB, wsb=need - 1) == 1       # workspace too small
    assert call(ws=BASE + 8 * MB + 8, wsb=need) == 1       # misaligned workspace
    assert call(ws=BASE + 6 * MB, wsb=need) == 1           # workspace overlaps dv
    assert call(ws=BASE + 2 * MB - 16, wsb=need) == 1      # workspace overlaps v


def _split(BH, N, sms=152):
    """The work split of the tensor-core kernels (piece slots per head), as the
    header describes it: G = min(chunks, SMs) runs, MPH = ceil(NC / L) + 1."""
    NC = (N + 127) // 128
    tc = BH * NC
    G = min(tc, sms)
    L = tc // G
    return NC, tc, (NC + L - 1) // L + 1


def test_tensor_core_variant_workspace_sizes(lib):
    # the workspace of each tensor-core form, from the split alone (the CPU has
    # no device, so the library takes a 152-SM GPU)
    B, H, N = 4, 8, 4096
    BH = B * H
    NC, tc, mph = _split(BH, N)
    slot64, slot128 = (64 * 64 + 64) * 4, (128 * 128 + 128) * 4
    simt = lambda d: lib.la_prefill_variant_workspace_bytes(B, H, N, d, d, 0, 1, 0)  # fp32: CUDA cores
    prefix64 = BH * mph * slot64 + tc * 66 * 128 + BH * N * 64 * 2
    # la_prefill: header, then the two-launch form's totals, prefix tiles and phi(K)
    assert lib.la_prefill_workspace_bytes(B, H, N, 64, 64, 1, 0) == 256 + prefix64
    # d = 128: header, then two slot arrays (no phi(K) copy)
    assert lib.la_prefill_workspace_bytes(B, H, N, 128, 128, 1, 0) == 256 + 2 * BH * mph * slot128
    # read before write at d = 64 (two-launch form): the prefill's workspace, no header
    assert lib.la_prefill_variant_workspace_bytes(B, H, N, 64, 64, 1, 1, 0) == max(prefix64, simt(64))
    # non-causal at d = 64: that plus one [80 x 64] bf16 state tile per head
    assert lib.la_prefill_variant_workspace_bytes(B, H, N, 64, 64, 1, 2, 0) == max(prefix64 + BH * 80 * 128,
                                                                                 simt(64))
    # non-causal at d = 128: the totals, then one [144 x 128] bf16 tile per head
    assert lib.la_prefill_variant_workspace_bytes(B, H, N, 128, 128, 1, 2, 0) == max(
        BH * mph * slot128 + BH * 2 * 144 * 128, simt(128))
    # read before write at d = 128: the three-launch prefill's workspace with its header
    assert lib.la_prefill_variant_workspace_bytes(B, H, N, 128, 128, 1, 1, 0) == max(
        256 + 2 * BH * mph * slot128, simt(128))
    # decayed at d = 128, either order: totals, entry states and one decay per slot
    dec128 = (2 * BH * mph * (128 * 128 + 128) + BH * mph) * 4
    assert lib.la_prefill_variant_workspace_bytes(B, H, N, 128, 128, 1, 0, 1) == max(dec128, simt(128))
    assert lib.la_prefill_variant_workspace_bytes(B, H, N, 128, 128, 1, 1, 1) == max(dec128, simt(128))
