"""Host-side checks of the C ABI: the library loads, exports what include/kda.h
declares, and rejects bad arguments before making any CUDA call.

No call here reaches a kernel: every argument set is invalid, so validation
returns first. These run without a GPU.
"""
import ctypes
import re

import pytest

from gated_delta_rule_57_gb300 import build, kda

ST = kda


@pytest.fixture(scope="module")
def L():
    return kda.lib()


def test_exports_every_header_symbol(L):
    names = kda.header_functions()
    assert {"kda_chunk_fwd", "kda_chunk_fwd_ckpt", "kda_decode_step", "kda_decode_multi",
            "kda_chunk_fwd_workspace_size",
            "kda_status_string", "kda_abi_version", "kda_last_error_string"} <= set(names)
    for n in names:
        assert hasattr(L, n), f"libkda.so does not export {n}"


def test_abi_version_matches_header(L):
    text = open(build.INCLUDE + "/kda.h").read()
    ver = int(re.search(r"#define KDA_ABI_VERSION (\d+)", text).group(1))
    assert L.kda_abi_version() == ver


def test_status_enum_matches_header():
    text = open(build.INCLUDE + "/kda.h").read()
    for name, val in re.findall(r"(KDA_(?:OK|ERR_\w+))\s*=\s*(\d+)", text):
        assert getattr(kda, name) == int(val), name
        assert kda.status_string(int(val)) == name
    for name, val in re.findall(r"#define (KDA_DEV_\w+) (0x[0-9a-f]+)", text):
        assert getattr(kda, name) == int(val, 16), name
    assert kda.status_string(99) == "KDA_ERR_UNKNOWN"


def test_workspace_size(L):
    # the tensor-core path's handoff buffer for the balanced schedule: one
    # 128 x 128 fp32 state and one int per sequence (ints padded to 256 bytes)
    assert L.kda_chunk_fwd_workspace_size(8, 8192, 32, 128, 128, kda.KDA_BF16) == 256 * 65536 + 1024
    assert L.kda_chunk_fwd_workspace_size(3, 64, 100, 128, 128, kda.KDA_BF16) == 300 * 65536 + 1280
    assert L.kda_chunk_fwd_workspace_size(8, 8192, 32, 128, 128, kda.KDA_F32) == 0
    # bf16 d = 64 runs the same kernel at d = 128: the same handoff buffer
    assert L.kda_chunk_fwd_workspace_size(8, 8192, 32, 64, 64, kda.KDA_BF16) == 256 * 65536 + 1024
    assert L.kda_chunk_fwd_workspace_size(8, 0, 32, 128, 128, kda.KDA_BF16) == 0
    assert L.kda_chunk_fwd_workspace_size(1, 64, 1, 128, 128, kda.KDA_BF16) == 0
    bad = ctypes.c_size_t(-1).value
    assert L.kda_chunk_fwd_workspace_size(1, 16, 1, 96, 96, kda.KDA_BF16) == bad
    assert L.kda_chunk_fwd_workspace_size(1, 16, 1, 128, 64, kda.KDA_F32) == bad
    assert L.kda_chunk_fwd_workspace_size(-1, 16, 1, 128, 128, kda.KDA_F32) == bad
    assert L.kda_chunk_fwd_workspace_size(1, 16, 1, 64, 64, 7) == bad


# Fake, 16-byte aligned addresses: never dereferenced, validation rejects first.
A = [0x10000 * (i + 1) for i in range(8)]


def call_fwd(L, q=A[0], k=A[1], v=A[2], g=A[3], beta=A[4], h0=None, o=A[5], hT=A[6], B=1,
             T=16, H=1, dk=64, dv=64, io=kda.KDA_BF16):
    return L.kda_chunk_fwd(q, k, v, g, beta, h0, o, hT, B, T, H, dk, dv, io, None, 0, None,
                           None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), ST.KDA_ERR_INVALID_ARG),
    (dict(T=-3), ST.KDA_ERR_INVALID_ARG),
    (dict(dk=96, dv=96), ST.KDA_ERR_UNSUPPORTED),
    (dict(dk=128, dv=64), ST.KDA_ERR_UNSUPPORTED),
    (dict(dk=0, dv=0), ST.KDA_ERR_INVALID_ARG),
    (dict(io=5), ST.KDA_ERR_INVALID_ARG),
    (dict(q=None), ST.KDA_ERR_INVALID_ARG),
    (dict(beta=None), ST.KDA_ERR_INVALID_ARG),
    (dict(o=None), ST.KDA_ERR_INVALID_ARG),
    (dict(k=A[1] + 8), ST.KDA_ERR_INVALID_ARG),     # misaligned
    (dict(beta=A[4] + 2), ST.KDA_ERR_INVALID_ARG),  # beta needs 4 bytes
    (dict(o=A[0]), ST.KDA_ERR_INVALID_ARG),         # o aliases q
    (dict(hT=A[3]), ST.KDA_ERR_INVALID_ARG),        # hT aliases g
    (dict(B=1 << 16, H=1 << 16), ST.KDA_ERR_INVALID_ARG),  # B*H >= 2^31
])
def test_chunk_fwd_rejects(L, kw, code):
    assert call_fwd(L, **kw) == code
    assert L.kda_last_error_string()  # a reason is recorded


def test_empty_batch_is_a_no_op(L):
    # B = 0 or H = 0: nothing to do, nothing launched, even with NULL pointers.
    assert L.kda_chunk_fwd(None, None, None, None, None, None, None, None, 0, 16, 4, 64, 64,
                           kda.KDA_BF16, None, 0, None, None) == ST.KDA_OK
    assert L.kda_decode_step(None, None, None, None, None, None, None, 0, 4, 128, 128,
                             kda.KDA_F32, None, None) == ST.KDA_OK


def call_dec(L, q=A[0], k=A[1], v=A[2], g=A[3], beta=A[4], S=A[5], o=A[6], N=2, H=1, dk=128,
             dv=128, io=kda.KDA_BF16):
    return L.kda_decode_step(q, k, v, g, beta, S, o, N, H, dk, dv, io, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(N=-1), ST.KDA_ERR_INVALID_ARG),
    (dict(dk=32, dv=32), ST.KDA_ERR_UNSUPPORTED),
    (dict(S=None), ST.KDA_ERR_INVALID_ARG),
    (dict(o=A[2]), ST.KDA_ERR_INVALID_ARG),
    (dict(S=A[5] + 4), ST.KDA_ERR_INVALID_ARG),
    (dict(io=3), ST.KDA_ERR_INVALID_ARG),
    (dict(N=1 << 15, H=1 << 15), ST.KDA_ERR_INVALID_ARG),  # 2 N H blocks >= 2^31
])
def test_decode_rejects(L, kw, code):
    assert call_dec(L, **kw) == code


def call_multi(L, q=A[0], k=A[1], v=A[2], g=A[3], beta=A[4], S=A[5], o=A[6], ntok=None, N=2,
               K=4, H=1, dk=128, dv=128, io=kda.KDA_BF16, commit=0):
    return L.kda_decode_multi(q, k, v, g, beta, S, o, ntok, N, K, H, dk, dv, io, commit, None,
                              None)


@pytest.mark.parametrize("kw,code", [
    (dict(K=-1), ST.KDA_ERR_INVALID_ARG),
    (dict(o=None), ST.KDA_ERR_INVALID_ARG),          # verify needs o
    (dict(dk=128, dv=64), ST.KDA_ERR_UNSUPPORTED),
    (dict(ntok=A[7] + 2), ST.KDA_ERR_INVALID_ARG),   # misaligned ntok
    (dict(S=A[2]), ST.KDA_ERR_INVALID_ARG),          # S aliases v
    (dict(q=None), ST.KDA_ERR_INVALID_ARG),
])
def test_decode_multi_rejects(L, kw, code):
    assert call_multi(L, **kw) == code


def test_decode_multi_empty_is_a_no_op(L):
    assert call_multi(L, K=0, q=None) == ST.KDA_OK


def call_ckpt(L, ckpt=A[7], every=128, T=256, **kw):
    a = dict(q=A[0], k=A[1], v=A[2], g=A[3], beta=A[4], h0=None, o=A[5], hT=A[6], B=1, H=1,
             dk=128, dv=128, io=kda.KDA_BF16)
    a.update(kw)
    return L.kda_chunk_fwd_ckpt(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], a["o"],
                                a["hT"], ckpt, every, a["B"], T, a["H"], a["dk"], a["dv"],
                                a["io"], None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(ckpt=None), ST.KDA_ERR_INVALID_ARG),
    (dict(every=100), ST.KDA_ERR_INVALID_ARG),     # not a multiple of the chunk
    (dict(every=0), ST.KDA_ERR_INVALID_ARG),
    (dict(ckpt=A[7] + 4), ST.KDA_ERR_INVALID_ARG),  # misaligned
    (dict(ckpt=A[2]), ST.KDA_ERR_INVALID_ARG),      # overlaps v
])
def test_chunk_fwd_ckpt_rejects(L, kw, code):
    assert call_ckpt(L, **kw) == code


def test_segmented_workspace_size(L):
    sz = ctypes.c_size_t(-1).value
    f = L.kda_chunk_fwd_segmented_workspace_size
    f.restype = ctypes.c_size_t
    per = 128 * 128 * 4
    assert f(1, 4096, 32, 128, 128, kda.KDA_BF16, 5) == 32 * 13 * per  # 64 chunks -> 5 x 13
    assert f(2, 640, 3, 128, 128, kda.KDA_BF16, 10) == 6 * 28 * per    # one chunk each
    assert f(1, 1000, 2, 128, 128, kda.KDA_BF16, 7) == 2 * 16 * per    # 16 chunks -> 6 x 3
    assert f(1, 4096, 32, 128, 128, kda.KDA_BF16, 1) == 0
    assert f(1, 64, 1, 128, 128, kda.KDA_BF16, 1) == 0
    # nseg = 0 (planned on the device): states for min(32, chunks) segments, then
    # 16 x B x H probe floats (16-byte multiple) and a 16-byte plan
    assert f(1, 4096, 32, 128, 128, kda.KDA_BF16, 0) == 32 * 94 * per + 16 * 32 * 4 + 16
    assert f(3, 1000, 1, 128, 128, kda.KDA_BF16, 0) == 3 * 46 * per + 48 * 4 + 16   # 16 chunks
    assert f(1, 65, 5, 128, 128, kda.KDA_BF16, 0) == 5 * 4 * per + 80 * 4 + 16      # 2 chunks
    assert f(1, 64, 5, 128, 128, kda.KDA_BF16, 0) == 0   # one chunk: no split
    assert f(1, 4096, 32, 128, 128, kda.KDA_F32, 0) == sz
    assert f(1, 4096, 32, 128, 128, kda.KDA_BF16, 65) == sz             # more segments than chunks
    assert f(1, 4096, 32, 128, 128, kda.KDA_F32, 2) == sz               # no segmented fp32 path
    assert f(1, 4096, 32, 64, 64, kda.KDA_BF16, 2) == sz
    assert f(-1, 4096, 32, 128, 128, kda.KDA_BF16, 2) == sz


def test_segments_hint(L):
    n = L.kda_chunk_fwd_segments_hint(1, 1 << 20, 32, 128, 128, kda.KDA_BF16)
    assert 1 <= n <= 32  # 1 without a visible GPU
    assert L.kda_chunk_fwd_segments_hint(1, 4096, 32, 128, 128, kda.KDA_F32) == 1
    assert L.kda_chunk_fwd_segments_hint(1, 4096, 32, 96, 96, kda.KDA_BF16) == -1
    assert L.kda_chunk_fwd_segments_hint(-1, 4096, 32, 128, 128, kda.KDA_BF16) == -1


def test_segment_plan(L):
    f = L.kda_chunk_fwd_segment_plan
    f.restype = ctypes.c_int
    sc, lead = ctypes.c_int(0), ctypes.c_int(0)

    def plan(B, T, H, nseg, dk=128, io=kda.KDA_BF16, lead_in=0):
        return f(B, T, H, dk, dk, io, nseg, lead_in, ctypes.byref(sc), ctypes.byref(lead))

    # covers the chunks with the workspace's segment count, whatever the lead
    for B, T, H, nseg in ((1, 1 << 20, 32, 10), (1, 1000, 2, 7), (1, 2048, 32, 8), (2, 640, 3, 10)):
        n = plan(B, T, H, nseg)
        nch = (T + 63) // 64
        even = -(-nch // nseg)
        assert n == -(-nch // even)  # non-empty segments of the even split
        assert lead.value >= 1 and (lead.value + n - 1) * sc.value >= nch
        assert (lead.value + n - 2) * sc.value < nch  # the last segment is not empty
        ws = L.kda_chunk_fwd_segmented_workspace_size
        ws.restype = ctypes.c_size_t
        assert ws(B, T, H, 128, 128, kda.KDA_BF16, nseg) == B * H * (3 * n - 2) * 128 * 128 * 4
    assert plan(1, 4096, 32, 1) == 1 and sc.value == 64 and lead.value == 1
    assert plan(1, 0, 32, 3) == 1
    assert plan(1, 4096, 32, 0) == -1
    assert plan(1, 4096, 32, 65) == -1  # more segments than chunks
    assert plan(1, 4096, 32, 2, io=kda.KDA_F32) == -1
    assert plan(1, 4096, 32, 2, dk=64) == -1
    assert plan(-1, 4096, 32, 2) == -1
    assert f(1, 4096, 32, 128, 128, kda.KDA_BF16, 4, 0, None, None) == 4  # outputs optional
    # an explicit lead: the first segment spans lead segment lengths
    assert plan(1, 1 << 20, 32, 16, lead_in=4) == 16 and lead.value == 4 and sc.value == 863
    assert plan(1, 1 << 20, 32, 8, lead_in=2) == 8 and (lead.value, sc.value) == (2, 1821)
    assert plan(1, 4096, 32, 16, lead_in=4) == 13 and (lead.value, sc.value) == (4, 4)
    assert plan(1, 4096, 32, 2, lead_in=64) == 1  # the first segment covers everything
    assert plan(1, 4096, 32, 2, lead_in=65) == -1  # longer than the sequence
    assert plan(1, 4096, 32, 0) == -1  # planned on the device


def test_segments_hint_decay(L):
    f = L.kda_chunk_fwd_segments_hint_decay
    f.argtypes = [ctypes.c_int] * 6 + [ctypes.POINTER(ctypes.c_float), ctypes.c_int,
                                       ctypes.POINTER(ctypes.c_int)]
    probe = (ctypes.c_float * 3)(-30.0, -25.0, -40.0)
    lead = ctypes.c_int(7)
    n = f(1, 1 << 20, 32, 128, 128, kda.KDA_BF16, probe, 3, ctypes.byref(lead))
    assert 1 <= n <= 32 and lead.value >= 1  # 1 and 1 without a visible GPU
    assert f(1, 4096, 32, 128, 128, kda.KDA_F32, probe, 3, ctypes.byref(lead)) == 1
    assert lead.value == 1
    assert f(1, 4096, 32, 96, 96, kda.KDA_BF16, probe, 3, None) == -1
    assert f(-1, 4096, 32, 128, 128, kda.KDA_BF16, probe, 3, None) == -1
    assert f(1, 4096, 32, 128, 128, kda.KDA_BF16, None, 3, None) == -1   # no probe
    assert f(1, 4096, 32, 128, 128, kda.KDA_BF16, probe, -1, None) == -1
    assert f(1, 4096, 32, 128, 128, kda.KDA_BF16, None, 0, None) >= 1    # empty sample


def call_probe(L, g=A[3], B=1, T=128, H=1, dk=128, nsample=4, out=A[6]):
    L.kda_chunk_fwd_decay_probe.argtypes = [ctypes.c_void_p] + [ctypes.c_int] * 5 + \
        [ctypes.c_void_p, ctypes.c_void_p]
    return L.kda_chunk_fwd_decay_probe(g, B, T, H, dk, nsample, out, None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=-1), ST.KDA_ERR_INVALID_ARG),
    (dict(dk=96), ST.KDA_ERR_UNSUPPORTED),
    (dict(nsample=0), ST.KDA_ERR_INVALID_ARG),
    (dict(nsample=4097), ST.KDA_ERR_INVALID_ARG),
    (dict(B=65536), ST.KDA_ERR_INVALID_ARG),
    (dict(g=None), ST.KDA_ERR_INVALID_ARG),
    (dict(out=None), ST.KDA_ERR_INVALID_ARG),
    (dict(g=A[3] + 2), ST.KDA_ERR_INVALID_ARG),   # misaligned
    (dict(g=A[3] + 4), ST.KDA_ERR_INVALID_ARG),   # g not 16-byte aligned
    (dict(H=8 * 65535 + 1, T=1, B=1), ST.KDA_ERR_INVALID_ARG),
    (dict(out=A[3] + 64), ST.KDA_ERR_INVALID_ARG),  # inside g
    (dict(B=0), ST.KDA_OK),                        # nothing to do: no launch
    (dict(T=0), ST.KDA_OK),
])
def test_decay_probe_rejects(L, kw, code):
    assert call_probe(L, **kw) == code


def call_seg(L, nseg=2, ws=None, ws_bytes=0, T=128, dk=128, io=kda.KDA_BF16, q=A[0], lead=0):
    # T = 128: two chunks; every tensor fits the 64 KB spacing of the fake addresses
    return L.kda_chunk_fwd_segmented(q, A[1], A[2], A[3], A[4], None, A[5], A[6], 1, T, 1, dk,
                                     dk, io, nseg, lead, ws, ws_bytes, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(nseg=3), ST.KDA_ERR_INVALID_ARG),                       # 2 chunks
    (dict(io=kda.KDA_F32), ST.KDA_ERR_UNSUPPORTED),
    (dict(dk=64), ST.KDA_ERR_UNSUPPORTED),
    (dict(ws=None, ws_bytes=0), ST.KDA_ERR_WORKSPACE),
    (dict(ws=A[7], ws_bytes=1024), ST.KDA_ERR_WORKSPACE),         # short
    (dict(ws=A[7] + 8, ws_bytes=1 << 22), ST.KDA_ERR_INVALID_ARG),  # misaligned
    (dict(ws=A[0], ws_bytes=1 << 22), ST.KDA_ERR_INVALID_ARG),    # overlaps q
    (dict(q=None), ST.KDA_ERR_INVALID_ARG),
    (dict(lead=3), ST.KDA_ERR_INVALID_ARG),                       # longer than the 2 chunks
    (dict(nseg=0, lead=1), ST.KDA_ERR_INVALID_ARG),               # a device plan takes no lead
    (dict(nseg=0, ws=None, ws_bytes=0), ST.KDA_ERR_WORKSPACE),
    (dict(nseg=-1), ST.KDA_ERR_INVALID_ARG),
])
def test_segmented_rejects(L, kw, code):
    assert call_seg(L, **kw) == code


@pytest.mark.parametrize("clocks,status", [(0, A[0]), ((1 << 31) + 1, A[0]), (1000, None),
                                           (1000, A[0] + 2)])
def test_selftest_wait_rejects(L, clocks, status):
    L.kda_selftest_wait_timeout.argtypes = [ctypes.c_longlong, ctypes.c_void_p, ctypes.c_void_p]
    assert L.kda_selftest_wait_timeout(clocks, status, None) == ST.KDA_ERR_INVALID_ARG
