"""Host-side checks of the C-ABI library (no GPU needed).

The library must build for sm_103a, load, export every function declared in
include/mxs.h, and reject bad arguments on the host before any launch.
"""
import ctypes

import pytest

import mxfp4_speculative_verification_gb300 as mxs


@pytest.fixture(scope="module")
def L():
    mxs.build()
    return mxs.lib()


def test_every_declared_symbol_is_exported(L):
    names = mxs.declared_symbols()
    assert {"mxfp4_pack", "mxfp4_verify_gemm", "spec_accept",
            "mxfp4_verify_gemm_workspace_size"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_version_and_status_strings(L):
    assert L.mxs_version() == 100
    assert L.mxs_status_string(0) == b"MXS_OK"
    assert L.mxs_status_string(5) == b"MXS_ERR_WORKSPACE"
    assert L.mxs_status_string(99) == b"MXS_ERR_UNKNOWN"


def test_workspace_size_rules(L):
    assert L.mxfp4_verify_gemm_workspace_size(5, 4096, 4096) > 0
    assert L.mxfp4_verify_gemm_workspace_size(0, 4096, 4096) == 0
    assert L.mxfp4_verify_gemm_workspace_size(5, 4096, 4100) == 0  # K % 32
    # K % 512 != 0 adds room for realigned scale rows
    a = L.mxfp4_verify_gemm_workspace_size(5, 1000, 544)
    b = L.mxfp4_verify_gemm_workspace_size(5, 1000, 512)
    assert a >= b + 1000 * 32


FAKE = 0x100000  # never dereferenced: validation fails first


def test_gemm_rejects_bad_arguments_on_host(L):
    ws = 1 << 30
    f = L.mxfp4_verify_gemm
    assert f(None, FAKE, FAKE, FAKE, 5, 64, 512, FAKE, ws, None, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, 0, 64, 512, FAKE, ws, None, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, 5, 64, 500, FAKE, ws, None, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, 1 << 20, 64, 512, FAKE, ws, None, None) == 3
    assert f(FAKE, FAKE + 8, FAKE, FAKE, 5, 64, 512, FAKE, ws, None, None) == 2   # nibbles 16B
    assert f(FAKE, FAKE, FAKE + 1, FAKE, 5, 64, 512, FAKE, ws, None, None) == 2   # scales, K%512==0
    assert f(FAKE, FAKE, FAKE, FAKE, 5, 64, 512, None, ws, None, None) == 5
    assert f(FAKE, FAKE, FAKE, FAKE, 5, 64, 512, FAKE, 16, None, None) == 5


def test_w4a4_gemm_rules_on_host(L):
    assert L.mxfp4_verify_gemm_w4a4_workspace_size(5, 4096, 4096) > 0
    assert L.mxfp4_verify_gemm_w4a4_workspace_size(0, 4096, 4096) == 0
    assert L.mxfp4_verify_gemm_w4a4_workspace_size(5, 4096, 4100) == 0  # K % 32
    # passes of up to 256 rows: the quantised X of one pass, whatever M
    assert (L.mxfp4_verify_gemm_w4a4_workspace_size(256, 4096, 4096)
            == L.mxfp4_verify_gemm_w4a4_workspace_size(1000, 4096, 4096))
    assert (L.mxfp4_verify_gemm_w4a4_workspace_size(16, 4096, 4096)
            < L.mxfp4_verify_gemm_w4a4_workspace_size(256, 4096, 4096))
    a = L.mxfp4_verify_gemm_w4a4_workspace_size(80, 1000, 544)
    b = L.mxfp4_verify_gemm_w4a4_workspace_size(80, 1000, 512)
    assert a >= b + 1000 * 32  # realigned scale rows
    ws = 1 << 30
    f = L.mxfp4_verify_gemm_w4a4
    assert f(None, FAKE, FAKE, FAKE, 5, 64, 512, FAKE, ws, None, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, 0, 64, 512, FAKE, ws, None, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, 5, 64, 500, FAKE, ws, None, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, 1 << 20, 64, 512, FAKE, ws, None, None) == 3
    assert f(FAKE + 1, FAKE, FAKE, FAKE, 5, 64, 512, FAKE, ws, None, None) == 2   # x 2B
    assert f(FAKE, FAKE + 8, FAKE, FAKE, 5, 64, 512, FAKE, ws, None, None) == 2   # nibbles 16B
    assert f(FAKE, FAKE, FAKE + 1, FAKE, 5, 64, 512, FAKE, ws, None, None) == 2   # scales, K%512==0
    assert f(FAKE, FAKE, FAKE, FAKE, 5, 64, 512, None, ws, None, None) == 5
    assert f(FAKE, FAKE, FAKE, FAKE, 5, 64, 512, FAKE, 16, None, None) == 5
    assert f(FAKE, FAKE, FAKE, FAKE, 5, 64, 512, FAKE + 8, ws, None, None) == 2   # workspace 16B


def test_nvfp4_gemm_rules_on_host(L):
    assert L.nvfp4_verify_gemm_workspace_size(5, 4096, 4096) > 0
    assert L.nvfp4_verify_gemm_workspace_size(5, 4096, 4100) == 0  # K % 32
    # scale rows are realigned unless K % 256 == 0 (K/16 bytes a multiple of 16)
    a = L.nvfp4_verify_gemm_workspace_size(5, 1000, 288)
    b = L.nvfp4_verify_gemm_workspace_size(5, 1000, 256)
    assert a >= b + 1000 * 32
    ws = 1 << 30
    f = L.nvfp4_verify_gemm
    assert f(None, FAKE, FAKE, 1.0, FAKE, 5, 64, 512, FAKE, ws, None, None) == 1
    assert f(FAKE, FAKE, FAKE, 1.0, FAKE, 5, 64, 496, FAKE, ws, None, None) == 1   # K % 32
    assert f(FAKE, FAKE, FAKE, 1.0, FAKE, 1 << 20, 64, 512, FAKE, ws, None, None) == 3
    assert f(FAKE, FAKE + 8, FAKE, 1.0, FAKE, 5, 64, 512, FAKE, ws, None, None) == 2
    assert f(FAKE, FAKE, FAKE + 4, 1.0, FAKE, 5, 64, 256, FAKE, ws, None, None) == 2   # scales, K%256==0
    assert f(FAKE, FAKE, FAKE, 1.0, FAKE, 5, 64, 512, FAKE, 16, None, None) == 5


def test_kv_cache_calls_reject_bad_arguments_on_host(L):
    f = L.mxfp4_kv_append
    assert f(FAKE, 2, 2, 5, 1024, FAKE, FAKE, 64, FAKE, None, None) == 1           # dtype
    assert f(FAKE, 0, 2, 5, 1000, FAKE, FAKE, 64, FAKE, None, None) == 1           # W % 32
    assert f(FAKE, 0, 2, 5, 1024, FAKE, FAKE, 0, FAKE, None, None) == 1            # L
    assert f(FAKE, 0, -1, 5, 1024, FAKE, FAKE, 64, FAKE, None, None) == 1
    assert f(FAKE, 0, 2, 0, 1024, None, None, 64, None, None, None) == 0           # nothing to append
    assert f(None, 0, 2, 5, 1024, FAKE, FAKE, 64, FAKE, None, None) == 1
    assert f(FAKE + 4, 0, 2, 5, 1024, FAKE, FAKE, 64, FAKE, None, None) == 2       # kv 16 B
    assert f(FAKE, 0, 2, 5, 1024, FAKE, FAKE, 64, FAKE + 2, None, None) == 2       # lens 4 B
    g = L.spec_kv_commit
    assert g(FAKE, FAKE, 4, 0, None) == 1 and g(None, FAKE, 4, 64, None) == 1 and g(FAKE + 1, FAKE, 4, 64, None) == 2
    assert g(None, None, 0, 64, None) == 0
    h = L.mxfp4_kv_dequant
    assert h(FAKE, FAKE, 2, 64, 100, FAKE, FAKE, None) == 1                        # W % 32
    assert h(FAKE, FAKE, 2, 64, 1024, FAKE, None, None) == 1
    assert h(FAKE, FAKE, 2, 64, 1024, FAKE, FAKE + 4, None) == 2                   # out 16 B
    assert h(FAKE, FAKE, 1 << 20, 1 << 20, 1024, FAKE, FAKE, None) == 1            # size limit


def test_accept_rejects_bad_arguments_on_host(L):
    f = L.spec_accept
    assert f(FAKE, FAKE, FAKE, FAKE, 0, 3, 8, FAKE, FAKE, None, None, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, 1, 33, 8, FAKE, FAKE, None, None, None) == 3
    assert f(FAKE, FAKE, FAKE, FAKE, 1, 3, (1 << 21) + 1, FAKE, FAKE, None, None, None) == 3
    assert f(FAKE, None, FAKE, FAKE, 1, 3, 8, FAKE, FAKE, None, None, None) == 1
    assert f(FAKE + 2, FAKE, FAKE, FAKE, 1, 3, 8, FAKE, FAKE, None, None, None) == 2


def test_pack_rejects_bad_arguments_on_host(L):
    f = L.mxfp4_pack
    assert f(FAKE, 0, 4, 33, FAKE, FAKE, None, None) == 1
    assert f(FAKE, 7, 4, 32, FAKE, FAKE, None, None) == 1
    assert f(FAKE + 2, 0, 4, 32, FAKE, FAKE, None, None) == 2
    assert f(None, 0, 0, 32, None, None, None, None) == 0  # empty: nothing to do


def test_grouped_rejects_bad_arguments_on_host(L):
    import mxfp4_speculative_verification_gb300 as m
    arr = (m.GemmProblem * 2)()
    arr[0] = m.GemmProblem(FAKE, FAKE, FAKE, FAKE, 64, 512)
    arr[1] = m.GemmProblem(FAKE, FAKE, FAKE, FAKE, 64, 4096)
    f = L.mxfp4_verify_gemm_grouped
    assert L.mxfp4_verify_gemm_grouped_workspace_size(arr, 2, 5) > 0
    assert f(None, 2, 5, FAKE, 1 << 30, None, None) == 1
    assert f(arr, 0, 5, FAKE, 1 << 30, None, None) == 1
    assert f(arr, 2, 65537, FAKE, 1 << 30, None, None) == 3
    assert f(arr, 2, 5, FAKE, 16, None, None) == 5
    arr[1] = m.GemmProblem(FAKE, FAKE, FAKE, FAKE, 64, 544)   # K % 512 != 0
    assert f(arr, 2, 5, FAKE, 1 << 30, None, None) == 3
    arr[1] = m.GemmProblem(FAKE, FAKE + 4, FAKE, FAKE, 64, 512)  # nibbles not 16-byte aligned
    assert f(arr, 2, 5, FAKE, 1 << 30, None, None) == 2


def test_grouped_w4a4_rules_on_host(L):
    P = mxs.GemmProblem
    arr = (P * 2)(P(FAKE, FAKE, FAKE, FAKE, 4096, 4096), P(FAKE, FAKE, FAKE, FAKE, 1000, 4096))
    a = L.mxfp4_verify_gemm_grouped_w4a4_workspace_size(arr, 2, 80)
    assert a > 0
    # one quantised X (both problems share x) of a pass of up to 256 rows
    assert a < L.mxfp4_verify_gemm_grouped_w4a4_workspace_size(arr, 2, 256)
    assert (L.mxfp4_verify_gemm_grouped_w4a4_workspace_size(arr, 2, 256)
            == L.mxfp4_verify_gemm_grouped_w4a4_workspace_size(arr, 2, 1000))
    f = L.mxfp4_verify_gemm_grouped_w4a4
    assert f(arr, 2, 80, None, 1 << 30, None, None) == 5
    assert f(arr, 2, 80, FAKE, 16, None, None) == 5
    assert f(arr, 0, 80, FAKE, 1 << 30, None, None) == 1
    bad = (P * 1)(P(FAKE, FAKE, FAKE, FAKE, 1000, 4000))
    assert f(bad, 1, 80, FAKE, 1 << 30, None, None) == 3  # grouped: K % 512
    bad = (P * 1)(P(FAKE, FAKE, FAKE, FAKE, 1000, 4001))
    assert f(bad, 1, 80, FAKE, 1 << 30, None, None) == 1  # K % 32


def test_grouped_workspace_layout(L):
    # problems sharing one X: the X space is counted once (16 rows of fp16 for a
    # 5-row pass, the wider of the two kernels' layouts, plus 64 unscale
    # factors), then one int claim counter per launch of up to 84 GEMMs, each
    # area rounded up to 256 bytes (4096 problems need 49 counters: one unit)
    import mxfp4_speculative_verification_gb300 as m

    def size(count, K=4096):
        arr = (m.GemmProblem * count)()
        for i in range(count):
            arr[i] = m.GemmProblem(FAKE, FAKE, FAKE, FAKE, 64, K)
        return L.mxfp4_verify_gemm_grouped_workspace_size(arr, count, 5)

    assert size(1) == 16 * 4096 * 2 + 256 + 256
    assert size(1) == size(84) == size(85) == size(4096)
    assert size(1, K=14336) == 16 * 14336 * 2 + 256 + 256


def test_hbm_probes_reject_bad_arguments_on_host(L):
    import ctypes
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    L.mxs_hbm_copy_probe.argtypes = [vp, vp, sz, vp]
    L.mxs_hbm_read_probe.argtypes = [vp, sz, vp, vp]
    copy, read = L.mxs_hbm_copy_probe, L.mxs_hbm_read_probe
    assert copy(FAKE, FAKE + (1 << 20), 0, None) == 1          # no bytes
    assert copy(FAKE, FAKE + (1 << 20), 1000, None) == 1       # not a multiple of 16
    assert copy(None, FAKE, 4096, None) == 1
    assert copy(FAKE + 8, FAKE + (1 << 20), 4096, None) == 2   # misaligned destination
    assert copy(FAKE, FAKE + 2048, 4096, None) == 1            # overlapping buffers
    assert read(FAKE, 0, FAKE, None) == 1
    assert read(FAKE + 4, 4096, FAKE, None) == 2


def test_law_calls_reject_bad_arguments_on_host(L):
    # fake, never-dereferenced device pointers: every case fails validation first
    p = ctypes.c_void_p(4096)
    s = mxs._Sampling(1.0, 0, 1.0)
    ok = ctypes.addressof(s)
    assert L.spec_sampling_law(p, 4, 1000, ok, None, None, None) == 1  # no output
    for bad in (mxs._Sampling(0.0, 0, 1.0), mxs._Sampling(1.0, -1, 1.0), mxs._Sampling(1.0, 0, 0.0),
                mxs._Sampling(1.0, 0, 1.5), mxs._Sampling(float("inf"), 0, 1.0)):
        assert L.spec_sampling_law(p, 4, 1000, ctypes.addressof(bad), p, None, None) == 1
    assert L.spec_sampling_law(p, 4, 131073, ok, p, None, None) == 3  # beyond one cluster per row
    assert L.spec_sampling_law(ctypes.c_void_p(4098), 4, 1000, ok, p, None, None) == 2
    assert L.spec_accept_logits_workspace_size(2, 4) == 2 * 9 * 16
    assert L.spec_accept_logits_workspace_size(0, 4) == 0
    ws = L.spec_accept_logits_workspace_size(2, 4)
    args = lambda **k: [k.get("tl", p), k.get("dl", p), k.get("d", p), k.get("u", p), k.get("B", 2), k.get("K", 4),
                        k.get("V", 1000), k.get("s", ok), k.get("ws", p), k.get("wsb", ws), p, p, None, None, None]
    assert L.spec_accept_logits(*args(wsb=ws - 1)) == 5
    assert L.spec_accept_logits(*args(ws=None)) == 5
    assert L.spec_accept_logits(*args(K=33)) == 3
    assert L.spec_accept_logits(*args(V=200000)) == 3
    assert L.spec_accept_logits(*args(dl=None)) == 1
    assert L.spec_accept_logits(*args(ws=ctypes.c_void_p(4104))) == 2
