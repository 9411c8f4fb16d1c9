"""Host-side checks of the C ABI (no GPU needed).

The library is cross-compiled here for sm_103a; these tests check that it
loads, exports every function include/slm_attn.h declares, answers the
workspace-size queries, and rejects bad arguments on the host before any
device work is enqueued.
"""
import ctypes
import os
import re

import pytest

from attention_packed_varlen_gb300 import _binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "slm_attn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(slm_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("slm_packed_prefill_attn", "slm_shared_prefix_decode_attn", "slm_beam_select"):
        assert required in names
    assert set(names) == set(_binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"
    assert lib.slm_abi_version() == 2
    assert lib.slm_last_error() == b""


def test_workspace_size_queries(lib):
    # one int32 count plus (start, length, pair of 64-token tiles) items,
    # rounded to 256 bytes
    n = _binding.slm_prefill_workspace_size(240, 130560, 1024, 16, 8)
    assert n > 0 and n % 256 == 0
    assert n >= 4 * (1 + 3 * (130560 // 128 + 240))
    assert _binding.slm_prefill_workspace_size(4, 320, 128, 4, 3) == 0      # Hq % Hkv != 0
    assert _binding.slm_beam_select_workspace_size(100, 151936, 100) > 0
    assert _binding.slm_beam_select_workspace_size(400, 151936, 400) > 0
    assert _binding.slm_beam_select_workspace_size(1, 151936, 400) > 0
    assert _binding.slm_beam_select_workspace_size(4, 10, 6) == 0           # 2W > V
    # decode key split: nothing to split in one key block of 128 rows
    assert _binding.slm_shared_prefix_decode_workspace_size(100, 96, 14, 2, 64) == 0
    assert _binding.slm_shared_prefix_decode_workspace_size(100, 128, 14, 2, 64) == 0
    assert _binding.slm_shared_prefix_decode_workspace_size(100, 1024, 14, 13, 64) == 0  # Hq % Hkv != 0
    assert _binding.slm_shared_prefix_decode_workspace_size(100, 1024, 14, 2, 80) == 0   # head_dim
    # W=400, Lp=1024, 14q/2kv, D=64: up to 8 splits x 48 sub-tiles x 128 rows x (64 fp32 + (max, sum))
    n = _binding.slm_shared_prefix_decode_workspace_size(400, 1024, 14, 2, 64)
    assert n >= 8 * 48 * 128 * (64 * 4 + 8) + 48 * 4 and n % 256 == 0
    # more key blocks or more beams never need less
    assert _binding.slm_shared_prefix_decode_workspace_size(400, 2048, 14, 2, 64) >= n
    assert _binding.slm_shared_prefix_decode_workspace_size(800, 1024, 14, 2, 64) >= n


NULL = None


def _prefill(lib, **kw):
    args = dict(q=ctypes.c_void_p(16), k=ctypes.c_void_p(16), v=ctypes.c_void_p(16), cu=ctypes.c_void_p(16),
                cu_host=NULL, B=1, T=8, max_seqlen=8, hq=4, hkv=2, d=64, scale=0.125, o=ctypes.c_void_p(32),
                lse=NULL, ws=ctypes.c_void_p(64), ws_bytes=1 << 20, status=NULL, stream=NULL)
    args.update(kw)
    return lib.slm_packed_prefill_attn(args["q"], args["k"], args["v"], args["cu"], args["cu_host"], args["B"],
                                       args["T"], args["max_seqlen"], args["hq"], args["hkv"], args["d"],
                                       args["scale"], args["o"], args["lse"], args["ws"], args["ws_bytes"],
                                       args["status"], args["stream"])


def test_prefill_rejects_bad_arguments_on_host(lib):
    assert _prefill(lib, d=96) == 2                                # unsupported head_dim
    assert b"head_dim" in lib.slm_last_error()
    assert _prefill(lib, hkv=3) == 1                               # Hq % Hkv
    assert _prefill(lib, scale=0.0) == 1
    assert _prefill(lib, q=ctypes.c_void_p(8)) == 1                # misaligned
    assert _prefill(lib, o=ctypes.c_void_p(16)) == 1               # o aliases q
    assert _prefill(lib, ws_bytes=4) == 4                          # workspace too small
    assert _prefill(lib, max_seqlen=4095 * 128 + 1) == 2
    bad = (ctypes.c_int32 * 3)(0, 5, 3)                            # host boundary decreases
    assert _prefill(lib, B=2, cu_host=bad) == 1
    short = (ctypes.c_int32 * 2)(0, 7)                             # does not end at T
    assert _prefill(lib, cu_host=short) == 1
    assert _prefill(lib, T=0, B=0, cu_host=(ctypes.c_int32 * 1)(0)) == 0   # nothing to do


def _decode(lib, **kw):
    p = ctypes.c_void_p
    args = dict(q=p(16), kp=p(32), vp=p(48), ks=p(64), vs=p(80), kn=p(96), vn=p(112), parent=NULL, W=4, Lp=8,
                L_prev=1, Smax=3, hq=14, hkv=2, d=64, scale=0.125, ks_out=p(128), vs_out=p(144), o=p(160),
                lse=NULL, status=NULL, ws=NULL, ws_bytes=0, stream=NULL)
    args.update(kw)
    a = args
    return lib.slm_shared_prefix_decode_attn(a["q"], a["kp"], a["vp"], a["ks"], a["vs"], a["kn"], a["vn"],
                                             a["parent"], a["W"], a["Lp"], a["L_prev"], a["Smax"], a["hq"],
                                             a["hkv"], a["d"], a["scale"], a["ks_out"], a["vs_out"], a["o"],
                                             a["lse"], a["status"], a["ws"], a["ws_bytes"], a["stream"])


def test_decode_rejects_bad_arguments_on_host(lib):
    assert _decode(lib, L_prev=3) == 1                 # L_prev + 1 > Smax
    assert _decode(lib, ks_out=ctypes.c_void_p(64)) == 1   # output aliases input suffix
    assert _decode(lib, kn=NULL) == 1                  # k_new without v_new
    assert _decode(lib, Lp=0, L_prev=0, kn=NULL, vn=NULL) == 1   # no keys at all
    assert _decode(lib, d=80) == 2
    assert _decode(lib, hq=13) == 1
    assert _decode(lib, W=0) == 0


def test_select_rejects_bad_arguments_on_host(lib):
    p = ctypes.c_void_p
    call = lambda W_in, V, W, ws_bytes=1 << 30, logits=p(16): lib.slm_beam_select(
        logits, p(32), W_in, V, W, p(48), p(64), p(80), NULL, NULL, NULL, NULL, p(256), ws_bytes, NULL)
    assert call(4, 10, 6) == 1            # 2W > V
    assert call(0, 10, 2) == 1
    assert call(4, 1000, 2, ws_bytes=8) == 4
    assert call(4, 1000, 2, logits=p(18)) == 1
