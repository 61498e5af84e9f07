"""Host-side tests of the C ABI: the library loads, exports every declared symbol, plans
layouts like the oracle's flat layout, and validates arguments before touching a GPU.
No kernel is launched here."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import muon_ref as ref
from muon_optimizer_step_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "muon.h")

capi = pytest.importorskip("muon_optimizer_step_gb300.capi",
                           reason="libmuon.so not built (run __graft_entry__.build())")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(muon_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = declared_symbols()
    assert len(names) >= 18
    for n in names:
        assert hasattr(capi.lib, n), n
    bound = {s[0] for s in capi.SIGNATURES}
    assert set(names) == bound


def test_abi_version():
    assert capi.muon_abi_version() == 1


@pytest.mark.parametrize("wl_name,n_shards", [("ragged_small", 1), ("ragged_small", 3),
                                              ("ragged_small", 8), ("llama3_8b_8shards", 8),
                                              ("gpt2_small_x12", 1), ("moe_64e", 5)])
def test_layout_matches_oracle(wl_name, n_shards):
    wl = inputs.WORKLOADS[wl_name]
    lay = capi.muon_layout_create(wl.shapes, n_shards, capi.MUON_NS_BF16, wl.is_matrix)
    o = ref.flat_layout(wl.shapes, n_shards, wl.is_matrix)
    assert lay.numel == o["N"]
    assert lay.shard_len == o["L"]
    # full layout: matrices only, row-major, each start a multiple of 4, no overlap
    prev_end = 0
    for i, (r, c) in enumerate(wl.shapes):
        off = lay.full_offsets[i]
        if not wl.is_matrix[i]:
            assert off == -1
            continue
        assert off % 4 == 0 and off >= prev_end
        prev_end = off + r * c
    assert lay.full_numel == prev_end
    assert lay.workspace_bytes > 0
    lay.close()


def test_workspace_bytes_cover_buffers():
    # bf16: X ping-pong (2 * r * ldx * 2 B) + A and B (2 * m * lda * 2 B) per matrix.
    lay = capi.muon_layout_create([(256, 128)], 1, capi.MUON_NS_BF16)
    assert lay.workspace_bytes >= 2 * 256 * 128 * 2 + 2 * 128 * 128 * 2
    lay32 = capi.muon_layout_create([(256, 128)], 1, capi.MUON_NS_FP32)
    assert lay32.workspace_bytes >= 2 * 256 * 128 * 4 + 2 * 128 * 128 * 4
    # split fp32: every buffer as three bf16 parts (h, m, l)
    lay3 = capi.muon_layout_create([(256, 128)], 1, capi.MUON_NS_SPLIT_FP32)
    assert lay3.workspace_bytes >= 3 * (2 * 256 * 128 * 2 + 2 * 128 * 128 * 2)
    assert lay3.workspace_bytes - lay.workspace_bytes == 2 * (2 * 256 * 128 * 2 + 2 * 128 * 128 * 2)


@pytest.mark.parametrize("shapes,n_shards,dtype,flags", [
    ([(0, 5)], 1, 0, None),          # zero rows
    ([(5, -1)], 1, 0, None),         # negative
    ([(4, 4)], 0, 0, None),          # no shards
    ([(4, 4)], 129, 0, None),        # too many shards
    ([(4, 4)], 1, 3, None),          # unknown dtype
    ([(70000, 70000)], 1, 0, None),  # > 2^31 - 1 elements in one matrix
])
def test_layout_rejects_bad_arguments(shapes, n_shards, dtype, flags):
    with pytest.raises(capi.MuonError) as e:
        capi.muon_layout_create(shapes, n_shards, dtype, flags)
    assert e.value.status == capi.MUON_ERR_INVALID_ARG
    assert capi.muon_last_error()


def test_non_matrix_zero_length_and_empty_layouts_are_accepted():
    lay = capi.muon_layout_create([(0, 1), (3, 4)], 2, 0, [False, True])
    assert lay.numel == 12 and lay.shard_len == 6
    empty = capi.muon_layout_create([], 4, 0)
    assert empty.numel == 0 and empty.shard_len == 0 and empty.full_numel == 0


def test_step_validates_before_any_launch():
    lay = capi.muon_layout_create([(8, 8)], 2, 0)
    null2 = (ctypes.c_void_p * 2)(None, None)
    st = capi.lib.muon_step(null2, null2, null2, lay.handle, None, 0.02, 0.01, 0.95, 1, 5, None)
    assert st == capi.MUON_ERR_INVALID_ARG
    odd = (ctypes.c_void_p * 2)(0x1004, 0x2000)
    ok = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    st = capi.lib.muon_step(odd, ok, ok, lay.handle, ctypes.c_void_p(0x10000), 0.02, 0.01, 0.95, 1,
                            5, None)
    assert st == capi.MUON_ERR_ALIGNMENT
    st = capi.lib.muon_step(ok, ok, ok, lay.handle, ctypes.c_void_p(0x10010), 0.02, 0.01, 0.95, 1,
                            5, None)
    assert st == capi.MUON_ERR_ALIGNMENT
    st = capi.lib.muon_step(ok, ok, ok, lay.handle, ctypes.c_void_p(0x10000), 0.02, 0.01, 0.95, 1,
                            101, None)
    assert st == capi.MUON_ERR_INVALID_ARG
    st = capi.lib.muon_step(ok, ok, ok, lay.handle, ctypes.c_void_p(0x10000), float("nan"), 0.01,
                            0.95, 1, 5, None)
    assert st == capi.MUON_ERR_INVALID_ARG
    st = capi.lib.muon_step(ok, ok, ok, None, ctypes.c_void_p(0x10000), 0.02, 0.01, 0.95, 1, 5,
                            None)
    assert st == capi.MUON_ERR_INVALID_ARG
    assert capi.lib.muon_selftest_wait_timeout(0, None) == capi.MUON_ERR_INVALID_ARG


def test_set_groups_validation_on_host():
    lay = capi.muon_layout_create([(4, 4), (3, 1)], 1, 0, [True, False])
    with pytest.raises(capi.MuonError):
        capi.muon_layout_set_groups(lay, [2, 0], 2)
    capi.muon_layout_set_groups(lay, [1, 99], 2)  # non-matrix entry is ignored
    with pytest.raises(capi.MuonError):
        capi.muon_layout_set_groups(lay, [0, 0], 33)
    with pytest.raises(capi.MuonError):
        capi.muon_layout_set_groups(lay, [0, 0], 0)


def test_header_constants_match_the_binding():
    """Every enum value and #define of the C header has the same value in the binding."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    consts = {}
    for name, val in re.findall(r"\b(MUON_[A-Z0-9_]+)\s*=\s*(\d+)", text):
        consts[name] = int(val)
    for name, val in re.findall(r"#define\s+(MUON_[A-Z0-9_]+)\s+(\d+)", text):
        consts[name] = int(val)
    assert {"MUON_OK", "MUON_ERR_UNSUPPORTED", "MUON_NS_SPLIT_FP32", "MUON_MAX_SHARDS"} <= set(consts)
    for name, val in consts.items():
        if name == "MUON_ABI_VERSION":
            assert capi.muon_abi_version() == val
        else:
            assert getattr(capi, name) == val, name


def test_debug_build_links_and_exports_the_same_symbols(tmp_path):
    """The debug build (-DMUON_DEBUG) compiles, exports every declared symbol and says it
    is a debug build; the release library says it is not.  No kernel runs."""
    import subprocess
    import sys
    from muon_optimizer_step_gb300.csrc import build
    lib = build.build(debug=True)
    names = declared_symbols()
    code = ("import ctypes, sys\n"
            f"lib = ctypes.CDLL({lib!r})\n"
            f"missing = [n for n in {names!r} if not hasattr(lib, n)]\n"
            "assert not missing, missing\n"
            "lib.muon_debug_build.restype = ctypes.c_int32\n"
            "assert lib.muon_debug_build() == 1\n"
            "print('ok')\n")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr
    assert not capi.muon_debug_build()
