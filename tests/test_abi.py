"""CPU checks of the C ABI: the library builds for sm_103a, loads, exports
every function include/ep.h declares, and its host-only entry points behave
(argument validation, workspace sizing, rank masks) without a GPU."""
import ctypes
import os
import re

import pytest

import combine_topk_ids_dest_gb300 as ep
from combine_topk_ids_dest_gb300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ep.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ep_[a-z_]+)\s*\(", text)))


def test_header_and_exports_agree():
    decl = declared_functions()
    assert decl == sorted(_lib.EXPORTS)
    L = _lib.load()
    for name in decl:
        assert hasattr(L, name), name


def test_library_is_the_in_tree_build():
    path = _lib.load()._name
    assert os.path.basename(path) == os.path.basename(_lib.lib_path())
    assert os.path.basename(path) in ("libep_gb300.so", "libep_gb300_checked.so")
    assert os.path.dirname(path).endswith(os.path.join("combine_topk_ids_dest_gb300", "_build"))


@pytest.mark.gpu
def test_loaded_kernels_are_sm103a_code(cuda_device):
    """The runtime's own report (cudaFuncGetAttributes.binaryVersion) for every
    kernel of the loaded library: code built for sm_103."""
    import torch
    torch.cuda.set_device(cuda_device)
    v = ctypes.c_int(0)
    L = _lib.load()
    assert L.ep_binary_version(ctypes.byref(v)) == ep.EP_OK, L.ep_last_error()
    assert v.value == 103


def _size(*args):
    n = ctypes.c_size_t(0)
    st = _lib.load().ep_workspace_size(*args, ctypes.byref(n))
    return st, n.value


def _align(x):
    return (x + 255) // 256 * 256


@pytest.mark.parametrize("ep_size,E,K,H,C,dt", [(32, 256, 8, 7168, 1024, 1), (8, 8, 2, 4096, 256, 0),
                                                (2, 8, 2, 256, 16, 0), (3, 6, 3, 136, 5, 0),
                                                (4, 8, 2, 256, 0, 0)])
def test_workspace_size_formula(ep_size, E, K, H, C, dt):
    st, n = _size(ep_size, E, K, H, C, dt)
    assert st == ep.EP_OK
    rows = ep_size * C
    elem = 2 if dt == 0 else 1
    G = H // 128 if H % 128 == 0 else 0
    want = ep_size * (_align(rows * H * elem) + _align(rows * G * 4) + _align(rows * K * 4) * 2 +
                      _align(rows * H * 2)) + _align(rows * 8) + _align(ep_size * 4)
    assert n == max(want, 256)


@pytest.mark.parametrize("args,frag", [
    ((0, 8, 2, 256, 16, 0), "ep_size"),
    ((65, 65, 2, 256, 16, 0), "ep_size"),
    ((3, 8, 2, 256, 16, 0), "multiple"),
    ((2, 8, 0, 256, 16, 0), "top_k"),
    ((2, 8, 33, 256, 16, 0), "top_k"),
    ((2, 8, 2, 12, 16, 0), "16 bytes"),
    ((2, 8, 2, 8, 16, 1), "16 bytes"),
    ((2, 8, 2, 256, -1, 0), "max_tokens_per_rank"),
    ((64, 64, 2, 256, (1 << 24) + 1, 0), "2^30"),
    ((1, 8, 2, (1 << 28) + 8, 1, 0), "2^28"),
    ((1, 8, 2, (1 << 28) + 16, 1, 1), "2^28"),
    ((2, 8, 2, 256, 16, 7), "dtype"),
])
def test_workspace_size_rejects(args, frag):
    st, _ = _size(*args)
    assert st == ep.EP_ERR_INVALID_ARG
    assert frag in _lib.load().ep_last_error().decode()


def test_workspace_size_accepts_the_widest_rows():
    st, n = _size(1, 8, 2, 1 << 28, 1, 3)  # fp32 rows of 2^30 bytes
    assert st == ep.EP_OK
    assert n >= (1 << 30) + (1 << 29)  # the hidden row plus its bf16 combine row


def test_rank_mask_helper():
    L = _lib.load()
    arr = (ctypes.c_int * 5)(0, 3, 63, 64, -1)
    assert L.ep_rank_mask(arr, 5) == (1 | (1 << 3) | (1 << 63))
    assert int(ep.EpComm.active_rank_mask([1, 2]).item()) == 6


def test_null_handle_calls_fail_cleanly():
    L = _lib.load()
    assert L.ep_destroy(None) == ep.EP_OK
    res = _lib.EpDispatchResultC()
    assert L.ep_dispatch(None, None, None, None, None, None, -1, 0, None, ctypes.byref(res)) == \
        ep.EP_ERR_INVALID_ARG
    assert L.ep_combine(None, None, None, 0, None) == ep.EP_ERR_INVALID_ARG
    p = ctypes.c_void_p()
    assert L.ep_get_combine_input_buffer(None, 0, ctypes.byref(p)) == ep.EP_ERR_INVALID_ARG


def test_create_without_gpu_reports_error():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    L = _lib.load()
    h = ctypes.c_void_p(1)
    st = L.ep_create(2, 8, 2, 256, 16, 0, 0, ctypes.byref(h))
    assert st in (ep.EP_ERR_CUDA, ep.EP_ERR_UNSUPPORTED)
    assert h.value is None
    assert L.ep_is_supported() == 0
    assert not ep.EpComm.is_platform_supported()


def _size_ex(**kw):
    base = dict(ep_size=4, num_experts=8, top_k=2, hidden=256, max_tokens_per_rank=16, dtype=0,
                enable_rank_mask=0, scale_cols=-1, eplb_stats_max_bytes=0, combine_dtype=0, launch_flags=0,
                num_partitions=0, partition=0)
    base.update(kw)
    cfg = _lib.EpConfigC(*[base[f] for f, _ in _lib.EpConfigC._fields_])
    n = ctypes.c_size_t(0)
    st = _lib.load().ep_workspace_size_ex(ctypes.byref(cfg), ctypes.byref(n))
    return st, n.value


@pytest.mark.parametrize("dtype,elem", [(0, 2), (1, 1), (2, 2), (3, 4)])
@pytest.mark.parametrize("scale_cols,G", [(-1, 2), (0, 0), (7, 7)])
@pytest.mark.parametrize("eplb", [0, 1024])
def test_workspace_size_ex_formula(dtype, elem, scale_cols, G, eplb):
    st, n = _size_ex(dtype=dtype, scale_cols=scale_cols, eplb_stats_max_bytes=eplb)
    assert st == ep.EP_OK
    ep_size, K, H, C = 4, 2, 256, 16
    rows = ep_size * C
    want = ep_size * (_align(rows * H * elem) + _align(rows * G * 4) + _align(rows * K * 4) * 2 +
                      _align(rows * H * 2)) + _align(rows * 8) + _align(ep_size * 4) + \
        _align(ep_size * eplb)
    assert n == want


@pytest.mark.parametrize("cdt,ce", [(0, 2), (2, 2), (3, 4)])
def test_workspace_size_ex_combine_dtype(cdt, ce):
    st, n = _size_ex(combine_dtype=cdt)
    assert st == ep.EP_OK
    rows = 4 * 16
    want = 4 * (_align(rows * 256 * 2) + _align(rows * 2 * 4) + _align(rows * 2 * 4) * 2 +
                _align(rows * 256 * ce)) + _align(rows * 8) + _align(4 * 4)
    assert n == want


def test_combine_dtype_rules():
    st, _ = _size_ex(combine_dtype=1)  # fp8 is not a combine type
    assert st == ep.EP_ERR_INVALID_ARG and b"combine_dtype" in _lib.load().ep_last_error()
    st, _ = _size_ex(combine_dtype=3, dtype=3, hidden=12)  # 48-byte fp32 rows: fine
    assert st == ep.EP_OK
    st, _ = _size_ex(combine_dtype=2, dtype=3, hidden=12)  # 24-byte fp16 combine rows: not
    assert st == ep.EP_ERR_INVALID_ARG and b"hidden % 8" in _lib.load().ep_last_error()


def test_default_config_matches_plain_workspace_size():
    assert _size_ex() == _size(4, 8, 2, 256, 16, 0)


def test_launch_flags():
    assert _size_ex(launch_flags=_lib.EP_LAUNCH_PDL) == _size_ex()  # no workspace of its own
    st, _ = _size_ex(launch_flags=2)
    assert st == ep.EP_ERR_INVALID_ARG and b"launch_flags" in _lib.load().ep_last_error()


@pytest.mark.parametrize("kw,frag", [
    (dict(scale_cols=-2), "scale_cols"),
    (dict(eplb_stats_max_bytes=6), "eplb_stats_max_bytes"),
    (dict(eplb_stats_max_bytes=-4), "eplb_stats_max_bytes"),
    (dict(dtype=4), "dtype"),
    (dict(dtype=3, hidden=12), "hidden % 8"),   # 48-byte fp32 rows, but a bf16 combine needs 8 | hidden
    (dict(dtype=1, hidden=24), "16 bytes"),     # 24-byte fp8 rows
])
def test_workspace_size_ex_rejects(kw, frag):
    st, _ = _size_ex(**kw)
    assert st == ep.EP_ERR_INVALID_ARG
    assert frag in _lib.load().ep_last_error().decode()


def test_null_config_and_args_rejected():
    L = _lib.load()
    n = ctypes.c_size_t(0)
    assert L.ep_workspace_size_ex(None, ctypes.byref(n)) == ep.EP_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert L.ep_create_ex(None, None, 0, ctypes.byref(h)) == ep.EP_ERR_INVALID_ARG
    res = _lib.EpDispatchResultC()
    assert L.ep_dispatch_ex(None, None, None, ctypes.byref(res)) == ep.EP_ERR_INVALID_ARG


def test_device_check_status_matches_header():
    text = open(HEADER).read()
    assert re.search(r"EP_ERR_DEVICE_CHECK\s*=\s*6\b", text)
    assert _lib.EP_ERR_DEVICE_CHECK == 6 and _lib.STATUS_NAMES[6] == "EP_ERR_DEVICE_CHECK"


def test_check_sites_match_the_kernels_enum():
    internal = os.path.join(os.path.dirname(HEADER), "..", "combine_topk_ids_dest_gb300", "csrc", "ep_internal.h")
    body = re.search(r"enum CheckSite \{(.*?)\};", open(internal).read(), flags=re.S).group(1)
    names = [n.split("=")[0].strip() for n in body.split(",") if n.strip()]
    assert names[-1] == "kNumSites"
    snake = [re.sub(r"(?<!^)([A-Z])", r"_\1", n[len("kSite"):]).lower() for n in names[:-1]]
    assert tuple(snake) == _lib.CHECK_SITES


def test_checked_build_loads_and_exports_the_abi():
    # In a child process: the loader picks the checked library under EP_GB300_CHECKED=1.
    import subprocess
    import sys
    code = ("import os; from combine_topk_ids_dest_gb300 import _lib; L = _lib.load(); "
            "print(os.path.basename(L._name)); "
            "print(all(hasattr(L, n) for n in _lib.EXPORTS)); "
            "print(L.ep_checked_trim_extent(99, 0), L.ep_checked_trim_extent(0, -1), "
            "L.ep_checked_trim_extent(3, 64), L.ep_checked_trim_extent(-1, 0))")
    root = os.path.dirname(os.path.dirname(HEADER))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, EP_GB300_CHECKED="1"))
    assert r.returncode == 0, r.stderr[-3000:]
    lines = r.stdout.split()
    assert lines[0] == "libep_gb300_checked.so" and lines[1] == "True"
    assert lines[2:] == ["1", "1", "0", "0"]  # bad site, negative bytes, then two valid calls


def test_normal_build_has_no_test_hook():
    assert not hasattr(_lib.load(), "ep_checked_trim_extent") or _lib.checked()


def test_binding_pointer_arrays():
    """The binding's host arrays of per-rank device pointers: uint64 words, 0 for
    NULL, and for a stacked [ep, M, cols] tensor base + s * M*cols*element_size."""
    import numpy as np
    import torch

    from combine_topk_ids_dest_gb300 import ep as epmod
    a = epmod._addr_array([0x1000, None, 0, 0x7FFF_FFFF_F000])
    assert a.dtype == np.uint64 and a.tolist() == [0x1000, 0, 0, 0x7FFF_FFFF_F000]
    assert epmod._data(None) is None and epmod._data(a) == a.ctypes.data
    t = torch.zeros(3, 5, 7, dtype=torch.float32)
    p = epmod.EpComm._stacked_ptrs(t, 5, 7)
    assert p.dtype == np.uint64
    assert p.tolist() == [t[s].data_ptr() for s in range(3)]
    assert epmod.EpComm._stacked_ptrs(t, 5, 7)[2] == t.data_ptr() + 2 * 5 * 7 * 4
