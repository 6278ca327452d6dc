"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every function include/lf_decode.h declares, and rejects bad arguments on the
host before touching CUDA."""
import ctypes
import os
import re

import pytest

import decode_kv_cache_step_gb300 as lf
from decode_kv_cache_step_gb300 import build as lfbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lf_decode.h")


@pytest.fixture(scope="module")
def lib():
    lfbuild.build()
    return lf.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lf_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_surface():
    assert set(declared_functions()) == set(lf.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported by {lf.library_path()}"


def test_library_is_built_for_sm_103a():
    # The build passes exactly one -gencode, for sm_103a.
    assert lfbuild.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert os.path.getsize(lf.library_path()) > 0


def test_version_and_status_strings(lib):
    assert lf.version() == 100
    assert "INVALID" in lf.status_string(lf.LF_ERR_INVALID_ARG)
    assert lf.status_string(lf.LF_OK) == "LF_OK"


FAKE = 0x10000  # a 64 KiB-aligned stand-in address; validation never dereferences it


def call_step(lib, **kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, mask=FAKE, nk=FAKE, nv=FAKE, ws=FAKE, out=FAKE,
                nxt=FAKE, B=1, Hq=4, Hkv=2, d=128, S=16, W=2, scale=0.1)
    args.update(kw)
    return lib.lf_decode_step(args["q"], args["k"], args["v"], args["mask"], args["nk"],
                              args["nv"], args["ws"], args["out"], args["nxt"], args["B"],
                              args["Hq"], args["Hkv"], args["d"], args["S"], args["W"],
                              args["scale"], None)


@pytest.mark.parametrize("kw,status", [
    ({"q": None}, lf.LF_ERR_INVALID_ARG),
    ({"k": FAKE + 8}, lf.LF_ERR_INVALID_ARG),
    ({"mask": FAKE + 2}, lf.LF_ERR_INVALID_ARG),
    ({"nxt": None}, lf.LF_ERR_INVALID_ARG),
    ({"B": 0}, lf.LF_ERR_INVALID_ARG),
    ({"S": 0}, lf.LF_ERR_INVALID_ARG),
    ({"Hq": 6, "Hkv": 4}, lf.LF_ERR_INVALID_ARG),
    ({"W": -1}, lf.LF_ERR_INVALID_ARG),
    ({"scale": float("inf")}, lf.LF_ERR_INVALID_ARG),
    ({"d": 96}, lf.LF_ERR_UNSUPPORTED),
    ({"Hq": 6, "Hkv": 2}, lf.LF_ERR_UNSUPPORTED),
    ({"Hq": 32, "Hkv": 2}, lf.LF_ERR_UNSUPPORTED),
    ({"S": (1 << 20) + 1}, lf.LF_ERR_UNSUPPORTED),
    ({"B": 40000, "Hkv": 2}, lf.LF_ERR_UNSUPPORTED),
])
def test_host_side_argument_errors(lib, kw, status):
    assert call_step(lib, **kw) == status
    assert lib.lf_last_error().decode() != ""


def test_scores_and_host_variants_validate_too(lib):
    assert lib.lf_decode_step_scores(*([FAKE] * 9), None, 1, 4, 2, 128, 16, 2,
                                     ctypes.c_float(0.1), None) == lf.LF_ERR_INVALID_ARG
    assert lib.lf_decode_step_host(None, *([FAKE] * 8), 1, 4, 2, 128, 16, 2,
                                   ctypes.c_float(0.1), None) == lf.LF_ERR_INVALID_ARG
    assert lib.lf_decode_step_host(*([FAKE] * 9), 1, 4, 2, 64, 16, -5, ctypes.c_float(0.1),
                                   None) == lf.LF_ERR_INVALID_ARG


def test_profile_api_without_launches(lib):
    lf.profile_enable(True)
    assert lf.profile_collect(lf.LF_KERNEL_DECODE_STEP) == (0.0, 0)
    lf.profile_enable(False)
    with pytest.raises(lf.LFError):
        lf.profile_collect(7)


def test_prepared_step_and_plan_validate_on_the_host(lib):
    h = ctypes.c_void_p(0)
    args = [FAKE] * 9 + [1, 4, 2, 128, 16, 2, ctypes.c_float(0.1), None]
    assert lib.lf_step_prepare(*args, None) == lf.LF_ERR_INVALID_ARG          # no handle slot
    bad = list(args)
    bad[0] = None                                                             # q missing
    assert lib.lf_step_prepare(*bad, ctypes.byref(h)) == lf.LF_ERR_INVALID_ARG
    bad = list(args)
    bad[1] = FAKE + 8                                                         # misaligned k_cache
    assert lib.lf_step_prepare(*bad, ctypes.byref(h)) == lf.LF_ERR_INVALID_ARG
    bad = list(args)
    bad[12] = 96                                                              # head dim 96
    assert lib.lf_step_prepare(*bad, ctypes.byref(h)) == lf.LF_ERR_UNSUPPORTED
    assert h.value is None
    assert lib.lf_step_run(None) == lf.LF_ERR_INVALID_ARG
    assert lib.lf_step_errors(None, None, 0) == lf.LF_ERR_INVALID_ARG
    assert lib.lf_step_destroy(None) == lf.LF_OK
    plan = (ctypes.c_int32 * 6)()
    assert lib.lf_step_plan(1, 4, 2, 128, 16, 1, None) == lf.LF_ERR_INVALID_ARG
    assert lib.lf_step_plan(1, 6, 4, 128, 16, 1, plan) == lf.LF_ERR_INVALID_ARG
    assert lib.lf_step_plan(1, 4, 2, 128, 16, 0, plan) == lf.LF_ERR_INVALID_ARG
    assert lib.lf_step_plan(1, 4, 2, 96, 16, 1, plan) == lf.LF_ERR_UNSUPPORTED


def test_prepared_step_binding_checks_tensors():
    import torch
    bf = torch.bfloat16
    q = torch.zeros(1, 4, 64, dtype=bf)
    k = torch.zeros(1, 2, 16, 64, dtype=bf)            # host caches: refused before the ABI
    mask = torch.zeros(1, 2, 16, dtype=torch.int32)
    nk = torch.zeros(1, 2, 64, dtype=bf)
    ws = torch.zeros(1, 2, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        lf.PreparedStep(q, k, k, mask, nk, nk, ws, q, ws, 2, 0.1)
