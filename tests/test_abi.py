"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every function include/hc_read.h declares, and answers without a device."""
import ctypes
import os
import re

import pytest

import hyper_connection_residual_read_gb300 as hc
from hyper_connection_residual_read_gb300 import build as hcbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(hcbuild.LIB):
        hcbuild.build()
    return hc.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "hc_read.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hc_read\w*)\s*\(", text)))


def test_header_declares_the_binding(lib):
    assert declared_functions() == sorted(hc.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_version_and_strerror(lib):
    assert hc.hc_read_version() == 102
    assert hc.hc_read_bounds_checked() is False     # the default build has no checks
    for code in range(0, -9, -1):
        assert hc.strerror(code) != "unknown status"
    assert hc.strerror(-99) == "unknown status"


def test_binding_constants_match_the_header():
    """Every enumerator and size macro of include/hc_read.h has the same value in
    the binding (parsed from the header text, so a renumbering on either side fails)."""
    from hyper_connection_residual_read_gb300 import _lib
    text = open(os.path.join(ROOT, "include", "hc_read.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    enums = dict((k, int(v)) for k, v in re.findall(r"\b(HC_(?:OK|ERR_\w+|PATH_\w+))\s*=\s*(-?\d+)", text))
    assert len(enums) == 15, sorted(enums)
    for name, value in enums.items():
        assert getattr(_lib, name) == value, name
    macros = dict((k, int(v)) for k, v in re.findall(r"#define\s+HC_READ_(\w+)\s+(\d+)", text))
    assert (macros["STREAMS"], macros["WIDTH"], macros["RANK"]) == (_lib.STREAMS, _lib.WIDTH, _lib.RANK)


def test_calls_without_a_device_fail_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU tests")
    # no kernel can be launched here: every entry point must return an error code
    assert lib.hc_read_init(0, 8, 1e-6) in (hc._lib.HC_ERR_CUDA, hc._lib.HC_ERR_ARCH)
    rc = lib.hc_read(1, None, None, None, None, None, None, None, None, None, None)
    assert rc in (hc._lib.HC_ERR_CUDA, hc._lib.HC_ERR_NOT_INIT)
    assert lib.hc_read_init(0, 0, 1e-6) == hc._lib.HC_ERR_ARG


def test_synth_recipe_shapes_and_statistics():
    from hyper_connection_residual_read_gb300 import synth
    import numpy as np
    w = synth.make_weights(0)
    assert w["W_down"].shape == (320, 10240) and w["W_down"].dtype == np.uint16
    assert w["W_up"].shape == (10240, 320) and w["w_norm"].shape == (4, 2560)
    a = synth.make_activations(1, 3, True)
    assert a["R"].shape == (3, 4, 2560) and a["P"].shape == (3, 4, 2560)
    assert np.allclose(a["Rmix"].sum(-1), 1.0, atol=1e-6) and (a["Rmix"] > 0).all()
    assert abs(float(a["R"].std()) - 1.0) < 0.02 and abs(float(a["P"].std()) - 0.1) < 0.005
    from oracle.hc_oracle import bf16_bits_to_f64
    assert abs(bf16_bits_to_f64(w["W_down"]).std() - 0.02) < 5e-4
    assert abs(bf16_bits_to_f64(w["w_norm"]).mean() - 1.0) < 0.01
    b = synth.make_activations(1, 3, True)
    assert (a["R"] == b["R"]).all()   # seeded
