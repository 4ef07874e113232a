"""The binding's C call path (``_hcpycall``) passes every argument to the entry point
unchanged: None as NULL, an int as that address, a tensor as its data_ptr(), the token
count, the path and the stream; and it returns the entry point's status code. Checked
on the CPU against a stub library with the same two entry points that records what it
receives."""
import ctypes
import os
import shutil
import subprocess

import pytest
import torch

import hyper_connection_residual_read_gb300._lib as hcl

STUB = r"""
#include <stdint.h>
static uintptr_t got[13];
int hc_read(int t, void* a, void* b, void* c, void* d, void* e, void* f, void* g, void* h,
            void* i, void* s) {
    void* p[10] = {a, b, c, d, e, f, g, h, i, s};
    got[0] = 1; got[1] = (uintptr_t)t; got[2] = 0;
    for (int k = 0; k < 10; ++k) got[3 + k] = (uintptr_t)p[k];
    return t == 99 ? -1 : 0;
}
int hc_read_path(int path, int t, void* a, void* b, void* c, void* d, void* e, void* f,
                 void* g, void* h, void* i, void* s) {
    void* p[10] = {a, b, c, d, e, f, g, h, i, s};
    got[0] = 2; got[1] = (uintptr_t)t; got[2] = (uintptr_t)path;
    for (int k = 0; k < 10; ++k) got[3 + k] = (uintptr_t)p[k];
    return -3;
}
uintptr_t stub_got(int k) { return got[k]; }
"""


@pytest.fixture()
def stub(tmp_path):
    try:
        from hyper_connection_residual_read_gb300 import _hcpycall
    except ImportError:
        pytest.skip("the Python call module is not built")
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "stub.c"
    src.write_text(STUB)
    so = tmp_path / "libstub.so"
    subprocess.run([cc, "-O1", "-shared", "-fPIC", str(src), "-o", str(so)], check=True)
    lib = ctypes.CDLL(os.fspath(so))
    lib.stub_got.restype = ctypes.c_uint64
    lib.stub_got.argtypes = [ctypes.c_int]
    addr = lambda f: ctypes.cast(f, ctypes.c_void_p).value  # noqa: E731
    _hcpycall.bind(addr(lib.hc_read), addr(lib.hc_read_path))
    yield _hcpycall, lib
    # back to the library the binding loaded, if any
    if hcl._lib is not None:
        hcl._bind_call(hcl._lib)


def test_read_passes_arguments_unchanged(stub):
    call, lib = stub
    t = torch.arange(16, dtype=torch.float32)
    u = torch.zeros(8, dtype=torch.int16)
    args = [t, None, u, 0x1000, t, u, 0x7FFF0000, None, t, 12345]
    rc = call.read(5, *args)
    assert rc == 0
    want = [t.data_ptr(), 0, u.data_ptr(), 0x1000, t.data_ptr(), u.data_ptr(), 0x7FFF0000, 0,
            t.data_ptr(), 12345]
    assert lib.stub_got(0) == 1 and lib.stub_got(1) == 5
    assert [lib.stub_got(3 + k) for k in range(10)] == want
    assert call.read(99, *args) == -1          # the entry point's code comes back


def test_read_path_passes_path_and_code(stub):
    call, lib = stub
    t = torch.ones(4)
    rc = call.read_path(4, 7, t, t, None, None, t, t, t, t, t, None)
    assert rc == -3
    assert lib.stub_got(0) == 2 and lib.stub_got(1) == 7 and lib.stub_got(2) == 4
    assert lib.stub_got(3) == t.data_ptr() and lib.stub_got(5) == 0 and lib.stub_got(12) == 0


def test_bad_arguments_raise(stub):
    call, _ = stub
    with pytest.raises(TypeError):
        call.read(1, None)                      # wrong count
    with pytest.raises(AttributeError):
        call.read(1, "not a tensor", *([None] * 9))
    with pytest.raises(OverflowError):               # not truncated into a small count
        call.read(2 ** 32 + 4, *([None] * 10))
    with pytest.raises(OverflowError):
        call.read_path(1, -(2 ** 40), *([None] * 10))
