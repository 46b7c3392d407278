"""The C-ABI library: it builds, loads without a GPU, exports every symbol the
header declares, and rejects bad host arguments before touching the device."""
import ctypes
import os
import re

import pytest

from tests.helpers import ROOT, ensure_built

HEADER = os.path.join(ROOT, "include", "fs_sampling.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fs_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def so():
    path = ensure_built()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ["fs_sampling_from_probs", "fs_top_k_sampling", "fs_top_p_sampling", "fs_min_p_sampling",
              "fs_top_k_top_p_sampling", "fs_top_k_renorm_probs", "fs_top_p_renorm_probs",
              "fs_top_k_mask_logits", "fs_philox4x32_10", "fs_status_string"]:
        assert n in names


def test_every_declared_symbol_is_exported(so):
    for name in _declared_functions():
        assert hasattr(so, name), name


def test_status_strings_and_limits(so):
    so.fs_status_string.restype = ctypes.c_char_p
    so.fs_max_vocab.restype = ctypes.c_int32
    assert so.fs_status_string(0) == b"FS_OK"
    assert b"INVALID" in so.fs_status_string(1)
    assert so.fs_max_vocab() == 2097152


P = ctypes.c_void_p
FAKE = P(0x1000)   # never dereferenced: every call below is rejected on the host


def _sample(so, probs=FAKE, b_in=4, V=16, idx=None, b_out=4, k=FAKE, p=FAKE, mp=None, order=0,
            tok=FAKE, valid=FAKE):
    f = so.fs_top_k_top_p_sampling
    f.argtypes = [P, ctypes.c_int32, ctypes.c_int32, P, ctypes.c_int32, P, P, P, ctypes.c_int32,
                  ctypes.c_uint64, ctypes.c_uint64, P, P, P, P]
    return f(probs, b_in, V, idx, b_out, k, p, mp, order, 1, 2, tok, valid, None, None)


def test_host_argument_checks(so):
    assert _sample(so, probs=None) == 1
    assert _sample(so, tok=None) == 1
    assert _sample(so, valid=None) == 1
    assert _sample(so, V=0) == 1
    assert _sample(so, V=2097153) == 2
    assert _sample(so, b_out=5) == 1            # no indices: batch_out must equal batch_in
    assert _sample(so, order=7) == 1
    assert _sample(so, k=None) == 1
    assert _sample(so, b_out=-1) == 1
    assert _sample(so, b_out=0, probs=None) == 0   # empty batch: nothing to do
    f = so.fs_top_k_renorm_probs
    f.argtypes = [P, ctypes.c_int32, ctypes.c_int32, P, P, P, P]
    assert f(None, 2, 8, FAKE, FAKE, None, None) == 1
    assert f(FAKE, 2, 8, None, FAKE, None, None) == 1
    assert f(FAKE, 0, 8, FAKE, FAKE, None, None) == 0
    g = so.fs_philox4x32_10
    g.argtypes = [P, P, ctypes.c_int64, P, P]
    assert g(None, FAKE, 4, FAKE, None) == 1
    assert g(FAKE, FAKE, 0, FAKE, None) == 0


def test_binding_imports_without_gpu():
    ensure_built()
    import min_sampling_gb300 as ms
    assert ms.MAX_VOCAB == 2097152
    with pytest.raises(ValueError):
        ms._order("sideways")


def test_binding_rejects_indices_the_kernels_cannot_read():
    """The kernels read `indices` on the device: a host tensor, another dtype or a
    strided view is refused before any call (every sampler goes through one check)."""
    ensure_built()
    import torch

    import min_sampling_gb300 as ms
    dev = torch.device("cuda", 0)
    assert ms._indices(None, 7, dev) == (None, 7)
    for bad in (torch.zeros(4, dtype=torch.int32),                  # host memory
                torch.zeros(4, dtype=torch.int64),                  # another dtype
                torch.zeros(8, dtype=torch.int32)[::2],             # not contiguous
                torch.zeros((2, 2), dtype=torch.int32),             # not 1-D
                [0, 1, 2]):
        with pytest.raises(ValueError):
            ms._indices(bad, 4, dev)
    cpu = torch.device("cpu")
    idx = torch.arange(6, dtype=torch.int32)
    got, b_out = ms._indices(idx, 3, cpu)
    assert got is idx and b_out == 6


def test_header_compiles_as_plain_c():
    """A C caller can use the boundary: the header compiles as C99 with warnings as
    errors, and every declared entry point is a function it can take the address of.
    The source goes to the compiler on stdin and the object to /dev/null."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = _declared_functions()
    src = ('#include "fs_sampling.h"\n'
           "typedef void (*fs_any_fn)(void);\n"
           "fs_any_fn fs_entry_points[] = {\n" + "".join(f"    (fs_any_fn)&{n},\n" for n in names) + "};\n"
           "int fs_order_values[] = {FS_ORDER_TOP_K_FIRST, FS_ORDER_JOINT, FS_OK, FS_ERR_CUDA};\n")
    r = subprocess.run([cc, "-pipe", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-x", "c", "-c", "-",
                        "-I", os.path.dirname(HEADER), "-o", os.devnull],
                       input=src, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_binding_rejects_tensors_on_another_device():
    """The binding checks that every tensor of a call lives on the call's device
    before anything reaches the library (cpu and meta stand in for two devices)."""
    import torch
    from min_sampling_gb300 import _same_device
    a = torch.zeros(3)
    _same_device(a.device, x=a, y=None)
    with pytest.raises(ValueError):
        _same_device(a.device, draft_probs=a, draft_tokens=torch.zeros(3, device="meta"))


def test_workspace_bytes_follow_the_documented_layout(so):
    """fs_workspace_bytes: 2 KB of counters, then per row 8 bytes per segment of the
    plan (rounded up to 4 segments), 16 bytes per 512 values and, for the joint
    order's run codes, one byte per 4 values (per 512-value unit, 128 bytes)."""
    f = so.fs_workspace_bytes
    f.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)]
    f.restype = ctypes.c_int

    def expect(B, V):
        shift = 0 if V <= 4096 * 128 else (1 if V <= 4096 * 256 else 2)
        seg = 128 << shift
        ns = (V + seg - 1) // seg
        ls = (ns + 3) // 4 * 4
        nu = (V + 511) // 512
        return 2048 + B * (2 * ls * 4 + nu * (16 + 128))

    for B, V in ((1, 1), (64, 151936), (256, 256000), (3, 32000), (5, 600001)):
        out = ctypes.c_size_t(0)
        assert f(B, V, ctypes.byref(out)) == 0
        assert out.value == expect(B, V), (B, V)
    out = ctypes.c_size_t(0)
    f(64, 151936, ctypes.byref(out))
    assert abs(out.value / 1e6 - 3.35) < 0.01   # the header's example: 3.3 MB in the joint order


def test_noalloc_rejects_a_joint_batch_that_fits_only_top_k_first(so):
    """256 rows of 256000 values: 6.1 MB of summaries top-k-first (within the fixed
    array), 22.5 MB with the joint order's run codes (rejected before any CUDA call)."""
    f = so.fs_top_k_top_p_sampling_noalloc
    P = ctypes.c_void_p
    f.argtypes = [P, ctypes.c_int32, ctypes.c_int32, P, ctypes.c_int32, P, P, P, ctypes.c_int32, ctypes.c_uint64,
                  ctypes.c_uint64, P, P, P, P]
    f.restype = ctypes.c_int
    so.fs_last_error_string.restype = ctypes.c_char_p
    fake = P(0x1000)   # never dereferenced: the size check comes first
    st = f(fake, 256, 256000, None, 256, fake, fake, None, 1, 1, 2, fake, fake, None, None)
    assert st == 2
    assert b"FS_NOALLOC_SCRATCH_BYTES" in so.fs_last_error_string()
