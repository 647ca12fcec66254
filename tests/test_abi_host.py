"""Host-side checks of the C ABI (no GPU needed): the library builds, loads and
exports every entry point include/*.h declares, and argument validation
rejects bad calls before anything touches the device."""
import ctypes
import glob
import os
import re

import pytest

import gated_softmax_kv_gb300 as gsk
from gated_softmax_kv_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gsk.build()
    return binding.load()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b(csa_[A-Za-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_two_calls():
    names = declared_functions()
    assert "csa_compress_fwd" in names and "csa_compress_bwd" in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for st in range(6):
        s = lib.csa_status_string(st)
        assert s and len(s) > 0
    assert lib.csa_status_string(99) == b"unknown status"


# Fake, well-aligned device addresses: validation must reject these calls
# before any CUDA call is made, so they are never dereferenced.
A = 0x10000


def fwd(lib, exact=False, **kw):
    args = dict(kv=A, score=A, ape=A, cu=A, cuc=A, nseq=1, T=64, C=8, r=4, coff=2, d=64, out=A)
    args.update(kw)
    fn = lib.csa_compress_fwd_exact if exact else lib.csa_compress_fwd
    return fn(args["kv"], args["score"], args["ape"], args["cu"], args["cuc"],
                                args["nseq"], args["T"], args["C"], args["r"], args["coff"],
                                args["d"], args["out"], None)


def bwd(lib, exact=False, **kw):
    args = dict(kv=A, score=A, ape=A, cu=A, cuc=A, nseq=1, T=64, C=8, r=4, coff=2, d=64, go=A,
                dkv=A, ds=A, dape=A)
    args.update(kw)
    fn = lib.csa_compress_bwd_exact if exact else lib.csa_compress_bwd
    return fn(args["kv"], args["score"], args["ape"], args["cu"], args["cuc"],
                                args["nseq"], args["T"], args["C"], args["r"], args["coff"],
                                args["d"], args["go"], args["dkv"], args["ds"], args["dape"], None)


def fwd_exact(lib, **kw):
    return fwd(lib, exact=True, **kw)


def bwd_exact(lib, **kw):
    return bwd(lib, exact=True, **kw)


@pytest.mark.parametrize("call", [fwd, bwd, fwd_exact, bwd_exact])
def test_validation_rejects_before_launch(lib, call):
    assert call(lib, r=3) == 3                  # unsupported ratio
    assert call(lib, r=256) == 3
    assert call(lib, coff=0) == 3
    assert call(lib, d=12) == 3                 # head_dim % 8 != 0
    assert call(lib, d=0) == 3
    assert call(lib, nseq=0) == 4
    assert call(lib, T=-1) == 4
    assert call(lib, C=-1) == 4
    assert call(lib, T=1 << 21, d=1024) == 4    # T * coff * d >= 2^31
    assert call(lib, C=1 << 22, d=512) == 4     # capacity * d >= 2^31
    assert call(lib, T=3, C=1) == 4             # capacity > 0 needs T >= ratio
    assert call(lib, kv=0) == 1
    assert call(lib, cu=0) == 1
    assert call(lib, ape=0) == 1
    assert call(lib, kv=A + 8) == 2             # 16-byte alignment
    assert call(lib, ape=A + 4) == 2
    assert call(lib, cuc=A + 2) == 2            # 4-byte alignment


def test_bwd_output_pointers_validated(lib):
    assert bwd(lib, go=0) == 1
    assert bwd(lib, dkv=0) == 1
    assert bwd(lib, dape=0) == 1
    assert bwd(lib, ds=A + 8) == 2
    assert fwd(lib, out=0) == 1
    assert fwd(lib, out=A + 2) == 2


def test_fwd_zero_capacity_launches_nothing(lib):
    # capacity == 0: valid, no launch, no CUDA call (works without a GPU)
    assert fwd(lib, C=0, out=0) == 0
    assert fwd(lib, exact=True, C=0, out=0) == 0


@pytest.mark.parametrize("exact", [True, False])
def test_exact_mode_envelope(lib, exact):
    # the exact mode covers windows of at most 8 slots; wider ones are
    # rejected before any CUDA call (zero capacity: nothing would launch)
    for r, coff in [(2, 1), (4, 1), (8, 1), (2, 2), (4, 2)]:
        assert fwd(lib, exact=exact, r=r, coff=coff, C=0, out=0) == 0
    for r, coff in [(8, 2), (16, 1), (16, 2), (128, 1), (128, 2)]:
        want = 3 if exact else 0
        assert fwd(lib, exact=exact, r=r, coff=coff, C=0, out=0) == want
        # the shape is checked before the output pointers
        assert bwd(lib, exact=exact, r=r, coff=coff, T=256, d=64, go=0) == (3 if exact else 1)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        binding.load()


def test_plain_c_client(lib, tmp_path):
    """include/csa_compress.h compiles as C99 and a C program linked against
    libcsa_compress.so gets the documented status codes (no GPU needed)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    from gated_softmax_kv_gb300 import nvbuild
    build_dir = os.path.dirname(nvbuild.LIB)
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(nvbuild.nvcc())), "include")
    exe = str(tmp_path / "abi_client")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", cuda_inc, os.path.join(ROOT, "tests", "abi_client.c"), "-L", build_dir,
                    "-lcsa_compress", "-Wl,-rpath," + build_dir, "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok")


def test_binding_rejects_host_tensors():
    """The kernels take device pointers: the binding refuses CPU tensors before
    anything reaches the library."""
    torch = pytest.importorskip("torch")
    kv = torch.zeros(8, 128, dtype=torch.bfloat16)
    ape = torch.zeros(4, 128, dtype=torch.float32)
    cu = torch.tensor([0, 8], dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        gsk.csa_compress_fwd(kv, kv, ape, cu, torch.tensor([0, 2], dtype=torch.int32), 2, 4, 2, 64)
    with pytest.raises(TypeError):
        gsk.csa_compress_fwd(kv.float(), kv, ape, cu, cu, 2, 4, 2, 64)
    go = torch.zeros(2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        gsk.csa_compress_bwd(kv, kv, ape, cu, cu, 2, 4, 2, 64, go)


def test_segment_check_validation(lib):
    # rejected before any CUDA call
    seg = ctypes.c_void_p(A)
    f = lib.csa_check_segments
    assert f(seg, seg, 1, 64, 8, 3, seg, None) == 3          # ratio 3
    assert f(seg, seg, 0, 64, 8, 4, seg, None) == 4          # num_seqs 0
    assert f(seg, seg, 1, -1, 8, 4, seg, None) == 4
    assert f(None, seg, 1, 64, 8, 4, seg, None) == 1
    assert f(seg, seg, 1, 64, 8, 4, None, None) == 1
    assert f(seg, ctypes.c_void_p(A + 2), 1, 64, 8, 4, seg, None) == 2


def _expected_status(nseq, T, C, r, coff, d, ptrs_ok=True):
    """The envelope of include/csa_compress.h, written out from its comment."""
    if r not in (2, 4, 8, 16, 32, 64, 128) or coff not in (1, 2):
        return 3
    if d < 8 or d % 8 != 0:
        return 3
    if nseq < 1 or T < 0 or C < 0:
        return 4
    if T * coff * d >= (1 << 31) or C * d >= (1 << 31):
        return 4
    if C > 0 and T < r:
        return 4
    return 0


def test_forward_validation_matches_the_documented_envelope(lib):
    """Seeded random argument tuples, valid and invalid: the forward's status
    is the one the header's envelope gives (no call launches anything: valid
    tuples use capacity 0)."""
    import numpy as np
    rng = np.random.default_rng(17)
    for _ in range(3000):
        r = int(rng.choice([0, 1, 2, 3, 4, 8, 16, 32, 64, 128, 256]))
        coff = int(rng.integers(0, 4))
        d = int(rng.choice([0, 4, 8, 12, 64, 512, 1024, 4096, 1 << 20]))
        nseq = int(rng.integers(-1, 4))
        T = int(rng.choice([-1, 0, 1, 3, 64, 1 << 20, 1 << 30]))
        C = int(rng.choice([-1, 0, 1, 8, 1 << 22]))
        want = _expected_status(nseq, T, C, r, coff, d)
        if want == 0:
            C = 0  # keep the call launch-free
            want = _expected_status(nseq, T, C, r, coff, d)
        got = fwd(lib, nseq=nseq, T=T, C=C, r=r, coff=coff, d=d, out=0 if C == 0 else A)
        assert got == want, (nseq, T, C, r, coff, d, got, want)
