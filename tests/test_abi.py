"""The C ABI boundary without a GPU: the library builds and loads, exports
every entry point ``include/pagedkv.h`` declares, answers host-only calls,
and rejects bad arguments before touching the device.  Also checks that the
product and the oracle share no code."""
import ctypes
import glob
import json
import os
import re

import pytest

import gqa_decode_attention_paged_gb300 as pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = glob.glob(os.path.join(ROOT, "include", "*.h"))


def _declared_functions():
    names = []
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?(?:pkv_status|double|char|uint64_t|int64_t|void)\s*\*?\s*(\w+)\s*\(",
                             text, flags=re.M):
            names.append(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    return pkv.load()


def test_header_declares_the_pool_append_and_decode_calls():
    names = _declared_functions()
    for n in ("kv_pool_create", "paged_kv_append", "paged_decode_attention", "kv_bytes_per_token"):
        assert n in names
    assert len(names) >= 14


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_library_targets_sm103a_only():
    # The shared object embeds sm_103a SASS only (checked through the build
    # flags, not by reading the binary).
    from gqa_decode_attention_paged_gb300 import _build

    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_kv_bytes_per_token_through_the_abi():
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "kv_bytes_per_token.json")))
    for case in g["cases"]:
        L, nkv, d, b = case["args"]
        assert pkv.kv_bytes_per_token(L, nkv, d, b) * case["times"] == case["bytes"], case["cite"]
    assert pkv.kv_bytes_per_token(-1, 8, 128, 2) < 0


def test_status_strings(lib):
    for code, name in pkv.STATUS.items():
        assert lib.pkv_status_string(code).decode() == name
    assert lib.pkv_status_string(99).decode() == "PKV_UNKNOWN"


@pytest.mark.parametrize("args,status", [
    ((0, 16, 8, 128, 0), 1),      # no blocks
    ((64, 32, 8, 128, 0), 5),     # block size
    ((64, 16, 8, 96, 0), 5),      # head dim
    ((64, 16, 0, 128, 0), 1),     # no heads
    ((64, 16, 8, 128, 7), 1),     # dtype
])
def test_pool_create_rejects_bad_shapes_on_host(lib, args, status):
    h = ctypes.c_void_p()
    assert lib.kv_pool_create(*args, ctypes.byref(h)) == status
    assert not h.value
    assert lib.pkv_last_error_message().decode()


def test_calls_with_null_pool_fail_cleanly(lib):
    assert lib.paged_kv_append(None, None, None, None, 1, None) == 1
    assert lib.paged_decode_attention(None, None, 8, None, 1, None, 1, 1.0, None, None) == 1
    assert lib.kv_pool_layout(None, None) == 1
    assert lib.kv_pool_destroy(None) == 0
    assert lib.pkv_get_error(None, 0, None) == 1


def test_pool_create_without_gpu_reports_cuda_error(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    st = lib.kv_pool_create(64, 16, 8, 128, 0, ctypes.byref(h))
    assert st in (4, 5) and not h.value


def test_product_and_oracle_share_no_code():
    prod = glob.glob(os.path.join(ROOT, "gqa_decode_attention_paged_gb300", "**", "*.*"), recursive=True)
    for f in prod:
        if f.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
            txt = open(f).read()
            assert not re.search(r"^\s*(import|from)\s+oracle\b", txt, flags=re.M), f
            assert "pagedkv_oracle" not in txt and "liboracle" not in txt, f
    for f in glob.glob(os.path.join(ROOT, "oracle", "*.*")):
        if f.endswith((".py", ".c", ".h")):
            txt = open(f).read()
            assert not re.search(r"^\s*(import|from)\s+gqa_decode_attention_paged_gb300\b", txt,
                                 flags=re.M), f
            assert not re.search(r"#\s*include\s*[<\"]pagedkv\.h", txt), f
            assert "libpagedkv" not in txt, f


def test_binding_structs_match_the_header(tmp_path):
    """The binding's ctypes mirrors of pkv_layout and pkv_timing have the
    header's size and field offsets (a C program built from the header
    prints them)."""
    import shutil
    import subprocess

    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    structs = {"pkv_layout": pkv._Layout, "pkv_timing": pkv._Timing}
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "pagedkv.h"', "int main(void) {"]
    for cname, py in structs.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {tuple(line.split()[:2]): int(line.split()[2]) for line in out if line}
    for cname, py in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(py), cname
        for f, _ in py._fields_:
            assert got[(cname, f)] == getattr(py, f).offset, (cname, f)
