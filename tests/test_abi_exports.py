"""The C-ABI library builds, loads and exports every entry point the header
declares; host-side argument checks answer without touching a GPU (no GPU)."""

import ctypes
import os
import re
import shutil
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "pagedkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:kv_status|const\s+char\s*\*)\s+(\w+)\s*\(", text, flags=re.M)
    assert names, "no declarations found"
    return names


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_68_gb300 import pagedkv
    return pagedkv.load()


def test_header_declares_the_hot_path():
    names = set(declared_functions())
    for must in ("kv_pool_create", "kv_pool_destroy", "kv_append", "copy_blocks",
                 "paged_attention_decode", "paged_attention_workspace_size",
                 "kv_pool_get_error", "kv_strerror"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    from paged_kv_cache_68_gb300 import pagedkv
    out = subprocess.run(["nm", "-D", "--defined-only", pagedkv.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, f"{name} declared in pagedkv.h but not exported"
        assert hasattr(lib, name)


def test_strerror_texts(lib):
    for code in range(6):
        assert lib.kv_strerror(code)
    assert lib.kv_strerror(99) == b"unknown status"


def test_create_rejects_bad_arguments_on_host(lib):
    h = ctypes.c_void_p()
    fake = ctypes.c_void_p(0x1000)
    mis = ctypes.c_void_p(0x1008)
    assert lib.kv_pool_create(4, 16, 8, 96, 2, fake, fake, ctypes.byref(h)) == 2   # head_dim
    assert lib.kv_pool_create(4, 16, 8, 128, 7, fake, fake, ctypes.byref(h)) == 2  # dtype
    assert lib.kv_pool_create(0, 16, 8, 128, 2, fake, fake, ctypes.byref(h)) == 1  # no blocks
    assert lib.kv_pool_create(4, 512, 8, 128, 2, fake, fake, ctypes.byref(h)) == 1  # block size
    assert lib.kv_pool_create(4, 16, 8, 128, 2, None, fake, ctypes.byref(h)) == 1
    assert lib.kv_pool_create(4, 16, 8, 128, 2, mis, fake, ctypes.byref(h)) == 1   # alignment
    assert lib.kv_pool_create(4, 16, 8, 128, 2, fake, fake, None) == 1
    assert h.value is None


def test_calls_on_null_pool_are_rejected(lib):
    assert lib.kv_append(None, None, None, None, 1, None) == 1
    assert lib.copy_blocks(None, None, 1, None) == 1
    assert lib.kv_pool_destroy(None) == 0
    size = ctypes.c_size_t()
    assert lib.paged_attention_workspace_size(None, 1, 1, ctypes.byref(size)) == 1


def test_build_is_sm103a_only():
    from paged_kv_cache_68_gb300 import _build
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_header_is_plain_c_and_links_from_c(lib, tmp_path):
    """A C99 program (pedantic, warnings as errors) that includes the header,
    takes the address of every declared entry point, links against the
    library and calls kv_strerror: the boundary is a C ABI, not a C++ one."""
    from paged_kv_cache_68_gb300 import pagedkv
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = declared_functions()
    src = tmp_path / "abi.c"
    src.write_text(
        '#include "pagedkv.h"\n#include <stdio.h>\n'
        "typedef void (*entry)(void);\n"
        "int main(void) {\n  entry fns[] = {\n"
        + "".join(f"    (entry)&{n},\n" for n in names)
        + "  };\n"
        '  printf("%d %s\\n", (int)(sizeof fns / sizeof fns[0]), kv_strerror(KV_OK));\n'
        "  return 0;\n}\n")
    exe = tmp_path / "abi"
    libdir = os.path.dirname(pagedkv.library_path())
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.dirname(HEADER), str(src), "-o", str(exe), "-L", libdir,
                    "-lpagedkv", f"-Wl,-rpath,{libdir}"], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    assert out.split() == [str(len(names)), "ok"]
