"""Every compute entry point of the C ABI opens a named range in the
"pagedkv" NVTX domain and closes it on return (early returns included), seen
through a recording NVTX tool injected the way profilers inject themselves
(no GPU: the calls are rejected on the host)."""

import os
import shutil
import subprocess
import sys
import textwrap

import pytest

from conftest import ROOT

ENTRY_CALLS = {
    "kv_append": "(None, None, None, None, I(1), None)",
    "copy_blocks": "(None, None, I(1), None)",
    "kv_swap_blocks": "(None, None, None, None, None, I(1), None, I(1), I(0), None)",
    "paged_attention_decode": "(None, None, None, None, I(1), None, I(1), I(1), F(1.0), I(1), "
                              "None, S(0), None)",
    "paged_attention_decode_cascade": "(None, None, None, None, I(1), None, I(1), I(1), F(1.0), "
                                      "I(1), None, None, None, I(0), None, S(0), None)",
    "paged_attention_prefill": "(None, None, None, None, I(1), I(1), None, I(1), None, I(1), "
                               "I(1), F(1.0), I(1), None)",
    "paged_attention_decode_noalloc": "(None, None, None, None, I(1), None, I(1), I(1), F(1.0), "
                                      "I(1), None)",
}


def test_each_entry_point_is_one_nvtx_range(tmp_path):
    from paged_kv_cache_68_gb300 import _build, pagedkv
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(_build._nvcc())), "include")
    if not os.path.exists(os.path.join(cuda_inc, "nvtx3", "nvToolsExt.h")):
        pytest.skip("no NVTX headers")
    pagedkv.load()
    tool = tmp_path / "libnvtx_record.so"
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-fPIC", "-shared", "-I", cuda_inc,
                    os.path.join(ROOT, "tests", "nvtx_record.c"), "-o", str(tool)],
                   check=True, capture_output=True)
    calls = "\n".join(f"print('{n}', lib.{n}{a})" for n, a in ENTRY_CALLS.items())
    script = textwrap.dedent(f"""\
        import ctypes
        I, F, S = ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib = ctypes.CDLL({pagedkv.library_path()!r})
        tool = ctypes.CDLL({str(tool)!r})
        tool.injection_log.restype = ctypes.c_char_p
        """) + calls + "\nprint(tool.injection_log().decode(), end='')\n"
    env = dict(os.environ, NVTX_INJECTION64_PATH=str(tool))
    out = subprocess.run([sys.executable, "-c", script], env=env, check=True,
                         capture_output=True, text=True).stdout.splitlines()
    n = len(ENTRY_CALLS)
    status, events = out[:n], out[n:]
    for line, name in zip(status, ENTRY_CALLS):
        assert line == f"{name} 1", line          # KV_EINVAL: a null pool
    expect = ["domain pagedkv"]
    for name in ENTRY_CALLS:
        expect += [f"push pagedkv {name}", "pop pagedkv"]
    assert events == expect
