"""The ctypes mirrors of the C ABI structs (hstu_fwd_desc, hstu_fwd_kv, hstu_fwd_descale,
hstu_fwd_args) must match
include/hstu_fwd.h field by field: a small C program built with gcc prints every field's
offset and each struct's size, compared with the ctypes layout. CPU only."""
import ctypes
import os
import subprocess

import pytest

from hstu_dense_forward_gb300 import _abi

HEADER_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


def _c_layout(tmp_path, struct, fields):
    src = tmp_path / "layout.c"
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "hstu_fwd.h"',
             "int main(void) {",
             f'  printf("size %zu\\n", sizeof({struct}));']
    lines += [f'  printf("{f} %zu\\n", offsetof({struct}, {f}));' for f in fields]
    lines += ["  return 0;", "}"]
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c11", "-I", HEADER_DIR, "-o", str(exe), str(src)])
    out = subprocess.check_output([str(exe)]).decode().split("\n")
    return {k: int(v) for k, v in (line.split() for line in out if line)}


@pytest.mark.parametrize("struct,cls", [("hstu_fwd_desc", _abi.Desc), ("hstu_fwd_kv", _abi.KV),
                                        ("hstu_fwd_descale", _abi.Descale),
                                        ("hstu_fwd_args", _abi.Args)])
def test_ctypes_mirror_matches_header(tmp_path, struct, cls):
    fields = [f for f, _ in cls._fields_]
    c = _c_layout(tmp_path, struct, fields)
    assert c["size"] == ctypes.sizeof(cls)
    for f in fields:
        assert c[f] == getattr(cls, f).offset, f


def test_enum_values_match_header(tmp_path):
    src = tmp_path / "enums.c"
    names = ["HSTU_OK", "HSTU_ERR_INVALID_ARG", "HSTU_ERR_UNSUPPORTED", "HSTU_ERR_CUDA",
             "HSTU_ERR_TIMEOUT", "HSTU_ERR_DEVICE_CHECK", "HSTU_F32", "HSTU_F16", "HSTU_BF16",
             "HSTU_FP8_E4M3", "HSTU_MASK_CAUSAL", "HSTU_MASK_UPPER", "HSTU_MASK_NONE",
             "HSTU_MASK_CUSTOM", "HSTU_DEVERR_NONE", "HSTU_DEVERR_OFFSETS",
             "HSTU_DEVERR_TIMEOUT", "HSTU_LAYOUT_JAGGED", "HSTU_LAYOUT_NORMAL",
             "HSTU_DESCALE_CAST", "HSTU_DESCALE_TENSOR", "HSTU_DESCALE_BATCH",
             "HSTU_DESCALE_HEAD", "HSTU_DESCALE_BLOCK"]
    body = "\n".join(f'  printf("{n} %d\\n", (int){n});' for n in names)
    src.write_text('#include <stdio.h>\n#include "hstu_fwd.h"\nint main(void) {\n' + body +
                   "\n  return 0;\n}\n")
    exe = tmp_path / "enums"
    subprocess.check_call(["gcc", "-std=c11", "-I", HEADER_DIR, "-o", str(exe), str(src)])
    out = subprocess.check_output([str(exe)]).decode().split("\n")
    for line in out:
        if line:
            n, v = line.split()
            assert getattr(_abi, n) == int(v), n
