"""The Python binding against the C header, on the CPU: the ctypes mirrors of the
parameter structs have the C compiler's size and field offsets (compiled from
include/sp.h with the host C compiler), and every function's declared argument types
have as many entries as its prototype in the header has parameters.  Drift between the
header and the binding would otherwise pass arguments in the wrong places silently."""
import ctypes
import json
import os
import re
import subprocess

import pytest

from sequence_head_attention_seq_b300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sp.h")

MIRRORS = {"sp_attn_params": binding.SpAttnParams, "sp_merge_params": binding.SpMergeParams,
           "sp_ulysses_host_params": binding.SpUlyssesHostParams}


def _c_layout(tmp_path):
    """sizeof and offsetof of every mirrored field, from gcc on the header."""
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "sp.h"', "int main(void) {",
             '  printf("{");']
    first = True
    for cname, mirror in MIRRORS.items():
        sep = "" if first else ","
        first = False
        lines.append(f'  printf("{sep}\\"{cname}\\": {{\\"size\\": %zu", sizeof({cname}));')
        for field, _ in mirror._fields_:
            lines.append(f'  printf(", \\"{field}\\": %zu", offsetof({cname}, {field}));')
        lines.append('  printf("}");')
    lines += ['  printf("}\\n");', "  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), "-o", str(exe), str(src)],
                   check=True, capture_output=True, text=True)
    return json.loads(subprocess.run([str(exe)], check=True, capture_output=True,
                                     text=True).stdout)


def test_struct_mirrors_match_the_header(tmp_path):
    c = _c_layout(tmp_path)
    for cname, mirror in MIRRORS.items():
        assert ctypes.sizeof(mirror) == c[cname]["size"], cname
        for field, _ in mirror._fields_:
            assert getattr(mirror, field).offset == c[cname][field], f"{cname}.{field}"


def _prototypes():
    """Function name -> parameter count, from the header's declarations."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    protos = {}
    for m in re.finditer(r"\b(sp_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text):
        name, params = m.group(1), m.group(2).strip()
        protos[name] = 0 if params in ("", "void") else params.count(",") + 1
    return protos


def test_argument_counts_match_the_prototypes():
    lib = binding.load()
    protos = _prototypes()
    assert sorted(protos) == sorted(binding.EXPORTS)
    for name, count in protos.items():
        argtypes = getattr(lib, name).argtypes
        if count == 0:
            assert not argtypes, name
        else:
            assert argtypes is not None and len(argtypes) == count, (name, count, argtypes)


@pytest.mark.parametrize("name,value", [("SP_NOALLOC_SCRATCH_BYTES",
                                         binding.NOALLOC_SCRATCH_BYTES),
                                        ("SP_MAX_RELAYOUT_TENSORS",
                                         binding.MAX_RELAYOUT_TENSORS)])
def test_constants_match_the_header(tmp_path, name, value):
    src = tmp_path / "c.c"
    src.write_text(f'#include <stdio.h>\n#include "sp.h"\n'
                   f'int main(void) {{ printf("%llu", (unsigned long long)({name})); return 0; }}\n')
    exe = tmp_path / "c"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), "-o", str(exe), str(src)],
                   check=True, capture_output=True, text=True)
    assert int(subprocess.run([str(exe)], check=True, capture_output=True,
                              text=True).stdout) == value
