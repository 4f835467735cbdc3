"""The Python binding's view of the C ABI agrees with include/kvrp.h.

Every prototype of the header is parsed and compared, argument by argument,
with the ctypes argtypes and restype the binding declares: the same count, the
same scalar widths (int32 / int64 / size_t / float / double), and a pointer
wherever the header has one.  The argument structs are compiled with the
host C compiler, and their size and every field offset are compared with the
ctypes Structures.  Nothing here needs a GPU."""
import ctypes as C
import os
import re
import shutil
import subprocess

import pytest

import position_invariant_kv_gb300._abi as abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvrp.h")

SCALARS = {"int32_t": C.c_int32, "int64_t": C.c_int64, "size_t": C.c_size_t, "double": C.c_double,
           "float": C.c_float, "kvrp_status": C.c_int, "uint32_t": C.c_uint32}


def _prototypes():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    out = {}
    for m in re.finditer(r"(kvrp_status|size_t|const char\*|int32_t|void)\s+(k\w+)\s*\(([^;]*?)\)\s*;", text):
        ret, name, args = m.group(1), m.group(2), " ".join(m.group(3).split())
        params = [] if args in ("", "void") else [a.strip() for a in args.split(",")]
        out[name] = (ret, params)
    return out


def _kind(param: str):
    """('ptr', None) for any pointer or array parameter, else ('scalar', ctype)."""
    if "*" in param or "[" in param or param.split()[0] == "kvrp_stream_t":
        return "ptr", None
    words = param.replace("const ", "").split()
    return "scalar", SCALARS[words[0]]


def _ctype_kind(t):
    if t in (C.c_void_p, C.c_char_p) or (isinstance(t, type) and issubclass(t, C._Pointer)):
        return "ptr", None
    return "scalar", t


def test_every_header_function_is_declared_alike_in_the_binding():
    lib = abi.lib()
    protos = _prototypes()
    assert set(protos) == set(abi.EXPORTED_SYMBOLS), set(protos) ^ set(abi.EXPORTED_SYMBOLS)
    for name, (ret, params) in protos.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, name
        assert len(fn.argtypes) == len(params), (name, len(fn.argtypes), len(params))
        for i, (p, t) in enumerate(zip(params, fn.argtypes)):
            want, got = _kind(p), _ctype_kind(t)
            assert want[0] == got[0], (name, i, p, t)
            if want[0] == "scalar":
                assert C.sizeof(want[1]) == C.sizeof(got[1]), (name, i, p, t)
                assert (want[1] in (C.c_float, C.c_double)) == (got[1] in (C.c_float, C.c_double)), (name, i, p, t)
        if ret == "void":
            assert fn.restype is None, name
            continue
        rt = {"kvrp_status": C.c_int, "size_t": C.c_size_t, "const char*": C.c_char_p, "int32_t": C.c_int32}[ret]
        assert C.sizeof(fn.restype) == C.sizeof(rt) and (fn.restype is C.c_char_p) == (rt is C.c_char_p), name


STRUCTS = {"kvrp_dst": abi.kvrp_dst, "kvrp_chunk": abi.kvrp_chunk, "kvrp_attn_chunk": abi.kvrp_attn_chunk,
           "kvrp_mla_chunk": abi.kvrp_mla_chunk}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs a host C compiler")
def test_struct_layouts_match_the_compiled_header(tmp_path):
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "kvrp.h"', "int main(void) {"]
    for sname, cls in STRUCTS.items():
        lines.append(f'  printf("{sname} size %zu\\n", sizeof({sname}));')
        for fname, _ in cls._fields_:
            lines.append(f'  printf("{sname} {fname} %zu\\n", offsetof({sname}, {fname}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = {}
    for ln in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines():
        s, f, v = ln.split()
        got[(s, f)] = int(v)
    for sname, cls in STRUCTS.items():
        assert got[(sname, "size")] == C.sizeof(cls), sname
        for fname, _ in cls._fields_:
            assert got[(sname, fname)] == getattr(cls, fname).offset, (sname, fname)
