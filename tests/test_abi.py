"""The C-ABI library loads and exports every entry point include/*.h
declares; host-side argument checks return statuses without a GPU."""
import ctypes
import glob
import os
import re

import state_space_sequence_06_b300 as m3
from state_space_sequence_06_b300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        for m in re.finditer(r"^M3_API\s+[^;(]*?\b(m3_\w+)\s*\(", open(h).read(), re.M):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_symbol():
    build.build()
    lib = m3.load_library()
    declared = declared_symbols()
    assert declared >= set(m3.SYMBOLS)
    for name in declared:
        assert hasattr(lib, name), f"{name} not exported"


def test_status_strings():
    assert m3.m3_status_string(m3.M3_OK) == "ok"
    assert "timed out" in m3.m3_status_string(m3.M3_ERR_TIMEOUT)
    assert m3.m3_status_string(99) == "unknown status"


def test_host_argument_checks_without_gpu():
    lib = m3.load_library()
    # null args / bad dims are rejected before any CUDA call
    assert lib.m3_scan_prefill(None, None, None) == m3.M3_ERR_INVALID_ARG
    assert lib.m3_decode_step(None, None, None) == m3.M3_ERR_INVALID_ARG
    out = ctypes.c_void_p()
    bad = m3.m3_dims(1, 1, 16, 15, 1, m3.M3_F32)  # odd N
    assert lib.m3_state_alloc(ctypes.byref(bad), ctypes.byref(out), None) == m3.M3_ERR_INVALID_ARG
    bad = m3.m3_dims(1, 1, 16, 16, 1, 7)  # unknown dtype
    assert lib.m3_state_alloc(ctypes.byref(bad), ctypes.byref(out), None) == m3.M3_ERR_INVALID_ARG
    a = m3.m3_prefill_args()
    a.dims = m3.m3_dims(1, 1, 16, 16, 1, m3.M3_F32)
    a.seqlen = 4
    assert lib.m3_scan_prefill(ctypes.byref(a), None, None) == m3.M3_ERR_INVALID_ARG  # null tensors
    for f in ("x", "B", "C", "dt", "lam", "theta", "A", "D", "y"):
        setattr(a, f, 4096)
    a.x = 4096 + 8  # misaligned
    assert lib.m3_scan_prefill(ctypes.byref(a), None, None) == m3.M3_ERR_INVALID_ARG
    a.x = 4096
    a.algo = 9
    assert lib.m3_scan_prefill(ctypes.byref(a), None, None) == m3.M3_ERR_INVALID_ARG
    assert lib.m3_state_view(None, None) == m3.M3_ERR_INVALID_ARG
    assert lib.m3_state_free(None) == m3.M3_OK
    # test hooks: unknown faults and negative limits are refused, NULL output too
    assert lib.m3_test_set_fault(7, 0) == m3.M3_ERR_INVALID_ARG
    assert lib.m3_test_set_fault(0, -1) == m3.M3_ERR_INVALID_ARG
    assert lib.m3_test_set_fault(0, 0) == m3.M3_OK
    assert lib.m3_test_last_launch(None) == m3.M3_ERR_INVALID_ARG


def _c_layout(tmp_path, structs):
    """sizeof and offsetof of each field, from the C compiler on the header."""
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "m3scan.h"', '#include "m3scan_backward.h"',
             '#include "m3scan_testing.h"', "int main(void) {"]
    for st, fields in structs.items():
        lines.append(f'  printf("{st} %zu\\n", sizeof({st}));')
        for f in fields:
            lines.append(f'  printf("{st}.{f} %zu\\n", offsetof({st}, {f}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    import subprocess

    subprocess.check_call(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)])
    out = subprocess.check_output([str(exe)], text=True)
    return dict((k, int(v)) for k, v in (ln.split() for ln in out.splitlines()))


def test_binding_structs_match_the_header_layout(tmp_path):
    """The ctypes argument structs the binding passes have the header's
    size and field offsets (a mismatch would hand the library garbage)."""
    structs = {"m3_dims": m3.m3_dims, "m3_state_ptrs": m3.m3_state_ptrs,
               "m3_prefill_args": m3.m3_prefill_args, "m3_decode_args": m3.m3_decode_args,
               "m3_backward_args": m3.m3_backward_args, "m3_launch_info": m3.m3_launch_info}
    layout = _c_layout(tmp_path, {name: [f for f, _ in cls._fields_] for name, cls in structs.items()})
    for name, cls in structs.items():
        assert layout[name] == ctypes.sizeof(cls), name
        for f, _ in cls._fields_:
            assert layout[f"{name}.{f}"] == getattr(cls, f).offset, f"{name}.{f}"
