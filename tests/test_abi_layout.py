"""Every structure the binding passes across the C ABI has the layout the C
compiler gives the header's declaration: field offsets and sizes, and the
structure's size (CPU; gcc compiles a probe against include/gpuos.h)."""
import ctypes as C
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _layouts(G):
    """{C struct name: (total size, [(field, offset, size)])} as the binding sees it."""
    out = {}
    for cname, cls in (("gpuos_config", G.Config), ("gpuos_record", G.Record),
                       ("gpuos_stats_t", G.Stats), ("gpuos_tile_profile", G.TileProfile)):
        out[cname] = (C.sizeof(cls), [(f, getattr(cls, f).offset, getattr(cls, f).size) for f, _ in cls._fields_])
    d = G.DESC_DTYPE
    out["gpuos_desc"] = (d.itemsize, [(f, d.fields[f][1], d.fields[f][0].itemsize) for f in d.names])
    return out


def test_binding_layouts_match_the_header(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    from persistent_micro_dispatch_gb300 import gpuos as G
    lay = _layouts(G)
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "gpuos.h"', "int main(void) {"]
    for t, (_, fields) in lay.items():
        lines.append(f'printf("{t} size %zu\\n", sizeof({t}));')
        for f, _, _ in fields:
            lines.append(f'printf("{t} {f} %zu %zu\\n", offsetof({t}, {f}), sizeof((({t} *)0)->{f}));')
    lines += ["return 0; }"]
    src = tmp_path / "probe.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = {}
    for line in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.splitlines():
        parts = line.split()
        if parts[1] == "size":
            got[(parts[0], "size")] = int(parts[2])
        else:
            got[(parts[0], parts[1])] = (int(parts[2]), int(parts[3]))
    for cname, (size, fields) in lay.items():
        assert got[(cname, "size")] == size, cname
        for f, off, sz in fields:
            assert got[(cname, f)] == (off, sz), (cname, f, got[(cname, f)], (off, sz))
