"""The C ABI on the host: the library loads, exports every declared symbol,
and rejects bad arguments before enqueueing anything (no GPU needed).

Every call below fails host-side validation, so none of them reaches a CUDA
launch even on a machine with a GPU; the launch counter proves it.
"""
import ctypes
import os
import re

import pytest

import perfectly_balanced_token_gb300 as mx
from perfectly_balanced_token_gb300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "moonep.h")


@pytest.fixture(scope="module", autouse=True)
def lib():
    from perfectly_balanced_token_gb300.build import build
    build()
    return mx.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moonep_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) == 20, names
    for n in names:
        assert hasattr(lib, n), n


def test_dims_validation():
    good = mx.dims(8, 384, 48, 8, 8192, 7168, 2048)
    assert mx.moonep_plan_workspace_bytes(good) > 0
    cases = {
        _lib.ERR_SLOTS: mx.dims(8, 384, 47, 8, 8192, 7168, 2048, 0),
        _lib.ERR_SHAPE: mx.dims(8, 380, 48, 8, 8192, 7168, 2048),
        _lib.ERR_ARG: mx.dims(8, 384, 48, 8, 8192, 7168, 2048, 2),
    }
    for code, d in cases.items():
        with pytest.raises(mx.MoonepError) as ei:
            mx.moonep_plan_workspace_bytes(d)
        assert ei.value.status == code
    shape_bad = [mx.dims(8, 384, 48, 385, 8192, 7168, 2048),   # K > E
                 mx.dims(8, 384, 48, 8, 8192, 7100, 2048),     # H % 64
                 mx.dims(8, 384, 48, 8, 8192, 7168, 2000),     # Hp % 64
                 mx.dims(2, 8192, 4096, 8, 16, 64, 64),        # E > 4096
                 mx.dims(8, 64, 65, 4, 16, 64, 64, 1),         # B > E
                 mx.dims(8, 64, 8, 64, 1 << 23, 64, 64)]       # N >= 2^31
    for d in shape_bad:
        with pytest.raises(mx.MoonepError) as ei:
            mx.moonep_plan_workspace_bytes(d)
        assert ei.value.status == _lib.ERR_SHAPE
    for d in [mx.dims(0, 8, 2, 2, 16, 64, 64), mx.dims(4, 8, -1, 2, 16, 64, 64, 1),
              mx.dims(4, 8, 2, 2, 0, 64, 64), mx.dims(4, 8, 2, 0, 16, 64, 64),  # S = 0, K = 0
              mx.dims(4, 0, 0, 2, 16, 64, 64, 1), mx.dims(4, 8, 2, 2, 16, 0, 64),
              mx.dims(4, 8, 2, 2, 16, 64, 0),
              mx.dims(4, 8, 2, 2, 16, 64, 64, 0, 2), mx.dims(4, 8, 2, 2, 16, 64, 64, 0, 0, 64),
              mx.dims(4, 8, 2, 2, 16, 64, 64, 0, 0, 512)]:
        with pytest.raises(mx.MoonepError) as ei:
            mx.moonep_plan_workspace_bytes(d)
        assert ei.value.status == _lib.ERR_ARG
    # inference mode accepts B < E/R, including B = 0
    assert mx.moonep_plan_workspace_bytes(mx.dims(8, 384, 0, 8, 8192, 7168, 2048, 1)) > 0
    # the work-tile height may be left to the plan or fixed; the workspace has
    # room for the longer tile list either way
    sizes = {r: mx.moonep_plan_workspace_bytes(mx.dims(8, 384, 48, 8, 8192, 7168, 2048, 0, 0, r))
             for r in (0, 128, 256)}
    assert sizes[0] == sizes[128] == sizes[256] > 0


def test_layout_tables_are_aligned_and_inside():
    d = mx.dims(64, 896, 14, 16, 1024, 4096, 1024)
    lay = mx.moonep_get_plan_layout(d)
    offs = [getattr(lay, f) for f in _lib._LAYOUT_FIELDS[1:]]
    assert lay.counters == 64 and lay.status == 0
    for o in offs[2:]:
        assert o % 256 == 0 and o < lay.total_bytes
    assert lay.nchunk == 4 and lay.max_mtiles >= d.N // 128
    # the GEMMs' scratch is the workspace's tail, past every table
    assert max(offs) + 4 <= lay.total_bytes - mx.GEMM_SCRATCH_BYTES
    hdr = open(HEADER).read()
    m = re.search(r"#define MOONEP_GEMM_SCRATCH_BYTES \((\d+)u << (\d+)\)", hdr)
    assert m and int(m.group(1)) << int(m.group(2)) == mx.GEMM_SCRATCH_BYTES


def test_bad_pointers_rejected_before_launch(lib):
    n0 = mx.moonep_launch_count()
    d = mx.dims(4, 8, 2, 2, 16, 64, 128)
    D = ctypes.byref(d)
    P = ctypes.c_void_p
    ws, ok, odd = P(0x10000), P(0x20000), P(0x20004)
    assert lib.moonep_plan(D, None, ws, None) == _lib.ERR_ARG
    assert lib.moonep_plan(D, odd, ws, None) == _lib.ERR_ALIGN
    assert lib.moonep_plan(D, ok, None, None) == _lib.ERR_ARG
    assert lib.moonep_plan(D, ok, P(0x10008), None) == _lib.ERR_ALIGN
    assert lib.moonep_dispatch(D, ws, ok, None, None) == _lib.ERR_ARG
    assert lib.moonep_dispatch(D, ws, odd, ok, None) == _lib.ERR_ALIGN
    assert lib.moonep_dispatch_send_once(D, ws, ok, ok, ok, None, None) == _lib.ERR_ARG
    assert lib.moonep_dispatch_send_once(D, ws, ok, odd, ok, ok, None) == _lib.ERR_ALIGN
    assert lib.moonep_prefetch_weights(D, ws, ok, None, None) == _lib.ERR_ARG
    assert lib.moonep_grouped_gemm(D, ws, ok, ok, None, ok, None) == _lib.ERR_ARG
    assert lib.moonep_grouped_gemm(D, ws, ok, odd, ok, ok, None) == _lib.ERR_ALIGN
    assert lib.moonep_combine(D, ws, ok, None, ok, None) == _lib.ERR_ARG
    assert lib.moonep_reduce_grad(D, ws, ok, None, None) == _lib.ERR_ARG
    assert lib.moonep_read_status(D, ws, None, None) == _lib.ERR_ARG
    assert lib.moonep_plan_export(D, ws, None, None) == _lib.ERR_ARG
    assert lib.moonep_combine_backward(D, ws, ok, ok, ok, ok, None, None) == _lib.ERR_ARG
    assert lib.moonep_grouped_gemm_dx(D, ws, ok, ok, ok, None, None) == _lib.ERR_ARG
    assert lib.moonep_grouped_gemm_dw(D, ws, ok, ok, ok, None, None) == _lib.ERR_ARG
    assert lib.moonep_dispatch_backward(D, ws, odd, ok, None) == _lib.ERR_ALIGN
    infer = mx.dims(4, 8, 2, 2, 16, 128, 128, 1)
    assert lib.moonep_grouped_gemm_dw(ctypes.byref(infer), ws, ok, ok, ok, ok, None) == _lib.ERR_ARG
    h64 = mx.dims(4, 8, 2, 2, 16, 64, 128, 0)
    assert lib.moonep_grouped_gemm_dw(ctypes.byref(h64), ws, ok, ok, ok, ok, None) == _lib.ERR_SHAPE
    bad = mx.dims(4, 8, 1, 2, 16, 64, 128, 0)
    assert lib.moonep_plan(ctypes.byref(bad), ok, ws, None) == _lib.ERR_SLOTS
    assert lib.moonep_plan(None, ok, ws, None) == _lib.ERR_ARG
    assert mx.moonep_launch_count() == n0


def test_noalloc_planner_rejects_dims_beyond_its_scratch(lib):
    # R*nchunk*E = 64*10*4096 chunk counters alone exceed the 4 MiB array
    n0 = mx.moonep_launch_count()
    big = mx.dims(64, 4096, 64, 1, 40960, 64, 64)
    rc = lib.moonep_plan_noalloc(ctypes.byref(big), ctypes.c_void_p(0x20000),
                                 ctypes.c_void_p(0x10000), None)
    assert rc == _lib.ERR_SCRATCH
    assert "scratch" in mx.status_string(rc)
    assert mx.moonep_launch_count() == n0


def test_selftest_wait_rejects_bad_arguments(lib):
    n0 = mx.moonep_launch_count()
    P = ctypes.c_void_p
    assert lib.moonep_selftest_bounded_wait(None, 1000, P(0x1000), None) == _lib.ERR_ARG
    assert lib.moonep_selftest_bounded_wait(P(0x1000), 0, P(0x1004), None) == _lib.ERR_ARG
    assert lib.moonep_selftest_bounded_wait(P(0x1000), 1000001, P(0x1004), None) == _lib.ERR_ARG
    assert lib.moonep_selftest_bounded_wait(P(0x1002), 1000, P(0x1004), None) == _lib.ERR_ALIGN
    assert mx.moonep_launch_count() == n0


def test_status_strings():
    for code in (0, 1, 2, 3, 4, 5, 6, 0x100, 0x200, 0x400, 0x300):
        s = mx.status_string(code)
        assert s and s != "unknown status"


def test_binding_requires_cuda_tensors():
    import torch
    d = mx.dims(4, 8, 2, 2, 16, 64, 128)
    with pytest.raises(ValueError):
        mx.moonep_plan(d, torch.zeros(4 * 16 * 2, dtype=torch.int32),
                       torch.zeros(mx.moonep_plan_workspace_bytes(d), dtype=torch.uint8))


def test_missing_library_fails_loudly(monkeypatch):
    # no fallback: with the shared library absent the first call raises
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", "/nonexistent/libmoonep.so")
    with pytest.raises(ImportError):
        _lib.library()
    with pytest.raises(ImportError):
        mx.moonep_plan_workspace_bytes(mx.dims(4, 8, 2, 2, 16, 64, 64))


C_CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "moonep.h"

int main(void) {
  moonep_dims d;
  size_t bytes = 0;
  moonep_plan_layout lay;
  memset(&d, 0, sizeof d);
  d.R = 8; d.E = 384; d.B = 48; d.K = 8; d.S = 8192; d.H = 7168; d.Hp = 2048;
  if (moonep_plan_workspace_bytes(&d, &bytes) != MOONEP_OK || bytes == 0) return 1;
  const size_t total = bytes;
  if (moonep_get_plan_layout(&d, &lay) != MOONEP_OK || lay.total_bytes != total) return 2;
  if (lay.cu_seqlens % 256 != 0 || lay.dst % 256 != 0 || lay.route + 4 > total) return 3;
  d.B = 47; /* training needs B >= E/R */
  if (moonep_plan_workspace_bytes(&d, &bytes) != MOONEP_ERR_SLOTS) return 4;
  if (moonep_plan_workspace_bytes(NULL, &bytes) != MOONEP_ERR_ARG) return 5;
  if (strlen(moonep_status_string(MOONEP_ERR_ROUTING)) == 0) return 6;
  {
    /* views are host arithmetic on the layout: no GPU work, any aligned base */
    moonep_plan_view v;
    const char* base = (const char*)0 + 4096;
    d.B = 48;
    if (moonep_plan_views(&d, base, &v) != MOONEP_OK) return 7;
    if ((const char*)v.cu_seqlens != base + lay.cu_seqlens || (const char*)v.dst != base + lay.dst ||
        (const char*)v.inverse != base + lay.inverse || (const char*)v.slot_expert != base + lay.slot_expert ||
        (const char*)v.status != base + lay.status) return 8;
    if (moonep_plan_views(&d, base + 8, &v) != MOONEP_ERR_ALIGN) return 9;
    if (moonep_plan_views(&d, NULL, &v) != MOONEP_ERR_ARG) return 10;
  }
  printf("%zu\n", total);
  return 0;
}
"""


def test_header_is_plain_c_and_links(tmp_path, lib):
    # a C99 program against the public header and the shared library alone
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from perfectly_balanced_token_gb300.build import LIB
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER),
                        str(src), LIB, f"-Wl,-rpath,{os.path.dirname(LIB)}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stderr)
    total = mx.moonep_plan_workspace_bytes(mx.dims(8, 384, 48, 8, 8192, 7168, 2048))
    assert r.stdout.split()[0] == str(total)


def test_binding_structs_match_the_header(tmp_path):
    # field offsets and sizes of the ctypes structures equal the C compiler's
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"moonep_dims": _lib.moonep_dims, "moonep_plan_layout": _lib.moonep_plan_layout,
               "moonep_plan_view": _lib.moonep_plan_view}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "moonep.h"', 'int main(void) {']
    for sname, cls in structs.items():
        lines.append(f'  printf("{sname} sizeof %zu\\n", sizeof({sname}));')
        for fname, _ in cls._fields_:
            lines.append(f'  printf("{sname} {fname} %zu\\n", offsetof({sname}, {fname}));')
    lines += ['  return 0;', '}']
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    r = subprocess.run([cc, "-std=c99", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60).stdout.split("\n")
    got = {tuple(ln.split()[:2]): int(ln.split()[2]) for ln in out if ln.strip()}
    for sname, cls in structs.items():
        assert got[(sname, "sizeof")] == ctypes.sizeof(cls), sname
        for fname, _ in cls._fields_:
            assert got[(sname, fname)] == getattr(cls, fname).offset, (sname, fname)
    # and every field the header declares is in the binding
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct moonep_plan_layout \{(.*?)\}", text, flags=re.S).group(1)
    declared = re.findall(r"\b(\w+)\s*;", body)
    assert declared == [f for f, _ in _lib.moonep_plan_layout._fields_]


def test_plan_views_point_at_the_layout_tables(lib):
    # host-only: the view of a workspace at any aligned device address is that
    # address plus the layout's offsets
    d = mx.dims(8, 64, 8, 4, 1024, 1024, 512)
    lay = mx.moonep_get_plan_layout(d)
    base = 1 << 30
    v = mx.moonep_plan_views(d, base)
    assert v == {"cu_seqlens": base + lay.cu_seqlens, "dst": base + lay.dst,
                 "inverse": base + lay.inverse, "slot_expert": base + lay.slot_expert,
                 "status": base + lay.status}
    with pytest.raises(mx.MoonepError):
        mx.moonep_plan_views(d, base + 4)
