"""The C-ABI library loads and exports every entry point that include/pa.h declares;
host-side validation answers without a GPU. No compute call is made here."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_107_gb300 as pk
from paged_kv_cache_107_gb300 import build as lib_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "pa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(pa_[a-z_0-9]+)\s*\(", text, re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    path = lib_build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("pa_store_kvcache", "pa_decode", "pa_decode_step", "pa_decode_workspace_size",
                 "pa_prefill_varlen", "pa_status_str", "pa_version"):
        assert must in names, names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} missing from {lib_build.LIB_PATH}"


def test_binding_has_same_names():
    for name in declared_functions():
        assert hasattr(pk, name), name


def test_status_strings_and_version():
    pk.load_library()
    assert pk.pa_status_str(0) == "PA_OK"
    assert "SHAPE" in pk.pa_status_str(2)
    assert pk.pa_version() >> 16 == 1


def test_validation_without_launch(lib):
    """Shape errors are caught before any CUDA call, so they answer on a CPU machine too."""
    lib.pa_decode.restype = ctypes.c_int
    vp = ctypes.c_void_p(16)
    # H % Hk != 0
    rc = lib.pa_decode(vp, vp, vp, vp, vp, 1, vp, 2, 12, 8, 128, 1, 16, ctypes.c_int64(4),
                       ctypes.c_float(0), 0, vp, ctypes.c_size_t(1 << 20), None, None)
    assert rc == 2
    # head_dim 96; element type F32 (not an attention type)
    rc = lib.pa_decode(vp, vp, vp, vp, vp, 1, vp, 2, 16, 8, 96, 1, 16, ctypes.c_int64(4),
                       ctypes.c_float(0), 0, vp, ctypes.c_size_t(1 << 20), None, None)
    assert rc == 3
    rc = lib.pa_decode(vp, vp, vp, vp, vp, 1, vp, 2, 16, 8, 64, 0, 16, ctypes.c_int64(4),
                       ctypes.c_float(0), 0, vp, ctypes.c_size_t(1 << 20), None, None)
    assert rc == 3
    # store: negative token count, bad stride
    lib.pa_store_kvcache.restype = ctypes.c_int
    rc = lib.pa_store_kvcache(vp, vp, ctypes.c_int64(1024), ctypes.c_int64(1024), vp, vp, vp, -1,
                              8, 128, 16, ctypes.c_int64(4), None, None)
    assert rc == 2
    rc = lib.pa_store_kvcache(vp, vp, ctypes.c_int64(10), ctypes.c_int64(1024), vp, vp, vp, 3, 8,
                              128, 16, ctypes.c_int64(4), None, None)
    assert rc == 2
    # zero tokens is a successful no-op without touching CUDA
    rc = lib.pa_store_kvcache(None, None, ctypes.c_int64(1024), ctypes.c_int64(1024), None, None,
                              None, 0, 8, 128, 16, ctypes.c_int64(4), None, None)
    assert rc == 0
    # fused step: token stride below one row; head_dim 64; zero sequences is a no-op
    lib.pa_decode_step.restype = ctypes.c_int
    i64 = ctypes.c_int64

    def step(kstride, head_dim, B):
        return lib.pa_decode_step(vp, vp, vp, vp, i64(kstride), i64(1024), vp, vp, vp, vp, 1, vp,
                                  B, 16, 8, head_dim, 1, 16, i64(4), ctypes.c_float(0), 0, vp,
                                  ctypes.c_size_t(1 << 20), None, None)
    assert step(1000, 128, 2) == 2
    assert step(1024, 32, 2) == 3
    assert step(1024, 128, 0) == 0
    # sampler: row stride below the vocabulary, unknown dtype, zero rows
    lib.pa_gumbel_sample.restype = ctypes.c_int
    lib.pa_sample_workspace_size.restype = ctypes.c_size_t

    def sample(stride, dtype, B):
        return lib.pa_gumbel_sample(vp, vp, i64(stride), dtype, B, 100, vp, vp, vp, vp,
                                    ctypes.c_size_t(1 << 20), None, None)
    assert sample(99, 0, 4) == 2
    assert sample(100, 7, 4) == 3
    assert sample(100, 0, 0) == 0
    assert lib.pa_sample_workspace_size(-1) == 0 and lib.pa_sample_workspace_size(256) >= 256 * 12
    # prefill: max_seqlen_k beyond what the table maps
    lib.pa_prefill_varlen.restype = ctypes.c_int
    rc = lib.pa_prefill_varlen(vp, vp, vp, vp, vp, 2, vp, vp, 1, 10, 600, 16, 8, 128, 1, 256,
                               ctypes.c_int64(4), 1, ctypes.c_float(0), None, None)
    assert rc in (2, 3)
    # empty batches are successful no-ops that touch neither the pointers nor CUDA
    rc = lib.pa_decode(None, None, None, None, None, 0, None, 0, 16, 8, 128, 1, 16,
                       ctypes.c_int64(4), ctypes.c_float(0), 0, None, ctypes.c_size_t(0), None,
                       None)
    assert rc == 0
    rc = lib.pa_prefill_varlen(None, None, None, None, None, 0, None, None, 0, 0, 0, 16, 8, 128,
                               1, 256, ctypes.c_int64(4), 1, ctypes.c_float(0), None, None)
    assert rc == 0


def test_header_is_plain_c_and_links(lib, tmp_path):
    """include/pa.h compiles as C99 with every warning an error, and a C program that takes
    the address of every declared function links against the library: the boundary
    needs no C++ and no torch."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = declared_functions()
    src = tmp_path / "uses_pa.c"
    body = "\n".join(f"  fns[{i}] = (void (*)(void)){n};" for i, n in enumerate(names))
    src.write_text('#include "pa.h"\n#include <stdio.h>\n'
                   "int main(void) {\n"
                   f"  void (*fns[{len(names)}])(void);\n{body}\n"
                   f"  printf(\"%s %d\\n\", pa_status_str(PA_OK), {len(names)});\n"
                   "  return fns[0] == 0;\n}\n")
    exe = tmp_path / "uses_pa"
    libdir = os.path.dirname(lib_build.LIB_PATH)
    libname = os.path.basename(lib_build.LIB_PATH)[3:-3]  # libX.so -> X
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.dirname(HEADER), str(src), "-o", str(exe),
           "-L", libdir, f"-l{libname}", f"-Wl,-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_runs_the_host_paths(lib, tmp_path):
    """A C program, linked against the library, runs the entry points that need no GPU and
    checks their results: version and status strings, empty batches and shape errors
    answered before any CUDA call, and pa_staged_pack, whose packed runs, applied to a
    host table, must equal the staged writes applied one after another in staging order
    (later writes win where they overlap)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "host_paths.c"
    src.write_text(r'''
#include "pa.h"
#include <stdio.h>
#include <string.h>

#define CHECK(c) do { if (!(c)) { printf("failed: %s (line %d)\n", #c, __LINE__); return 1; } } while (0)

int main(void) {
  CHECK(pa_version() >> 16 == 1);
  CHECK(strcmp(pa_status_str(PA_OK), "PA_OK") == 0);
  CHECK(pa_store_kvcache(NULL, NULL, 1024, 1024, NULL, NULL, NULL, 0, 8, 128, 16, 4, NULL,
                         NULL) == PA_OK);
  CHECK(pa_decode(NULL, NULL, NULL, NULL, NULL, 0, NULL, 0, 16, 8, 128, PA_DTYPE_BF16, 16, 4,
                  0.f, 0, NULL, 0, NULL, NULL) == PA_OK);
  CHECK(pa_decode(NULL, NULL, NULL, NULL, NULL, 1, NULL, 2, 12, 8, 128, PA_DTYPE_BF16, 16, 4,
                  0.f, 0, NULL, 0, NULL, NULL) == PA_ERR_SHAPE);
  CHECK(pa_prefill_varlen(NULL, NULL, NULL, NULL, NULL, 0, NULL, NULL, 0, 0, 0, 16, 8, 128,
                          PA_DTYPE_BF16, 256, 4, 1, 0.f, NULL, NULL) == PA_OK);
  CHECK(pa_sample_workspace_size(-1) == 0);

  /* staged writes, in staging order: later ones win where they overlap */
  enum { R = 6, C = 12, W = 5 };
  const int32_t rows[W] = {3, 0, 3, 5, 3};
  const int32_t starts[W] = {4, 0, 2, 10, 6};
  const int32_t lens[W] = {3, 2, 3, 2, 1};
  const int32_t vals[11] = {10, 11, 12, 20, 21, 30, 31, 32, 40, 41, 50};
  int32_t expect[R][C], got[R][C];
  memset(expect, 0xff, sizeof expect);
  memcpy(got, expect, sizeof got);
  int v = 0;
  for (int w = 0; w < W; ++w)
    for (int i = 0; i < lens[w]; ++i) expect[rows[w]][starts[w] + i] = vals[v++];
  unsigned char packed[1024] __attribute__((aligned(16)));
  pa_staged_layout lay;
  CHECK(pa_staged_pack_bound(W, 11, 4) <= sizeof packed);
  CHECK(pa_staged_pack(rows, starts, lens, vals, W, 4, packed, sizeof packed, &lay) == PA_OK);
  CHECK(lay.num_writes >= 1 && lay.num_writes <= W && lay.bytes <= (int64_t)sizeof packed);
  const int32_t* pr = (const int32_t*)(packed + lay.rows_offset);
  const int32_t* ps = (const int32_t*)(packed + lay.starts_offset);
  const int32_t* po = (const int32_t*)(packed + lay.offsets_offset);
  const int32_t* pv = (const int32_t*)(packed + lay.values_offset);
  CHECK(lay.values_offset % 16 == 0 && po[0] == 0 && po[lay.num_writes] == lay.num_values);
  for (int w = 0; w < lay.num_writes; ++w) {
    CHECK(po[w + 1] >= po[w]);
    for (int i = 0; i < po[w + 1] - po[w]; ++i) got[pr[w]][ps[w] + i] = pv[po[w] + i];
  }
  CHECK(memcmp(got, expect, sizeof got) == 0);
  /* a buffer too small reports the size it needs */
  pa_staged_layout small;
  CHECK(pa_staged_pack(rows, starts, lens, vals, W, 4, packed, 8, &small) == PA_ERR_WORKSPACE);
  CHECK(small.bytes == lay.bytes);
  printf("ok %d runs\n", lay.num_writes);
  return 0;
}
''')
    exe = tmp_path / "host_paths"
    libdir = os.path.dirname(lib_build.LIB_PATH)
    libname = os.path.basename(lib_build.LIB_PATH)[3:-3]
    cmd = [cc, "-std=gnu99", "-Wall", "-Wextra", "-Werror", "-I", os.path.dirname(HEADER),
           str(src), "-o", str(exe), "-L", libdir, f"-l{libname}", f"-Wl,-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok")
