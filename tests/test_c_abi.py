"""The boundary is a C ABI: include/fab.h compiles as strict C99 and as C++17,
and programs in both languages link against libfab.so and call its host-only
entry points (layout and sizing, validation, status text) without a GPU.
The values they print must match what the ctypes binding reads."""
import os
import shutil
import subprocess

import pytest

from attention_backward_tcgen05_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <stdio.h>
#include "fab.h"

int main(void) {
  /* the packing test shape of the ggmlR test file: DK = 3, DV = 5 */
  fab_dims d = {2, 4, 2, 2, 4, 3, 5};
  size_t off_k = 0, off_v = 0, end = 0;
  int rc = fab_packed_offsets(&d, &off_k, &off_v, &end);
  fab_dims g = {4, 32, 8, 2048, 2048, 128, 128};
  fab_dims bad = {1, 3, 2, 1, 1, 1, 1}; /* H % Hkv != 0 */
  printf("%d %d %zu %zu %zu %zu %zu %zu %zu\n", fab_version(), rc, off_k, off_v, end, fab_packed_bytes(&d),
         fab_backward_workspace_bytes(&g, FAB_BF16), fab_backward_recompute_workspace_bytes(&g, FAB_BF16),
         fab_backward_workspace_bytes(&bad, FAB_BF16));
  /* validation runs on the host before anything is enqueued */
  printf("%d\n", fab_backward(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, 1.0f, FAB_BF16, &g, NULL, 0, NULL, NULL));
  printf("%s\n", fab_status_string(FAB_ERR_WORKSPACE));
  return 0;
}
"""


def _compile_and_run(tmp_path, compiler, std, suffix):
    cc = shutil.which(compiler)
    if cc is None:
        pytest.skip(f"{compiler} not installed")
    lib = binding.lib()  # builds nothing: loads (and so checks) the in-tree library
    del lib
    libdir = os.path.dirname(binding.LIB_PATH)
    src = tmp_path / f"abi{suffix}"
    src.write_text(PROGRAM)
    exe = tmp_path / f"abi_{compiler.replace('+', 'x')}"
    cmd = [cc, f"-std={std}", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE, str(src), "-o", str(exe),
           "-L", libdir, "-lfab", f"-Wl,-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    return out.stdout.splitlines()


def _expected():
    d = binding.make_dims(2, 4, 2, 2, 4, 3, 5)
    off_k, off_v, end = binding.fab_packed_offsets(d)
    g = binding.make_dims(4, 32, 8, 2048, 2048, 128, 128)
    bad = binding.make_dims(1, 3, 2, 1, 1, 1, 1)
    first = [binding.fab_version(), binding.FAB_OK, off_k, off_v, end, binding.fab_packed_bytes(d),
             binding.fab_backward_workspace_bytes(g, binding.FAB_BF16),
             binding.fab_backward_recompute_workspace_bytes(g, binding.FAB_BF16),
             binding.fab_backward_workspace_bytes(bad, binding.FAB_BF16)]
    return [" ".join(str(x) for x in first), str(binding.FAB_ERR_INVALID),
            binding.status_string(binding.FAB_ERR_WORKSPACE)]


@pytest.mark.parametrize("compiler,std,suffix", [("gcc", "c99", ".c"), ("g++", "c++17", ".cpp")])
def test_header_compiles_links_and_runs(tmp_path, compiler, std, suffix):
    lines = _compile_and_run(tmp_path, compiler, std, suffix)
    assert lines == _expected()
    # the ggmlR packing shape, worked by hand: q has 2*4*2*3 = 48 floats (192
    # bytes), k 2*2*4*3 = 48 (192), v 2*2*4*5 = 80 (320)
    off_k, off_v, end = (int(x) for x in lines[0].split()[2:5])
    assert (off_k, off_v, end) == (192, 384, 704)
