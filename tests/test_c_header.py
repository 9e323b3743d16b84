"""The boundary from plain C, without a GPU: include/gdn.h compiles as strict
C11 (warnings as errors), a C program that takes the address of every entry
point the header declares links against libgdn.so, and its host-only calls
answer.  A declared entry point the library does not export fails the link."""
from __future__ import annotations

import os
import re
import shutil
import subprocess

import pytest

from chunkwise_gated_delta_gdn_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    with open(os.path.join(ROOT, "include", "gdn.h")) as f:
        src = f.read()
    return sorted(set(re.findall(r"GDN_API\s+[\w\s\*]*?\b(gdn_\w+)\s*\(", src)))


PROGRAM = r"""
#include <stdio.h>
#include <string.h>

#include "gdn.h"

typedef void (*entry_fn)(void);

int main(void) {
  const entry_fn entries[] = {
%(entries)s
  };
  size_t i;
  for (i = 0; i < sizeof entries / sizeof entries[0]; i++)
    if (!entries[i]) return 2;
  if (gdn_version() <= 0) return 3;
  if (strcmp(gdn_status_string(GDN_OK), "GDN_OK") != 0) return 4;
  if (strcmp(gdn_status_string(GDN_ERR_UNSUPPORTED), "GDN_ERR_UNSUPPORTED") != 0) return 5;
  printf("%%d %%u\n", gdn_version(), (unsigned)(sizeof entries / sizeof entries[0]));
  return 0;
}
"""


def test_header_compiles_and_links_as_c(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = cuda_build.build()
    names = declared_symbols()
    assert names, "no entry points found in include/gdn.h"
    src = tmp_path / "use_gdn.c"
    src.write_text(PROGRAM % {"entries": "\n".join(f"      (entry_fn){n}," for n in names)})
    exe = tmp_path / "use_gdn"
    libdir = os.path.dirname(lib)
    cmd = [cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
           "-L", libdir, "-lgdn", f"-Wl,-rpath,{libdir}"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr[-3000:]
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, (run.returncode, run.stderr[-2000:])
    version, count = run.stdout.split()
    assert int(version) > 0 and int(count) == len(names)
