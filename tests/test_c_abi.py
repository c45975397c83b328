"""The C ABI from C: include/zero.h compiles as C99 and a C program links the
library and calls its host-only entry points (no GPU needed). The layout it
reports is checked against the worked case of the layout pins."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "mixed_precision_gb300")

PROGRAM = r"""
#include <stdio.h>
#include <stdint.h>
#include "zero.h"

int main(void) {
  /* sizes 100, 30, 200; W = 2; 512-byte buckets of bf16 (256 elements) */
  int64_t s0[1] = {100}, s1[1] = {30}, s2[2] = {10, 20};
  const int64_t* shapes[3] = {s0, s1, s2};
  int ndims[3] = {1, 1, 2};
  zero_config cfg = {2, 2, 512, ZERO_BF16, ZERO_BF16, -1, 0};
  zero_layout_t* L = NULL;
  if (zero_layout_create(shapes, ndims, 3, &cfg, &L) != ZERO_OK) {
    printf("create failed: %s\n", zero_last_error());
    return 1;
  }
  zero_layout_info info;
  if (zero_layout_query(L, &info) != ZERO_OK) return 2;
  int64_t off[3];
  for (int p = 0; p < 3; ++p)
    if (zero_param_offset(L, p, &off[p]) != ZERO_OK) return 3;
  int64_t f0, s, n;
  if (zero_shard_range(L, 1, 1, &f0, &s, &n) != ZERO_OK) return 4;
  printf("%lld %lld %lld %lld %lld %lld %lld %lld %lld\n", (long long)info.n_real,
         (long long)info.n_padded, (long long)info.n_buckets, (long long)off[0],
         (long long)off[1], (long long)off[2], (long long)f0, (long long)s, (long long)n);
  /* errors come back as codes with a message, never as a crash */
  zero_config bad = cfg;
  bad.world = 0;
  zero_layout_t* L2 = NULL;
  int rc = zero_layout_create(shapes, ndims, 3, &bad, &L2);
  printf("%d %d\n", rc, L2 == NULL);
  zero_layout_destroy(L);
  zero_layout_destroy(NULL);
  return 0;
}
"""


@pytest.fixture(scope="module")
def lib_path():
    from mixed_precision_gb300 import build
    build.build()
    return os.path.join(PKG, "libzero_gb300.so")


def test_header_compiles_as_c99_and_links(tmp_path, lib_path):
    src = tmp_path / "use_zero.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_zero"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", PKG, "-lzero_gb300", f"-Wl,-rpath,{PKG}"],
                   check=True, capture_output=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert res.returncode == 0, res.stdout + res.stderr
    first, second = res.stdout.strip().splitlines()
    n_real, n_padded, n_buckets, o0, o1, o2, f0, s, n = map(int, first.split())
    # 330 elements; p0 at 0, p1 at 128 (span 158 <= 256), p2 (200 elements)
    # would end at 392 > 256 and opens bucket 1 at 256; both buckets padded
    # to 2 * 128
    assert (n_real, n_padded, n_buckets) == (330, 512, 2)
    assert (o0, o1, o2) == (0, 128, 256)
    # rank 1's slice of bucket 1: flat [384, 512), shard offset 384
    assert (f0, s, n) == (384, 384, 128)
    rc, null_out = map(int, second.split())
    assert rc == 1 and null_out == 1  # ZERO_ERR_INVALID, *out untouched
