"""The C ABI from plain C: a C99 program that includes include/rmsnorm_train.h and
include/layernorm_train.h, links against the library and calls its host-only entry points
(launch plans, workspace sizes, status strings, argument rejection).  This shows that the
headers are valid C, that every symbol links without torch or C++, and that the values a
C caller sees equal the Python binding's.  No GPU: none of these calls reaches CUDA."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include "layernorm_train.h"   /* includes rmsnorm_train.h */

int main(void) {
  int64_t p[16];
  int i;
  if (rmsnorm_train_launch_plan(4096, RMSN_PLAN_BWD, p, RMSN_PLAN_FIELDS) != RMSN_OK) return 1;
  printf("rms_bwd_plan");
  for (i = 0; i < RMSN_PLAN_FIELDS; ++i) printf(" %lld", (long long)p[i]);
  printf("\n");
  if (layernorm_train_launch_plan(4096, LN_PLAN_FWD, p, LN_PLAN_FIELDS) != RMSN_OK) return 2;
  printf("ln_fwd_plan");
  for (i = 0; i < LN_PLAN_FIELDS; ++i) printf(" %lld", (long long)p[i]);
  printf("\n");
  printf("rms_ws %zu\n", rmsnorm_train_bwd_workspace_bytes(65536, 1, 4096, 1));
  printf("ln_ws %zu\n", layernorm_train_bwd_workspace_bytes(8192, 4096, 1));
  printf("status3 %s\n", rmsnorm_train_status_str(RMSN_ERR_WORKSPACE));
  printf("rms_fwd_null %d\n", rmsnorm_train_fwd(NULL, NULL, NULL, RMSN_W_BF16, NULL, NULL,
                                                NULL, 4, 1, 64, 64, 64, 1e-6f, NULL));
  printf("ln_fwd_wide %d\n", layernorm_train_fwd(NULL, NULL, NULL, RMSN_W_BF16, NULL, NULL,
                                                 NULL, 4, 16400, 1e-5f, NULL));
  return 0;
}
"""


@pytest.fixture(scope="module")
def libdir():
    from rmsnorm_fwd_02_gb300 import build as B
    return os.path.dirname(B.build())


def test_c_program_links_and_sees_the_bindings_values(tmp_path, libdir):
    from rmsnorm_fwd_02_gb300 import _native as N
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L", libdir, "-lrmsnorm_train", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = dict(line.split(" ", 1) for line in out.strip().splitlines())
    rp = N.rmsnorm_train_launch_plan(4096, N.PLAN_BWD)
    assert [int(v) for v in got["rms_bwd_plan"].split()] == [rp[k] for k in N.PLAN_FIELDS]
    lp = N.layernorm_train_launch_plan(4096, N.LN_PLAN_FWD)
    assert [int(v) for v in got["ln_fwd_plan"].split()] == [lp[k] for k in N.LN_PLAN_FIELDS]
    assert int(got["rms_ws"]) == N.rmsnorm_train_bwd_workspace_bytes(65536, 1, 4096, 1)
    assert int(got["ln_ws"]) == N.layernorm_train_bwd_workspace_bytes(8192, 4096, 1)
    assert got["status3"] == N.status_str(3)
    assert int(got["rms_fwd_null"]) == 1          # RMSN_ERR_INVALID_ARG
    assert int(got["ln_fwd_wide"]) == 2           # RMSN_ERR_UNSUPPORTED (H > 16384)
