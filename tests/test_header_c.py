"""The boundary as a C caller sees it: include/gf.h compiles as strict C99
and C++17, and a C program linked against libgf.so gets the documented
answers from the calls that need no GPU (version, status strings, argument
validation with NULL or unsupported arguments, workspace-size queries)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "gf.h"

static int fails = 0;
#define EXPECT(cond) do { if (!(cond)) { printf("FAIL line %d: %s\n", __LINE__, #cond); ++fails; } } while (0)

int main(void) {
  EXPECT(gf_abi_version() == 2);
  EXPECT(strcmp(gf_status_string(GF_OK), "ok") == 0 || strlen(gf_status_string(GF_OK)) > 0);
  EXPECT(strlen(gf_status_string(GF_ERR_SHAPE)) > 0);
  /* NULL pointers are rejected before anything touches a device */
  EXPECT(gf_linear_swish_bias_groupnorm(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 256, 1024, 4096, 64, 1e-5f,
                                        GF_MODE_FP32_3XTF32, NULL, 0, NULL) == GF_ERR_NULL);
  EXPECT(gf_linear_lse_act(NULL, NULL, NULL, NULL, 1024, 8192, 8192, 0.01f, GF_MODE_FP32_3XTF32, NULL, 0, NULL)
         == GF_ERR_NULL);
  EXPECT(gf_ln_gelu_dconv1d_res(NULL, NULL, NULL, NULL, NULL, NULL, 32, 256, 4096, 3, 4, 4, 1e-5f,
                                GF_MODE_FP32_3XTF32, NULL, 0, NULL) == GF_ERR_NULL);
  EXPECT(gf_convt3d_swish_gn_hswish(NULL, NULL, NULL, NULL, NULL, NULL, 128, 3, 16, 16, 32, 32, 3, 2, 1, 4, 1e-5f,
                                    NULL, 0, NULL) == GF_ERR_NULL);
  /* workspace queries: sizes for supported shapes, 0 for unsupported ones */
  EXPECT(gf_linear_swish_bias_groupnorm_workspace_size(32768, 1024, 4096, 64, GF_MODE_FP32_3XTF32) ==
         (size_t)4 * (32768 * 1024 + 4096 * 1024));
  EXPECT(gf_linear_swish_bias_groupnorm_workspace_size(32768, 1024, 4096, 3, GF_MODE_FP32_3XTF32) == 0);
  EXPECT(gf_ln_gelu_dconv1d_res_workspace_size(32, 256, 4096, 3, 4, GF_MODE_FP32_3XTF32 | GF_FLAG_GELU_TANH) > 0);
  EXPECT(gf_convt3d_swish_gn_hswish_workspace_size(128, 3, 16, 16, 32, 32, 3, 2, 1, 4) > 0);
  EXPECT(gf_convt3d_swish_gn_hswish_workspace_size(128, 3, 16, 16, 32, 32, 9, 2, 1, 4) == 0);
  printf("%s\n", fails ? "failed" : "ok");
  return fails != 0;
}
"""


def _compiler(name):
    path = shutil.which(name)
    if path is None:
        pytest.skip(f"{name} not found")
    return path


@pytest.mark.parametrize("lang,cc,std", [("c", "gcc", "-std=c99"), ("c++", "g++", "-std=c++17")])
def test_header_compiles_strictly(tmp_path, lang, cc, std):
    src = tmp_path / ("h.c" if lang == "c" else "h.cpp")
    src.write_text('#include "gf.h"\nint main(void) { return gf_abi_version() == 2 ? 0 : 1; }\n')
    r = subprocess.run([_compiler(cc), std, "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                        "-I", INCLUDE, str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_against_the_library(tmp_path):
    from conv_activation_normalization_gb300 import binding, build
    build.build()
    lib = binding.LIB_PATH
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    r = subprocess.run([_compiler("gcc"), "-std=c99", "-Wall", "-Werror", "-I", INCLUDE, str(src), lib,
                        "-Wl,-rpath," + os.path.dirname(lib), "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
