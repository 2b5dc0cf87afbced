"""The ABI from plain C (CPU only): tests/c_abi_smoke.c is compiled with gcc against
include/sagebwd.h, linked with libsagebwd.so and run; its answers must equal the
Python binding's.  Only size queries and argument checks run, none of which touch
a GPU."""
import os
import shutil
import subprocess

import pytest

import bit_trainable_attention_gb300 as sb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
def test_plain_c_program(tmp_path):
    lib = sb.load_library()
    lib_path = lib._name
    exe = tmp_path / "c_abi_smoke"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi_smoke.c"), "-o", str(exe), lib_path,
                    "-Wl,-rpath," + os.path.dirname(lib_path)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = dict(line.split(" ", 1) for line in out.strip().splitlines())
    p = sb.Problem.make(1, 12, 2, 16384, 128, True)
    assert int(got["version"]) == sb.sagebwd_version()
    assert int(got["saved"]) == sb.sagebwd_saved_bytes(p) > 0
    assert int(got["ws0"]) == sb.sagebwd_workspace_bytes(p, 0) > 0
    assert int(got["ws1"]) == sb.sagebwd_workspace_bytes(p, 1) > 0
    assert int(got["bad_d_saved"]) == 0 and int(got["bad_g_saved"]) == 0
    assert int(got["fwd_null"]) == 1  # SAGEBWD_ERR_INVALID_ARG
    assert int(got["fwd_misaligned"]) == 3  # SAGEBWD_ERR_MISALIGNED
    assert got["status_string_2"] == lib.sagebwd_status_string(2).decode()
