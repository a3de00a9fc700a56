"""Host code under AddressSanitizer and UndefinedBehaviorSanitizer (no GPU).

compute-sanitizer is not available for the device code here; these builds
check the C that runs on the host instead: the oracle and the input
generator (their pin and generator suites), and the library's host side
(argument checks, status strings, the host-buffer entry point's offset
checks), each built with -fsanitize=address,undefined and run in a child
process with the ASan runtime preloaded.  Any sanitizer report fails the
test."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SAN = ["-fsanitize=address,undefined", "-fno-omit-frame-pointer", "-fno-sanitize-recover=all"]


def _asan_runtime():
    try:
        p = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True,
                           text=True).stdout.strip()
    except OSError:
        p = ""
    if not p or not os.path.isabs(p) or not os.path.exists(p):
        pytest.skip("gcc's AddressSanitizer runtime is not installed")
    return p


def _run_sanitized(env_extra, args, timeout=900):
    env = dict(os.environ)
    env.update(env_extra)
    env["LD_PRELOAD"] = _asan_runtime()
    # CUDA's runtime needs the address range ASan would reserve; Python leaks by design.
    env["ASAN_OPTIONS"] = "detect_leaks=0:protect_shadow_gap=0:abort_on_error=1"
    env["UBSAN_OPTIONS"] = "print_stacktrace=1:halt_on_error=1"
    env["PYTHONPATH"] = ROOT
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", *args],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)
    out = r.stdout + r.stderr
    assert "AddressSanitizer" not in out and "runtime error:" not in out, out[-4000:]
    assert r.returncode == 0, out[-4000:]
    return out


def test_oracle_and_input_generator(tmp_path):
    import inputgen
    import oracle
    _asan_runtime()
    olib = oracle.build_lib(extra_flags=["-O1", *SAN], out_path=str(tmp_path / "oracle_san.so"))
    glib = inputgen.build_lib(extra_flags=["-O1", *SAN], out_path=str(tmp_path / "gen_san.so"))
    out = _run_sanitized({"ORACLE_LIB_PATH": olib, "INPUTGEN_LIB_PATH": glib},
                         ["tests/test_oracle_pins.py", "tests/test_inputgen.py", "-m", "not gpu",
                          "-k", "not planted_mistakes"])
    assert "passed" in out


def test_library_host_side(tmp_path):
    from gqa_attention_prefill_gb300 import build
    _asan_runtime()
    # (nvcc splits -Xcompiler arguments at commas: one sanitizer per flag)
    lib = build.build(out=str(tmp_path / "libtsk_mha_san.so"),
                      host_flags=["-fsanitize=address", "-fsanitize=undefined", *SAN[1:]])
    # (the test that compiles another build runs the compiler: not under the ASan runtime)
    out = _run_sanitized({"TSK_LIB_PATH": lib}, ["tests/test_abi.py", "-m", "not gpu",
                                                 "-k", "not bounds_checked_build"])
    assert "passed" in out
