"""The host's choice of decode path and of the persistent kernel's launch form.

Both live in paged_expert_cache_gb300/csrc/decode_policy.h, free of CUDA; a
small driver (tests/native/decode_policy_check.cpp) is compiled with the host
compiler and fed cases, so no GPU is needed. The rules checked:
  * MOE_DECODE_AUTO takes one kernel for one token, and for two tokens on
    per-layer pools; ONE_KERNEL for every call that fits; THREE_KERNELS never;
    speculation, the MEMCPY upload, a call that does not fit one CTA per SM and
    a handle whose persistent launch was refused keep to three kernels;
  * the persistent kernel goes out as a cooperative launch with programmatic
    dependent launch, then as a cooperative launch alone; a refused form is not
    tried again, and once both are refused every later call is refused without
    an attempt (the forward then keeps to three kernels).
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
AUTO, THREE, ONE = 0, 1, 2
PER_LAYER, SHARED = 0, 1
PULL, MEMCPY = 0, 1


@pytest.fixture(scope="module")
def policy(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path_factory.mktemp("policy") / "decode_policy_check")
    subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-Werror",
                    "-I", os.path.join(ROOT, "paged_expert_cache_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "native", "decode_policy_check.cpp"), "-o", exe], check=True)

    def run(lines):
        r = subprocess.run([exe], input="\n".join(lines) + "\n", capture_output=True, text=True, check=True)
        return r.stdout.split("\n")[:len(lines)]
    return run


def path_case(mode, T, pool=PER_LAYER, upload=PULL, spec=0, fused_ok=1, fits=1):
    return f"path {mode} {T} {pool} {upload} {spec} {fused_ok} {fits}"


def test_auto_rule(policy):
    cases = {
        path_case(AUTO, 1): "1",
        path_case(AUTO, 1, pool=SHARED): "1",
        path_case(AUTO, 2): "1",
        path_case(AUTO, 2, pool=SHARED): "0",
        path_case(AUTO, 3): "0",
        path_case(AUTO, 8): "0",
        path_case(ONE, 8): "1",
        path_case(ONE, 4, pool=SHARED): "1",
        path_case(THREE, 1): "0",
    }
    assert policy(list(cases)) == list(cases.values())


def test_what_keeps_a_call_on_three_kernels(policy):
    for mode in (AUTO, ONE):
        got = policy([path_case(mode, 1, spec=1), path_case(mode, 1, upload=MEMCPY),
                      path_case(mode, 1, fits=0), path_case(mode, 1, fused_ok=0)])
        assert got == ["0", "0", "0", "0"], mode


def test_launch_forms_in_order(policy):
    got = policy([
        "coop 0 1 AA",     # both calls accepted with PDL
        "coop 0 1 RAA",    # PDL refused once: the cooperative launch alone from then on
        "coop 0 1 RR",     # both refused: final
        "coop 0 0 AA",     # without PDL the first form is the cooperative launch alone
        "coop 0 0 R",      # and its refusal is final
        "coop 2 1 A",      # refused earlier: no attempt at all
    ])
    assert got[0] == "p:1:0 p:1:0 "
    assert got[1] == "pc:1:1 c:1:1 "
    assert got[2] == "pc:0:2 "
    assert got[3] == "c:1:0 c:1:0 "
    assert got[4] == "c:0:2 "
    assert got[5] == ":0:2 "
