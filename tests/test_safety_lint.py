"""Source rules that keep the kernels from hanging or faulting a GPU, checked
on the text of csrc/ (no GPU needed):

- no device-side trap or assert (failures are reported through the error
  word and a status code, never by killing the context);
- mbarrier polling only inside the bounded wait helpers of ptx.cuh, whose
  every loop ends on a %globaltimer limit and a round cap;
- no endless loop form outside those helpers;
- none of the batched host-copy calls anywhere in the sources.
"""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_io_aware_40_gb300", "csrc")


def sources():
    out = {}
    for f in sorted(os.listdir(CSRC)):
        if f.endswith((".cu", ".cuh", ".h")):
            out[f] = open(os.path.join(CSRC, f)).read()
    return out


def strip_comments(text):
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.sub(r"//[^\n]*", "", text)


def test_no_device_trap_or_assert():
    for f, text in sources().items():
        code = strip_comments(text)
        assert "__trap" not in code, f
        assert not re.search(r"\btrap\s*;", code), f
        assert not re.search(r"(?<!static_)\bassert\s*\(", code), f


def test_mbarrier_polling_only_in_the_bounded_helpers():
    for f, text in sources().items():
        code = strip_comments(text)
        if f == "ptx.cuh":
            continue
        assert "mbarrier.try_wait" not in code and "mbarrier.test_wait" not in code, f
        assert "mbar_try_wait" not in code, f


def test_bounded_helpers_check_time_and_rounds():
    code = strip_comments(sources()["ptx.cuh"])
    for helper in ("mbar_wait", "mbar_wait_drain"):
        m = re.search(r"bool\s+%s\s*\(.*?\n}\n" % helper, code, flags=re.S)
        assert m, helper
        body = m.group(0)
        assert "globaltimer()" in body and "kWaitLimitNs" in body, helper
        assert "kMaxWaitRounds" in body, helper


def test_no_endless_loop_outside_the_helpers():
    for f, text in sources().items():
        if f == "ptx.cuh":
            continue
        code = strip_comments(text)
        assert not re.search(r"while\s*\(\s*(true|1)\s*\)", code), f
        assert not re.search(r"for\s*\([^;)]*;\s*;", code), f


def test_no_batched_host_copies():
    pattern = re.compile(r"Memcpy(3D)?" + "Batch")
    for base in (CSRC, os.path.join(ROOT, "include"), os.path.join(ROOT, "exact_io_aware_40_gb300")):
        for f in os.listdir(base):
            if f.endswith((".cu", ".cuh", ".h", ".py")):
                assert not pattern.search(open(os.path.join(base, f)).read()), f
    for f in ("bench.py", "__graft_entry__.py"):
        assert not pattern.search(open(os.path.join(ROOT, f)).read()), f
