"""Every bounded wait in the kernels records its own status code.

The device status word tells the host which wait ran out (codes 101..199,
reported as ATTN_ERR_TIMEOUT) or which index check of a debug build failed
(codes >= 200, ATTN_ERR_DEVICE_CHECK).  A wait numbered past 99 would be
misread as a failed index check, and two waits sharing a number could not be
told apart, so each number is used once, in 1..99.  (The wait_code template
rejects out-of-range numbers at compile time; this test also covers
uniqueness, without a GPU.)
"""
import collections
import os
import re

CSRC = os.path.join(os.path.dirname(__file__), "..", "bwd_flashattention_fwd_gb300", "csrc")


def _sources():
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(CSRC, name)) as f:
                yield name, f.read()


def test_wait_codes_unique_and_in_range():
    uses = collections.defaultdict(list)
    for name, text in _sources():
        for m in re.finditer(r"wait_code<(\d+)>\(\)", text):
            uses[int(m.group(1))].append(name)
    assert uses, "no wait codes found"
    assert all(1 <= c <= 99 for c in uses), sorted(uses)
    dup = {c: f for c, f in uses.items() if len(f) > 1}
    assert not dup, f"wait codes used more than once: {dup}"


def test_no_raw_timeout_arithmetic():
    # codes are formed only through the range-checked template
    for name, text in _sources():
        if name == "kernel_common.cuh":
            continue
        assert "kDevTimeoutBase +" not in text, name
