"""The committed ncu records describe the committed kernels: every summary under profiles/ that states the
hash of its kernel's source files (the key bench.py checks before it reports a record's DRAM traffic) states
the hash of the sources as they are now. A kernel edit without its records taken again fails here."""
import hashlib
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "zero_gradient_reduction_gb300", "csrc")
PROFILES = os.path.join(ROOT, "profiles")

# the source files behind each kind of record, as bench.py hashes them
REGISTER = ("zr_step_kernel.cuh", "zr_device.cuh")
BULK = ("zr_step_bulk.cuh", "zr_step_kernel.cuh", "zr_device.cuh")
CHUNKED = ("zr_step_bulk_chunked.cuh", "zr_step_bulk.cuh", "zr_step_kernel.cuh", "zr_device.cuh")


def _digest(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _sources(name):
    if name.startswith("fused_bulk_chunked_"):
        return CHUNKED
    if name.startswith("fused_bulk_"):
        return BULK
    if name.startswith(("fused_step_", "inplace_step_")):
        return REGISTER
    raise AssertionError(f"{name}: a hashed record of an unknown kind")


def _hashed():
    out = []
    for name in sorted(os.listdir(PROFILES)):
        text = open(os.path.join(PROFILES, name)).read()
        m = re.findall(r"kernel_source_sha256_16: `([0-9a-f]+)`", text)
        if m:
            out.append((name, m))
    return out


def test_some_records_are_hashed():
    assert len(_hashed()) >= 10


@pytest.mark.parametrize("name,hashes", _hashed())
def test_record_matches_current_sources(name, hashes):
    want = _digest(_sources(name))
    assert all(h == want for h in hashes), f"{name}: records {hashes}, sources now {want}; retake its ncu capture"
