"""The bounds-checked build (MX_BOUNDS_CHECK=1 at build and test time): its
kernels check every plain global load and store computed from an index against
the extent of its buffer, skip an access outside it and record it in the
device status word, which the suite's conftest reads after every GPU test.  So
`MX_BOUNDS_CHECK=1 python -m pytest tests -m gpu` runs the whole GPU suite as a
bounds check of every kernel it exercises, as a memory checker would.

These tests confirm that the library the process loaded is the build the
environment asked for, so that such a run cannot pass on the release build by
mistake."""
import os

import pytest

import block_scaled_fp4_bf16_gb300 as mx

pytestmark = pytest.mark.gpu


def test_loaded_library_is_the_requested_build():
    want = mx.MX_BUILD_BOUNDS_CHECK if os.environ.get("MX_BOUNDS_CHECK") == "1" else 0
    assert mx.mx_build_flags() == want
    assert mx.mx_available()


def test_status_word_starts_clean():
    assert mx.mx_device_status() == mx.MX_OK
