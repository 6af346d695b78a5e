"""The product path stands alone: importing and loading the library pulls in nothing from the
oracle package, and a missing libmgw.so makes every call fail loudly instead of falling back."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_product_import_does_not_touch_the_oracle():
    code = ("import sys; from moe_grouped_gemm_wgrad_gb300 import mgw, synth; mgw.load(); "
            "bad = [m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')]; "
            "print(bad); sys.exit(1 if bad else 0)")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stdout + out.stderr


def test_csrc_never_includes_oracle_sources():
    csrc = os.path.join(ROOT, "moe_grouped_gemm_wgrad_gb300", "csrc")
    for name in os.listdir(csrc):
        with open(os.path.join(csrc, name), errors="replace") as f:
            text = f.read()
        assert "oracle" not in text.lower(), name


def test_missing_library_raises(monkeypatch):
    from moe_grouped_gemm_wgrad_gb300 import mgw

    monkeypatch.setattr(mgw, "_lib", None)
    monkeypatch.setattr(mgw, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libmgw.so"))
    with pytest.raises(mgw.MgwError):
        mgw.load()
    with pytest.raises(mgw.MgwError):
        mgw.token_capacity(10, 2)


def test_time_limit_test_switch_only_in_the_test_build():
    """The device time-limit test drops a pipeline stage through MGW_TEST_DROP_LOAD; only the
    test build of the library reads that variable, libmgw.so does not contain it."""
    from moe_grouped_gemm_wgrad_gb300 import build

    build.build()
    with open(build.LIB, "rb") as f:
        assert b"MGW_TEST_DROP_LOAD" not in f.read()
    with open(build.LIB_TESTHOOKS, "rb") as f:
        assert b"MGW_TEST_DROP_LOAD" in f.read()
