"""The C-ABI library builds for sm_103a, loads without a GPU, and exports every entry point
that include/spec_verify.h declares (no compute call is made here)."""
import ctypes
import re

import numpy as np
import pytest

import speculative_decoding_verification_rejection_gb300 as sv


def test_header_declares_the_boundary():
    names = sv.declared_symbols()
    for required in ("spec_verify_init", "spec_verify_run", "spec_verify_free",
                     "spec_verify_last_error", "spec_verify_run_host"):
        assert required in names


def test_library_exports_every_declared_symbol():
    L = sv.lib()
    missing = [n for n in sv.declared_symbols() if not hasattr(L, n)]
    assert not missing, missing


def test_status_strings_and_constants():
    assert sv.spec_verify_status_string(sv.SV_OK) == "ok"
    assert "capacity" in sv.spec_verify_status_string(sv.SV_ECAPACITY)
    assert sv.spec_verify_launches_per_run() == 2
    assert len(sv.KERNELS) == 3                       # profiling slots: stats, verify, select
    with open(sv._HEADER, encoding="utf-8") as f:
        text = f.read()
    for name, val in (("SV_OK", 0), ("SV_EINVAL", -1), ("SV_ECAPACITY", -2), ("SV_EDTYPE", -3),
                      ("SV_ECUDA", -4), ("SV_EDEVICE", -5), ("SV_F32", 0), ("SV_BF16", 1)):
        m = re.search(rf"#define {name} \(?(-?\d+)\)?", text)
        assert m and int(m.group(1)) == val == getattr(sv, name)


def test_argument_errors_need_no_device():
    L = sv.lib()
    ctx = ctypes.c_void_p()
    assert L.spec_verify_init(None, 1, 1, 8, sv.SV_F32, 0, 0) == sv.SV_EINVAL
    assert L.spec_verify_init(ctypes.byref(ctx), 0, 1, 8, sv.SV_F32, 0, 0) == sv.SV_EINVAL
    assert L.spec_verify_init(ctypes.byref(ctx), 4, 1, 8, 7, 0, 0) == sv.SV_EDTYPE
    # argmax candidates hold twice an index in an int: vocabularies from 2^30 on are refused
    assert L.spec_verify_init(ctypes.byref(ctx), 1, 0, 1 << 30, sv.SV_F32, 0, 0) == sv.SV_ECAPACITY
    assert ctx.value is None
    assert L.spec_verify_run(None, *([None] * 6), 0, 0, 1, 0, 0, None, None, None, None, None,
                             None, None) == sv.SV_EINVAL
    rc = L.spec_verify_init(ctypes.byref(ctx), 4, 3, 1024, sv.SV_F32, 1, 0)
    assert rc in (sv.SV_OK, sv.SV_EDEVICE)      # EDEVICE where no sm_103 GPU is present
    if rc == sv.SV_OK:
        sv.spec_verify_free(ctx.value)
    sv.spec_verify_free(None)


def test_product_path_does_not_use_the_oracle():
    import pathlib
    pkg = pathlib.Path(sv.__file__).parent
    for f in list(pkg.rglob("*.py")) + list(pkg.rglob("*.cu")) + list(pkg.rglob("*.cuh")):
        text = f.read_text(encoding="utf-8")
        assert "import oracle" not in text and "from oracle" not in text, f
        assert "sv_oracle" not in text and "spec_verify_ref" not in text, f


def test_synthetic_rates_helper_matches_the_oracle():
    """The library's host helper (no device involved) against the oracle's own conversion."""
    import oracle

    for K in (0, 1, 3, 5, 8):
        for L in np.linspace(1.0, K + 1.0, 17):
            got = sv.spec_verify_synthetic_rates(L, K)
            np.testing.assert_array_equal(got, oracle.synthetic_rates(L, K))
    for L, K in ((0.5, 3), (4.5, 3), (float("nan"), 2), (2.0, sv.SV_MAX_SYNTHETIC + 1)):
        with pytest.raises(sv.SpecVerifyError):
            sv.spec_verify_synthetic_rates(L, K)
