"""The binding never loads a library older than its sources: a failed rebuild raises instead of
silently loading (and measuring) the previous binary. No GPU and no real compile involved."""
import os
import time

import pytest

import speculative_decoding_verification_rejection_gb300 as sv


def test_failed_rebuild_raises_instead_of_loading_the_old_library(tmp_path, monkeypatch):
    sv.build()                                  # a library exists (the case that used to pass)
    assert os.path.exists(sv.LIB_PATH)
    fake = tmp_path / "nvcc"
    fake.write_text("#!/bin/sh\necho 'error: broken compiler' >&2\nexit 1\n")
    fake.chmod(0o755)
    newer = tmp_path / "edited_source.cu"       # a source newer than the library
    newer.write_text("// edited after the last build\n")
    later = time.time() + 3600
    os.utime(newer, (later, later))
    monkeypatch.setenv("NVCC", str(fake))
    monkeypatch.setattr(sv, "_SOURCES", sv._SOURCES + [str(newer)])
    monkeypatch.setattr(sv, "_lib", None)
    with pytest.raises(RuntimeError, match="could not be rebuilt"):
        sv.lib()
    assert sv._lib is None                      # nothing was loaded


def test_up_to_date_library_loads_without_a_compiler(monkeypatch):
    sv.build()
    monkeypatch.setenv("NVCC", "/nonexistent/nvcc")
    monkeypatch.setattr(sv, "_lib", None)
    assert sv.lib() is not None                 # not stale: no rebuild is attempted
