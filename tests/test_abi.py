"""The C ABI library loads and exports what include/hs.h declares (no GPU needed).

Only host-side paths run here: argument validation returns before any CUDA call.
"""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "hs.h")).read()
    return sorted(set(re.findall(r"HS_API\s+[\w\s\*]*?\b(hs_\w+)\s*\(", text)))


def test_header_declarations_match_binding():
    import hierarchical_sparse_attention_gb300 as hs
    assert declared_symbols() == sorted(hs.EXPORTS)


def test_library_exports_every_declared_symbol():
    import hierarchical_sparse_attention_gb300 as hs
    lib = ctypes.CDLL(hs.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", hs.LIB_PATH], capture_output=True, text=True).stdout
    exported = sorted({l.split()[-1] for l in out.splitlines() if re.search(r" T hs_", l)})
    assert exported == declared_symbols(), "the library exports exactly the declared hs_* entry points"


def test_workspace_and_config_validation():
    import hierarchical_sparse_attention_gb300 as hs
    good = hs.make_config(32, 2048, 4096, 656, 1, 0, 131136, 0)
    assert hs.hs_workspace_bytes(good) >= 16
    bad = [hs.make_config(32, 2048, 1024, 656),  # H < K
           hs.make_config(32, 0, 4096, 656),  # K = 0
           hs.make_config(32, 8192, 16384, 656),  # K over the limit
           hs.make_config(32, 64, 128, 656, 9),  # too many layers
           hs.make_config(0, 64, 128, 656),  # no requests
           hs.make_config(4, 64, 128, 656, 1, 64, 4096, 10)]  # page table too short
    for c in bad:
        if c.max_context == 0:
            c.max_context = 1024
        assert hs.hs_workspace_bytes(c) == 0


def test_host_side_errors_without_gpu():
    import hierarchical_sparse_attention_gb300 as hs
    cfg = hs.make_config(4, 64, 128, 576, 1, 0, 1024, 0)
    with pytest.raises(hs.HsError) as e:
        hs.hs_create(cfg, [None], [None], 100, 100, None)
    assert e.value.status == hs.HS_ERR_INVALID_ARG
    bad = hs.make_config(4, 64, 32, 576, 1, 0, 1024, 0)
    with pytest.raises(hs.HsError) as e:
        hs.hs_create(bad, [1 << 20], [1 << 20], 100, 100, 1 << 20)
    assert e.value.status == hs.HS_ERR_INVALID_CONFIG
    with pytest.raises(hs.HsError) as e:
        hs.hs_resolve(None, 1, *([None] * 10))
    assert e.value.status == hs.HS_ERR_INVALID_ARG
    with pytest.raises(hs.HsError) as e:
        hs.hs_backup(None, 1, None, None, None, None)
    assert e.value.status == hs.HS_ERR_INVALID_ARG
    # the calls added for split layer groups and launch shapes refuse a missing handle too
    for call in (lambda: hs.hs_launch_shape(None),
                 lambda: hs.hs_gather(None, 1, None, 0, 1),
                 lambda: hs.hs_gather_spec(None, 1, None, 0, 0, 1),
                 lambda: hs.hs_resolve_layers(None, 1, *([None] * 10), 1),
                 lambda: hs.hs_resolve_spec_layers(None, 1, 1, *([None] * 10), 1)):
        with pytest.raises(hs.HsError) as e:
            call()
        assert e.value.status == hs.HS_ERR_INVALID_ARG
    for s in range(6):
        assert hs.hs_status_str(s)


def test_product_path_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "hierarchical_sparse_attention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cuh", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\boracle\b", text), f"{f} mentions the oracle"
