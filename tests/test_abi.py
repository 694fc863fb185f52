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
                 lambda: hs.hs_resolve_spec_layers(None, 1, 1, *([None] * 10), 1),
                 lambda: hs.hs_resolve_spec(None, 1, 1, *([None] * 10)),
                 lambda: hs.hs_backup_spec(None, 1, 1, *([None] * 5)),
                 lambda: hs.hs_invalidate_tokens(None, 1, *([None] * 5)),
                 lambda: hs.hs_invalidate_host_rows(None, 1, None, None, None, 0, None, None),
                 lambda: hs.hs_reset_hints(None)):
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


def test_consumer_host_side_validation_without_gpu():
    """hs_sparse_mla_workspace_bytes sizes the split workspace (0 where none is needed or the
    shape is refused); hs_sparse_mla_decode refuses bad shapes, missing or misaligned buffers
    and a short workspace before any launch, and does nothing for zero requests."""
    import hierarchical_sparse_attention_gb300 as hs
    ws = hs.hs_sparse_mla_workspace_bytes
    assert ws(32, 128, 2) == 2 * 32 * 128 * (512 + 1) * 4  # partial outputs and lse per split
    assert hs.hs_sparse_mla_launches(32, 128, 1) == 1  # one split: one launch, no device query
    for bad in ((0, 128, 2), (32, 0, 2), (32, 129, 2), (32, 128, 0), (32, 128, hs.HS_MAX_MLA_SPLITS + 1)):
        assert hs.hs_sparse_mla_launches(*bad) == 0
    assert ws(32, 128, 1) == 0  # one split writes o and lse directly
    for bad in ((0, 128, 2), (32, 0, 2), (32, 129, 2), (32, 128, 0), (32, 128, hs.HS_MAX_MLA_SPLITS + 1)):
        assert ws(*bad) == 0
    A = 1 << 20  # a 16-byte aligned stand-in address: nothing is launched in these calls
    good = dict(R=2, H=128, K=64, splits=2, q=A, pool=A, rows_n=100, out_rows=A, o=A, lse=A, wsp=A,
                wsb=ws(2, 128, 2), err=A)

    def call(**kw):
        a = dict(good, **kw)
        hs.hs_sparse_mla_decode(a["R"], a["H"], a["K"], a["splits"], a["q"], a["pool"], a["rows_n"],
                                a["out_rows"], 0.1, a["o"], a["lse"], a["wsp"], a["wsb"], a["err"])

    refused = [dict(R=-1), dict(H=0), dict(H=129), dict(K=0), dict(K=hs.HS_MAX_TOP_K + 1), dict(splits=0),
               dict(splits=hs.HS_MAX_MLA_SPLITS + 1), dict(rows_n=0), dict(q=None), dict(pool=None),
               dict(out_rows=None), dict(o=None), dict(lse=None), dict(err=None), dict(q=A + 8),
               dict(pool=A + 4), dict(o=A + 8), dict(wsp=None), dict(wsb=good["wsb"] - 1), dict(wsp=A + 8)]
    for kw in refused:
        with pytest.raises(hs.HsError) as e:
            call(**kw)
        assert e.value.status == hs.HS_ERR_INVALID_ARG, kw
    call(R=0, q=None, pool=A, out_rows=None, o=None, lse=None, wsp=None, wsb=0, err=None)  # no work, no launch
