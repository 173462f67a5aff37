"""The compiled-in tuned-shape table (csrc/tuned_shapes.inc) against the host
planner: every entry plans, for its own shape and a 152-SM GB300, to exactly
the options it records, and tune.py writes entries in the field order the
library reads.  No GPU: tgemm_plan does not touch the device."""
import importlib
import importlib.util
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TABLE = os.path.join(ROOT, "tiled_dense_gemm_02_gb300", "csrc", "tuned_shapes.inc")
FIELDS = ("kernel", "cta_group", "tile_n", "tile_m", "swap_ab", "tile_k", "group_m")
A0, B0, C0 = 0x1000_0000, 0x2000_0000, 0x4000_0000


@pytest.fixture(scope="module")
def tg():
    return importlib.import_module("tiled_dense_gemm_02_gb300")


def entries(path=TABLE):
    out = []
    for line in open(path):
        m = re.match(r"\s*\{([^}]*)\}", line)
        if m:
            vals = [int(v) for v in m.group(1).split(",")]
            assert len(vals) == 4 + len(FIELDS), line
            out.append((tuple(vals[:4]), dict(zip(FIELDS, vals[4:]))))
    return out


def test_table_is_not_empty_and_shapes_are_unique():
    e = entries()
    assert len(e) >= 5
    assert len({k for k, _ in e}) == len(e)


@pytest.mark.parametrize("key,opts", entries(), ids=lambda x: "x".join(map(str, x)) if isinstance(x, tuple) else "")
def test_entry_plans_to_its_options(tg, key, opts):
    M, N, K, dtype = key
    st, p = tg.plan(M, N, K, A0, K, B0, N, C0, N, dtype, None, sm_count=152)
    assert st == tg.OK and p.tuned == 1
    if opts["cta_group"]:
        assert p.cta_group == opts["cta_group"]
    if opts["swap_ab"] == 2:
        assert p.swap_ab == 1 and p.tile_m == opts["tile_m"]
    if opts["tile_n"]:
        assert p.tile_n == opts["tile_n"]
    if opts["tile_k"]:
        assert p.tile_k == opts["tile_k"]
    if opts["group_m"]:
        assert p.group_m == min(opts["group_m"], p.tiles_m)
    # the same options given explicitly are a valid plan of their own
    given = {k: v for k, v in opts.items() if v}
    if given:
        st2, q = tg.plan(M, N, K, A0, K, B0, N, C0, N, dtype, given, sm_count=152)
        assert st2 == tg.OK and q.tuned == 0
        assert (q.tile_m, q.tile_n, q.tile_k, q.cta_group, q.swap_ab) == (p.tile_m, p.tile_n, p.tile_k, p.cta_group,
                                                                         p.swap_ab)


def test_tune_writes_entries_the_library_reads(tmp_path):
    spec = importlib.util.spec_from_file_location("tgemm_tune", os.path.join(ROOT, "tiled_dense_gemm_02_gb300", "tune.py"))
    tune = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(tune)
    assert tune.FIELDS == FIELDS
    results = [{"shape": "300x400x500:bf16", "M": 300, "N": 400, "K": 500, "dtype": 2, "best_us": 9.5, "auto_us": 10.0,
                "options": {"swap_ab": 2, "tile_m": 192, "tile_n": 256, "tile_k": 64, "group_m": 4}, "tflops": 12.6},
               {"shape": "64x64x64:f16", "M": 64, "N": 64, "K": 64, "dtype": 1, "best_us": 5.0, "auto_us": 5.0,
                "options": {}, "tflops": 0.1}]
    out = tmp_path / "t.inc"
    tune.write_table(results, "test device", str(out))
    got = entries(str(out))
    assert got[0] == ((300, 400, 500, 2), {"kernel": 0, "cta_group": 0, "tile_n": 256, "tile_m": 192, "swap_ab": 2,
                                           "tile_k": 64, "group_m": 4})
    assert got[1] == ((64, 64, 64, 1), dict.fromkeys(FIELDS, 0))
