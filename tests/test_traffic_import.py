"""bench.import_traffic on a synthetic ncu CSV (CPU only): the library's launches are told
apart from other kernels (templates by '<', plain kernels such as the register-held final
aggregation by '('), classified in the step's per-chunk order, converted from the unit ncu
printed, and scaled to a 16384-token launch."""
import csv
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from synth import inputs as I  # noqa: E402

HDR = ["ID", "Process ID", "Process Name", "Host Name", "Kernel Name", "Context", "Stream",
       "Block Size", "Grid Size", "Device", "CC", "Section Name", "Metric Name", "Metric Unit",
       "Metric Value"]
NAMES = {
    "phase1": "unnamed>::phase1_tc_kernel<9, 0, 1>(CUtensorMap_st, CUtensorMap_st, Phase1Args)",
    "phase2": "unnamed>::phase2_kernel<__nv_bfloat16, __nv_bfloat16, 4, 0>(Phase2Args)",
    "close": "unnamed>::add_kernel<__nv_bfloat16>(const T1 *, const T1 *, T1 *, long)",
    "final": "unnamed>::full_hold_kernel(FullArgs, int)",
    "other": "void at::native::vectorized_elementwise_kernel<4, at::FillFunctor<float>>(int)",
}


def _write_csv(path, chunks, mb_units):
    S = I.LONGCTX_PREFILL_BF16.S
    kinds = ["phase1"] + ["phase2"] * S + ["close", "final"]
    # read / write MB per kind of launch in the chunk (phase 2: first, partial, fused)
    mb = {"phase1": (900.0, 1300.0), "close": (117.0, 7.0), "final": (587.0, 50.0)}
    rows, lid = [], 0
    for _ in range(chunks):
        for i, k in enumerate(kinds):
            if k == "phase1":  # a foreign kernel between ours must be skipped
                for metric in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
                    rows.append([str(lid), "1", "py", "h", NAMES["other"], "1", "7", "(1,1,1)",
                                 "(1,1,1)", "0", "10.3", "m", metric, "byte", "5"])
                lid += 1
            if k == "phase2":
                j = i - 1
                rd, wr = (58.0, 6.0) if j == 0 else (117.0, 6.0) if j == 1 else (176.0, 57.0)
            else:
                rd, wr = mb[k]
            for metric, val in (("dram__bytes_read.sum", rd), ("dram__bytes_write.sum", wr),
                                ("gpu__time_duration.sum", 100.0)):
                if metric == "gpu__time_duration.sum":
                    unit, v = "us", val
                elif mb_units:
                    unit, v = "Mbyte", val
                else:
                    unit, v = "byte", val * 1e6
                rows.append([str(lid), "1", "py", "h", NAMES[k], "1", "7", "(1,1,1)", "(1,1,1)",
                             "0", "10.3", "m", metric, unit, f"{v:,.3f}"])
            lid += 1
    with open(path, "w", newline="") as f:
        f.write("==PROF== Connected to process 1\n")
        w = csv.writer(f, quoting=csv.QUOTE_ALL)
        w.writerow(HDR)
        w.writerows(rows)


@pytest.mark.parametrize("mb_units", [False, True])
def test_import_classifies_scales_and_converts(tmp_path, mb_units):
    p = tmp_path / "dram.csv"
    _write_csv(p, chunks=2, mb_units=mb_units)
    bench.import_traffic(str(p), tokens=4096, out_dir=str(tmp_path))
    out = json.load(open(tmp_path / "dram_traffic_longctx_T4096.json"))
    S = I.LONGCTX_PREFILL_BF16.S
    want = {"phase1": (2, 2200.0), "phase2_first": (2, 64.0), "phase2": (2, 123.0),
            "phase2_fused": (2 * (S - 2), 233.0), "close": (2, 124.0), "final": (2, 637.0)}
    assert set(out) == set(want)
    for kind, (launches, mb_per_launch) in want.items():
        e = out[kind]
        assert e["launches_captured"] == launches, kind
        assert e["bytes_per_launch"] == pytest.approx(mb_per_launch * 1e6 * 16384 / 4096), kind
        assert e["ncu_duration_ns_captured"] == pytest.approx(1e5), kind
        assert e["src_hash"] == bench.kernel_hash(kind)
    assert "full_hold_kernel" in out["final"]["kernel"]


def test_import_rejects_unknown_units(tmp_path):
    p = tmp_path / "dram.csv"
    _write_csv(p, chunks=1, mb_units=True)
    text = open(p).read().replace('"Mbyte"', '"furlong"')
    open(p, "w").write(text)
    with pytest.raises(ValueError):
        bench.import_traffic(str(p), tokens=4096, out_dir=str(tmp_path))
