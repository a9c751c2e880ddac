"""Host side of bench.py without a GPU: workload names and shapes under the
--batch / --layout / --size / --crop overrides (the names key the committed
traffic figures), and the reference arm (the CPU oracle) on an overridden
image size."""
import json
import os
import subprocess
import sys
from types import SimpleNamespace

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _args(**kw):
    a = dict(config=3, layout=None, batch=None, size=None, crop=0)
    a.update(kw)
    return SimpleNamespace(**a)


def test_workload_names_and_shapes():
    assert bench.workload(_args())["workload"] == "n256_224x224x3_f16_nhwc_flip_erase"
    cfg = bench.workload(_args(size="299x299"))
    assert cfg["workload"] == "n256_299x299x3_f16_nhwc_flip_erase"
    assert (cfg["N"], cfg["H"], cfg["W"], cfg["C"]) == (256, 299, 299, 3)
    cfg = bench.workload(_args(size="227x300", batch=64, layout="nhwc4"))
    assert cfg["workload"] == "n64_227x300x3_f16_nhwc_flip_erase_nhwc4"
    assert (cfg["N"], cfg["H"], cfg["W"], cfg["layout"]) == (64, 227, 300, "nhwc4")
    assert bench.workload(_args(crop=256))["workload"] == "n256_224x224x3_f16_nhwc_flip_erase_crop_from_256x256"


def test_traffic_only_for_the_profiled_source():
    # every committed figure names the kernel source it was taken on; a name
    # that was never profiled has none
    assert bench.profiled_traffic("n7_1x1x3_nothing") is None
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    for name, e in d.items():
        assert len(e["kernel_source_sha256_16"]) == 16
        assert e["dram_bytes_per_launch"] == e["dram_read_bytes"] + e["dram_write_bytes"]


def test_reference_arm_on_an_overridden_size():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "1", "--size", "33x35",
           "--steps", "1", "--warmup", "0"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["config"]["workload"].startswith("n16_33x35x3_")
    assert (line["config"]["H"], line["config"]["W"]) == (33, 35)
    assert line["value"] > 0


def test_l2_note_counts_the_sets_the_timed_region_touches():
    l2 = 136 * 2**20
    # the headline: 20 launches over five 115.6 MB sets touch all of them
    assert bench.l2_note(20, 5, 115_605_504, l2).startswith("inputs larger than L2: 5 rotating")
    # 40 launches of a 0.94 MB workload touch 40 of 692 sets: L2-resident
    note = bench.l2_note(40, 692, 940_800, l2)
    assert note.startswith("L2-resident") and "40 of the 692" in note
    # the same workload over every set is not
    assert bench.l2_note(692, 692, 940_800, l2).startswith("inputs larger than L2")
