"""bench.py's roofline bookkeeping on CPU: every kernel name libswe's per-kernel
timing can report (the names set in csrc/swe_api.cu) has an algorithmic
model in bench.kernel_model for each precision and layer count it runs with,
and a traffic record that bench.traffic_per_launch can read; every committed
traffic record is well formed and names only such kernels."""
import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

API = os.path.join(ROOT, "finite_volume_shallow_gb300", "csrc", "swe_api.cu")

# the layer counts each kernel runs with
LAYERS = {
    "cart1_step_kernel": (1,),
    "cart2_march_kernel<plain>": (2,),
    "cart2_march_kernel<fused>": (2,),
    "cart2_update_kernel": (2,),
    "mesh_tile_kernel": (1, 2),
    "mesh_update_kernel": (1, 2),
    "wd_speed_kernel": (1,),
    "wd_tile_kernel": (1,),
}


def reported_names():
    return sorted(set(re.findall(r'names\[\d\]\s*=\s*"([^"]+)"', open(API).read())))


def test_the_library_reports_the_kernels_modelled_here():
    assert reported_names() == sorted(LAYERS)


@pytest.mark.parametrize("name", sorted(LAYERS))
def test_every_reported_kernel_has_a_model_and_a_record(name):
    assert name in bench.KERNEL_SOURCES
    srcs, rec = bench.KERNEL_SOURCES[name]
    for f in srcs:
        assert os.path.exists(os.path.join(bench.CSRC, f)), f
    assert os.path.exists(os.path.join(ROOT, "profiles", rec)), rec
    for nl in LAYERS[name]:
        for precision in (32, 64):
            bound, amount, unit = bench.kernel_model(name, precision, nl, 1000, 2000)
            assert bound in ("hbm", "alu")
            assert unit == ("B" if bound == "hbm" else "flop")
            assert amount > 0


def test_traffic_records_are_well_formed():
    known = set(LAYERS)
    for rec in sorted({r for _, r in bench.KERNEL_SOURCES.values()}):
        lines = [ln for ln in open(os.path.join(ROOT, "profiles", rec)) if not ln.startswith("#")]
        vals = dict(ln.split(":", 1) for ln in lines if ":" in ln)
        vals = {k.strip(): v.strip() for k, v in vals.items()}
        assert re.fullmatch(r"[0-9a-f]{16}", vals.pop("source_sha256_16")), rec
        assert vals, rec
        for key, v in vals.items():
            assert key.startswith("bytes_per_launch_"), (rec, key)
            assert int(v) > 0, (rec, key)
            kern = key[len("bytes_per_launch_"):]
            if rec != "cart1_step_traffic.txt":  # keyed by workload alone
                assert any(kern.startswith(k + "_") for k in known), (rec, key)
            assert re.search(r"_f(32|64)$", kern), (rec, key)


def test_a_record_is_read_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    # a copy of the mesh record under another hash reads as missing
    src = os.path.join(ROOT, "profiles", "mesh_traffic.txt")
    text = re.sub(r"source_sha256_16: [0-9a-f]+", "source_sha256_16: 0000000000000000",
                  open(src).read())
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "mesh_traffic.txt").write_text(text)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_per_launch("mesh_tile_kernel", 32, "tri1024") is None
