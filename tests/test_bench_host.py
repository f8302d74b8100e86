"""Host logic of bench.py on CPU: the DRAM traffic a bench line reports comes
from the committed ncu summary only when that summary was taken on the
current kernel sources, from a capture of the same launch size when there is
one, else scaled by steps from the nearest launch size of the same workload."""
import hashlib
import json
import os

import bench


def _tree(tmp_path, records, sources=(("a.cu", b"kernel"), ("b.h", b"header"))):
    csrc = tmp_path / "decode_megakernel_sm_gb300" / "csrc"
    csrc.mkdir(parents=True)
    h = hashlib.sha256()
    for name, body in sorted(sources):
        (csrc / name).write_bytes(body)
        h.update(body)
    sha = h.hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    recs = {k: dict(v, kernel_src_sha=v.get("kernel_src_sha", sha)) for k, v in records.items()}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(recs))
    return sha


def test_source_hash_covers_every_kernel_source_in_name_order(tmp_path, monkeypatch):
    sha = _tree(tmp_path, {}, sources=(("z.cuh", b"2"), ("a.cu", b"1")))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_src_hash() == sha == hashlib.sha256(b"12").hexdigest()[:16]


def test_exact_launch_size_is_taken_as_is(tmp_path, monkeypatch):
    _tree(tmp_path, {"w@4": {"dram_bytes_per_launch": 4000}, "w@16": {"dram_bytes_per_launch": 1}})
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    v, how = bench.traffic_record("w", 4)
    assert v == 4000.0 and "launches of 4" in how


def test_one_step_launches_use_the_bare_key(tmp_path, monkeypatch):
    _tree(tmp_path, {"w": {"dram_bytes_per_launch": 250}, "w@4": {"dram_bytes_per_launch": 1}})
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("w", 1)[0] == 250.0


def test_other_launch_size_is_scaled_by_steps_from_the_nearest(tmp_path, monkeypatch):
    _tree(tmp_path, {"w": {"dram_bytes_per_launch": 100},          # 1 step: 100 per step
                     "w@16": {"dram_bytes_per_launch": 16 * 90},   # 16 steps: 90 per step
                     "other@8": {"dram_bytes_per_launch": 1}})
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    v, how = bench.traffic_record("w", 12)  # 16 is nearer to 12 than 1 is
    assert v == 12 * 90.0 and "scaled to 12" in how
    v, _ = bench.traffic_record("w", 2)     # 1 is nearer to 2
    assert v == 2 * 100.0


def test_a_capture_of_older_sources_is_never_used(tmp_path, monkeypatch):
    _tree(tmp_path, {"w@4": {"dram_bytes_per_launch": 4000, "kernel_src_sha": "0" * 16},
                     "w@16": {"dram_bytes_per_launch": 16000, "kernel_src_sha": "0" * 16}})
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("w", 4) == (None, "no capture on this kernel source")


def test_missing_summary_is_reported(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("w", 4) == (None, "no profiles/traffic.json")


def test_committed_summary_names_its_sources_and_commands():
    # every record says which sources and which command it came from
    recs = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    assert recs
    for key, r in recs.items():
        assert len(r["kernel_src_sha"]) == 16 and r["dram_bytes_per_launch"] > 0, key
        assert r["from"].startswith("ncu --metrics") and "--clock-control none" in r["from"], key
