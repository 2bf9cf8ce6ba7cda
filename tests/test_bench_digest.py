"""The bench reports ncu traffic only for the kernel sources it was taken on.

bench.source_digest(unit) hashes one translation unit under csrc/ and every
local header it includes, recursively.  It must change when that unit or any
header it reaches changes, and must not change for files the unit does not
include.  ncu_traffic_per_launch() must give the recorded bytes (scaled by
tokens) only while the digest matches."""
import json

import bench


def _tree(tmp_path):
    csrc = tmp_path / "hyper_connection_residual_mixes_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "include").mkdir()
    (csrc / "a.cu").write_text('#include "h1.h"\n#include <cstdint>\nint a;\n')
    (csrc / "h1.h").write_text('#include "h2.cuh"\n#include "../../include/api.h"\n')
    (csrc / "h2.cuh").write_text('#include "h1.h"\nint h2;\n')  # a cycle: must terminate
    (csrc / "b.cu").write_text('#include "other.h"\nint b;\n')
    (csrc / "other.h").write_text("int other;\n")
    (tmp_path / "include" / "api.h").write_text("int api;\n")
    return csrc


def test_digest_follows_local_includes_only(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    csrc = _tree(tmp_path)
    d0 = bench.source_digest("a.cu")
    (csrc / "other.h").write_text("int other2;\n")
    (csrc / "b.cu").write_text("int b2;\n")
    assert bench.source_digest("a.cu") == d0
    (csrc / "h2.cuh").write_text('#include "h1.h"\nint h2_changed;\n')
    d1 = bench.source_digest("a.cu")
    assert d1 != d0
    (tmp_path / "include" / "api.h").write_text("int api_changed;\n")
    assert bench.source_digest("a.cu") != d1


def test_traffic_used_only_while_the_digest_matches(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    csrc = _tree(tmp_path)
    (csrc / "hc_slices.cu").write_text('#include "h1.h"\nint chain;\n')
    (tmp_path / "profiles").mkdir()
    rec = {"source_digest": bench.source_digest("hc_slices.cu"), "dram_bytes_per_token": 100.5,
           "dram_bytes_fixed": 7}
    (tmp_path / "profiles" / "hc_chain_side_traffic.json").write_text(json.dumps(rec))
    assert bench.ncu_traffic_per_launch(1000, "chain") == int(100.5 * 1000 + 7)
    (csrc / "h1.h").write_text('#include "h2.cuh"\nint edited;\n')
    assert bench.ncu_traffic_per_launch(1000, "chain") is None
    assert bench.ncu_traffic_per_launch(1000, "step") is None  # no record (nor source) for the step kernel here
    (csrc / "hc_slices.cu").unlink()
    assert bench.ncu_traffic_per_launch(1000, "chain") is None  # no source: no figure

