"""Host logic of the measurement tools (no GPU): kernel labels of the ncu captures, the
source digest that ties a capture to the CUDA sources, and the clock summary that decides
whether a timed region ran throttled."""
import json
import os

import bench
import capture_profile


def test_kernel_labels():
    assert capture_profile.kernel_label("void ds_split_kernel<unsigned short, 1, 0>(ScanParams)") == \
        "ds_split_kernel_u16"
    # ncu shows some launches with the namespace; the label (a file name) never has it
    assert capture_profile.kernel_label("void dsk::ds_split_kernel<unsigned short, 1, 0>(dsk::ScanParams)") == \
        "ds_split_kernel_u16"
    assert capture_profile.kernel_label("dsk::ds_merge_kernel<unsigned int>(dsk::MergeParams)") == "ds_merge_kernel_u32"
    assert capture_profile.kernel_label("ds_sort_kernel(int)") == "ds_sort_kernel"


def _tree(tmp_path, kernel_text):
    csrc = tmp_path / "top_selection_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text(kernel_text)
    (csrc / "notes.txt").write_text("not a source")
    (tmp_path / "profiles").mkdir()
    return tmp_path


class _Shape:
    name = "indexer"
    k = 512


def test_traffic_only_while_the_sources_match(tmp_path, monkeypatch):
    root = _tree(tmp_path, "__global__ void k() {}\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    digest = bench._source_digest()
    assert len(digest) == 16 and int(digest, 16) >= 0
    assert bench._source_digest() == digest  # deterministic
    prof = {"source_digest": digest, "traffic_bytes_per_launch": 16853760}
    (root / "profiles" / "ds_split_kernel_u16_indexer_k512.json").write_text(json.dumps(prof))
    assert bench._traffic_from_profile("ds_split_kernel_u16", _Shape) == 16853760
    # a file that is not a CUDA source does not count; an edited kernel does
    (root / "top_selection_gb300" / "csrc" / "notes.txt").write_text("edited")
    assert bench._source_digest() == digest
    (root / "top_selection_gb300" / "csrc" / "k.cu").write_text("__global__ void k() { }\n")
    assert bench._source_digest() != digest
    assert bench._traffic_from_profile("ds_split_kernel_u16", _Shape) is None
    # no capture for this kernel and workload at all
    assert bench._traffic_from_profile("ds_scan_kernel_u16", _Shape) is None


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _samples(tmp_path, lines):
    s = bench.ClockSampler(0)
    s.proc = _Done()
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    return s.stop()


def test_clock_summary_under_load_and_throttle_reasons(tmp_path):
    # index, sm, max sm, power, active mask, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
    idle = "0, 345, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active"
    busy = "0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active"
    capped = "0, 1980, 2070, 1400.0, 0x4, Not Active, Not Active, Not Active, Active"
    got = _samples(tmp_path, [idle, busy, busy, capped, "garbage line"])
    assert got["samples"] == 4
    assert got["sm_max_mhz"] == 2070.0
    assert got["sm_mhz"] == 2070.0  # the median of the samples under load (idle ones left out)
    assert got["reasons"] == ["sw_power_cap"]
    slowed = "0, 1200, 2070, 700.0, 0x8, Active, Not Active, Not Active, Not Active"
    got = _samples(tmp_path, [busy, slowed, busy])
    assert got["reasons"] == ["hw_slowdown"]
    assert not os.path.exists(str(tmp_path / "clocks.csv"))  # the sample file is removed


def test_clock_summary_without_nvidia_smi():
    s = bench.ClockSampler(0)
    s.proc = None
    assert s.stop() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
