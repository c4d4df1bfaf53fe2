"""Host logic of bench.py that needs no GPU: the roofline's DRAM traffic is read from a
committed ncu summary only while the kernel's source is the one the counters were taken on."""
import hashlib
import os

import bench


def _layout(tmp_path, source_text: str, line: str):
    csrc = tmp_path / "serving_router_top_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k_fake.cu").write_text(source_text)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "k_fake__decode_t4_fake.md").write_text("# summary\n\nsome figures\n\n" + line + "\n")
    return csrc / "k_fake.cu"


def _sha(text: str) -> str:
    return hashlib.sha1(text.encode()).hexdigest()


def test_traffic_used_while_the_source_matches(tmp_path, monkeypatch):
    src = "__global__ void k() {}\n"
    _layout(tmp_path, src, f"bench-traffic: kernel=fake source=k_fake.cu sha1={_sha(src)} bytes=12345")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("decode_t4_fake", "fake") == 12345


def test_traffic_dropped_once_the_source_changes(tmp_path, monkeypatch):
    src = "__global__ void k() {}\n"
    path = _layout(tmp_path, src, f"bench-traffic: kernel=fake source=k_fake.cu sha1={_sha(src)} bytes=12345")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    path.write_text(src + "// edited\n")
    assert bench.profiled_traffic("decode_t4_fake", "fake") is None


def test_traffic_of_another_kernel_or_workload_or_missing_source(tmp_path, monkeypatch):
    src = "__global__ void k() {}\n"
    _layout(tmp_path, src, f"bench-traffic: kernel=fake source=k_gone.cu sha1={_sha(src)} bytes=7")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("decode_t4_fake", "other") is None      # no line for this kernel
    assert bench.profiled_traffic("prefill_t8192_fake", "fake") is None   # no summary of this workload
    assert bench.profiled_traffic("decode_t4_fake", "fake") is None       # its source file is gone


def test_committed_summaries_name_existing_sources():
    """Every traffic line committed under profiles/ names a kernel source of this tree."""
    import re
    pat = re.compile(r"bench-traffic:\s*kernel=(\S+)\s+source=(\S+)\s+sha1=(\w+)\s+bytes=(\d+)")
    found = 0
    for name in sorted(os.listdir(os.path.join(bench.ROOT, "profiles"))):
        with open(os.path.join(bench.ROOT, "profiles", name)) as f:
            for line in f:
                m = pat.search(line)
                if m:
                    found += 1
                    assert os.path.exists(os.path.join(bench.ROOT, "serving_router_top_gb300", "csrc", m.group(2))), line
                    assert len(m.group(3)) == 40 and int(m.group(4)) > 0, line
    assert found >= 1
