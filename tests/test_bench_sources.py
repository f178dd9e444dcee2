"""The bench reports an ncu traffic figure for a kernel only while that
kernel's sources hash to the value the figure was captured on.  These checks
keep that guard honest: each kernel family's hash covers every header its
source includes (directly or through another header), and every recorded
traffic entry names a family the bench knows, with a well-formed hash."""
import os
import re

import bench

CSRC = os.path.join(bench.ROOT, "softmax_tree_reduction_gb300", "csrc")
INCLUDE = re.compile(r'^\s*#\s*include\s+"([^"]+)"', re.M)


def local_includes(name, seen=None):
    """The csrc files `name` pulls in through quoted includes, transitively."""
    seen = set() if seen is None else seen
    with open(os.path.join(CSRC, name)) as fh:
        text = fh.read()
    for inc in INCLUDE.findall(text):
        base = os.path.basename(inc)
        if os.path.exists(os.path.join(CSRC, base)) and base not in seen:
            seen.add(base)
            local_includes(base, seen)
    return seen


def test_each_family_hashes_every_file_it_includes():
    for family, files in bench.KERNEL_SOURCES.items():
        root = files[0]
        assert os.path.exists(os.path.join(CSRC, root)), (family, root)
        missing = local_includes(root) - set(files)
        assert not missing, f"{family}: {sorted(missing)} not in its source hash"


def test_traffic_entries_name_known_families():
    for (family, workload, queries), entry in bench.NCU_TRAFFIC.items():
        assert family in bench.KERNEL_SOURCES, family
        assert isinstance(workload, str) and queries >= 1
        assert re.fullmatch(r"[0-9a-f]{64}", entry["src_sha256"]), (family, workload, queries)
        assert entry["bytes_per_launch"] > 0 and entry["num_splits"] >= 1


def test_hash_changes_with_any_listed_file(tmp_path, monkeypatch):
    """A change to any file of a family (or to the launch code) changes its hash."""
    import shutil
    fake_root = tmp_path / "repo"
    shutil.copytree(CSRC, fake_root / "softmax_tree_reduction_gb300" / "csrc")
    monkeypatch.setattr(bench, "ROOT", str(fake_root))
    base = bench.kernel_source_hash("tc05")
    for f in bench.KERNEL_SOURCES["tc05"] + ("api.cu",):
        path = fake_root / "softmax_tree_reduction_gb300" / "csrc" / f
        original = path.read_bytes()
        path.write_bytes(original + b"\n")
        assert bench.kernel_source_hash("tc05") != base, f
        path.write_bytes(original)
    assert bench.kernel_source_hash("tc05") == base
